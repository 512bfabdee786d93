// Step a8, the FP32 weight update w += Y^T alpha, and step a9, the full-data loss.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): weight updates run in high precision; the method's accuracy claim
// is stated on the training loss of logistic, linear and Poisson problems.
//
// Both are streaming reductions bound by HBM (the loss) or L2 (the update, whose Y was
// written one step earlier).  Both reduce in a fixed order so that results do not
// depend on scheduling: the update writes one FP32 partial row per CTA and a second
// kernel sums them column by column; the loss keeps FP32 per-row values, FP64 per-CTA
// partials, and the last CTA to finish sums the partials in CTA order.
#include "casgd_internal.cuh"
#include "ptx_async.cuh"

namespace casgd {

namespace {


// CTA p sums alpha_i * Y_i over its row range into part[p][:] (ldY floats).
// Threads form TR row-lanes x TV vector-lanes (TV a power of two, TR = 256/TV); a thread
// holds kV 16-byte column vectors (kV = ceil(nvec / TV), a template parameter so that
// only the accumulators in use take registers).  kUnroll rows are loaded before any is
// used, so several loads per thread are in flight; the FMA order per column stays
// row-ascending.
template <int kV>
__global__ void __launch_bounds__(256) update_partial_kernel(
    const uint16_t* __restrict__ Y, const float* __restrict__ alpha, int64_t S, int64_t ldY,
    float* __restrict__ part, int TV) {
  extern __shared__ float red[];  // [TR][TV*8] when TR > 1
  constexpr int kUnroll = kV <= 2 ? 4 : 2;
  const int64_t nvec = ldY / 8;
  const int TR = 256 / TV;
  const int tv = threadIdx.x % TV, tr = threadIdx.x / TV;
  const int64_t r_lo = S * blockIdx.x / gridDim.x;
  const int64_t r_hi = S * (blockIdx.x + 1) / gridDim.x;
  float acc[kV][8];
#pragma unroll
  for (int v = 0; v < kV; ++v)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[v][e] = 0.0f;

  for (int64_t i0 = r_lo + tr; i0 < r_hi; i0 += (int64_t)TR * kUnroll) {
    float a[kUnroll];
    uint4 q[kUnroll][kV];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + (int64_t)u * TR;
      const bool in = i < r_hi;
      a[u] = in ? __ldg(alpha + i) : 0.0f;
      const uint16_t* yr = Y + (in ? i : r_lo) * ldY;
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const int64_t vec = tv + (int64_t)v * TV;
        q[u][v] = vec < nvec ? __ldg(reinterpret_cast<const uint4*>(yr + vec * 8))
                             : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const uint32_t pw[4] = {q[u][v].x, q[u][v].y, q[u][v].z, q[u][v].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          acc[v][2 * h] = fmaf(a[u], bf16_bits_to_float(pw[h] & 0xFFFFu), acc[v][2 * h]);
          acc[v][2 * h + 1] = fmaf(a[u], bf16_bits_to_float(pw[h] >> 16), acc[v][2 * h + 1]);
        }
      }
    }
  }

  float* out = part + (int64_t)blockIdx.x * ldY;
  if (TR == 1) {
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      const int64_t vec = tv + (int64_t)v * TV;
      if (vec < nvec)
#pragma unroll
        for (int e = 0; e < 8; ++e) out[vec * 8 + e] = acc[v][e];
    }
    return;
  }
  // TR > 1 means TV*8 >= ldY fits one vector per thread (v = 0 only).
  for (int e = 0; e < 8; ++e) red[tr * TV * 8 + tv * 8 + e] = acc[0][e];
  __syncthreads();
  for (int col = threadIdx.x; col < TV * 8; col += 256) {
    float sum = 0.0f;
    for (int q = 0; q < TR; ++q) sum += red[q * TV * 8 + col];
    if (col < ldY) out[col] = sum;
  }
}

// w[c] += sum_p part[p][c].  A CTA covers 32 columns with 8 warps; warp q sums the
// partial rows p = q, q+8, ... of its column (eight loads in flight), and the eight
// warp sums are combined in warp order: a fixed association, so the result is
// deterministic.
__global__ void __launch_bounds__(256) update_reduce_kernel(const float* __restrict__ part,
                                                            int P, int64_t n, int64_t ldY,
                                                            float* __restrict__ w, Ctrl* ctrl) {
  __shared__ float red[8][32];
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  float acc = 0.0f;
  if (c < n) {
    int p = q;
    for (; p + 56 < P; p += 64) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(part + (int64_t)(p + 8 * u) * ldY + c);
#pragma unroll
      for (int u = 0; u < 8; ++u) acc += v[u];
    }
    for (; p < P; p += 8) acc += __ldg(part + (int64_t)p * ldY + c);
  }
  red[q][lane] = acc;
  __syncthreads();
  if (q == 0 && c < n) {
    float sum = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; ++u) sum += red[u][lane];
    const float v = w[c] + sum;
    w[c] = v;
    if (!isfinite(v)) atomicOr(&ctrl->status, ST_NONFINITE);
  }
}

// Loss: the rows are streamed, never gathered -- each CTA owns a contiguous range of
// rows and reads each of its rows once, straight from HBM into registers.  G lanes per
// row (a power of two; a lane holds at most eight of the row's 16-byte vectors for
// n <= 2048): lane g takes the vectors g, g+G, ..., all of a lane's loads for a row
// issued together.  For n <= 2048 (kPipe) a lane issues the loads of its next row
// before it uses those of the current one, so each SM keeps about 128 KB of X in flight
// without pause; wider rows are read eight vectors per lane at a time.  No staging in
// shared memory and no hand-off between warps.  w is staged once in shared memory; the
// row's label is loaded with its vectors.  Per row the FP32 dot product takes eight
// sums (element e of every vector into sum e, vectors in increasing order), a fixed
// tree, then a shuffle tree over the row's lanes -- the order of the margins; the row's
// loss is added in FP64, the CTA's values in warp order, and the last CTA to finish
// sums the CTA partials in CTA order.
constexpr int kLossThreads = 256;
constexpr int kLossV = 8;  // at most a lane's 16-byte loads per row (per batch of a wider row)
// CTAs per SM the register budget is sized for (kV loads of two rows per lane in kPipe)
constexpr int loss_min_ctas(int kV, bool pipe) { return pipe ? (kV >= 8 ? 2 : 4) : 3; }

struct LossArgs {
  const uint16_t* X;
  const float* y;
  int64_t m, n, ld;
  int loss, G;
  const float* w;
  double* part;
  double* out;
  Ctrl* ctrl;
};

template <int kV, bool kPipe>
__global__ void __launch_bounds__(kLossThreads, loss_min_ctas(kV, kPipe)) loss_kernel(LossArgs a) {
  extern __shared__ __align__(16) float loss_w[];
  __shared__ double red[kLossThreads / 32];
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // w in two planes of ld/2 floats: plane 0 holds columns 8v..8v+3 of each 16-byte
  // vector v at 4v, plane 1 columns 8v+4..8v+7, so a warp's 16-byte reads of w for
  // consecutive vectors are contiguous (zero past n)
  float* w_s = loss_w;
  float* w_s1 = loss_w + a.ld / 2;
  for (int64_t c = threadIdx.x; c < a.ld; c += blockDim.x)
    ((c & 4) ? w_s1 : w_s)[(c >> 3) * 4 + (c & 3)] = c < a.n ? a.w[c] : 0.0f;
  __syncthreads();

  const int G = a.G;
  const int g = lane & (G - 1);
  const int rows_per_pass = (kLossThreads / 32) * (32 / G);
  const int my = warp * (32 / G) + lane / G;  // row slot within a pass
  const int64_t r_lo = a.m * blockIdx.x / gridDim.x;
  const int64_t r_hi = a.m * (blockIdx.x + 1) / gridDim.x;
  const int nfull = (int)(a.n / 8);     // vectors wholly inside the n columns
  const int nv = (int)((a.n + 7) / 8);  // vectors holding data

  // the lane's vectors v0, v0+G, ... (at most kV) of row `row` (zeros if !live)
  auto load = [&](int64_t row, bool live, int v0, uint4 (&xv)[kV]) {
    const uint4* xr = reinterpret_cast<const uint4*>(a.X + (live ? row : 0) * a.ld);
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      const int v = v0 + k * G;
      xv[k] = (live && v < nv) ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // adds those vectors times w into the eight sums
  auto add = [&](const uint4 (&xv)[kV], int v0, float (&sum)[8]) {
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      const int v = v0 + k * G;
      if (v >= nv) break;
      const float4 w0 = *reinterpret_cast<const float4*>(w_s + v * 4);
      const float4 w1 = *reinterpret_cast<const float4*>(w_s1 + v * 4);
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t pw[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
      if (v >= nfull) {  // the partial last vector: columns from n on are not data
        const int64_t c0 = (int64_t)v * 8;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int64_t cc = c0 + 2 * h;
          if (cc >= a.n) pw[h] = 0;
          else if (cc + 1 >= a.n) pw[h] &= 0xFFFFu;
        }
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        sum[2 * h] = fmaf(__uint_as_float(pw[h] << 16), wv[2 * h], sum[2 * h]);
        sum[2 * h + 1] = fmaf(__uint_as_float(pw[h] & 0xFFFF0000u), wv[2 * h + 1], sum[2 * h + 1]);
      }
    }
  };
  // the row's margin (eight sums, tree, shuffle tree) and, on its first lane, its loss
  double mine = 0.0;
  auto finish = [&](const float (&sum)[8], bool live, float label) {
    float acc = ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
    for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
    if (live && g == 0) mine += (double)loss_value(a.loss, acc, label);
  };

  if (kPipe) {  // one batch per row (nv <= kV * G); the next row's loads go first
    int64_t row = r_lo + my;
    bool live = row < r_hi;
    uint4 xa[kV];
    load(row, live, g, xa);
    float la = (live && g == 0) ? __ldg(a.y + row) : 0.0f;
    for (int64_t p0 = r_lo; p0 < r_hi; p0 += rows_per_pass) {  // CTA-uniform
      const int64_t nrow = row + rows_per_pass;
      const bool nlive = nrow < r_hi;
      uint4 xb[kV];
      load(nrow, nlive, g, xb);
      const float lb = (nlive && g == 0) ? __ldg(a.y + nrow) : 0.0f;
      float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      add(xa, g, sum);
      finish(sum, live, la);
#pragma unroll
      for (int k = 0; k < kV; ++k) xa[k] = xb[k];
      la = lb;
      row = nrow;
      live = nlive;
    }
  } else {
    for (int64_t p0 = r_lo; p0 < r_hi; p0 += rows_per_pass) {  // CTA-uniform
      const int64_t row = p0 + my;
      const bool live = row < r_hi;
      const float label = (live && g == 0) ? __ldg(a.y + row) : 0.0f;
      float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int v0 = g; v0 < nv; v0 += kV * G) {
        uint4 xv[kV];
        load(row, live, v0, xv);
        add(xv, v0, sum);
      }
      finish(sum, live, label);
    }
  }
  for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
  if (lane == 0) red[warp] = mine;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int q = 0; q < kLossThreads / 32; ++q) t += red[q];
    a.part[blockIdx.x] = t;
    __threadfence();
    const uint32_t done = atomicAdd(&a.ctrl->loss_done, 1u);
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    double t = 0.0;
    for (unsigned q = 0; q < gridDim.x; ++q) t += __ldcg(a.part + q);
    *a.out = t / (double)a.m;
    a.ctrl->loss_done = 0;
  }
}

int pow2_at_least(int64_t v, int cap) {
  int g = 1;
  while (g < v && g < cap) g <<= 1;
  return g;
}

}  // namespace

cudaError_t launch_update(const uint16_t* Y, const float* alpha, int64_t S, int64_t n,
                          int64_t ldY, float* w, float* part, int upd_ctas, Ctrl* ctrl,
                          Ctx& c) {
  const int64_t nvec = ldY / 8;
  const int TV = pow2_at_least(nvec, 256);
  const int TR = 256 / TV;
  const size_t smem = TR > 1 ? (size_t)TR * TV * 8 * sizeof(float) : 0;
  const int64_t vpt = (nvec + TV - 1) / TV;  // <= 8 since ldY <= 16384
  if (vpt <= 1)
    update_partial_kernel<1><<<upd_ctas, 256, smem, c.stream>>>(Y, alpha, S, ldY, part, TV);
  else if (vpt <= 2)
    update_partial_kernel<2><<<upd_ctas, 256, smem, c.stream>>>(Y, alpha, S, ldY, part, TV);
  else if (vpt <= 4)
    update_partial_kernel<4><<<upd_ctas, 256, smem, c.stream>>>(Y, alpha, S, ldY, part, TV);
  else
    update_partial_kernel<8><<<upd_ctas, 256, smem, c.stream>>>(Y, alpha, S, ldY, part, TV);
  ++c.launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_update_reduce(part, upd_ctas, n, ldY, w, ctrl, c);
}

cudaError_t launch_update_reduce(const float* part, int upd_ctas, int64_t n, int64_t ldY,
                                 float* w, Ctrl* ctrl, Ctx& c) {
  const unsigned blocks = (unsigned)((n + 31) / 32);
  update_reduce_kernel<<<blocks, 256, 0, c.stream>>>(part, upd_ctas, n, ldY, w, ctrl);
  ++c.launches;
  return cudaGetLastError();
}

int loss_ctas(int num_sms) {
  const int v = num_sms * loss_min_ctas(kLossV, false);
  return v > kLossCtas ? kLossCtas : v;
}

cudaError_t launch_loss(const casgd_data_t& d, int loss, const float* w, double* part,
                        double* out_dev, Ctrl* ctrl, Ctx& c) {
  LossArgs a;
  a.X = static_cast<const uint16_t*>(d.X);
  a.y = d.y;
  a.m = d.m;
  a.n = d.n;
  a.ld = d.ld;
  a.loss = loss;
  // G lanes per row, each with at most eight of the row's 16-byte vectors where that
  // fits in 32 lanes
  const int64_t nv = (d.n + 7) / 8;
  a.G = pow2_at_least((nv + kLossV - 1) / kLossV, 32);
  a.w = w;
  a.part = part;
  a.out = out_dev;
  a.ctrl = ctrl;
  // a lane's loads per row: kV (a power of two) covers its ceil(nv / G) vectors; wider
  // rows (n > 2048) are read in batches of kLossV
  const int64_t per_lane = (nv + a.G - 1) / a.G;
  const bool pipe = per_lane <= kLossV;
  const int kv = pipe ? pow2_at_least(per_lane, kLossV) : kLossV;
  const size_t smem = (size_t)d.ld * 4;  // w's two planes (ld % 8 == 0)
  void (*const fn)(LossArgs) = !pipe    ? loss_kernel<kLossV, false>
                               : kv == 1 ? loss_kernel<1, true>
                               : kv == 2 ? loss_kernel<2, true>
                               : kv == 4 ? loss_kernel<4, true>
                                         : loss_kernel<8, true>;
  int dummy = 0;
  cudaError_t e = cached_query(c, (const void*)fn, [&](int& v) {
    v = 1;
    return cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(64 * 1024));
  }, dummy);
  if (e != cudaSuccess) return e;
  int64_t blocks = (int64_t)c.num_sms * loss_min_ctas(kv, pipe);
  if (blocks > kLossCtas) blocks = kLossCtas;
  if (blocks > d.m) blocks = d.m;
  fn<<<(unsigned)blocks, kLossThreads, smem, c.stream>>>(a);
  ++c.launches;
  return cudaGetLastError();
}

}  // namespace casgd
