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

// Loss: groups of G lanes per row (as in the gather), grid-stride over rows; w is
// staged in shared memory once per CTA, and each warp issues its next row's loads
// before it sums the current row.
__global__ void __launch_bounds__(256, 2) loss_kernel(const uint16_t* __restrict__ X,
                                                   const float* __restrict__ y, int64_t m,
                                                   int64_t n, int64_t ld, int loss,
                                                   const float* __restrict__ w,
                                                   double* __restrict__ part,
                                                   double* __restrict__ out, Ctrl* ctrl,
                                                   int G) {
  __shared__ double red[8];
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane & (G - 1);
  const int rows_per_warp = 32 / G;
  const int64_t nvec = (n + 7) / 8;
  const int64_t rows_per_pass = (int64_t)gridDim.x * 8 * rows_per_warp;
  constexpr int kBatch = 8;
  extern __shared__ __align__(16) float w_s[];  // w, zero padded to a multiple of 8
  for (int64_t c = threadIdx.x; c < nvec * 8; c += blockDim.x) w_s[c] = c < n ? w[c] : 0.0f;
  __syncthreads();
  double mine = 0.0;
  // FP32 dot of row `row` with w from the kBatch vectors in q starting at vector v0
  auto dot_batch = [&](const uint4 (&q)[kBatch], int64_t v0, float acc) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t c0 = (v0 + (int64_t)u * G) * 8;
      if (c0 >= n) break;
      float wv[8];
      const float4 w0 = *reinterpret_cast<const float4*>(w_s + c0);
      const float4 w1 = *reinterpret_cast<const float4*>(w_s + c0 + 4);
      wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
      wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
      const uint32_t pw[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
      if (c0 + 8 <= n) {  // the whole vector holds features
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          acc = fmaf(__uint_as_float(pw[h] << 16), wv[2 * h], acc);
          acc = fmaf(__uint_as_float(pw[h] & 0xFFFF0000u), wv[2 * h + 1], acc);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int64_t c = c0 + 2 * h;
          if (c < n) acc = fmaf(bf16_bits_to_float(pw[h] & 0xFFFFu), wv[2 * h], acc);
          if (c + 1 < n) acc = fmaf(bf16_bits_to_float(pw[h] >> 16), wv[2 * h + 1], acc);
        }
      }
    }
    return acc;
  };
  auto load_batch = [&](uint4 (&q)[kBatch], int64_t row, int64_t v0) {
    const uint16_t* xr = X + row * ld;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t v = v0 + (int64_t)u * G;
      q[u] = (row < m && v < nvec) ? __ldg(reinterpret_cast<const uint4*>(xr + v * 8))
                                   : make_uint4(0, 0, 0, 0);
    }
  };
  auto finish_row = [&](float acc, int64_t row) {
    for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
    if (row < m && g == 0) mine += (double)loss_value(loss, acc, __ldg(y + row));
  };
  const int64_t first = ((int64_t)blockIdx.x * 8 + warp) * rows_per_warp + lane / G;
  if (nvec <= (int64_t)G * kBatch) {
    // one batch per row: the next row's loads are issued before this row is summed
    uint4 q[kBatch], qn[kBatch];
    load_batch(q, first, g);
    for (int64_t row = first; row - lane / G < m; row += rows_per_pass) {
      load_batch(qn, row + rows_per_pass, g);
      finish_row(dot_batch(q, g, 0.0f), row);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) q[u] = qn[u];
    }
  } else {
    for (int64_t row = first; row - lane / G < m; row += rows_per_pass) {
      float acc = 0.0f;
      // Issue up to kBatch 16-byte loads of the row before using any of them.
      for (int64_t v0 = g; v0 < nvec; v0 += (int64_t)G * kBatch) {
        uint4 q[kBatch];
        load_batch(q, row, v0);
        acc = dot_batch(q, v0, acc);
      }
      finish_row(acc, row);
    }
  }
  for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
  if (lane == 0) red[warp] = mine;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int q = 0; q < 8; ++q) t += red[q];
    part[blockIdx.x] = t;
    __threadfence();
    const uint32_t done = atomicAdd(&ctrl->loss_done, 1u);
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    double t = 0.0;
    for (unsigned q = 0; q < gridDim.x; ++q) t += __ldcg(part + q);
    *out = t / (double)m;
    ctrl->loss_done = 0;
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
  int v = num_sms * 4;
  return v > kLossCtas ? kLossCtas : v;
}

cudaError_t launch_loss(const casgd_data_t& d, int loss, const float* w, double* part,
                        double* out_dev, Ctrl* ctrl, Ctx& c) {
  const int G = pow2_at_least((d.n + 7) / 8, 32);
  const int64_t rows_per_cta = 8 * (32 / G);
  int64_t blocks = (d.m + rows_per_cta - 1) / rows_per_cta;
  const size_t smem = (size_t)((d.n + 7) / 8 * 8) * sizeof(float);
  int per_sm = 0;
  cudaError_t e = cached_query(c, (const void*)loss_kernel, [&](int& v) {
    if (smem > 48 * 1024) {
      cudaError_t r = cudaFuncSetAttribute(loss_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (r != cudaSuccess) return r;
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, loss_kernel, 256, smem);
  }, per_sm);
  if (e != cudaSuccess) return e;
  int cap = (per_sm > 0 ? per_sm : 1) * c.num_sms;  // one resident wave
  if (cap > loss_ctas(c.num_sms)) cap = loss_ctas(c.num_sms);
  if (blocks > cap) blocks = cap;
  loss_kernel<<<(unsigned)blocks, 256, smem, c.stream>>>(static_cast<const uint16_t*>(d.X), d.y,
                                                         d.m, d.n, d.ld, loss, w, part, out_dev,
                                                         ctrl, G);
  ++c.launches;
  return cudaGetLastError();
}

}  // namespace casgd
