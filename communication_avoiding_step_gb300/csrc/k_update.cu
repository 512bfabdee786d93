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
// rows, and because X is row-major with a 16-byte-multiple pitch, R consecutive rows are
// one contiguous block that a single bulk copy (cp.async.bulk) moves into shared memory.
// A producer lane keeps nst such stages in flight (a shared-memory ring with full/empty
// barriers), so the bytes in flight per SM do not cost registers; eight consumer warps
// take G lanes per row from the landed stage: lane g sums the row's 16-byte vectors g,
// g+G, ... with w (staged in shared memory once), the row's lanes add by a shuffle tree,
// and the row's loss is added in FP64.  Per row the FP32 dot product has the same order
// as the margins.  Every wait is bounded; on expiry the CTA records ST_TIMEOUT, stops
// consuming, and its producer waits (bounded) for its copies in flight before exiting.
constexpr int kLossWarps = 16;                       // consumer warps
constexpr int kLossThreads = 32 * (kLossWarps + 1);  // + one producer warp
constexpr int kLossMaxStages = 8;
constexpr uint32_t kLossStageBytes = 64 * 1024;
constexpr int kLabelAhead = 8;                 // passes a label is copied ahead of its use
constexpr int kLabelSlots = kLabelAhead + 1;   // ring slots per row slot of a pass

struct LossArgs {
  const uint16_t* X;
  const float* y;
  int64_t m, n, ld;
  int loss, G;
  int R;            // rows per stage
  int nst;          // stages in the ring
  uint32_t stage;   // bytes per stage slot (multiple of 128)
  uint32_t lring;   // bytes of the label ring (rows per pass x kLabelSlots floats)
  const float* w;
  double* part;
  double* out;
  Ctrl* ctrl;
  uint64_t timeout_ns;
};

__device__ __forceinline__ bool loss_wait(uint64_t* bar, uint32_t parity, const LossArgs& a,
                                          volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      *abort_flag = 1;
      atomicOr(&a.ctrl->status, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kLossThreads, 1) loss_kernel(LossArgs a) {
  extern __shared__ __align__(128) uint8_t loss_smem[];
  __shared__ uint64_t full[kLossMaxStages], empty[kLossMaxStages];
  __shared__ double red[kLossWarps];
  __shared__ volatile int s_abort;
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ldv = a.ld / 8;                         // 16-byte vectors per row
  // w in two planes of ld/2 floats: plane 0 holds columns 8v..8v+3 of each 16-byte
  // vector v at 4v, plane 1 columns 8v+4..8v+7, so a warp's 16-byte reads of w for
  // consecutive vectors are contiguous (zero past n)
  float* w_s = reinterpret_cast<float*>(loss_smem);
  float* w_s1 = w_s + a.ld / 2;
  float* label_ring = reinterpret_cast<float*>(loss_smem + ((a.ld * 4 + 127) / 128) * 128);
  uint8_t* ring = reinterpret_cast<uint8_t*>(label_ring) + a.lring;
  const int64_t r_lo = a.m * blockIdx.x / gridDim.x;
  const int64_t r_hi = a.m * (blockIdx.x + 1) / gridDim.x;
  const int64_t nchunk = (r_hi - r_lo + a.R - 1) / a.R;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kLossWarps);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int64_t c = threadIdx.x; c < a.ld; c += blockDim.x)
    ((c & 4) ? w_s1 : w_s)[(c >> 3) * 4 + (c & 3)] = c < a.n ? a.w[c] : 0.0f;
  __syncthreads();

  double mine = 0.0;
  if (warp == kLossWarps) {
    // ---------------------------------------------------------------- producer lane
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t ch = 0; ch < nchunk && !s_abort; ++ch) {
        const int st = (int)(ch % a.nst);
        const uint32_t ph = (uint32_t)((ch / a.nst) & 1);
        if (!loss_wait(&empty[st], ph ^ 1u, a, &s_abort)) break;
        const int64_t row0 = r_lo + ch * a.R;
        const int64_t rows = r_hi - row0 < a.R ? r_hi - row0 : a.R;
        const uint32_t bytes = (uint32_t)(rows * a.ld * 2);
        mbar_expect_tx(&full[st], bytes);
        bulk_load(ring + (size_t)st * a.stage, a.X + row0 * a.ld, bytes, &full[st]);
        issued = ch + 1;
      }
      // every copy issued has landed before the CTA may exit
      for (int64_t ch = issued - a.nst < 0 ? 0 : issued - a.nst; ch < issued; ++ch) {
        const int st = (int)(ch % a.nst);
        const uint32_t ph = (uint32_t)((ch / a.nst) & 1);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[st], ph) && globaltimer_ns() - t0 < a.timeout_ns) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumer warps
    const int G = a.G;
    const int g = lane & (G - 1);
    const int rows_per_pass = kLossWarps * (32 / G);
    const int my = warp * (32 / G) + lane / G;  // row slot within a pass
    const int nfull = (int)(a.n / 8);             // vectors wholly inside the n columns
    // Labels: pass P of the CTA is pass P % ppc of chunk P / ppc.  Lane g == 0 of each row
    // slot copies its row's label kLabelAhead passes ahead into the slot's shared-memory
    // ring with a 4-byte cp.async (one commit group per pass, empty where the row does
    // not exist), so the label's memory latency never stalls a pass.  The ring has one
    // slot more than the distance: the copy for pass P + kLabelAhead goes into the slot
    // pass P - 1 read, never into the one the current pass is reading.
    const int ppc = (a.R + rows_per_pass - 1) / rows_per_pass;
    float* lring = label_ring + (size_t)my * kLabelSlots;
    auto issue_label = [&](int64_t P) {
      const int64_t ch = P / ppc;
      const int64_t row = r_lo + ch * a.R + (P - ch * ppc) * rows_per_pass + my;
      const int64_t end = r_lo + (ch + 1) * a.R < r_hi ? r_lo + (ch + 1) * a.R : r_hi;
      if (g == 0 && ch < nchunk && row < end)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                         smem_u32(lring + (P % kLabelSlots))),
                     "l"(a.y + row)
                     : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    for (int64_t P = 0; P < kLabelAhead; ++P) issue_label(P);
    for (int64_t ch = 0; ch < nchunk; ++ch) {
      const int st = (int)(ch % a.nst);
      const uint32_t ph = (uint32_t)((ch / a.nst) & 1);
      int ok = 1;
      if (lane == 0) ok = loss_wait(&full[st], ph, a, &s_abort) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int64_t row0 = r_lo + ch * a.R;
      const int rows = (int)(r_hi - row0 < a.R ? r_hi - row0 : a.R);
      const uint8_t* stg = ring + (size_t)st * a.stage;
      for (int pp = 0; pp * rows_per_pass < rows; ++pp) {  // warp-uniform
        const int64_t P = ch * ppc + pp;
        const int q = pp * rows_per_pass + my;
        const bool live = q < rows;
        const uint4* xr = reinterpret_cast<const uint4*>(stg + (size_t)(live ? q : 0) * a.ld * 2);
        // eight independent sums (element e of every vector into sum e), then a fixed tree
        float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        auto add_full = [&](const uint4 xv, const float (&wv)[8]) {
          const uint32_t pw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            sum[2 * h] = fmaf(__uint_as_float(pw[h] << 16), wv[2 * h], sum[2 * h]);
            sum[2 * h + 1] = fmaf(__uint_as_float(pw[h] & 0xFFFF0000u), wv[2 * h + 1], sum[2 * h + 1]);
          }
        };
        auto add_vec = [&](const uint4 xv, const float (&wv)[8], int64_t c0) {
          uint32_t pw[4] = {xv.x, xv.y, xv.z, xv.w};
          if (c0 + 8 > a.n) {  // columns from n on are not data: zero them
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
        };
        // whole vectors (no masking), two at a time; then the partial last vector
        if (live) {
          int v = g;
          for (; v + G < nfull; v += 2 * G) {
            const uint4 x0 = xr[v], x1 = xr[v + G];
            const float4 a0 = *reinterpret_cast<const float4*>(w_s + v * 4);
            const float4 a1 = *reinterpret_cast<const float4*>(w_s1 + v * 4);
            const float4 b0 = *reinterpret_cast<const float4*>(w_s + (v + G) * 4);
            const float4 b1 = *reinterpret_cast<const float4*>(w_s1 + (v + G) * 4);
            const float wva[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float wvb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            add_full(x0, wva);
            add_full(x1, wvb);
          }
          for (; v < nfull; v += G) {
            const float4 a0 = *reinterpret_cast<const float4*>(w_s + v * 4);
            const float4 a1 = *reinterpret_cast<const float4*>(w_s1 + v * 4);
            const float wva[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            add_full(xr[v], wva);
          }
          if (v == nfull && nfull * 8 < a.n) {  // this lane holds the partial vector
            const float4 a0 = *reinterpret_cast<const float4*>(w_s + v * 4);
            const float4 a1 = *reinterpret_cast<const float4*>(w_s1 + v * 4);
            const float wva[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            add_vec(xr[v], wva, (int64_t)v * 8);
          }
        }
        float acc = ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
        for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
        // this pass's label: every group but the newest kLabelAhead - 1 has landed
        asm volatile("cp.async.wait_group %0;" ::"n"(kLabelAhead - 1) : "memory");
        if (live && g == 0) mine += (double)loss_value(a.loss, acc, lring[P % kLabelSlots]);
        issue_label(P + kLabelAhead);  // into the slot pass P - 1 read
      }
      // passes the last chunk does not have keep the pass count (and the ring) in step
      for (int pp = (rows + rows_per_pass - 1) / rows_per_pass; pp < ppc; ++pp) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kLabelAhead - 1) : "memory");
        issue_label(ch * ppc + pp + kLabelAhead);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no label copy outlives the CTA
    for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
    if (lane == 0) red[warp] = mine;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int q = 0; q < kLossWarps; ++q) t += red[q];
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
  int v = num_sms;
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
  a.G = pow2_at_least((nv + 7) / 8, 32);
  a.w = w;
  a.part = part;
  a.out = out_dev;
  a.ctrl = ctrl;
  a.timeout_ns = 1000000000ull;
  // stages of at least one row, 128-byte aligned slots; as many as fit beside w
  const size_t row_bytes = (size_t)d.ld * 2;
  size_t stage = row_bytes > kLossStageBytes ? row_bytes : kLossStageBytes;
  stage = (stage + 127) / 128 * 128;
  a.R = (int)(stage / row_bytes);
  a.stage = (uint32_t)stage;
  const size_t w_bytes = ((size_t)d.ld * 4 + 127) / 128 * 128;
  const size_t rows_per_pass = (size_t)kLossWarps * (32 / a.G);
  a.lring = (uint32_t)((rows_per_pass * kLabelSlots * 4 + 127) / 128 * 128);
  const size_t budget = 216 * 1024;
  int nst = (int)((budget - w_bytes - a.lring) / stage);
  if (nst > 4) nst = 4;
  if (nst < 2) return cudaErrorInvalidValue;  // (n <= 16384 keeps at least 2 stages)
  a.nst = nst;
  const size_t smem = w_bytes + a.lring + (size_t)nst * stage;
  void (*const fn)(LossArgs) = loss_kernel;
  int dummy = 0;
  cudaError_t e = cached_query(c, (const void*)fn, [&](int& v) {
    v = 1;
    return cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(224 * 1024));
  }, dummy);
  if (e != cudaSuccess) return e;
  int64_t blocks = loss_ctas(c.num_sms);
  if (blocks > d.m) blocks = d.m;
  fn<<<(unsigned)blocks, kLossThreads, smem, c.stream>>>(a);
  ++c.launches;
  return cudaGetLastError();
}

}  // namespace casgd
