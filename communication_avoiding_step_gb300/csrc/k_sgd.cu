// FP32 plain minibatch SGD on FP32 X: the baseline the paper measures CA-SGD against.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): CA-SGD is reported faster than FP32 SGD and its final loss within
// 0.5% of it.  Step q (counters q*b .. q*b+b-1, the rows CA-SGD's outer iteration uses
// for the same minibatch) does
//     z_i = x_i . w,  alpha_i = -(eta/b) l'(z_i, y_i),  w <- w + sum_i alpha_i x_i
// in FP32.
//
// One cooperative persistent launch runs all steps; two grid barriers per step (after
// the margins, after the update) keep every CTA on the same w.  Margins: w staged in
// shared memory, a warp per minibatch row, all float4 chunks of the row requested
// before they are used.  Update: alpha and the row indices staged in shared memory; a
// CTA owns 16 columns at a time; its 16 row-groups of threads each sum 1/16 of the rows
// in order (loads issued together), then the 16 partial sums are added in group order
// — the result does not depend on timing.  Barrier waits are bounded (status TIMEOUT, abort word).
#include "casgd_internal.cuh"

namespace casgd {

namespace {

constexpr int kSgdThreads = 256;
constexpr int kColsPerCta = 16;   // update: columns per CTA (16 row-groups x 16 columns)

struct SgdArgs {
  const float* X;
  const float* y;
  int64_t m, n, ld;
  float* w;
  float* alpha;      // [b]
  int32_t* idx;      // [b]
  uint32_t* bar;     // [2]: arrivals, generation
  Ctrl* ctrl;
  uint64_t seed, q0;
  int steps, b, loss;
  int perm_d;  // sampling: 0 with replacement, else perm_width(m)
  float coef;
  uint64_t timeout_ns;
};

// Grid barrier for a cooperative launch; false after a timeout (recorded) or an abort.
__device__ bool grid_barrier(const SgdArgs& a) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint32_t gen = ld_volatile_u32(a.bar + 1);
    __threadfence();
    if (atomicAdd(a.bar, 1u) == gridDim.x - 1) {
      a.bar[0] = 0;
      __threadfence();
      atomicExch(a.bar + 1, gen + 1);
    } else {
      const uint64_t t_start = globaltimer_ns();
      while (ld_volatile_u32(a.bar + 1) == gen) {
        __nanosleep(64);
        if (ld_volatile_u32(&a.ctrl->abort)) { ok = 0; break; }
        if (globaltimer_ns() - t_start > a.timeout_ns) {
          atomicOr(&a.ctrl->status, ST_TIMEOUT);
          atomicExch(&a.ctrl->abort, 1u);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__global__ void __launch_bounds__(kSgdThreads, 1) sgd_kernel(SgdArgs a) {
  extern __shared__ __align__(16) float sm[];  // w (ldw floats), then alpha[b], idx[b]
  __shared__ float part[16][kColsPerCta];
  const int ldw = (int)((a.n + 127) / 128 * 128);
  float* w_s = sm;
  float* al_s = sm + ldw;
  int32_t* idx_s = reinterpret_cast<int32_t*>(al_s + a.b);
  const int lane = threadIdx.x & 31;
  const int gwarp = (int)(blockIdx.x * (kSgdThreads / 32) + (threadIdx.x >> 5));
  const int nwarps = (int)(gridDim.x * (kSgdThreads / 32));
  const bool vec = (a.ld % 4) == 0 && (reinterpret_cast<uintptr_t>(a.X) & 15u) == 0;
  const int nv = ldw / 128;  // float4 chunks per lane and row
  const int rows_per_group = (a.b + 15) / 16;
  for (int q = 0; q < a.steps; ++q) {
    // ---- margins and alpha: w into shared memory, then a warp per row of the minibatch
    for (int c = threadIdx.x; c < ldw; c += kSgdThreads) w_s[c] = c < a.n ? __ldcg(a.w + c) : 0.0f;
    __syncthreads();
    for (int i = gwarp; i < a.b; i += nwarps) {
      const int32_t row = draw_row(a.seed, (a.q0 + (uint64_t)q) * (uint64_t)a.b + (uint64_t)i,
                                   (uint32_t)a.m, a.perm_d);
      const float* x = a.X + (int64_t)row * a.ld;
      float acc = 0.0f;
      if (vec) {
        // every chunk of the row is requested before any is used (8 per round)
        for (int v0 = 0; v0 < nv; v0 += 8) {
          float4 xv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int64_t c = (int64_t)(v0 + u) * 128 + lane * 4;
            xv[u] = (v0 + u < nv && c + 4 <= a.n) ? __ldg(reinterpret_cast<const float4*>(x + c))
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            if (v0 + u < nv && c < a.n && c + 4 > a.n) {  // the row's last, partial chunk
              float e[4] = {0.f, 0.f, 0.f, 0.f};
              for (int k = 0; c + k < a.n; ++k) e[k] = __ldg(x + c + k);
              xv[u] = make_float4(e[0], e[1], e[2], e[3]);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (v0 + u < nv) {
              const float4 wv = *reinterpret_cast<const float4*>(w_s + (v0 + u) * 128 + lane * 4);
              acc = fmaf(xv[u].x, wv.x, acc);
              acc = fmaf(xv[u].y, wv.y, acc);
              acc = fmaf(xv[u].z, wv.z, acc);
              acc = fmaf(xv[u].w, wv.w, acc);
            }
          }
        }
      } else {
        for (int64_t c = lane; c < a.n; c += 32) acc = fmaf(__ldg(x + c), w_s[c], acc);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) {
        a.alpha[i] = a.coef * loss_deriv(a.loss, acc, __ldg(a.y + row));
        a.idx[i] = row;
      }
    }
    if (!grid_barrier(a)) return;
    // ---- update: alpha and the rows in shared memory, then a CTA block of 16 columns
    // with 16 row-groups of threads, all of a thread's rows requested at once
    for (int i = threadIdx.x; i < a.b; i += kSgdThreads) {
      al_s[i] = __ldcg(a.alpha + i);
      // the row index is a pure function of the counter: recomputed, not read back
      idx_s[i] = draw_row(a.seed, (a.q0 + (uint64_t)q) * (uint64_t)a.b + (uint64_t)i,
                          (uint32_t)a.m, a.perm_d);
    }
    __syncthreads();
    const int col_in = threadIdx.x % kColsPerCta, grp = threadIdx.x / kColsPerCta;
    for (int64_t c0 = (int64_t)blockIdx.x * kColsPerCta; c0 < a.n;
         c0 += (int64_t)gridDim.x * kColsPerCta) {
      const int64_t c = c0 + col_in;
      float sum = 0.0f;
      if (c < a.n) {
        const int i0 = grp * rows_per_group;
        const int i1 = min(i0 + rows_per_group, a.b);
        for (int i = i0; i < i1; i += 16) {
          float v[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            v[u] = i + u < i1 ? __ldg(a.X + (int64_t)idx_s[i + u] * a.ld + c) : 0.0f;
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (i + u < i1) sum = fmaf(al_s[i + u], v[u], sum);
        }
      }
      part[grp][col_in] = sum;
      __syncthreads();
      if (grp == 0 && c < a.n) {
        float tot = 0.0f;
        for (int g2 = 0; g2 < 16; ++g2) tot += part[g2][col_in];
        const float wv = a.w[c] + tot;
        a.w[c] = wv;
        if (!isfinite(wv)) atomicOr(&a.ctrl->status, ST_NONFINITE);
      }
      __syncthreads();
    }
    if (!grid_barrier(a)) return;
  }
}

}  // namespace

size_t sgd_workspace_bytes(int b) {
  return 512 + 256 + (size_t)b * 8 + 256;
}

cudaError_t launch_sgd_fp32(const float* X, int64_t m, int64_t n, int64_t ld, const float* y,
                            const casgd_params_t& p, float* w, uint64_t q0, int steps, void* ws,
                            Ctx& c) {
  char* base = static_cast<char*>(ws);
  SgdArgs a;
  a.X = X;
  a.y = y;
  a.m = m;
  a.n = n;
  a.ld = ld;
  a.w = w;
  a.ctrl = reinterpret_cast<Ctrl*>(base);
  a.bar = reinterpret_cast<uint32_t*>(base + 512);
  a.alpha = reinterpret_cast<float*>(base + 768);
  a.idx = reinterpret_cast<int32_t*>(base + 768 + ((size_t)p.b * 4 + 255) / 256 * 256);
  a.seed = p.seed;
  a.perm_d = (p.flags & CASGD_FLAG_SAMPLE_PERMUTED) ? perm_width(m) : 0;
  a.q0 = q0;
  a.steps = steps;
  a.b = p.b;
  a.loss = p.loss;
  a.coef = -(p.eta / (float)p.b);
  a.timeout_ns = (uint64_t)(p.timeout_us ? p.timeout_us : 1000000u) * 1000ull;
  if (steps <= 0) return cudaSuccess;
  // re-arm the abort word and the barrier (stream-ordered before the launch)
  cudaError_t e = cudaMemsetAsync(a.bar, 0, 2 * sizeof(uint32_t), c.stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(&a.ctrl->abort, 0, sizeof(uint32_t), c.stream);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)((n + 127) / 128 * 128) * 4 + (size_t)p.b * 8;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(sgd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sgd_kernel, kSgdThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorLaunchOutOfResources;
  // enough CTAs for one warp per minibatch row and 16 columns per CTA, within one wave
  int64_t grid = (n + kColsPerCta - 1) / kColsPerCta;
  const int64_t warps_needed = (p.b + 7) / 8;
  if (grid < warps_needed) grid = warps_needed;
  const int64_t cap = (int64_t)per_sm * c.num_sms;
  if (grid > cap) grid = cap;
  if (grid > c.num_sms) grid = c.num_sms;  // one CTA per SM keeps the barrier short
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel((const void*)sgd_kernel, dim3((unsigned)grid),
                                  dim3(kSgdThreads), args, smem, c.stream);
  ++c.launches;
  return e;
}

}  // namespace casgd
