// Steps a6/a7: the FP32 inner s-step recurrence
//     z_j = r_j + sum_{t<j} G_{j,t} alpha_t,   alpha_j = -(eta/b) * l'(z_j, y_j).
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the inner recurrence runs in high precision, from the BF16 margins
// and the FP32 Gram matrix.  alpha of one row depends only on that row's z, so rows
// are independent once all earlier blocks are known; the s blocks form a serial chain.
//
// Design: one persistent cooperative launch (all CTAs co-resident) with two roles.
//  * Chain CTAs (the first C CTAs) each own 8-row groups of every block and walk the
//    phases j = 0..s-1 in order.  Phase j needs only the band
//        band_j = sum_{t=j-B}^{j-1} G_{j,t} alpha_t      (B = 1 or 2 blocks)
//    on top of far_j (below).  A chain CTA loads its rows of the band blocks into
//    registers before it waits for alpha_{j-1}, so after the wait only alpha_{j-1}
//    (from L2), a short dot product and l' remain on the critical path.
//  * Bulk CTAs take units (block j >= B+1, 16 rows) from an atomic queue in increasing
//    j and compute far_j = sum_{t<j-B} G_{j,t} alpha_t for their rows, streaming G with
//    coalesced float4 reads as each alpha_t becomes available.  far_j is needed only B
//    phases after its last input is known, so most of G is read off the critical path.
// Completion is published with device-scope fences and atomic counters
// (block_done[j]: chain CTAs finished with phase j; far_done[j]: bulk units of block j
// finished) and read with acquire loads.  Every wait is bounded by `timeout_ns`; on
// expiry the waiter records ST_TIMEOUT, which wait gave up (Ctrl::diag), and the abort
// word, and every other waiter stops.  Sums are taken in a fixed order (far_j over t
// ascending, then the band, then r), so results are deterministic.
#include "casgd_internal.cuh"

namespace casgd {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;       // rows per bulk unit
constexpr int kChainRows = 8;   // rows per chain group (a warp per row)
constexpr int kPrefetch = 8;    // float4 of band G (and of alpha) a chain lane keeps in registers

struct RecArgs {
  const float* G;
  const uint16_t* r;
  const float* yY;
  float* alpha;
  float* far;
  uint32_t* far_done;
  uint64_t* trace;  // [kMaxS][4] timestamps of chain CTA 0 (see chain_role)
  Ctrl* ctrl;
  uint64_t timeout_ns;
  int b, s, loss, U, Uc, C, B, bulk_units;
  float coef;
  bool diag, stall_test, vec4;
};

// One thread waits until *p >= need; false on timeout or abort.  `where` is recorded
// in Ctrl::diag when this wait is the one that gives up.
__device__ bool spin_until(const uint32_t* p, uint32_t need, const RecArgs& a, bool backoff,
                           uint32_t where) {
  if (ld_acquire_u32(p) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (backoff) __nanosleep(128);
    if (ld_acquire_u32(p) >= need) return true;
    if (ld_volatile_u32(&a.ctrl->abort)) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      atomicOr(&a.ctrl->status, ST_TIMEOUT);
      atomicExch(&a.ctrl->diag, where | (ld_volatile_u32(p) & 0xFFFu));
      atomicExch(&a.ctrl->abort, 1u);
      return false;
    }
  }
}

// Release add: orders every write this CTA made before the preceding barrier (the
// barrier makes them visible to thread 0, the release makes them visible device-wide)
// before the counter changes.
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Whole-CTA wait: thread 0 spins; the barrier orders everyone's later reads.
__device__ bool cta_wait(const uint32_t* p, uint32_t need, const RecArgs& a, bool backoff,
                         uint32_t where) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) s_ok = spin_until(p, need, a, backoff, where) ? 1 : 0;
  __syncthreads();
  const int ok = s_ok;
  __syncthreads();
  return ok != 0;
}

// Ctrl::diag codes: kind << 24 | block << 12 | counter value seen.
__device__ __forceinline__ uint32_t where_code(uint32_t kind, int j) {
  return (kind << 24) | ((uint32_t)j << 12);
}

__device__ __forceinline__ float dot4(float4 g, float4 v, float acc) {
  acc = fmaf(g.x, v.x, acc);
  acc = fmaf(g.y, v.y, acc);
  acc = fmaf(g.z, v.z, acc);
  return fmaf(g.w, v.w, acc);
}

// ------------------------------------------------------------------ chain role
// A warp per row (8 rows per group); a lane's columns are lane*4 + 128k.  Chain CTA c
// owns the 8-row groups c, c+C, ... of every block.  Per phase, everything that does
// not depend on alpha_{j-1} is issued as asynchronous loads before the wait (band rows
// of G, alpha of the older band block, r and y of the row), the far part is checked
// only after the wait (the bulk had B phases to produce it), and completion is
// published by one release-add after the CTA barrier.
__device__ void chain_role(const RecArgs& a, int c) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = a.vec4 ? (a.b + 127) / 128 : 0;  // float4 slots per band block
  // Chain CTA 0 keeps a per-phase timeline (globaltimer ns): phase start, alpha_{j-1}
  // ready, far part ready, alpha_j published.
  const bool tracer = (c == 0 && threadIdx.x == 0);
  for (int j = 0; j < a.s; ++j) {
    if (tracer) a.trace[4 * j] = globaltimer_ns();
    const int t0 = j - a.B > 0 ? j - a.B : 0;
    const int nq = nk * (j - t0);       // band slots, t ascending then column ascending
    const int nq_old = nk * (j - 1 - t0 > 0 ? j - 1 - t0 : 0);  // slots with t < j-1
    const bool has_far = j >= a.B + 1;
    for (int grp = c; grp < a.Uc; grp += a.C) {
      const int i = grp * kChainRows + warp;  // row within block j
      const bool live = i < a.b;
      const int64_t p = (int64_t)j * a.b + (live ? i : 0);
      const float* grow0 = a.G + (int64_t)i * a.b;
      // (a) asynchronous loads that do not need alpha_{j-1}
      float4 gv[kPrefetch], av[kPrefetch];
#pragma unroll
      for (int q = 0; q < kPrefetch; ++q) {
        gv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        av[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && q < nq) {
          const int t = t0 + q / nk, col = lane * 4 + 128 * (q % nk);
          if (col < a.b) {
            gv[q] = __ldg(reinterpret_cast<const float4*>(grow0 + packed_offset(j, t, a.b, a.diag) + col));
            if (q < nq_old)
              av[q] = __ldcg(reinterpret_cast<const float4*>(a.alpha + (int64_t)t * a.b + col));
          }
        }
      }
      float rj = 0.0f, yj = 0.0f;
      if (live && lane == 0) {
        rj = bf16_bits_to_float(a.r[p]);
        yj = a.yY[p];
      }
      // (b) the critical wait: every chain CTA done with phase j-1
      if (grp == c && j > 0 &&
          !cta_wait(&a.ctrl->block_done[j - 1], (uint32_t)a.C, a, false, where_code(2, j)))
        return;
      if (tracer) a.trace[4 * j + 1] = globaltimer_ns();
      // (c) alpha_{j-1}
      if (live) {
#pragma unroll
        for (int q = 0; q < kPrefetch; ++q) {
          if (q >= nq_old && q < nq) {
            const int t = t0 + q / nk, col = lane * 4 + 128 * (q % nk);
            if (col < a.b)
              av[q] = __ldcg(reinterpret_cast<const float4*>(a.alpha + (int64_t)t * a.b + col));
          }
        }
      }
      // (d) far part (normally complete long before)
      if (grp == c && has_far &&
          !cta_wait(&a.far_done[j], (uint32_t)a.U, a, false, where_code(1, j)))
        return;
      if (tracer) a.trace[4 * j + 2] = globaltimer_ns();
      float acc = 0.0f;
      if (live) {
        if (a.vec4) {
#pragma unroll
          for (int q = 0; q < kPrefetch; ++q)
            if (q < nq) acc = dot4(gv[q], av[q], acc);
          for (int q = kPrefetch; q < nq; ++q) {  // beyond the register budget
            const int t = t0 + q / nk, col = lane * 4 + 128 * (q % nk);
            if (col < a.b)
              acc = dot4(__ldg(reinterpret_cast<const float4*>(grow0 + packed_offset(j, t, a.b, a.diag) + col)),
                         __ldcg(reinterpret_cast<const float4*>(a.alpha + (int64_t)t * a.b + col)),
                         acc);
          }
        } else {
          for (int t = t0; t < j; ++t) {
            const float* al = a.alpha + (int64_t)t * a.b;
            const float* grow = grow0 + packed_offset(j, t, a.b, a.diag);
            for (int col = lane; col < a.b; col += 32)
              acc = fmaf(__ldg(grow + col), __ldcg(al + col), acc);
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (live && lane == 0) {
        float z = rj;
        if (has_far) z += __ldcg(a.far + p);
        z += acc;
        a.alpha[p] = a.coef * loss_deriv(a.loss, z, yj);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && !(a.stall_test && j == 0)) red_release_add(&a.ctrl->block_done[j], 1u);
    if (tracer) a.trace[4 * j + 3] = globaltimer_ns();
  }
}

// ------------------------------------------------------------------- bulk role
// Unit = (block j, 16 rows); each warp owns two rows; a lane's columns are lane*4 + 128k.
// Phases complete in order, so one look at the newest counter a unit needs tells it
// whether everything is already there (a unit claimed late then streams its blocks
// without further polling).  Up to four blocks t are processed per pass with all their
// loads issued together; each block's dot product is summed over columns first and
// then added in t order, so the result does not depend on how passes were grouped.
__device__ void bulk_role(const RecArgs& a) {
  __shared__ int s_unit;
  __shared__ int s_all;
  constexpr int kT = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  while (true) {
    if (threadIdx.x == 0) {
      int u = (int)atomicAdd(&a.ctrl->next_unit, 1u);
      if (ld_volatile_u32(&a.ctrl->abort)) u = a.bulk_units;
      s_unit = u;
    }
    __syncthreads();
    const int unit = s_unit;
    __syncthreads();
    if (unit >= a.bulk_units) return;
    const int j = a.B + 1 + unit / a.U;
    const int c = unit % a.U;
    const int i0 = c * kRows + warp * 2;
    const bool has0 = i0 < a.b, has1 = i0 + 1 < a.b;
    const int t_end = j - a.B;  // far_j covers t < j - B
    if (threadIdx.x == 0) s_all = ld_acquire_u32(&a.ctrl->block_done[t_end - 1]) >= (uint32_t)a.C;
    __syncthreads();
    int known = s_all ? t_end : 0;  // blocks of alpha known to be complete
    __syncthreads();
    float acc0 = 0.0f, acc1 = 0.0f;
    for (int t = 0; t < t_end;) {
      if (t >= known) {
        if (!cta_wait(&a.ctrl->block_done[t], (uint32_t)a.C, a, true, where_code(3, j))) return;
        known = t + 1;
      }
      const int nt = min(min(known, t_end) - t, kT);
      if (has0) {
        const float* g0 = a.G + (int64_t)i0 * a.b;
        float d0[kT] = {0.f, 0.f, 0.f, 0.f}, d1[kT] = {0.f, 0.f, 0.f, 0.f};
        if (a.vec4) {
          for (int col = lane * 4; col < a.b; col += 128) {
            float4 av[kT], x0[kT], x1[kT];
#pragma unroll
            for (int u = 0; u < kT; ++u) {
              if (u < nt) {
                const float* gb = g0 + packed_offset(j, t + u, a.b, a.diag) + col;
                av[u] = __ldcg(reinterpret_cast<const float4*>(a.alpha + (int64_t)(t + u) * a.b + col));
                x0[u] = __ldg(reinterpret_cast<const float4*>(gb));
                x1[u] = has1 ? __ldg(reinterpret_cast<const float4*>(gb + a.b))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
#pragma unroll
            for (int u = 0; u < kT; ++u) {
              if (u < nt) {
                d0[u] = dot4(x0[u], av[u], d0[u]);
                d1[u] = dot4(x1[u], av[u], d1[u]);
              }
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < kT; ++u) {
            if (u < nt) {
              const float* gb = g0 + packed_offset(j, t + u, a.b, a.diag);
              const float* al = a.alpha + (int64_t)(t + u) * a.b;
              for (int col = lane; col < a.b; col += 32) {
                const float av = __ldcg(al + col);
                d0[u] = fmaf(__ldg(gb + col), av, d0[u]);
                if (has1) d1[u] = fmaf(__ldg(gb + a.b + col), av, d1[u]);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kT; ++u) {
          if (u < nt) {
            acc0 += d0[u];
            acc1 += d1[u];
          }
        }
      }
      t += nt;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      acc0 += __shfl_xor_sync(0xffffffffu, acc0, off);
      acc1 += __shfl_xor_sync(0xffffffffu, acc1, off);
    }
    if (lane == 0 && has0) {
      const int64_t p0 = (int64_t)j * a.b + i0;
      a.far[p0] = acc0;
      if (has1) a.far[p0 + 1] = acc1;
    }
    __syncthreads();
    if (threadIdx.x == 0) red_release_add(&a.far_done[j], 1u);
  }
}

__global__ void __launch_bounds__(kThreads) recur_kernel(RecArgs a) {
  if ((int)blockIdx.x < a.C)
    chain_role(a, blockIdx.x);
  else
    bulk_role(a);
}

}  // namespace

cudaError_t launch_recur(const float* G, const uint16_t* r, const float* yY, float* alpha,
                         float* far, uint32_t* far_done, int b, int s, float eta, int loss,
                         uint32_t flags, uint32_t timeout_us, Ctrl* ctrl, Ctx& c) {
  RecArgs a;
  a.G = G;
  a.r = r;
  a.yY = yY;
  a.alpha = alpha;
  a.far = far;
  a.far_done = far_done;
  a.trace = reinterpret_cast<uint64_t*>(far_done + kMaxS);
  a.ctrl = ctrl;
  a.timeout_ns = (uint64_t)(timeout_us ? timeout_us : 1000000u) * 1000ull;
  a.b = b;
  a.s = s;
  a.loss = loss;
  a.U = (b + kRows - 1) / kRows;
  a.Uc = (b + kChainRows - 1) / kChainRows;
  a.vec4 = (b % 4) == 0;
  // band width: two blocks while a chain lane can hold both in registers
  a.B = (a.vec4 && 2 * ((b + 127) / 128) <= kPrefetch) ? 2 : 1;
  a.bulk_units = s > a.B + 1 ? (s - a.B - 1) * a.U : 0;
  a.coef = -(eta / (float)b);
  a.diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  a.stall_test = (flags & CASGD_FLAG_TEST_STALL) != 0;

  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, recur_kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorLaunchOutOfResources;
  const int64_t cap = (int64_t)per_sm * c.num_sms;
  // one chain CTA per 8-row group while that leaves room for the bulk CTAs
  int64_t cmax = a.bulk_units > 0 ? cap / 2 : cap;
  if (cmax < 1) cmax = 1;
  a.C = (int)(a.Uc < cmax ? a.Uc : cmax);
  if (a.C + (a.bulk_units > 0 ? 1 : 0) > cap) return cudaErrorNotSupported;
  int64_t grid = a.C + (int64_t)a.bulk_units;
  if (grid > cap) grid = cap;
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel((const void*)recur_kernel, dim3((unsigned)grid),
                                  dim3(kThreads), args, 0, c.stream);
  ++c.launches;
  return e;
}

}  // namespace casgd
