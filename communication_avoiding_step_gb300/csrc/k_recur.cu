// Steps a6/a7: the FP32 inner s-step recurrence
//     z_j = r_j + sum_{t<j} G_{j,t} alpha_t,   alpha_j = -(eta/b) * l'(z_j, y_j).
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the inner recurrence runs in high precision, from the BF16 margins
// and the FP32 Gram matrix.  alpha of one row depends only on that row's z, so rows
// are independent once all earlier blocks are known.
//
// Design: one persistent cooperative launch (all CTAs co-resident).  Work units are
// (block j, 16 consecutive rows of it), handed out in increasing j from an atomic
// queue, so a unit's dependencies are always held by running CTAs.  Each warp owns two
// rows and walks t = 0..j-1, reading its rows of G_{j,t} (coalesced float4) and
// alpha_t (from L2).  Blocks finish in order (block j needs block j-1), so a unit only
// polls the completion counter of a block it has not yet seen finished.  The last
// block's rows of G are prefetched into L2 before the wait.  Completion is published
// with a device-scope fence plus an atomic add; waits read with acquire semantics and
// give up after `timeout_ns`, setting ST_TIMEOUT and the abort word so that every other
// waiter stops too.  Per row the sum order is fixed, so results are deterministic.
#include <cooperative_groups.h>

#include "casgd_internal.cuh"

namespace casgd {

namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 2;
constexpr int kUnitRows = kWarps * kRowsPerWarp;

struct RecArgs {
  const float* G;
  const uint16_t* r;
  const float* yY;
  float* alpha;
  Ctrl* ctrl;
  uint64_t timeout_ns;
  int b, s, loss, units_per_block, unit_rows;
  float coef;
  bool diag, stall_test;
};

// Lane 0 spins until block t has all its units done; returns false on timeout/abort.
__device__ bool wait_block(const RecArgs& a, int t) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) {
    const uint32_t need = (uint32_t)a.units_per_block;
    if (ld_acquire_u32(&a.ctrl->block_done[t]) < need) {
      const uint64_t t0 = globaltimer_ns();
      while (true) {
        if (ld_acquire_u32(&a.ctrl->block_done[t]) >= need) break;
        if (ld_volatile_u32(&a.ctrl->abort)) { ok = 0; break; }
        if (globaltimer_ns() - t0 > a.timeout_ns) {
          atomicOr(&a.ctrl->status, ST_TIMEOUT);
          atomicExch(&a.ctrl->abort, 1u);
          ok = 0;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();  // orders lane 0's acquire before the other lanes' reads of alpha_t
  return ok != 0;
}

__global__ void __launch_bounds__(256) recur_kernel(RecArgs a) {
  __shared__ int s_unit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total_units = a.s * a.units_per_block;
  const bool vec4 = (a.b % 4) == 0;

  while (true) {
    if (threadIdx.x == 0) {
      int u = (int)atomicAdd(&a.ctrl->next_unit, 1u);
      if (ld_volatile_u32(&a.ctrl->abort)) u = total_units;
      s_unit = u;
    }
    __syncthreads();
    const int unit = s_unit;
    __syncthreads();
    if (unit >= total_units) break;

    const int j = unit / a.units_per_block;
    const int c = unit - j * a.units_per_block;
    const int row_lo = c * a.unit_rows;
    const int row_hi = min(a.b, row_lo + a.unit_rows);
    const int i0 = row_lo + warp * kRowsPerWarp;
    const bool has0 = i0 < row_hi, has1 = i0 + 1 < row_hi;
    bool alive = true;

    if (has0) {
      // Prefetch this warp's rows of G_{j,j-1}, the block most likely waited on.
      if (j > 0) {
        const float* gb = a.G + packed_offset(j, j - 1, a.b, a.diag);
        const int lines = (a.b * 4 + 127) / 128;
        for (int l = lane; l < 2 * lines; l += 32) {
          const int rr = l / lines;
          if (rr == 1 && !has1) continue;
          const float* pch = gb + (int64_t)(i0 + rr) * a.b + (l - rr * lines) * 32;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(pch));
        }
      }
      float acc0 = 0.0f, acc1 = 0.0f;
      int frontier = 0;
      if (j > 0 && lane == 0 &&
          ld_acquire_u32(&a.ctrl->block_done[j - 1]) >= (uint32_t)a.units_per_block)
        frontier = j;
      frontier = __shfl_sync(0xffffffffu, frontier, 0);
      for (int t = 0; t < j; ++t) {
        if (t >= frontier) {
          if (!wait_block(a, t)) { alive = false; break; }
          frontier = t + 1;
        }
        const float* g0 = a.G + packed_offset(j, t, a.b, a.diag) + (int64_t)i0 * a.b;
        const float* g1 = g0 + a.b;
        const float* al = a.alpha + (int64_t)t * a.b;
        if (vec4) {
          for (int col = lane * 4; col < a.b; col += 128) {
            const float4 av = __ldcg(reinterpret_cast<const float4*>(al + col));
            const float4 x0 = __ldg(reinterpret_cast<const float4*>(g0 + col));
            acc0 = fmaf(x0.x, av.x, acc0); acc0 = fmaf(x0.y, av.y, acc0);
            acc0 = fmaf(x0.z, av.z, acc0); acc0 = fmaf(x0.w, av.w, acc0);
            if (has1) {
              const float4 x1 = __ldg(reinterpret_cast<const float4*>(g1 + col));
              acc1 = fmaf(x1.x, av.x, acc1); acc1 = fmaf(x1.y, av.y, acc1);
              acc1 = fmaf(x1.z, av.z, acc1); acc1 = fmaf(x1.w, av.w, acc1);
            }
          }
        } else {
          for (int col = lane; col < a.b; col += 32) {
            const float av = __ldcg(al + col);
            acc0 = fmaf(__ldg(g0 + col), av, acc0);
            if (has1) acc1 = fmaf(__ldg(g1 + col), av, acc1);
          }
        }
      }
      if (alive) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          acc0 += __shfl_xor_sync(0xffffffffu, acc0, off);
          acc1 += __shfl_xor_sync(0xffffffffu, acc1, off);
        }
        if (lane == 0) {
          const int64_t p0 = (int64_t)j * a.b + i0;
          const float z0 = bf16_bits_to_float(a.r[p0]) + acc0;
          a.alpha[p0] = a.coef * loss_deriv(a.loss, z0, a.yY[p0]);
          if (has1) {
            const float z1 = bf16_bits_to_float(a.r[p0 + 1]) + acc1;
            a.alpha[p0 + 1] = a.coef * loss_deriv(a.loss, z1, a.yY[p0 + 1]);
          }
          __threadfence();
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && !(a.stall_test && j == 0)) {
      __threadfence();
      atomicAdd(&a.ctrl->block_done[j], 1u);
    }
  }
}

}  // namespace

cudaError_t launch_recur(const float* G, const uint16_t* r, const float* yY, float* alpha,
                         int b, int s, float eta, int loss, uint32_t flags,
                         uint32_t timeout_us, Ctrl* ctrl, Ctx& c) {
  RecArgs a;
  a.G = G;
  a.r = r;
  a.yY = yY;
  a.alpha = alpha;
  a.ctrl = ctrl;
  a.timeout_ns = (uint64_t)(timeout_us ? timeout_us : 1000000u) * 1000ull;
  a.b = b;
  a.s = s;
  a.loss = loss;
  a.unit_rows = b < kUnitRows ? b : kUnitRows;
  a.units_per_block = (b + a.unit_rows - 1) / a.unit_rows;
  a.coef = -(eta / (float)b);
  a.diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  a.stall_test = (flags & CASGD_FLAG_TEST_STALL) != 0;

  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, recur_kernel, 256, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorLaunchOutOfResources;
  int64_t grid = (int64_t)per_sm * c.num_sms;
  const int64_t units = (int64_t)s * a.units_per_block;
  if (grid > units) grid = units;
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel((const void*)recur_kernel, dim3((unsigned)grid), dim3(256),
                                  args, 0, c.stream);
  ++c.launches;
  return e;
}

}  // namespace casgd
