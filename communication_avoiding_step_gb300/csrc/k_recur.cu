// Steps a6/a7: the FP32 inner s-step recurrence
//     z_j = r_j + sum_{t<j} G_{j,t} alpha_t,   alpha_j = -(eta/b) * l'(z_j, y_j).
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the inner recurrence runs in high precision, from the BF16 margins
// and the FP32 Gram matrix.  alpha of one row depends only on that row's z, so rows
// are independent once all earlier blocks are known; the s blocks form a serial chain.
//
// Design: one persistent cooperative launch (all CTAs co-resident) with two roles.
//  * Chain CTAs (the first C CTAs): one warp per row, 8-row groups.  Phase j of a row
//    needs only the band  sum_{t=j-B}^{j-1} G_{j,t} alpha_t  (B = 1 or 2 blocks) on top
//    of far_j (below).  The warp loads its band rows of G, the older band alpha, r and
//    y before it waits, then waits for alpha_{j-1} and far_j by loading exactly those
//    values until none holds the pending pattern.
//  * Bulk CTAs take units (block j >= B+1, 16 rows) from an atomic queue in increasing
//    j and compute far_j = sum_{t<j-B} G_{j,t} alpha_t for their rows, streaming G with
//    coalesced float4 reads; they wait on alpha_t the same way.  far_j is needed only B
//    phases after its last input is known, so most of G is read off the critical path.
//    After the far units, the same queue hands out the first stage of the weight update
//    (step a8) when it is fused here: per block j and 64-column chunk, the partial row
//    of Y^T alpha over that block, each waiting on the alpha of its own rows.
// Synchronisation is through the data: the gather kernel fills alpha and far with
// kAlphaPending before this kernel runs, and a value is final once it differs from
// that pattern (32-bit stores are single-copy atomic, and a reader uses only the value
// it waited on, so no fences or counters are needed).  Warps of a chain CTA never wait
// on each other.  Every wait is bounded by `timeout_ns`; on expiry the waiter records
// ST_TIMEOUT, which wait gave up (Ctrl::diag) and the abort word, and every other
// waiter stops.  Sums are taken in a fixed order (far_j over t ascending; then
// r + far + band), so results are deterministic.
#include "casgd_internal.cuh"

namespace casgd {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;       // rows per bulk unit
constexpr int kChainRows = 8;   // rows per chain group (a warp per row)
constexpr int kPrefetch = 8;    // float4 of band G (and of alpha) a chain lane keeps in registers
constexpr int kT = 4;           // bulk: blocks t handled per pass

struct RecArgs {
  const float* G;
  const uint16_t* r;
  const float* yY;
  float* alpha;
  float* far;
  uint64_t* trace;  // [kMaxS][4] timestamps of chain CTA 0, warp 0
  // fused first stage of the weight update (upd_units > 0): partial rows of Y^T alpha
  const uint16_t* Y;
  float* part;
  int64_t ldY;
  int upd_units, TV;
  Ctrl* ctrl;
  uint64_t timeout_ns;
  int b, s, loss, U, Uc, C, B, bulk_units;
  float coef;
  bool diag, stall_test, vec4;
};

// Ctrl::diag codes: kind << 24 | block << 12 (kind 2: chain wait, 3: bulk wait).
__device__ __forceinline__ uint32_t where_code(uint32_t kind, int j) {
  return (kind << 24) | ((uint32_t)j << 12);
}

__device__ __forceinline__ float dot4(float4 g, float4 v, float acc) {
  acc = fmaf(g.x, v.x, acc);
  acc = fmaf(g.y, v.y, acc);
  acc = fmaf(g.z, v.z, acc);
  return fmaf(g.w, v.w, acc);
}

__device__ __forceinline__ bool pending1(float v) { return __float_as_uint(v) == kAlphaPending; }
__device__ __forceinline__ bool pending4(float4 v) {
  return pending1(v.x) || pending1(v.y) || pending1(v.z) || pending1(v.w);
}

__device__ __forceinline__ float4 ld_volatile_f4(const float* p) {
  float4 v;
  asm volatile("ld.volatile.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ float ld_volatile_f32(const float* p) {
  return *reinterpret_cast<const volatile float*>(p);
}

// Records a timeout (status, diag, abort); returns false.
__device__ bool give_up(const RecArgs& a, uint32_t where) {
  atomicOr(&a.ctrl->status, ST_TIMEOUT);
  atomicExch(&a.ctrl->diag, where);
  atomicExch(&a.ctrl->abort, 1u);
  return false;
}

// Bound check for a wait loop: false once the wait must end.
__device__ __forceinline__ bool keep_waiting(const RecArgs& a, uint64_t t_start, uint32_t where) {
  if (ld_volatile_u32(&a.ctrl->abort)) return false;
  if (globaltimer_ns() - t_start > a.timeout_ns) return give_up(a, where);
  return true;
}

// Scalar value wait (used where b is not a multiple of 4).
__device__ bool wait_value(const float* p, float& v, const RecArgs& a, uint32_t where) {
  v = ld_volatile_f32(p);
  if (!pending1(v)) return true;
  const uint64_t t_start = globaltimer_ns();
  while (true) {
    v = ld_volatile_f32(p);
    if (!pending1(v)) return true;
    if (!keep_waiting(a, t_start, where)) return false;
  }
}

// ------------------------------------------------------------------ chain role
// A warp per row; a lane's columns are lane*4 + 128k.  Chain CTA c owns the 8-row
// groups c, c+C, ... of every block.  The band is kB blocks wide; register slot
// (tb, k) holds band block j-1-tb at columns lane*4 + 128k, so every slot index is a
// compile-time constant (kKB = kPrefetch / kB slots per block).
template <int kB>
__device__ void chain_role(const RecArgs& a, int c) {
  constexpr int kKB = kPrefetch / kB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (a.b + 127) / 128;  // float4 slots per band block (vec4 path)
  // Chain CTA 0, warp 0 keeps a per-phase timeline (globaltimer ns): phase start, loads
  // issued, alpha_{j-1} and far_j arrived, alpha_j stored.
  const bool tracer = (c == 0 && threadIdx.x == 0);
  for (int j = 0; j < a.s; ++j) {
    if (tracer) a.trace[4 * j] = globaltimer_ns();
    const int t0 = j - kB > 0 ? j - kB : 0;
    const int nb = j - t0;             // band blocks this phase (the last is t = j-1)
    const bool has_far = j >= kB + 1;
    for (int grp = c; grp < a.Uc; grp += a.C) {
      const int i = grp * kChainRows + warp;  // row within block j
      if (i >= a.b) continue;                 // warp-uniform
      const int64_t p = (int64_t)j * a.b + i;
      const float* grow0 = a.G + (int64_t)i * a.b;
      // (a) loads that do not need alpha_{j-1}.  Slot row tb holds band block
      // t = j-1-tb (tb < nb): row 0 is the block waited on, rows >= 1 are complete.
      float4 gv[kB][kKB], av[kB][kKB];
#pragma unroll
      for (int tb = 0; tb < kB; ++tb) {
        const int t = j - 1 - tb;
        const bool in_band = tb < nb;
        const float* gb = grow0 + (in_band ? packed_offset(j, t, a.b, a.diag) : 0) + lane * 4;
        const float* ab = a.alpha + (int64_t)(in_band ? t : 0) * a.b + lane * 4;
#pragma unroll
        for (int k = 0; k < kKB; ++k) {
          gv[tb][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          av[tb][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (a.vec4 && in_band && lane * 4 + 128 * k < a.b) {
            gv[tb][k] = __ldg(reinterpret_cast<const float4*>(gb + 128 * k));
            if (tb >= 1)  // seen complete by this lane in an earlier phase
              av[tb][k] = __ldcg(reinterpret_cast<const float4*>(ab + 128 * k));
          }
        }
      }
      uint32_t rbits = 0;  // converted after the wait, so the load does not stall the issue
      float yj = 0.0f;
      if (lane == 0) {
        rbits = a.r[p];
        yj = a.yY[p];
      }
      if (tracer) a.trace[4 * j + 1] = globaltimer_ns();
      // (b) alpha_{j-1} (slot row 0) and far_j: load them until none is pending
      const float* aprev = a.alpha + (int64_t)(j - 1) * a.b + lane * 4;
      bool pend = false;
      float farv = 0.0f;
      if (a.vec4 && j > 0) {
#pragma unroll
        for (int k = 0; k < kKB; ++k) {
          if (lane * 4 + 128 * k < a.b) {
            av[0][k] = ld_volatile_f4(aprev + 128 * k);
            pend |= pending4(av[0][k]);
          }
        }
      }
      if (has_far && lane == 0) {
        farv = ld_volatile_f32(a.far + p);
        pend |= pending1(farv);
      }
      bool ok = true;
      if (__any_sync(0xffffffffu, pend)) {
        const uint64_t t_start = globaltimer_ns();
        while (true) {
          __nanosleep(32);  // eases the load on the few L2 lines every chain warp polls
          pend = false;
          if (a.vec4 && j > 0) {
#pragma unroll
            for (int k = 0; k < kKB; ++k) {
              if (lane * 4 + 128 * k < a.b && pending4(av[0][k])) {
                av[0][k] = ld_volatile_f4(aprev + 128 * k);
                pend |= pending4(av[0][k]);
              }
            }
          }
          if (has_far && lane == 0 && pending1(farv)) {
            farv = ld_volatile_f32(a.far + p);
            pend |= pending1(farv);
          }
          if (!__any_sync(0xffffffffu, pend)) break;
          ok = keep_waiting(a, t_start, where_code(2, j));
          if (!__all_sync(0xffffffffu, ok)) return;
        }
      }
      if (tracer) a.trace[4 * j + 2] = globaltimer_ns();
      float acc = 0.0f;
      if (a.vec4) {
#pragma unroll
        for (int tb = 0; tb < kB; ++tb)
#pragma unroll
          for (int k = 0; k < kKB; ++k)
            if (tb < nb) acc = dot4(gv[tb][k], av[tb][k], acc);
        // columns beyond the register slots (b > 128 * kKB)
        for (int tb = 0; tb < nb; ++tb) {
          const int t = j - 1 - tb;
          for (int k = kKB; k < nk; ++k) {
            const int col = lane * 4 + 128 * k;
            if (col >= a.b) break;
            const float* src = a.alpha + (int64_t)t * a.b + col;
            float4 v = ld_volatile_f4(src);
            if (pending4(v)) {
              const uint64_t t_start = globaltimer_ns();
              while (pending4(v) && (ok = keep_waiting(a, t_start, where_code(2, j)))) v = ld_volatile_f4(src);
            }
            acc = dot4(__ldg(reinterpret_cast<const float4*>(grow0 + packed_offset(j, t, a.b, a.diag) + col)),
                       v, acc);
          }
        }
      } else {
        for (int t = t0; t < j && ok; ++t) {
          const float* al = a.alpha + (int64_t)t * a.b;
          const float* grow = grow0 + packed_offset(j, t, a.b, a.diag);
          for (int col = lane; col < a.b; col += 32) {
            float v;
            if (!(ok = wait_value(al + col, v, a, where_code(2, j)))) break;
            acc = fmaf(__ldg(grow + col), v, acc);
          }
        }
      }
      if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0 && !(a.stall_test && j == 0)) {
        const float z = bf16_bits_to_float(rbits) + farv + acc;
        __stcg(a.alpha + p, a.coef * loss_deriv(a.loss, z, yj));
      }
    }
    if (tracer) a.trace[4 * j + 3] = globaltimer_ns();
  }
}

// --------------------------------------------------------------- update units
// Step a8's first stage, fused: unit (j, cc) sums alpha_i * Y_i over the b rows of block
// j for the 64 columns cc*64 .. cc*64+63 into part[j][...] (one partial row per block;
// the reduce kernel then adds the s rows to w).  Threads: 32 row-lanes x 8 column
// vectors; each waits on the alpha of its own rows.  Units of block j become workable
// as soon as phase j is done, so only the last block's units (spread over many CTAs)
// run after the chain ends.  Fixed order: rows ascending per row-lane, then row-lanes
// ascending in shared memory.
__device__ void update_unit(const RecArgs& a, int u) {
  __shared__ float red[32][64];
  const int nchunk = (int)((a.ldY / 8 + 7) / 8);
  const int j = u / nchunk, cc = u - j * nchunk;
  const int tv = threadIdx.x & 7, tr = threadIdx.x >> 3;  // vector-lane, row-lane
  const int64_t vec = (int64_t)cc * 8 + tv;
  const bool vin = vec < a.ldY / 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  for (int i0 = tr; i0 < a.b && ok; i0 += 32 * 4) {
    float al[4];
    uint4 q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = i0 + 32 * k;
      const bool in = i < a.b;
      const int64_t row = (int64_t)j * a.b + i;
      al[k] = in ? ld_volatile_f32(a.alpha + row) : 0.0f;
      q[k] = (in && vin) ? __ldg(reinterpret_cast<const uint4*>(a.Y + row * a.ldY + vec * 8))
                         : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (pending1(al[k])) {  // this row's alpha is not final yet
        const int64_t row = (int64_t)j * a.b + i0 + 32 * k;
        const uint64_t t_start = globaltimer_ns();
        while (pending1(al[k]) && ok) {
          __nanosleep(200);
          al[k] = ld_volatile_f32(a.alpha + row);
          if (pending1(al[k])) ok = keep_waiting(a, t_start, where_code(4, j));
        }
      }
      const uint32_t pw[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        acc[2 * h] = fmaf(al[k], bf16_bits_to_float(pw[h] & 0xFFFFu), acc[2 * h]);
        acc[2 * h + 1] = fmaf(al[k], bf16_bits_to_float(pw[h] >> 16), acc[2 * h + 1]);
      }
    }
  }
  __syncthreads();  // red may still be read by this CTA's previous unit
#pragma unroll
  for (int e = 0; e < 8; ++e) red[tr][tv * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < 64) {
    const int col = threadIdx.x;
    float sum = 0.0f;
    for (int r = 0; r < 32; ++r) sum += red[r][col];
    const int64_t c = (int64_t)cc * 64 + col;
    if (c < a.ldY) a.part[(int64_t)j * a.ldY + c] = sum;
  }
}

// ------------------------------------------------------------------- bulk role
// Unit = (block j, 16 rows); each warp owns two rows; a lane's columns are lane*4 + 128k.
// The CTA waits as a whole: a final alpha value of phase q implies that phase q-1 is
// complete (its row needed all of alpha_{q-1}), so thread 0 reads single values of the
// next phases (spread over the values by CTA index, with a back-off while the next
// phase is not done) and the CTA then processes every block known complete, up to kT
// per pass with all their loads issued together, reading alpha with plain loads.  Each
// block's dot product is summed over columns first and then added in t order, so the
// result does not depend on timing.
__device__ void bulk_role(const RecArgs& a) {
  __shared__ int s_unit, s_lead;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int probe_col = (int)((blockIdx.x * 37u) % (unsigned)a.b);
  while (true) {
    if (threadIdx.x == 0) {
      int u = (int)atomicAdd(&a.ctrl->next_unit, 1u);
      if (ld_volatile_u32(&a.ctrl->abort)) u = a.bulk_units + a.upd_units;
      s_unit = u;
    }
    __syncthreads();
    const int unit = s_unit;
    __syncthreads();
    if (unit >= a.bulk_units) {
      if (unit < a.bulk_units + a.upd_units) {
        update_unit(a, unit - a.bulk_units);
        __syncthreads();
        continue;
      }
      return;
    }
    const int j = a.B + 1 + unit / a.U;
    const int c = unit % a.U;
    const int i0 = c * kRows + warp * 2;
    const bool has0 = i0 < a.b, has1 = i0 + 1 < a.b;
    const int t_end = j - a.B;  // far_j covers t < j - B
    float acc0 = 0.0f, acc1 = 0.0f;
    bool ok = true;
    for (int t = 0; t < t_end;) {
      if (threadIdx.x == 0) {
        // leading run of complete phases t, t+1, ... (at most kT and t_end - t)
        const int lim = min(kT, t_end - t);
        int lead = 0;
        while (lead < lim && !pending1(ld_volatile_f32(a.alpha + (int64_t)(t + lead + 1) * a.b + probe_col)))
          ++lead;
        if (lead == 0) {  // wait for phase t, polling one value of phase t+1
          const float* pv = a.alpha + (int64_t)(t + 1) * a.b + probe_col;
          const uint64_t t_start = globaltimer_ns();
          while (pending1(ld_volatile_f32(pv))) {
            __nanosleep(200);
            if (!keep_waiting(a, t_start, where_code(3, j))) break;
          }
          lead = pending1(ld_volatile_f32(pv)) ? 0 : 1;
        }
        s_lead = lead;
      }
      __syncthreads();
      const int nt = s_lead;
      __syncthreads();
      if (nt == 0) { ok = false; break; }  // gave up (uniform)
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
                const float v = __ldcg(al + col);
                d0[u] = fmaf(__ldg(gb + col), v, d0[u]);
                if (has1) d1[u] = fmaf(__ldg(gb + a.b + col), v, d1[u]);
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
    if (has0) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        acc0 += __shfl_xor_sync(0xffffffffu, acc0, off);
        acc1 += __shfl_xor_sync(0xffffffffu, acc1, off);
      }
      if (lane == 0 && ok) {
        const int64_t p0 = (int64_t)j * a.b + i0;
        __stcg(a.far + p0, acc0);
        if (has1) __stcg(a.far + p0 + 1, acc1);
      }
    }
    __syncthreads();  // every warp of the unit is done before the CTA claims the next
  }
}

template <int kB>
__global__ void __launch_bounds__(kThreads) recur_kernel(RecArgs a) {
  if ((int)blockIdx.x < a.C)
    chain_role<kB>(a, blockIdx.x);
  else
    bulk_role(a);
}

}  // namespace

cudaError_t launch_recur(const float* G, const uint16_t* r, const float* yY, float* alpha,
                         float* far, uint32_t* far_done, int b, int s, float eta, int loss,
                         uint32_t flags, uint32_t timeout_us, Ctrl* ctrl, const uint16_t* Y,
                         int64_t ldY, float* part, int upd_units /* nonzero: fuse */, Ctx& c) {
  RecArgs a;
  a.G = G;
  a.r = r;
  a.yY = yY;
  a.alpha = alpha;
  a.far = far;
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
  const void* fn = a.B == 2 ? (const void*)recur_kernel<2> : (const void*)recur_kernel<1>;
  a.bulk_units = s > a.B + 1 ? (s - a.B - 1) * a.U : 0;
  a.coef = -(eta / (float)b);
  a.Y = Y;
  a.part = part;
  a.ldY = ldY;
  // update units: s blocks x ceil(ldY / 64) column chunks (0 = update not fused)
  a.upd_units = upd_units ? s * (int)((ldY / 8 + 7) / 8) : 0;
  a.TV = 0;
  a.diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  a.stall_test = (flags & CASGD_FLAG_TEST_STALL) != 0;

  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorLaunchOutOfResources;
  const int64_t cap = (int64_t)per_sm * c.num_sms;
  // one chain CTA per 8-row group while that leaves room for the bulk CTAs
  const int64_t queued = (int64_t)a.bulk_units + a.upd_units;  // units for non-chain CTAs
  int64_t cmax = queued > 0 ? cap / 2 : cap;
  if (cmax < 1) cmax = 1;
  a.C = (int)(a.Uc < cmax ? a.Uc : cmax);
  if (a.C + (queued > 0 ? 1 : 0) > cap) return cudaErrorNotSupported;
  int64_t grid = a.C + queued;
  if (grid > cap) grid = cap;
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel(fn, dim3((unsigned)grid), dim3(kThreads), args, 0, c.stream);
  ++c.launches;
  return e;
}

}  // namespace casgd
