// Roles of the inner s-step recurrence (steps a6/a7) and of the fused first stage of
// the weight update (a8), shared by the stand-alone recurrence kernel (k_recur.cu) and
// the kernel that runs them beside the paired-SM Gram (k_gram_tc.cu).
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the inner recurrence runs in high precision, from the BF16 margins
// and the FP32 Gram matrix,
//     z_j = r_j + sum_{t<j} G_{j,t} alpha_t,   alpha_j = -(eta/b) * l'(z_j, y_j).
// alpha of one row depends only on that row's z, so rows are independent once all
// earlier blocks are known; the s blocks form a serial chain.
//
// Two roles, each run by a group of 256 threads (a whole CTA in the stand-alone kernel,
// warps 6-13 of a CTA in the kernels shared with the Gram).  kMode: 0 own CTA, G
// complete; 1 shared CTA, rows of G still being stored by the same launch; 2 shared
// CTA, G complete (the launch computes the next iteration's Gram); 3 shared CTA, the
// Gram of the same launch stores only the band blocks and forms the far sums itself
// (partial sums per row and block t, see below); 4 as 3 with the band already
// complete (the launch's Gram stores the next iteration's band):
//  * chain groups (the first C): one warp per row, 8-row groups.  Phase j of a row
//    needs only the band  sum_{t=j-B}^{j-1} G_{j,t} alpha_t  (B = 1 to 3 blocks) on top
//    of far_j (below).  The warp has its band rows of G in registers before it waits
//    (loaded while it waited in the previous phase), then waits for alpha_{j-1} and
//    far_j by loading exactly those values until none holds the pending pattern.
//  * bulk groups take units from atomic queues.  Modes 0-2: far units (block j >= B+1,
//    16 rows) whose sum far_j = sum_{t<j-B} G_{j,t} alpha_t runs over t in runs of up to
//    four phases whose alpha is already final, streaming G with coalesced float4 reads.
//    Modes 3 and 4 have no far units: the Gram's epilogue multiplies each far tile
//    G_{j,t} by alpha_t once alpha_t is final and stores one partial sum per row, block
//    t and column group (npb groups per block), and the chain adds a row's (j-B) * npb
//    partials itself, in a fixed order; there the bulk units are margin units
//    (r = Y w for a run of rows, before the chain needs them).  A second queue hands
//    out the first stage of the weight update: per block j and 64-column chunk (and
//    row part), the partial row of Y^T alpha over that block, once its alpha is final.
//    far_j is needed only B phases after its last input is known, so most of the far
//    work is off the critical path.
// Synchronisation is through the data: the launch before the recurrence fills alpha and
// far (and r and the far partials where those are formed in the launch) with
// kAlphaPending, and a value is final once it differs from that pattern (32-bit stores
// are single-copy atomic, and a reader uses only the value it waited on, so no fences
// or counters are needed).  When the Gram of the same iteration runs in the same launch
// and stores the rows a reader needs (modes 1 and 3), those rows are guarded by
// per-32-row counters that the Gram's epilogue warps release once their stores of a
// tile are complete; a reader acquires the counter of its rows before loading them, and
// loads G through L2 only.  Every wait is bounded by `timeout_ns`; on expiry the waiter
// records ST_TIMEOUT, which wait gave up (Ctrl::diag) and the abort word, and every
// other waiter stops.  Sums are taken in a fixed order (far_j over t ascending, or the
// partials two per lane and then a fixed shuffle tree; then r + far + band), so results are deterministic.
#pragma once

#include "casgd_internal.cuh"

namespace casgd {

constexpr int kRecThreads = 256;  // threads of one role group
constexpr int kRecRows = 16;      // rows per bulk unit
constexpr int kChainRows = 8;     // rows per chain group (a warp per row)

struct RecArgs {
  const float* G;
  int gB;          // layout of G: 0 packed block-lower, B > 0 band layout (g_block_offset)
  const float* r;  // margins (BF16 values in the recipe)
  const float* yY;
  float* alpha;
  float* far;
  uint64_t* trace;  // [kMaxS][4] timestamps of chain group 0, warp 0 (null: not traced)
  // fused first stage of the weight update (upd_units > 0): partial rows of Y^T alpha
  const uint16_t* Y;
  // Rows of Y read straight from X (X non-null; the far-forming launch that gathers its
  // operands itself): row p of Y is row draw_row(xseed, xctr + p, xm, xperm) of X, whose
  // pitch is ldx; columns of X from n on are never read
  const uint16_t* X;
  int64_t ldx;
  uint64_t xseed, xctr;
  uint32_t xm;
  int xperm;
  float* part;
  int64_t ldY;
  int upd_units;
  int upd_R;  // row parts per block (upd_row_parts)
  // the update's counters: row parts of (block, column chunk) that have stored their
  // partial row (upd_blocks), and block sums of a column chunk formed (upd_chunks; the
  // last adds the chunk's s block sums to w)
  uint32_t* upd_chunks;
  uint32_t* upd_blocks;
  float* w;
  int64_t n;
  // Gram in the same launch: per-32-row completion counters of the paired-SM Gram
  const uint32_t* slab;
  // mode 3: far partial sums fpart[row * fs + t * npb + c], t < j - B, c < npb (column
  // groups of block t), written by the Gram
  const float* fpart;
  int fs, npb;
  // Gram in the same launch: Ctrl::band_done reaches band_total once every tile the Gram
  // stores is stored (each epilogue warp adds its tiles after its 32-row counter)
  uint32_t band_total;
  // Margins formed in this launch (with the far-forming Gram): the bulk groups' first
  // units (bulk_units of them, mrows rows each, mG lanes per row) write r (pending until
  // then) from Y and w.  The update writes w only once a column chunk's s block sums are
  // all formed, which needs alpha_{s-1}, so after the chain has read every margin.
  bool margins, r_fp32, wm_vec;  // wm_vec: w 16-byte aligned
  int mrows, mG;
  float* r_w;
  const float* wm;  // w as the launch starts (w_k), read by the margin units
  bool far_gram;  // the Gram stores only the band (and diagonal) tiles
  int64_t S;
  Ctrl* ctrl;  // status, abort word and diagnostics
  Ctrl* q;     // this iteration's queues and counters (next_unit, upd_next, band_done)
  uint64_t timeout_ns;
  int b, s, loss, U, Uc, C, B, bulk_units;
  int upd_groups;  // bulk groups that serve the update queue first
  float coef;
  bool diag, stall_test, vec4;
};

// Register layout of a chain lane: kB band blocks x kKB float4 slots per block.
// 1: (1, 8) for b > 512 or b % 4 != 0; 2: (2, 4) for 256 < b <= 512; 3: (3, 2) for
// b <= 256 (a wider band leaves the far sums one more phase of slack).
inline int chain_variant(const RecArgs& a) {
  if (a.B == 3) return 3;
  return a.B == 2 ? 2 : 1;
}

// Bulk groups that serve the update queue first, out of nbulk: the update's share of
// the bytes the bulk role streams (Y for the update, the far blocks of G), at least one.
inline int update_groups(const RecArgs& a, int nbulk) {
  if (a.upd_units <= 0 || nbulk <= 1) return 0;
  const double ub = (double)a.S * (double)a.ldY * 2.0;
  const double nfar = (a.s > a.B + 1) ? 0.5 * (a.s - a.B - 1) * (a.s - a.B) : 0.0;
  const double fb = nfar * (double)a.b * (double)a.b * 4.0;
  int g = (int)(nbulk * ub / (ub + fb) + 0.5);
  if (g < 1) g = 1;
  if (g > nbulk - 1) g = nbulk - 1;
  return g;
}

// Fills every field but C and upd_groups (chosen by the launcher from its grid) and slab.
// counters: the workspace's counters area (timeline_of); w: FP32[n], updated in place.
RecArgs make_rec_args(const float* G, const float* r, const float* yY, float* alpha,
                      float* far, uint32_t* counters, int b, int s, float eta, int loss,
                      uint32_t flags, uint32_t timeout_us, Ctrl* ctrl, const uint16_t* Y,
                      int64_t ldY, int64_t n, float* part, float* w);

namespace {

constexpr int kT = 4;         // bulk: blocks t handled per pass
constexpr int kUpdRows = 8;   // update unit: rows a thread loads per pass

// Ctrl::diag codes: kind << 24 | block << 12 (2: chain wait, 3: bulk wait, 4: update
// wait, 5: wait for rows of G, 6: wait for the CTA's own tiles).
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

// G is read through the read-only path when an earlier launch wrote it, and through L2
// only when the Gram of the same launch is still writing other rows of it.
template <bool kInFlight>
__device__ __forceinline__ float4 ldG4(const float* p) {
  if (kInFlight) return __ldcg(reinterpret_cast<const float4*>(p));
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <bool kInFlight>
__device__ __forceinline__ float ldG1(const float* p) {
  if (kInFlight) return __ldcg(p);
  return __ldg(p);
}

// Barrier of one role group: the whole CTA, or named barrier 1 over warps 6-13.
template <bool kShared>
__device__ __forceinline__ void group_sync() {
  if (kShared)
    asm volatile("bar.sync 1, %0;" ::"r"(kRecThreads) : "memory");
  else
    __syncthreads();
}

// Profiling (tracing on): latest time an event of kind e happened (summary row of the
// timeline: 0 last tile of G stored, 1 last far sum stored, 2 last update partial).
__device__ __forceinline__ void stamp_last(uint64_t* trace, int e) {
  if (trace)
    atomicMax(reinterpret_cast<unsigned long long*>(trace + kMaxS * 4 + e),
              (unsigned long long)globaltimer_ns());
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

// Tiles the Gram stores for the 256-row group holding 32-row slab `sl`.
__device__ __forceinline__ uint32_t slab_need(const RecArgs& a, int64_t sl) {
  const int g = (int)(sl >> 3);
  return (uint32_t)(a.far_gram ? far_gram_stored_tiles(a.b, a.diag, g)
                               : pair_group_tiles(a.S, a.b, a.diag, g));
}

// Waits (acquire) until every tile of the Gram's 256-row group holding absolute row
// `row` is stored: the counter of the row's 32-row slab reaches the group's tile count.
__device__ bool wait_rows_of_G(const RecArgs& a, int64_t row, uint32_t where) {
  const int64_t sl = row >> 5;
  const uint32_t need = slab_need(a, sl);
  if (ld_acquire_u32(a.slab + sl) >= need) return true;
  const uint64_t t_start = globaltimer_ns();
  while (true) {
    __nanosleep(256);
    if (ld_acquire_u32(a.slab + sl) >= need) return true;
    if (!keep_waiting(a, t_start, where)) return false;
  }
}

// ------------------------------------------------------------------ chain role
// A warp per row; a lane's columns are lane*4 + 128k.  Chain group c owns the 8-row
// groups c, c+C, ... of every block, so a warp's work is a sequence of items (phase j,
// row i): phases ascending, then its groups.  The band is kB blocks wide; register slot
// (tb, k) holds band block j-1-tb at columns lane*4 + 128k (k < kKB), so every slot
// index is a compile-time constant.
// Software pipeline: the band rows of G for the warp's next item are loaded while it
// waits for the current item's alpha (once the Gram has stored them, when it runs in
// the same launch), and the alpha vectors are kept in registers from item to item:
// alpha_{j-2} of phase j is the alpha_{j-1} the warp waited for in phase j-1, and the
// later items of a phase reuse the first item's.  So the only loads on the critical
// path are the polls of alpha_{j-1} and far_j.  `rt` is the thread's index within the
// role group.
template <int kB, int kKB, int kMode>
__device__ void chain_role(const RecArgs& a, int c, int rt) {
  constexpr bool kInFlight = kMode == 1 || kMode == 3;  // G stored by this launch
  constexpr bool kFarParts = kMode >= 3;                // far sums from the Gram's partials
  // the next item's row values are loaded with its band, except in the widest register
  // layout (eight float4 slots per block), which has no registers to spare for them
  constexpr bool kRowAhead = kKB < 8;
  const int warp = rt >> 5, lane = rt & 31;
  const int nk = (a.b + 127) / 128;  // float4 slots per band block (vec4 path)
  // With tracing on, chain group 0, warp 0 keeps a per-phase timeline (globaltimer ns):
  // phase start, loads issued, alpha_{j-1} and far_j arrived, alpha_j stored.
  const bool tracer = (c == 0 && rt == 0 && a.trace != nullptr);
  // groups of this warp with a row inside the block (the last group may be partial)
  int ng = 0;
  for (int grp = c; grp < a.Uc; grp += a.C)
    if (grp * kChainRows + warp < a.b) ++ng;
  if (ng == 0) return;

  // loads the band rows of G of item (j, i) into g (zeros outside the band)
  auto load_band = [&](float4 (&g)[kB][kKB], int j, int i) {
    const float* grow0 = a.G + (int64_t)i * a.b;
    const int nb = j < kB ? j : kB;
#pragma unroll
    for (int tb = 0; tb < kB; ++tb) {
      const float* gb = grow0 + (tb < nb ? g_block_offset(j, j - 1 - tb, a.b, a.diag, a.gB) : 0) + lane * 4;
#pragma unroll
      for (int k = 0; k < kKB; ++k) {
        g[tb][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.vec4 && tb < nb && lane * 4 + 128 * k < a.b) g[tb][k] = ldG4<kInFlight>(gb + 128 * k);
      }
    }
  };

  // loads the row values of item (j, i): margin and label (lane 0) and far_j (lane 0;
  // mode 3: the row's partials t = lane and t = lane + 32), possibly still pending
  auto load_row = [&](int j, int i, uint32_t& rb, float& yv, float& f0, float& f1) {
    const int64_t p = (int64_t)j * a.b + i;
    rb = 0;
    yv = f0 = f1 = 0.0f;
    if (lane == 0) {
      rb = __float_as_uint(ld_volatile_f32(a.r + p));  // pending while formed in this launch
      yv = a.yY[p];
    }
    if (j < kB + 1) return;
    if (kFarParts) {
      const int nfar = (j - kB) * a.npb;
      const float* fsrc = a.fpart + p * a.fs;
      if (lane < nfar) f0 = ld_volatile_f32(fsrc + lane);
      if (lane + 32 < nfar) f1 = ld_volatile_f32(fsrc + lane + 32);
    } else if (lane == 0) {
      f0 = ld_volatile_f32(a.far + p);
    }
  };
  // Gram in the same launch: whether rows of item (j, i) are stored; once every stored
  // tile is, no counter is read again
  bool all_stored = !kInFlight;
  auto rows_stored = [&](int j, int i) -> bool {
    int ready = 1;
    if (!all_stored) {
      if (lane == 0) {
        ready = ld_acquire_u32(&a.q->band_done) >= a.band_total;
        if (!ready) {
          const int64_t sl = ((int64_t)j * a.b + i) >> 5;
          ready = ld_acquire_u32(a.slab + sl) >= slab_need(a, sl) ? 2 : 0;
        }
      }
      ready = __shfl_sync(0xffffffffu, ready, 0);
      __syncwarp();
      if (ready == 1) all_stored = true;
    }
    return ready != 0;
  };

  float4 gv[kB][kKB], gn[kB][kKB], av[kB][kKB];
#pragma unroll
  for (int tb = 0; tb < kB; ++tb)
#pragma unroll
    for (int k = 0; k < kKB; ++k) av[tb][k] = make_float4(0.f, 0.f, 0.f, 0.f);
  bool cur_loaded = false;  // gv holds the current item's band
  bool row_loaded = false;  // rbits, yj, fv0, fv1 hold the current item's row values
  uint32_t rbits = 0;       // converted after the wait, so the load does not stall the issue
  float yj = 0.0f, fv0 = 0.0f, fv1 = 0.0f;
  int jprev = -1;
  int j = 0, gi = 0;        // item: phase j, gi-th valid group of the warp
  while (j < a.s) {
    const int i = (c + gi * a.C) * kChainRows + warp;  // row within block j
    const int64_t p = (int64_t)j * a.b + i;
    const int nb = j < kB ? j : kB;  // band blocks this phase (the first is t = j-1)
    const bool has_far = j >= kB + 1;
    if (tracer && gi == 0) a.trace[4 * j] = globaltimer_ns();
    if (!row_loaded) load_row(j, i, rbits, yj, fv0, fv1);
    if (!cur_loaded) {
      if (kInFlight && j > 0 && !rows_stored(j, i)) {  // block 0 reads no row of G
        int ok0 = 1;
        if (lane == 0) ok0 = wait_rows_of_G(a, p, where_code(5, j)) ? 1 : 0;
        ok0 = __shfl_sync(0xffffffffu, ok0, 0);
        __syncwarp();
        if (!ok0) return;
      }
      load_band(gv, j, i);
    }
    // the next item: its row values, and its band if its rows of G are already stored
    int j2 = j, gi2 = gi + 1;
    if (gi2 == ng) {
      gi2 = 0;
      ++j2;
    }
    bool next_loaded = false;
    uint32_t rbits_n = 0;
    float yj_n = 0.0f, fv0_n = 0.0f, fv1_n = 0.0f;
    if (j2 < a.s) {
      const int i2 = (c + gi2 * a.C) * kChainRows + warp;
      if (kRowAhead) load_row(j2, i2, rbits_n, yj_n, fv0_n, fv1_n);
      if (j2 > 0 && rows_stored(j2, i2)) {
        load_band(gn, j2, i2);
        next_loaded = true;
      }
    }
    if (tracer && gi == 0) a.trace[4 * j + 1] = globaltimer_ns();
    // alpha_{j-1} (slot row 0; polled once per phase) and far_j (mode 3: the row's
    // j-B partial sums, two per lane): load them until none is pending
    bool pend = false;
    const float* aprev = a.alpha + (int64_t)(j - 1) * a.b + lane * 4;
    const bool poll_alpha = a.vec4 && j > 0 && j != jprev;
    if (poll_alpha) {
      // slot row tb holds alpha_{j-1-tb}: shift the rows of the previous phase down
#pragma unroll
      for (int tb = kB - 1; tb >= 1; --tb)
#pragma unroll
        for (int k = 0; k < kKB; ++k) av[tb][k] = av[tb - 1][k];
#pragma unroll
      for (int k = 0; k < kKB; ++k) {
        if (lane * 4 + 128 * k < a.b) {
          av[0][k] = ld_volatile_f4(aprev + 128 * k);
          pend |= pending4(av[0][k]);
        }
      }
    }
    // far_j as loaded with the row values (lane 0; mode 3: partials t = lane and
    // t = lane + 32), reloaded below while pending
    float farv = kFarParts ? 0.0f : fv0;
    float fp0 = fv0, fp1 = fv1;
    const int nfar = (j - kB) * a.npb;  // partials of the row (has_far), at most 64
    const float* fsrc = kFarParts ? a.fpart + p * a.fs : nullptr;
    if (kFarParts) {
      if (has_far && lane < nfar) pend |= pending1(fp0);
      if (has_far && lane + 32 < nfar) pend |= pending1(fp1);
    } else if (has_far && lane == 0) {
      pend |= pending1(farv);
    }
    if (lane == 0) pend |= pending1(__uint_as_float(rbits));
    bool ok = true;
    if (__any_sync(0xffffffffu, pend)) {
      const uint64_t t_start = globaltimer_ns();
      while (true) {
        __nanosleep(32);  // eases the load on the few L2 lines every chain warp polls
        pend = false;
        if (poll_alpha) {
#pragma unroll
          for (int k = 0; k < kKB; ++k) {
            if (lane * 4 + 128 * k < a.b && pending4(av[0][k])) {
              av[0][k] = ld_volatile_f4(aprev + 128 * k);
              pend |= pending4(av[0][k]);
            }
          }
        }
        if (lane == 0 && pending1(__uint_as_float(rbits))) {
          rbits = __float_as_uint(ld_volatile_f32(a.r + p));
          pend |= pending1(__uint_as_float(rbits));
        }
        if (kFarParts) {
          if (has_far && lane < nfar && pending1(fp0)) {
            fp0 = ld_volatile_f32(fsrc + lane);
            pend |= pending1(fp0);
          }
          if (has_far && lane + 32 < nfar && pending1(fp1)) {
            fp1 = ld_volatile_f32(fsrc + lane + 32);
            pend |= pending1(fp1);
          }
        } else if (has_far && lane == 0 && pending1(farv)) {
          farv = ld_volatile_f32(a.far + p);
          pend |= pending1(farv);
        }
        if (!__any_sync(0xffffffffu, pend)) break;
        ok = keep_waiting(a, t_start, where_code(2, j));
        if (!__all_sync(0xffffffffu, ok)) return;
      }
    }
    if (tracer && gi == 0) a.trace[4 * j + 2] = globaltimer_ns();
    float acc = 0.0f;
    if (a.vec4) {
#pragma unroll
      for (int tb = 0; tb < kB; ++tb)
#pragma unroll
        for (int k = 0; k < kKB; ++k)
          if (tb < nb) acc = dot4(gv[tb][k], av[tb][k], acc);
      // columns beyond the register slots (b > 128 * kKB): kX float4 of G and of alpha
      // per lane requested together, then summed in column order
      const float* grow0 = a.G + (int64_t)i * a.b;
      for (int tb = 0; tb < nb && ok; ++tb) {
        const int t = j - 1 - tb;
        const float* gsrc = grow0 + g_block_offset(j, t, a.b, a.diag, a.gB);
        const float* asrc = a.alpha + (int64_t)t * a.b;
        constexpr int kX = 2;
        for (int k0 = kKB; k0 < nk && ok; k0 += kX) {
          float4 gx[kX], vx[kX];
#pragma unroll
          for (int u = 0; u < kX; ++u) {
            const int col = lane * 4 + 128 * (k0 + u);
            const bool in = k0 + u < nk && col < a.b;
            gx[u] = in ? ldG4<kInFlight>(gsrc + col) : make_float4(0.f, 0.f, 0.f, 0.f);
            vx[u] = in ? ld_volatile_f4(asrc + col) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < kX; ++u) {
            if (pending4(vx[u])) {
              const float* src = asrc + lane * 4 + 128 * (k0 + u);
              const uint64_t t_start = globaltimer_ns();
              while (pending4(vx[u]) && (ok = keep_waiting(a, t_start, where_code(2, j))))
                vx[u] = ld_volatile_f4(src);
            }
            acc = dot4(gx[u], vx[u], acc);
          }
        }
      }
    } else {
      const float* grow0 = a.G + (int64_t)i * a.b;
      const int t0 = j - nb;
      for (int t = t0; t < j && ok; ++t) {
        const float* al = a.alpha + (int64_t)t * a.b;
        const float* grow = grow0 + g_block_offset(j, t, a.b, a.diag, a.gB);
        for (int col = lane; col < a.b; col += 32) {
          float v;
          if (!(ok = wait_value(al + col, v, a, where_code(2, j)))) break;
          acc = fmaf(ldG1<kInFlight>(grow + col), v, acc);
        }
      }
    }
    if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (kFarParts) {  // far_j: the row's partials, lane sums then a fixed tree
      float fs = fp0 + fp1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) fs += __shfl_xor_sync(0xffffffffu, fs, off);
      farv = fs;
    }
    if (lane == 0 && !(a.stall_test && j == 0)) {
      const float z = __uint_as_float(rbits) + farv + acc;
      __stcg(a.alpha + p, a.coef * loss_deriv(a.loss, z, yj));
    }
    if (tracer && gi == ng - 1) a.trace[4 * j + 3] = globaltimer_ns();
    // advance
#pragma unroll
    for (int tb = 0; tb < kB; ++tb)
#pragma unroll
      for (int k = 0; k < kKB; ++k) gv[tb][k] = gn[tb][k];
    cur_loaded = next_loaded;
    row_loaded = kRowAhead;
    rbits = rbits_n;
    yj = yj_n;
    fv0 = fv0_n;
    fv1 = fv1_n;
    jprev = j;
    j = j2;
    gi = gi2;
  }
}

// --------------------------------------------------------------- update units
// Step a8, fused: unit (j, cc, rq) sums alpha_i * Y_i over row part rq (of R) of block j
// for the 64 columns cc*64 .. cc*64+63 into partial row j*R + rq.  With R > 1 the last of
// the R units of (j, cc) sums the R partial rows (four interleaved sums) into row j*R,
// the block's sum (R = 1: the unit's own row is).  The last of the s block sums of a
// column chunk (a per-chunk counter) adds them to w: block rows q, q+8, q+16, ... for
// each q < 8, then the eight sums in q order.  No unit waits on another (modes 0-2: the
// bulk groups also stream G), and w receives one addition per iteration whatever order
// the units finish in.
// Threads: 32 row-lanes x 8 column vectors.  The unit issues its first rows of Y, then
// waits as a whole for its rows of alpha_j: lane 0 of warp 0 polls one value with a
// back-off (of phase j+1; the part's last row for the last block and, in modes 3-4, the
// last two), then warp 0 loads
// the part's values until none is pending.  Fixed
// order: rows ascending per row-lane, then row-lanes ascending in shared memory.  Y was
// written by an earlier launch.  Returns, in thread 0 of the group, whether every update
// unit had been dealt once alpha_j was final (the queue's counter, read then; it only
// grows), so the group need not ask the queue again; false in the other threads.
template <int kMode, bool kFromX>
__device__ bool update_unit(const RecArgs& a, int u, int rt) {
  __shared__ float red[32][64];
  // one flag per stage, each written by thread 0 and read by the group after a barrier;
  // the next write of a flag comes after at least two more barriers of the group
  __shared__ int s_ready, s_last;
  const int nchunk = (int)((a.ldY / 8 + 7) / 8);
  const int per_j = nchunk * a.upd_R;
  const int j = u / per_j, cc = (u - j * per_j) / a.upd_R;
  const int rq = u - j * per_j - cc * a.upd_R;
  const int r0 = (int)((int64_t)rq * a.b / a.upd_R), r1 = (int)((int64_t)(rq + 1) * a.b / a.upd_R);
  const int tv = rt & 7, tr = rt >> 3;  // vector-lane, row-lane
  const int64_t vec = (int64_t)cc * 8 + tv;
  const bool vin = vec < a.ldY / 8;
  const float* al_j = a.alpha + (int64_t)j * a.b;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  uint4 q[kUpdRows];
  // (reading X: vectors from column n on are skipped, and the columns past n of the last
  // vector only reach partial-row columns that are never added to w)
  const bool xin = kFromX ? vec * 8 < a.n : vin;
  // warp 0 polls the part's alpha values (all of them in modes 3-4 and for the last
  // block) and then keeps them in red, which holds up to 2048
  const bool polled = kMode >= 3 || j + 1 == a.s;
  const bool al_sm = polled && r1 - r0 <= 32 * 64;
  float* red_f = &red[0][0];
  // w as the launch started (w_k): this column's value for the chunk's final sum, read
  // now (w changes only with that sum)
  const int64_t c = (int64_t)cc * 64 + (rt & 63);
  const float w_k = (rt < 64 && c < a.n) ? a.w[c] : 0.0f;
  uint32_t dealt = 0;
  auto drained = [&]() { return rt == 0 && dealt >= (uint32_t)a.upd_units; };
  auto load_rows = [&](int i0) {
#pragma unroll
    for (int k = 0; k < kUpdRows; ++k) {
      const int i = i0 + 32 * k;
      const int64_t row = (int64_t)j * a.b + i;
      const uint16_t* src =
          kFromX ? a.X + (int64_t)draw_row(a.xseed, a.xctr + (uint64_t)row, a.xm, a.xperm) * a.ldx
                 : a.Y + row * a.ldY;
      q[k] = (i < r1 && xin) ? __ldg(reinterpret_cast<const uint4*>(src + vec * 8))
                             : make_uint4(0, 0, 0, 0);
    }
  };
  load_rows(r0 + tr);
  if (rt < 32) {  // warp 0 waits for the part's alpha
    bool ok = true;
    const uint64_t t_start = globaltimer_ns();
    if (rt == 0) {
      // one value polled with a back-off: of phase j+1 (final there implies alpha_j
      // complete; the update of block j is off the critical path), or its own last row
      // for the last block and, in modes 3-4 (which poll the part's own values next),
      // for the last two: block s-2's sum is then formed before the last block's alpha
      const int probe_ahead = kMode >= 3 ? j + 2 < a.s : j + 1 < a.s;
      const float* pv = probe_ahead
                            ? a.alpha + (int64_t)(j + 1) * a.b + (int)((blockIdx.x * 37u) % (unsigned)a.b)
                            : al_j + r1 - 1;
      while (pending1(ld_volatile_f32(pv)) && ok) {
        __nanosleep(200);
        ok = keep_waiting(a, t_start, where_code(4, j));
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    // the part's own values, four per lane in flight (modes 0-2 rely on the probe of
    // phase j+1 for every block but the last, as the far units do), kept in shared
    // memory for the sums (al_sm)
    if (polled) {
      for (int i = r0 + rt; i < r1 && ok; i += 32 * 4) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = i + 32 * k < r1 ? ld_volatile_f32(al_j + i + 32 * k) : 0.0f;
        bool pend = pending1(v[0]) || pending1(v[1]) || pending1(v[2]) || pending1(v[3]);
        while (pend && ok) {
          __nanosleep(64);
          pend = false;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (pending1(v[k])) {
              v[k] = ld_volatile_f32(al_j + i + 32 * k);
              pend |= pending1(v[k]);
            }
          if (pend) ok = keep_waiting(a, t_start, where_code(4, j));
        }
        if (al_sm) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (i + 32 * k < r1) red_f[i + 32 * k - r0] = v[k];
        }
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (rt == 0) {
      s_ready = ok ? 1 : 0;
      dealt = ld_volatile_u32(&a.q->upd_next);  // used when the unit is done
    }
  }
  group_sync<kMode != 0>();
  const bool ready = s_ready != 0;  // rewritten only after the group syncs below
  if (ready) {
    for (int i0 = r0 + tr; i0 < r1; i0 += 32 * kUpdRows) {
      if (i0 != r0 + tr) load_rows(i0);
#pragma unroll
      for (int k = 0; k < kUpdRows; ++k) {
        const int i = i0 + 32 * k;
        const float al = i < r1 ? (al_sm ? red_f[i - r0] : __ldcg(al_j + i)) : 0.0f;
        const uint32_t pw[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          acc[2 * h] = fmaf(al, bf16_bits_to_float(pw[h] & 0xFFFFu), acc[2 * h]);
          acc[2 * h + 1] = fmaf(al, bf16_bits_to_float(pw[h] >> 16), acc[2 * h + 1]);
        }
      }
    }
  }
  group_sync<kMode != 0>();  // (red held alpha until here)
#pragma unroll
  for (int e = 0; e < 8; ++e) red[tr][tv * 8 + e] = acc[e];
  group_sync<kMode != 0>();
  const int R = a.upd_R;                          // 1 in modes 0-2
  float* brow = a.part + (int64_t)j * R * a.ldY;  // block j's partial rows
  if (rt < 64 && ready) {
    float sum = 0.0f;
    for (int r = 0; r < 32; ++r) sum += red[r][rt];
    if (rt == 0) stamp_last(a.trace, 2);
    if (c < a.ldY) brow[(int64_t)rq * a.ldY + c] = sum;
    __threadfence();  // the partial row is visible before this unit is counted
  }
  if (R > 1) {
    // the last of the R units of (j, cc): the block's sum (parts rq, rq+4, ... in four
    // sums, then combined) into the block's first partial row
    group_sync<kMode != 0>();
    if (rt == 0)
      s_last = ready && atomicAdd(a.upd_blocks + (int64_t)j * nchunk + cc, 1u) ==
                            (unsigned)(R - 1)
                   ? 1
                   : 0;
    group_sync<kMode != 0>();
    if (!s_last) return drained();  // group-uniform
    if (rt < 64 && c < a.ldY) {
      __threadfence();
      float p4[4] = {0.f, 0.f, 0.f, 0.f};
      for (int r0 = 0; r0 < R; r0 += 16) {  // 16 loads in flight, added in r order
        float v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          v[k] = r0 + k < R ? __ldcg(brow + (int64_t)(r0 + k) * a.ldY + c) : 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) p4[k & 3] += v[k];
      }
      brow[c] = (p4[0] + p4[1]) + (p4[2] + p4[3]);
      __threadfence();
    }
  }
  // the last of the s block sums of column chunk cc adds them to w: block rows q, q+8,
  // q+16, ... for each q < 8, then the eight sums in q order
  group_sync<kMode != 0>();
  if (rt == 0)
    s_last = ready && atomicAdd(a.upd_chunks + cc, 1u) == (unsigned)(a.s - 1) ? 1 : 0;
  group_sync<kMode != 0>();
  if (s_last && rt < 64 && c < a.n) {
    __threadfence();
    float acc_q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int p0 = 0; p0 < a.s; p0 += 16) {  // 16 loads in flight, added in row order
      float v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        v[k] = p0 + k < a.s ? __ldcg(a.part + (int64_t)(p0 + k) * R * a.ldY + c) : 0.0f;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc_q[k & 7] += v[k];
    }
    float sum = 0.0f;
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) sum += acc_q[q8];
    const float v = w_k + sum;
    a.w[c] = v;
    if (!isfinite(v)) atomicOr(&a.ctrl->status, ST_NONFINITE);
  }
  return drained();
}

// -------------------------------------------------------------- margin units
// Step a4 in the recurrence's launch (with the far-forming Gram): unit u forms the
// margins of rows u*mrows .. of Y with w (the launch's w_k: the update writes w only
// after the last phase).  mG lanes per row (a power of two covering the row's 16-byte vectors
// up to 32), 32/mG rows per warp and pass; lane g sums the vectors g, g+mG, ... in FP32,
// eight elements each in column order, the row's lanes then add by a shuffle tree, and
// its first lane stores the margin (rounded once to BF16, or FP32 with MARGINS_FP32).
template <bool kFromX>
__device__ void margin_unit(const RecArgs& a, int u, int rt) {
  const int G = a.mG;
  const int warp = rt >> 5, lane = rt & 31;
  const int g = lane & (G - 1);
  const int rows_pass = 8 * (32 / G);
  const int64_t nvec = a.ldY / 8;
  const int64_t p_end = (int64_t)(u + 1) * a.mrows < a.S ? (int64_t)(u + 1) * a.mrows : a.S;
  for (int64_t p0 = (int64_t)u * a.mrows; p0 < p_end; p0 += rows_pass) {
    const int64_t p = p0 + warp * (32 / G) + lane / G;
    const bool live = p < p_end;
    const uint16_t* yr =
        kFromX ? a.X + (int64_t)draw_row(a.xseed, a.xctr + (uint64_t)(live ? p : 0), a.xm,
                                         a.xperm) * a.ldx
               : a.Y + (live ? p : 0) * a.ldY;
    float acc = 0.0f;
    constexpr int kBatch = 8;
    for (int64_t v0 = g; v0 < nvec; v0 += (int64_t)G * kBatch) {
      uint4 q[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t v = v0 + (int64_t)k * G;
        q[k] = (live && v < nvec && (!kFromX || v * 8 < a.n))
                   ? __ldg(reinterpret_cast<const uint4*>(yr + v * 8))
                   : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t c0 = (v0 + (int64_t)k * G) * 8;
        if (c0 >= a.n) break;
        uint32_t pw[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
        if (kFromX && c0 + 8 > a.n) {  // columns from n on: zero (X's padding is not data)
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int64_t c = c0 + 2 * h;
            if (c >= a.n) pw[h] = 0;
            else if (c + 1 >= a.n) pw[h] &= 0xFFFFu;
          }
        }
        float wv[8];
        if (a.wm_vec && c0 + 8 <= a.n) {
          const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.wm + c0));
          const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.wm + c0 + 4));
          wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
          wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) wv[e] = c0 + e < a.n ? __ldg(a.wm + c0 + e) : 0.0f;
        }
        // elements in column order; past n the row holds zeros (stored padding)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          acc = fmaf(bf16_bits_to_float(pw[h] & 0xFFFFu), wv[2 * h], acc);
          acc = fmaf(bf16_bits_to_float(pw[h] >> 16), wv[2 * h + 1], acc);
        }
      }
    }
    for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
    if (live && g == 0) __stcg(a.r_w + p, a.r_fp32 ? acc : round_bf16(acc));
  }
}

// ------------------------------------------------------------------- bulk role
// Far units (block j, 16 rows) come first, in increasing j; each warp owns two rows; a
// lane's columns are lane*4 + 128k.  The group waits as a whole: a final alpha value of
// phase q implies that phase q-1 is complete (its row needed all of alpha_{q-1}), so
// thread 0 reads single values of the next phases (spread over the values by CTA
// index, with a back-off while the next phase is not done) and the group then
// processes every block known complete, up to kT per pass with all their loads issued
// together, reading alpha with plain loads.  Each block's dot product is summed over
// columns first and then added in t order, so the result does not depend on timing.
// The first upd_groups bulk groups (`upd_group`; their share of the bulk groups is the
// update's share of the bulk role's bytes) serve the update units from their own queue,
// in block order, so the update keeps pace with the chain instead of queueing behind
// the far units; when no update units are left they turn to far units, and the other
// groups turn to update units once the far units are gone.
template <int kMode, bool kFromX = false>
__device__ void bulk_role(const RecArgs& a, int rt, bool upd_group) {
  constexpr bool kInFlight = kMode == 1 || kMode == 3;
  __shared__ int s_unit, s_lead;
  const int warp = rt >> 5, lane = rt & 31;
  const int probe_col = (int)((blockIdx.x * 37u) % (unsigned)a.b);
  bool far_left = true, upd_left = a.upd_units > 0;
  while (true) {
    if (rt == 0) {
      int u = a.bulk_units + a.upd_units;  // none left
      for (int pass = 0; pass < 2; ++pass) {
        const bool take_upd = (pass == 0) == upd_group;
        if (take_upd && upd_left) {
          const int v = (int)atomicAdd(&a.q->upd_next, 1u);
          if (v < a.upd_units) { u = a.bulk_units + v; break; }
          upd_left = false;
        } else if (!take_upd && far_left) {
          const int v = (int)atomicAdd(&a.q->next_unit, 1u);
          if (v < a.bulk_units) { u = v; break; }
          far_left = false;
        }
      }
      // (nothing dealt: the group leaves without reading the abort word)
      if (u < a.bulk_units + a.upd_units && ld_volatile_u32(&a.ctrl->abort))
        u = a.bulk_units + a.upd_units;
      s_unit = u;
    }
    group_sync<kMode != 0>();
    const int unit = s_unit;
    group_sync<kMode != 0>();
    if (unit >= a.bulk_units) {
      if (unit < a.bulk_units + a.upd_units) {
        if (update_unit<kMode, kFromX>(a, unit - a.bulk_units, rt)) upd_left = false;
        group_sync<kMode != 0>();
        continue;
      }
      return;
    }
    if (a.margins) {  // the bulk units are margin units
      margin_unit<kFromX>(a, unit, rt);
      group_sync<kMode != 0>();
      continue;
    }
    const int j = a.B + 1 + unit / a.U;
    const int c = unit % a.U;
    const int i0 = c * kRecRows + warp * 2;
    const bool has0 = i0 < a.b, has1 = i0 + 1 < a.b;
    const int t_end = j - a.B;  // far_j covers t < j - B
    float acc0 = 0.0f, acc1 = 0.0f;
    bool ok = true;
    for (int t = 0; t < t_end;) {
      if (rt == 0) {
        bool rows_ok = true;
        if (kInFlight && t == 0) {  // the unit's rows of G are stored (first and last row)
          const int64_t r0 = (int64_t)j * a.b + c * kRecRows;
          const int last = min(c * kRecRows + kRecRows, a.b) - 1;
          rows_ok = wait_rows_of_G(a, r0, where_code(5, j)) &&
                    wait_rows_of_G(a, (int64_t)j * a.b + last, where_code(5, j));
        }
        // leading run of complete phases t, t+1, ... (at most kT and t_end - t)
        const int lim = min(kT, t_end - t);
        int lead = 0;
        while (rows_ok && lead < lim &&
               !pending1(ld_volatile_f32(a.alpha + (int64_t)(t + lead + 1) * a.b + probe_col)))
          ++lead;
        if (rows_ok && lead == 0) {  // wait for phase t, polling one value of phase t+1
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
      group_sync<kMode != 0>();
      const int nt = s_lead;
      group_sync<kMode != 0>();
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
                x0[u] = ldG4<kInFlight>(gb);
                x1[u] = has1 ? ldG4<kInFlight>(gb + a.b) : make_float4(0.f, 0.f, 0.f, 0.f);
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
                d0[u] = fmaf(ldG1<kInFlight>(gb + col), v, d0[u]);
                if (has1) d1[u] = fmaf(ldG1<kInFlight>(gb + a.b + col), v, d1[u]);
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
        if (warp == 0) stamp_last(a.trace, 1);
      }
    }
    group_sync<kMode != 0>();  // every warp of the unit is done before the group claims the next
  }
}

}  // namespace

}  // namespace casgd
