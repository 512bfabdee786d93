// Step a3 on the 5th-generation tensor cores of sm_103a: G_{j,t} = Y_j Y_t^T with BF16
// operands and FP32 accumulation in tensor memory (TMEM).
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): matrix hardware with low-precision formats accelerates the Gram
// GEMM, formed from low-precision inputs with high-precision accumulation.  Only the
// blocks the inner recurrence reads (t < j), plus the diagonal on request, are formed.
//
// Design (persistent, one CTA per SM, 6 warps):
//   warp 0      TMA producer: 128x64 (A) and 256x64 (B) BF16 tiles of Y, 128-byte
//               swizzled, into a 4-stage shared-memory ring (48 KB per stage);
//   warp 1      allocates 512 TMEM columns (two 128x256 FP32 accumulators) and one
//               elected lane issues tcgen05.mma (M=128, N=256, K=16) per 16 columns of
//               K, committing each stage back to the producer and each finished tile
//               to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one row per thread), masked
//               stores of the rows/columns that belong to needed blocks into the packed
//               block-lower G.  Two accumulators let the epilogue of one tile overlap
//               the MMAs of the next.
// Variants: the paired-SM kernel below (default) and this single-CTA kernel.  Every
// TMA copy lands in the shared memory of the CTA that issues it (no cluster multicast),
// so the same code runs unchanged in processes that each drive their own GPU.
// Both operands are K-major slices of the same Y (rows are samples, K the features);
// out-of-range rows and columns of K are zero-filled by TMA.  Tiles of the S x S
// product are visited row-tile by row-tile, skipping tiles wholly above the needed
// blocks.  Every wait is bounded: on timeout the kernel records ST_TIMEOUT, stops
// issuing work, waits (bounded) for its own copies and MMAs in flight, frees TMEM and
// returns.
#include <cuda.h>

#include <cstring>

#include "casgd_internal.cuh"
#include "ptx_async.cuh"
#include "recur_roles.cuh"

namespace casgd {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kStageOut = 2 * 32 * 32 * 4;  // per epilogue warp: two 32x32 FP32 chunks (8 KB)
constexpr int kOutBytes = 4 * kStageOut;     // four epilogue warps (32 KB)
constexpr size_t kSmemBytes =
    (size_t)kStages * kStageBytes + kOutBytes + 1024 /*barriers*/ + 1024 /*align*/;

struct TcArgs {
  float* G;
  Ctrl* ctrl;  // status and abort word
  Ctrl* q;     // this iteration's counters (band_done, ahead_next)
  int64_t S;
  int n, b, nkb;
  int TR, TC, ntiles;  // ntiles: work items (tiles; units of nb tiles when fpart is set)
  bool diag;
  bool g_bf16;     // entries rounded to BF16 before they are stored or used
  bool tma_store;  // b % 32 == 0: 32x32 chunks go out through a TMA tensor store
  int gB;          // layout of G: 0 packed block-lower, B > 0 band layout (g_block_offset)
  uint64_t timeout_ns;
  uint32_t* slab;  // recurrence in the same launch: per-32-row tile counters (else null)
  // Far-forming mode (fpart set; b a multiple of 256): only the band blocks (and the
  // diagonal on request) are stored; each far tile G_{j,t} (t < j-B) is multiplied by
  // alpha_t once alpha_t is final, and each row's sum over column group c of block t
  // (uq tiles) goes to fpart[row * fs + t * npb + c].
  float* fpart;
  const float* alpha;
  int s, B, nb;      // steps, band width, 256-wide column tiles per block
  int npb, uq, fs;   // column groups per block, tiles per group, fpart row stride
  bool stored_last;  // the stored units are the next iteration's band (see FarCursor)
  int n_stored;      // stored units in this launch
  int far_head;      // stored_last: far units before the stored ones
  int store_tail;    // stored_last: stored units moved behind every far unit
  // Rows read straight from X (kernels with kGather): row p of the Gram's own rows is
  // row draw_row(seed, ctr_g + p) of X, row p of the far tiles' rows (this iteration's)
  // draw_row(seed, ctr_f + p) -- the sampler is a pure function of its counter, so the
  // producer draws the indices itself and Y never exists
  uint64_t seed, ctr_g, ctr_f;
  uint32_t m;
  int perm_d;
  // Rows gathered ahead once this CTA's Gram work is done (gather_ahead; far-forming
  // launch with the next band only)
  bool ahead_on;
  int64_t ahead_ldY;
  AheadRows ahead;
  // The next iteration's state, reset during this launch (reset_next_set)
  bool nx_on;
  NextSet nx;
  // Weighted deal of the work items to the CTA pairs: the first pc pairs (those whose
  // CTAs also run the recurrence's chain) take wa items for every wb the other pairs
  // take (wa <= wb; wa == wb: plain round robin)
  int pc, wa, wb;
};

// The kq-th work item of pair cid of ncl, in increasing order: items are dealt in rounds
// of pc*wa + (ncl-pc)*wb; sub-round s < wa of a round gives one item to every pair (in
// pair order), sub-rounds wa..wb-1 one to every pair from pc on.
__device__ __forceinline__ int unit_of(const TcArgs& a, int cid, int ncl, int kq) {
  if (a.wa == a.wb) return cid + kq * ncl;
  const bool chain = cid < a.pc;
  const int W = chain ? a.wa : a.wb;
  const int r = kq / W, sub = kq - r * W;
  const int R = a.pc * a.wa + (ncl - a.pc) * a.wb;
  const int off = sub < a.wa ? sub * ncl : a.wa * ncl + (sub - a.wa) * (ncl - a.pc);
  const int pos = sub < a.wa ? cid : cid - a.pc;
  return r * R + off + pos;
}

struct SharedCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile uint32_t abort;
};

// Bounded wait: false (and the CTA's abort word set) if the phase does not complete in
// time or another role of this CTA already gave up.
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, SharedCtl* sc, const TcArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sc->abort) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      sc->abort = 1;
      atomicOr(&a.ctrl->status, ST_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, rows of 128 bytes, 128-byte swizzle,
// 8-row groups 1024 bytes apart (the layout a 64-column BF16 TMA box with 128-byte
// swizzle produces).  Bits: start>>4 [0,14), LBO>>4 [16,30), SBO>>4 [32,46), fixed
// 0b001 [46,49), swizzle mode [61,64) = 2 (128-byte).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor, kind::f16: D FP32 (bits 4-5 = 1), A and B BF16 (bits 7-9 and
// 10-12 = 1), both K-major (bits 15, 16 = 0), N>>3 at bits 17-22, M>>4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.ld of 32 columns without the wait; the registers are valid only after
// tmem_wait_ld on the same array (which takes them as operands, so no use of them can
// be scheduled before the wait).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]),
                 "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]),
                 "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// Number of needed column tiles in row tile `ra` (columns [0, count*BN) hold every
// entry of a needed block in those rows).
__device__ __forceinline__ int cols_needed(const TcArgs& a, int ra) {
  int64_t last = (int64_t)ra * BM + BM - 1;
  if (last > a.S - 1) last = a.S - 1;
  const int64_t jmax = last / a.b;
  const int64_t lim = (int64_t)a.b * (a.diag ? jmax + 1 : jmax);  // columns < lim needed
  int64_t c = (lim + BN - 1) / BN;
  return (int)(c < a.TC ? c : a.TC);
}

// Column tiles of row group g (row tiles kCl*g .. kCl*g+kCl-1; kCl = 1 for the
// single-CTA kernel, 2 for CTA pairs): those of its last row tile, which needs the
// most (the count grows with the row).
template <int kCl>
__device__ __forceinline__ int group_cols(const TcArgs& a, int g) {
  if (kCl == 2) return pair_group_tiles(a.S, a.b, a.diag, g);  // the count readers expect
  int last = kCl * g + kCl - 1;
  if (last > a.TR - 1) last = a.TR - 1;
  return cols_needed(a, last);
}

// Walks the linear tile index forward (tiles are visited in increasing order).
template <int kCl>
struct TileCursor {
  int g = 0;
  int base = 0;   // linear index of the first tile of row group g
  int cnt = -1;   // tiles in row group g
  __device__ void seek(const TcArgs& a, int tile, int& rg, int& cc) {
    if (cnt < 0) cnt = group_cols<kCl>(a, 0);
    while (tile >= base + cnt) {
      base += cnt;
      ++g;
      cnt = group_cols<kCl>(a, g);
    }
    rg = g;
    cc = tile - base;
  }
};

// Work order of the far-forming mode: units of uq column tiles (one 256-row group g
// against column group c of block t; npb groups of uq tiles per block).  Far units come
// by the phase j that needs them, t ascending within a phase (alpha_t is final earliest
// for small t); stored units (the band blocks t = j-1 down to j-B, then the diagonal on
// request) by phase.  Within a block t: column groups outer, row groups of block j inner.
// Same iteration: every stored unit first (they wait on nothing and the recurrence
// starts on them).  Band of the next iteration (stored_last): the first far_head far
// units (one round over the pairs), then the stored units but the last store_tail, which
// fill the MMAs while the first far tiles wait for alpha, then the other far units, then
// those store_tail stored units (nothing in this launch waits for them, so they overlap
// the recurrence's last phases).
struct UnitWalk {  // forward walk over the far units (far) or the stored units
  int j = 0, base = 0, cnt = -1;
  __device__ int count(const TcArgs& a, bool far) const {
    const int nband = j < a.B ? j : a.B;
    return a.nb * a.npb * (far ? j - nband : nband + (a.diag ? 1 : 0));
  }
  __device__ void seek(const TcArgs& a, bool far, int u, int& g, int& t, int& c) {
    if (cnt < 0) cnt = count(a, far);
    while (u >= base + cnt) {
      base += cnt;
      ++j;
      cnt = count(a, far);
    }
    const int per_t = a.nb * a.npb;
    const int v = u - base;
    const int tb = v / per_t;
    const int r = v - tb * per_t;
    c = r / a.nb;
    g = j * a.nb + (r - c * a.nb);
    const int nband = j < a.B ? j : a.B;
    t = far ? tb : (tb < nband ? j - 1 - tb : j);
  }
};

struct FarCursor {
  UnitWalk far_w, st_w;
  __device__ void seek(const TcArgs& a, int u, int& g, int& t, int& c, bool& far) {
    int lf;  // index among the far units, or -1
    int ls = -1;
    if (!a.stored_last) {
      lf = u < a.n_stored ? -1 : u - a.n_stored;
      if (lf < 0) ls = u;
    } else if (u < a.far_head) {
      lf = u;
    } else if (u < a.far_head + a.n_stored - a.store_tail) {
      lf = -1;
      ls = u - a.far_head;
    } else if (u < a.ntiles - a.store_tail) {
      lf = u - (a.n_stored - a.store_tail);
    } else {
      lf = -1;
      ls = u - (a.ntiles - a.n_stored);
    }
    far = lf >= 0;
    if (far)
      far_w.seek(a, true, lf, g, t, c);
    else
      st_w.seek(a, false, ls, g, t, c);
  }
};

// Work items of the paired kernel: single 256x256 tiles in row-group order, or (kFar)
// the units above.  seek gives the row group, the first column tile, the number of
// consecutive column tiles, the block t, the unit's partial index within the row
// (t * npb + c) and whether the unit is far.
template <bool kFar>
struct WorkCursor {
  TileCursor<2> tiles;
  FarCursor units;
  __device__ void seek(const TcArgs& a, int u, int& rg, int& ca0, int& nq, int& t, int& pidx,
                       bool& far) {
    if (kFar) {
      int c;
      units.seek(a, u, rg, t, c, far);
      ca0 = t * a.nb + c * a.uq;
      nq = a.uq;
      pidx = t * a.npb + c;
    } else {
      tiles.seek(a, u, rg, ca0);
      nq = 1;
      t = pidx = 0;
      far = false;
    }
  }
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read1() {  // at most one group still reading smem
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {  // no group still reading smem
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {  // every issued store has completed
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Epilogue of one tile for one warp: TMEM lanes 32*quarter.. hold rows ra*BM + 32*quarter
// + lane of the tile; the 256 accumulator columns of buffer `acc` are read 32 at a time
// and the entries that belong to needed blocks are stored into G (either layout) by
// each lane, one row each.  Without a.tma_store only; store_tile_tma otherwise.
__device__ __forceinline__ void store_tile_rows(const TcArgs& a, uint32_t tmem, int acc,
                                                int quarter, int lane, int ra, int ca,
                                                const CUtensorMap* tmG, uint8_t* stage,
                                                int& sbuf) {
  const bool vec_ok = (a.b % 4) == 0;
  const int64_t p = (int64_t)ra * BM + quarter * 32 + lane;
  const bool prow = p < a.S;
  const int64_t jb = prow ? p / a.b : 0;
  const int64_t ib = p - jb * a.b;
  const int64_t p0 = (int64_t)ra * BM + quarter * 32;  // the warp's first row
  for (int ch = 0; ch < BN / 32; ++ch) {
    uint32_t v[32];
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + ch * 32), v);
    if (a.g_bf16) {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(round_bf16(__uint_as_float(v[e])));
    }
    const int64_t q0 = (int64_t)ca * BN + ch * 32;
    if (!prow || q0 >= a.S) continue;
    const int64_t t0b = q0 / a.b;
    const int64_t q1 = q0 + 31;
    const int64_t t1b = q1 / a.b;
    const bool whole = (q1 < a.S) && (t0b == t1b) && (t0b < jb || (a.diag && t0b == jb));
    if (whole && vec_ok && ((q0 - t0b * a.b) % 4) == 0) {
      float* dst = a.G + g_block_offset(jb, t0b, a.b, a.diag, a.gB) + ib * a.b + (q0 - t0b * a.b);
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(dst + e) =
            make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                        __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int64_t q = q0 + e;
        if (q >= a.S) break;
        const int64_t tb = q / a.b;
        if (tb < jb || (a.diag && tb == jb))
          a.G[g_block_offset(jb, tb, a.b, a.diag, a.gB) + ib * a.b + (q - tb * a.b)] =
              __uint_as_float(v[e]);
      }
    }
  }
}

// One 32x32 chunk of store_tile_tma: columns q0.. of the warp's rows p0.. (block row j0),
// stored if the chunk lies in a needed block.  The warp writes it into one of its two
// 128-byte-swizzled staging buffers and lane 0 stores it with a TMA tensor store (whole
// 128-byte lines) through a 2D tensor map that views G as (blocks*b) rows of b columns.
__device__ __forceinline__ void store_chunk_tma(const TcArgs& a, const uint32_t (&v)[32],
                                                int lane, int64_t p0, int64_t j0, int64_t q0,
                                                const CUtensorMap* tmG, uint8_t* stage,
                                                int& sbuf) {
  if (q0 >= a.S) return;  // warp-uniform, as below
  const int64_t t0b = q0 / a.b;
  if (!(t0b < j0 || (a.diag && t0b == j0))) return;
  uint8_t* buf = stage + sbuf * (32 * 32 * 4);
  if (lane == 0) bulk_wait_read1();  // the store issued two chunks ago has read buf
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // row `lane`, 16-byte chunk c at swizzled slot c ^ (row % 8)
    uint32_t x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      x[e] = a.g_bf16 ? __float_as_uint(round_bf16(__uint_as_float(v[4 * c + e]))) : v[4 * c + e];
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) * 16)) =
        make_uint4(x[0], x[1], x[2], x[3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    const int64_t grow = (g_block_offset(j0, t0b, a.b, a.diag, a.gB) / a.b) + (p0 - j0 * a.b);
    tma_store_2d(tmG, smem_u32(buf), (int32_t)(q0 - t0b * a.b), (int32_t)grow);
    bulk_commit();
  }
  sbuf ^= 1;
}

// The epilogue of store_tile_rows with a.tma_store (b a multiple of 32, so every 32x32
// chunk lies inside one block of G), 32 columns of TMEM at a time.  (Keeping the next
// chunk's TMEM load in flight while one is stored measured no faster on n = 2000 and
// 10% slower per outer iteration on n = 18, where the launch stores mostly band tiles.)
__device__ __forceinline__ void store_tile_tma(const TcArgs& a, uint32_t tmem, int acc,
                                               int quarter, int lane, int ra, int ca,
                                               const CUtensorMap* tmG, uint8_t* stage,
                                               int& sbuf) {
  const int64_t p0 = (int64_t)ra * BM + quarter * 32;  // the warp's first row
  if (p0 >= a.S) return;                                // warp-uniform
  const int64_t j0 = p0 / a.b;
  const int64_t q00 = (int64_t)ca * BN;
  const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
  for (int ch = 0; ch < BN / 32; ++ch) {
    uint32_t v[32];
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
    tmem_ld32(base + (uint32_t)ch * 32, v);
    store_chunk_tma(a, v, lane, p0, j0, q00 + ch * 32, tmG, stage, sbuf);
  }
}

// Single-CTA variant: one CTA per 128x256 tile, A and both halves of B loaded by the
// CTA itself (48 KB per stage).
__global__ void __launch_bounds__(kThreads, 1)
    gram_tc_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmG,
                   TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* out_stage = smem + (size_t)kStages * kStageBytes;  // 1024-aligned
  SharedCtl* sc = reinterpret_cast<SharedCtl*>(out_stage + kOutBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = blockIdx.x, ncl = gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sc->full[i], 1);
      mbar_init(&sc->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc->tfull[i], 1);
      mbar_init(&sc->tempty[i], 4);
    }
    mbar_init(&sc->drain, 1);
    sc->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sc->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sc->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      TileCursor<1> cur;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // bit st: a load into stage st was issued; its parity below
      uint32_t last_par = 0;
      for (int tile = cid; tile < a.ntiles && !sc->abort; tile += ncl) {
        int rg, ca;
        cur.seek(a, tile, rg, ca);
        const int ra = rg;
        for (int kb = 0; kb < a.nkb; ++kb) {
          if (!mbar_wait(&sc->empty[stage], phase ^ 1u, sc, a)) break;
          uint8_t* sa = smem + (size_t)stage * kStageBytes;
          uint8_t* sb = sa + kABytes;
          // the tile's A and both halves of B: 48 KB land per stage
          mbar_expect_tx(&sc->full[stage], kStageBytes);
          tma_load_2d(smem_u32(sa), &tmY, &sc->full[stage], kb * BK, ra * BM);
          tma_load_2d(smem_u32(sb), &tmY, &sc->full[stage], kb * BK, ca * BN);
          tma_load_2d(smem_u32(sb + kBBytes / 2), &tmY, &sc->full[stage], kb * BK,
                      ca * BN + BN / 2);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every issued copy has landed before the CTA may exit.
      for (int st = 0; st < kStages; ++st)
        if (issued & (1u << st)) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&sc->full[st], (last_par >> st) & 1u) &&
                 globaltimer_ns() - t0 < a.timeout_ns) {
          }
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tphase[2] = {0, 0};
      int iter = 0;
      bool any = false;
      for (int tile = cid; tile < a.ntiles && !sc->abort; tile += ncl, ++iter) {
        const int acc = iter & 1;
        if (!mbar_wait(&sc->tempty[acc], tphase[acc] ^ 1u, sc, a)) break;
        tphase[acc] ^= 1u;
        tc_fence_after();
        const uint32_t tacc = tmem + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < a.nkb; ++kb) {
          if (!mbar_wait(&sc->full[stage], phase, sc, a)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          const uint64_t ad = sdesc_sw128(sa), bd = sdesc_sw128(sb);
          const int krem = a.n - kb * BK;
          const int ksteps = krem >= BK ? BK / 16 : (krem + 15) / 16;
          for (int kk = 0; kk < ksteps; ++kk)
            mma_bf16(tacc, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                     (kb > 0 || kk > 0) ? 1u : 0u);
          any = true;
          mma_commit(&sc->empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&sc->tfull[acc]);
      }
      if (any) {  // drain: all MMAs of this CTA complete before TMEM is freed
        mma_commit(&sc->drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&sc->drain, 0) && globaltimer_ns() - t0 < a.timeout_ns) {
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    uint8_t* stage = out_stage + (warp - 2) * kStageOut;
    int sbuf = 0;
    TileCursor<1> cur;
    uint32_t tphase[2] = {0, 0};
    int iter = 0;
    for (int tile = cid; tile < a.ntiles; tile += ncl, ++iter) {
      int rg, ca;
      cur.seek(a, tile, rg, ca);
      const int ra = rg;
      const int acc = iter & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sc->tfull[acc], tphase[acc], sc, a) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tphase[acc] ^= 1u;
      tc_fence_after();
      if (a.tma_store)
        store_tile_tma(a, tmem, acc, quarter, lane, ra, ca, &tmG, stage, sbuf);
      else
        store_tile_rows(a, tmem, acc, quarter, lane, ra, ca, &tmG, stage, sbuf);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc->tempty[acc]);
    }
    if (lane == 0) bulk_wait_all();  // this warp's tensor stores are complete
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  if (threadIdx.x == 0 && sc->abort) atomicExch(&a.ctrl->abort, 1u);
}

// ------------------------------------------------------------ paired-SM variant
// A 2-CTA cluster computes a 256x256 tile with tcgen05.mma.cta_group::2 (M = 256): each
// CTA loads its own 128 rows of A and its own 128-row half of B, so a stage costs a CTA
// 32 KB of shared memory and 32 KB of L2 reads for 128x256x64 of MMA work.  The leader
// CTA (rank 0) issues the MMAs; its full barrier receives both CTAs' copies
// (cta_group::2 TMA signals the leader's barrier); each commit multicasts to the
// barriers of both CTAs; each CTA's TMEM holds its 128 rows of the accumulator and its
// own epilogue warps store them.  Every tcgen05 operation of this kernel, the TMEM
// allocation included, uses cta_group::2.
//
// With kRecV > 0 the same launch also runs an inner recurrence (recur_roles.cuh) on
// eight more warps per CTA (warps 6-13; kRecV: the chain's register layout, see
// chain_variant).  With kNext the Gram is the next outer iteration's (its rows were
// sampled ahead; only the margins need the current w) and the recurrence reads this
// iteration's complete G, so the two only share the SMs; otherwise both work on the
// same iteration as follows.  After the stores of a tile are complete, each epilogue warp releases
// the counter of its 32 rows, and the recurrence acquires the counters of the rows it
// reads.  Row groups are visited in increasing order, so phase j of the recurrence can
// start as soon as block row j of G is stored instead of after the whole Gram.  The
// Gram warps never wait on the recurrence, so the Gram always completes; the
// recurrence needs every CTA resident (the grid is the number of co-resident clusters).
constexpr int kHalfB = 128 * BK * 2;              // 16 KB
constexpr int kStageBytes2 = kABytes + kHalfB;    // 32 KB per CTA per stage
constexpr int kStagesPair = 6;                    // Gram alone: 6 x 32 KB + 32 KB staging
constexpr int kStagesFused = 5;                   // with the recurrence's shared memory
constexpr int kAlphaStage = 4 * BN * 4;  // far tiles: alpha of a tile, per epilogue warp
template <int kSt, bool kFar = false>
constexpr size_t pair_smem_bytes() {
  return (size_t)kSt * kStageBytes2 + kOutBytes + 1024 + (kFar ? kAlphaStage : 0) + 1024;
}
static_assert(pair_smem_bytes<kStagesPair>() <= 232448, "dynamic shared memory per CTA");
static_assert(pair_smem_bytes<kStagesFused, true>() + 9 * 1024 <= 232448, "with the recurrence");
constexpr int kFusedThreads = kThreads + kRecThreads;  // 6 Gram warps + 8 recurrence warps
// Gram items per round of a pair that also runs the chain, and of the other pairs
constexpr int kChainPairShare = 1;
constexpr int kOtherPairShare = 1;
// Share (percent) of the next iteration's band tiles computed after every far tile
constexpr int kStoreTailPct = 50;
constexpr uint32_t kIdesc2 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                             ((uint32_t)(256 >> 4) << 24);

template <int kSt>
struct SharedCtl2 {
  uint64_t full[kSt];   // leader: both CTAs' copies of a stage have landed
  uint64_t empty[kSt];  // both CTAs: the leader's MMAs have read a stage
  uint64_t tfull[2];    // both CTAs: accumulator buffer complete
  uint64_t tempty[2];   // leader: both CTAs' epilogues done with a buffer (8 warps)
  uint64_t drain;       // leader: every MMA complete
  uint64_t gfull[kSt];  // gather_ahead: a stage's row copies have landed
  uint32_t tmem_base;
  volatile uint32_t abort;
};

__device__ __forceinline__ uint32_t mapa_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// TMA into this CTA's shared memory, completion signalled on a barrier that may live in
// the peer CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// Four rows r0..r3 of a 2D tensor (columns x .. x+63 of each, the map's box being one row
// high) into consecutive 128-byte rows of this CTA's shared memory, 128-byte swizzled by
// their shared-memory address (so four copies to dst, dst+512, ... build the same tile a
// 128-row box copy would); completion counted on a barrier that may be the pair leader's.
__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t r0,
                                                 int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(r0), "r"(r1), "r"(r2),
      "r"(r3)
      : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc2), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}


// Bounded wait; a timeout also raises the workspace abort word at once, so waiters of
// the recurrence (same launch or later) stop instead of running into their own bounds.
template <int kSt>
__device__ bool mbar_wait2(uint64_t* bar, uint32_t parity, SharedCtl2<kSt>* sc, const TcArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sc->abort) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      sc->abort = 1;
      atomicOr(&a.ctrl->status, ST_TIMEOUT);
      atomicExch(&a.ctrl->abort, 1u);
      return false;
    }
  }
}

// Narrow rows (ldY <= 64 columns) gathered ahead (TcArgs::ahead) by the producer warp
// once its Gram work is issued, with plain 16-byte loads and stores: one row per lane,
// chunks of 32 rows taken four at a time from Ctrl::ahead_next.  X's rows have at least
// ldY/8 whole vectors (ld >= n, ld % 8 == 0); the columns from n on are stored as zeros.
__device__ void gather_ahead_narrow(const TcArgs& a, int lane) {
  const AheadRows& h = a.ahead;
  const int ldv = (int)(a.ahead_ldY / 8);  // 16-byte vectors per row, at most 8
  const int64_t nch = (a.S + 31) / 32;
  constexpr int kGrab = 4;
  while (true) {
    int64_t c0 = 0;
    if (lane == 0) c0 = (int64_t)atomicAdd(&a.q->ahead_next, (unsigned)kGrab);
    c0 = __shfl_sync(0xffffffffu, c0, 0);
    if (c0 >= nch) break;
    for (int k = 0; k < kGrab; ++k) {
      const int64_t p = (c0 + k) * 32 + lane;
      if (c0 + k >= nch || p >= a.S) continue;
      const int32_t x = draw_row(h.seed, h.ctr + (uint64_t)p, h.m, h.perm_d);
      const uint4* src = reinterpret_cast<const uint4*>(h.X + (int64_t)x * h.ld);
      uint4* dst = reinterpret_cast<uint4*>(h.Y + p * a.ahead_ldY);
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < ldv) v[i] = __ldg(src + i);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i >= ldv) break;
        uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // columns i*8 + 2e and i*8 + 2e + 1
          const int c = i * 8 + 2 * e;
          if (c >= a.n) w4[e] = 0u;
          else if (c + 1 >= a.n) w4[e] &= 0xFFFFu;
        }
        dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
  }
}

// Resets TcArgs::nx (see NextSet), by warp 1 of every CTA that does not lead its pair
// (idle there: the leader's warp 1 issues the MMAs).  Pair cid's warp takes rows
// cid*32 + lane, + ncl*32, ...; pair 0's also the counters.
__device__ void reset_next_set(const NextSet& x, int64_t S, int cid, int ncl, int lane) {
  const float pend = __uint_as_float(kAlphaPending);
  if (cid == 0) {
    if (lane == 0) {
      x.q->next_unit = 0;
      x.q->upd_next = 0;
      x.q->band_done = 0;
      x.q->ahead_next = 0;
    }
    uint32_t* chunks = upd_chunk_counters(x.counters);
    for (int i = lane; i < x.nchunk; i += 32) chunks[i] = 0;
    uint32_t* blocks = upd_block_counters(x.counters);
    for (int i = lane; i < x.s * x.nchunk; i += 32) blocks[i] = 0;
  }
  for (int64_t p = (int64_t)cid * 32 + lane; p < S; p += (int64_t)ncl * 32) {
    x.alpha[p] = pend;
    x.far[p] = pend;
    x.r[p] = pend;
    if (x.fpart) {
      const int nfar = ((int)(p / x.fb) - x.fB) * x.fnp;
      float* row = x.fpart + p * x.fs;
      for (int t = 0; t < nfar; ++t) row[t] = pend;
    }
    if (x.yY) {
      const int32_t row = draw_row(x.seed, x.ctr + (uint64_t)p, x.m, x.perm_d);
      x.idx[p] = row;
      x.yY[p] = __ldg(x.y + row);
    }
  }
}

// Waits for a phase ignoring the abort word, at most timeout_ns: copies already issued
// into this CTA's shared memory land before it leaves.
__device__ __forceinline__ bool mbar_wait_quiet(uint64_t* bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > ns) return false;
  return true;
}

// Rows gathered ahead (TcArgs::ahead) by the producer warp of each CTA once the MMAs
// have read every stage of the CTA's ring, `stage`/`phase` being where the producer
// stopped.  Chunks of rps rows (one stage each) are taken from Ctrl::ahead_next, so the
// CTAs whose Gram work ends early take most of them.  For a chunk, lane r draws row r
// from the sampler and copies its n*2 bytes from X into the stage (cp.async.bulk,
// completion on the stage's gfull barrier); once landed the chunk goes out as
// full-pitch bulk stores into Y (the stages' bytes from n*2 to the pitch are zeroed
// once, so Y's padding stays zero).  The rows' indices and labels are written by the
// launch's reset of the next state (reset_next_set).  Waits are bounded; after a failed
// one the warp still lets the copies it issued land before it returns.
template <int kSt>
__device__ void gather_ahead(const TcArgs& a, SharedCtl2<kSt>* sc, uint8_t* smem, int lane,
                             int stage, uint32_t phase) {
  const AheadRows& h = a.ahead;
  int ok = 1;
  if (lane == 0) {  // every stage: the MMAs' reads of its last use are complete
    for (int i = 0; i < kSt && ok; ++i) {
      ok = mbar_wait2(&sc->empty[stage], phase ^ 1u, sc, a) ? 1 : 0;
      if (++stage == kSt) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  const uint32_t rowb = (uint32_t)a.n * 2;           // data bytes per row (n % 8 == 0)
  const uint32_t pitch = (uint32_t)a.ahead_ldY * 2;  // bytes per row in Y and in a stage
  const int rps = (int)(kStageBytes2 / pitch) < 32 ? (int)(kStageBytes2 / pitch) : 32;
  const int64_t nch = (a.S + rps - 1) / rps;
  for (int st = 0; st < kSt; ++st)
    for (int r = 0; r < rps; ++r)
      for (uint32_t o = rowb + (uint32_t)lane * 16; o < pitch; o += 32 * 16)
        *reinterpret_cast<uint4*>(smem + (size_t)st * kStageBytes2 + (size_t)r * pitch + o) =
            make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncwarp();
  // A ring over the stages: kSt-1 chunks' copies in flight while the oldest chunk is
  // stored; a stage is refilled once the stores issued from it have read it (all but
  // the newest store group).  Chunks enter the ring in stage order, so the first empty
  // stage in that order ends it.
  int64_t held[kSt];  // the chunk each stage holds (-1: none)
  for (int st = 0; st < kSt; ++st) held[st] = -1;
  // chunks are reserved kGrab at a time (one atomic per kGrab chunks)
  constexpr int kGrab = 4;
  int64_t res = 0;
  int res_left = 0;
  auto grab = [&]() -> int64_t {
    if (res_left == 0) {
      int64_t c = 0;
      if (lane == 0) c = (int64_t)atomicAdd(&a.q->ahead_next, (unsigned)kGrab);
      res = __shfl_sync(0xffffffffu, c, 0);
      res_left = kGrab;
    }
    --res_left;
    return res++;
  };
  // X's rows are read once here: evict them from L2 first (measured 126.3-128.1 ->
  // 125.6 us per outer iteration on n = 2000)
  const uint64_t pol = l2_evict_first_policy();
  auto issue = [&](int st, int64_t c) {  // chunk c's copies
    const int64_t p0 = c * rps;
    const int nr = (int)(a.S - p0 < rps ? a.S - p0 : rps);
    if (lane == 0) mbar_expect_tx(&sc->gfull[st], (uint32_t)nr * rowb);
    __syncwarp();
    if (lane < nr) {
      const int32_t x = draw_row(h.seed, h.ctr + (uint64_t)(p0 + lane), h.m, h.perm_d);
      bulk_load_hint(smem + (size_t)st * kStageBytes2 + (size_t)lane * pitch,
                     h.X + (int64_t)x * h.ld, rowb, &sc->gfull[st], pol);
    }
    held[st] = c;
  };
  bool more = true;
  for (int st = 0; st < kSt - 1 && more; ++st) {
    const int64_t c = grab();
    if (c >= nch)
      more = false;
    else
      issue(st, c);
  }
  uint32_t gph = 0;  // parity of each stage's gfull barrier
  bool live = true;
  for (int i = 0;; ++i) {
    const int st = i % kSt;
    const int64_t c = held[st];
    if (c < 0) break;
    held[st] = -1;
    const uint32_t par = (gph >> st) & 1u;
    gph ^= 1u << st;
    if (live) {
      int got = 1;
      if (lane == 0) got = mbar_wait2(&sc->gfull[st], par, sc, a) ? 1 : 0;
      live = __shfl_sync(0xffffffffu, got, 0) != 0;
      if (!live) more = false;
    }
    if (!live) {  // let the chunk's copies land, store nothing
      if (lane == 0) mbar_wait_quiet(&sc->gfull[st], par, a.timeout_ns);
      __syncwarp();
      continue;
    }
    const int64_t p0 = c * rps;
    const int nr = (int)(a.S - p0 < rps ? a.S - p0 : rps);
    if (lane < nr)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       reinterpret_cast<uint64_t>(h.Y + (p0 + lane) * a.ahead_ldY)),
                   "r"(smem_u32(smem + (size_t)st * kStageBytes2 + (size_t)lane * pitch)),
                   "r"(pitch)
                   : "memory");
    bulk_commit();
    if (more) {  // refill the stage stored last time
      bulk_wait_read1();  // every store group but this chunk's has read shared memory
      __syncwarp();
      const int64_t cn = grab();
      if (cn >= nch)
        more = false;
      else
        issue((st + kSt - 1) % kSt, cn);
    }
  }
  bulk_wait_all();  // this lane's stores are complete
  __syncwarp();
}

// Far tiles: waits until the 256 values of alpha that multiply the tile's columns are
// final (loading them until none holds the pending pattern), then stages them in the
// warp's shared-memory slot.  false when the wait ends without them: the workspace's
// abort word was raised, or the bound ran out (recorded as a timeout; diag kind 7).
__device__ __forceinline__ void load_alpha(const float* src, int lane, float4& v0, float4& v1) {
  v0 = ld_volatile_f4(src + lane * 4);
  v1 = ld_volatile_f4(src + 128 + lane * 4);
}
// v0, v1: this lane's values as loaded earlier (load_alpha), reloaded while pending.
// While values are pending, lane 0 first polls one of them alone (with a back-off), and
// the warp reloads its pending values only once that one is final: the chain stores a
// block's alpha within a short time, and hundreds of waiting warps then put one load
// each instead of 64 on the lines the chain writes.
__device__ bool stage_alpha(const TcArgs& a, const float* src, float* dst, int lane,
                            int where_j, float4 v0, float4 v1) {
  if (__any_sync(0xffffffffu, pending4(v0) || pending4(v1))) {
    const uint64_t t0 = globaltimer_ns();
    // the probe: the first pending value of the lowest lane with one
    const unsigned who = __ballot_sync(0xffffffffu, pending4(v0) || pending4(v1));
    const int pl = __ffs(who) - 1;
    const int pv = __shfl_sync(0xffffffffu, pending4(v0) ? 0 : 1, pl);
    const float* probe = src + pv * 128 + pl * 4;
    int fin = 0;  // the probe was seen final (warp-uniform)
    while (true) {
      if (!fin) {
        if (lane == 0) fin = !pending4(ld_volatile_f4(probe));
        fin = __shfl_sync(0xffffffffu, fin, 0);
      }
      if (fin) {
        if (pending4(v0)) v0 = ld_volatile_f4(src + lane * 4);
        if (pending4(v1)) v1 = ld_volatile_f4(src + 128 + lane * 4);
        if (!__any_sync(0xffffffffu, pending4(v0) || pending4(v1))) break;
      }
      // long sleeps while the probe is pending: hundreds of waiting warps polling the lines
      // the chain writes slowed the launch (measured: 128 ns 132 us, 512 ns 128 us)
      __nanosleep(fin ? 64 : 512);
      int stop = 0;
      if (lane == 0) {
        if (ld_volatile_u32(&a.ctrl->abort)) {
          stop = 1;
        } else if (globaltimer_ns() - t0 > a.timeout_ns) {
          atomicOr(&a.ctrl->status, ST_TIMEOUT);
          atomicExch(&a.ctrl->diag, (7u << 24) | ((uint32_t)where_j << 12));
          atomicExch(&a.ctrl->abort, 1u);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
  *reinterpret_cast<float4*>(dst + lane * 4) = v0;
  *reinterpret_cast<float4*>(dst + 128 + lane * 4) = v1;
  __syncwarp();
  return true;
}


// An accumulator entry as the recurrence uses it: FP32, or rounded to BF16 (G_BF16).
__device__ __forceinline__ float far_entry(uint32_t bits, bool g_bf16) {
  const float g = __uint_as_float(bits);
  return g_bf16 ? round_bf16(g) : g;
}

__device__ __forceinline__ void far_chunk(const uint32_t (&v)[32], const float* al, bool g_bf16,
                                          float (&sum)[8]) {
  const float4* a4 = reinterpret_cast<const float4*>(al);
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 w = a4[e4];
    const int o = (e4 & 1) * 4;
    sum[o + 0] = fmaf(far_entry(v[4 * e4 + 0], g_bf16), w.x, sum[o + 0]);
    sum[o + 1] = fmaf(far_entry(v[4 * e4 + 1], g_bf16), w.y, sum[o + 1]);
    sum[o + 2] = fmaf(far_entry(v[4 * e4 + 2], g_bf16), w.z, sum[o + 2]);
    sum[o + 3] = fmaf(far_entry(v[4 * e4 + 3], g_bf16), w.w, sum[o + 3]);
  }
}

// Adds one far tile's products into the row's eight running sums: accumulator row
// (TMEM lane 32*quarter + lane, buffer acc) times the staged alpha, columns ascending,
// column e into sum e % 8.  The load of the next 32 columns is in flight while the
// current ones are summed.
__device__ __forceinline__ void far_tile_dot(uint32_t tmem, int acc, int quarter,
                                             const float* al, bool g_bf16, float (&sum)[8]) {
  const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
  uint32_t va[32], vb[32];
  __syncwarp();
  tmem_ld32_issue(base, va);
  tmem_wait_ld(va);
#pragma unroll
  for (int ch = 0; ch < BN / 32; ch += 2) {
    tmem_ld32_issue(base + (uint32_t)(ch + 1) * 32, vb);
    far_chunk(va, al + ch * 32, g_bf16, sum);
    tmem_wait_ld(vb);
    if (ch + 2 < BN / 32) tmem_ld32_issue(base + (uint32_t)(ch + 2) * 32, va);
    far_chunk(vb, al + (ch + 1) * 32, g_bf16, sum);
    if (ch + 2 < BN / 32) tmem_wait_ld(va);
  }
}

// The same with the choice as a template parameter, so the FP32 loop carries no
// per-entry select: used by the launches with b >= 1024 (narrow n, where the far
// tiles' epilogue paces the launch; measured on n = 28, b = 2048, s = 32: 1142 -> 998
// us per outer iteration).  The other launches keep the form above (the change cost
// the n = 2000 launch ~1 us through its register allocation).
template <bool kGBf16>
__device__ __forceinline__ float far_entry(uint32_t bits) {
  const float g = __uint_as_float(bits);
  return kGBf16 ? round_bf16(g) : g;
}

template <bool kGBf16>
__device__ __forceinline__ void far_chunk(const uint32_t (&v)[32], const float* al,
                                          float (&sum)[8]) {
  const float4* a4 = reinterpret_cast<const float4*>(al);
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 w = a4[e4];
    const int o = (e4 & 1) * 4;
    sum[o + 0] = fmaf(far_entry<kGBf16>(v[4 * e4 + 0]), w.x, sum[o + 0]);
    sum[o + 1] = fmaf(far_entry<kGBf16>(v[4 * e4 + 1]), w.y, sum[o + 1]);
    sum[o + 2] = fmaf(far_entry<kGBf16>(v[4 * e4 + 2]), w.z, sum[o + 2]);
    sum[o + 3] = fmaf(far_entry<kGBf16>(v[4 * e4 + 3]), w.w, sum[o + 3]);
  }
}

template <bool kGBf16>
__device__ __forceinline__ void far_tile_dot(uint32_t tmem, int acc, int quarter,
                                             const float* al, float (&sum)[8]) {
  const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
  uint32_t va[32], vb[32];
  __syncwarp();
  tmem_ld32_issue(base, va);
  tmem_wait_ld(va);
#pragma unroll
  for (int ch = 0; ch < BN / 32; ch += 2) {
    tmem_ld32_issue(base + (uint32_t)(ch + 1) * 32, vb);
    far_chunk<kGBf16>(va, al + ch * 32, sum);
    tmem_wait_ld(vb);
    if (ch + 2 < BN / 32) tmem_ld32_issue(base + (uint32_t)(ch + 2) * 32, va);
    far_chunk<kGBf16>(vb, al + (ch + 1) * 32, sum);
    if (ch + 2 < BN / 32) tmem_wait_ld(va);
  }
}

template <int kSt, int kRecV, bool kNext, bool kFar, bool kGather = false>
__global__ void __launch_bounds__(kRecV ? kFusedThreads : kThreads, 1)
    gram_tc2sm_kernel(const __grid_constant__ CUtensorMap tmY,
                      const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmYf, TcArgs a, RecArgs rec) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* out_stage = smem + (size_t)kSt * kStageBytes2;  // 1024-aligned
  SharedCtl2<kSt>* sc = reinterpret_cast<SharedCtl2<kSt>*>(out_stage + kOutBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_rank();
  const bool leader = rank == 0;
  const int cid = (int)blockIdx.x / 2, ncl = (int)gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSt; ++i) {
      mbar_init(&sc->full[i], 1);
      mbar_init(&sc->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc->tfull[i], 1);
      mbar_init(&sc->tempty[i], 8);
    }
    mbar_init(&sc->drain, 1);
    for (int i = 0; i < kSt; ++i) mbar_init(&sc->gfull[i], 1);
    sc->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates collectively for the pair
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sc->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sc->tmem_base;
  // Launched behind the gather (programmatic dependent launch), the setup above
  // overlaps the gather's end; every global access follows this wait.
  wait_prior_grid();

  if (warp == 0 && kGather) {
    // ------------------------------------------------ row-gathering producer (both CTAs)
    // The whole warp: per tile, lane L draws the X rows of A rows 4L..4L+3 and of B rows
    // 4L..4L+3 (of this CTA's half) from the sampler, then per 64 columns of K issues one
    // four-row gather of each into the stage (lane 0 waits for the stage and, in the
    // leader, arms its barrier for both CTAs' bytes first).  Every tile is whole: S is a
    // multiple of 256 on this path.
    WorkCursor<kFar> cur;
    int stage = 0;
    uint32_t phase = 0;
    bool live = true;
    for (int kq = 0, u = unit_of(a, cid, ncl, 0); u < a.ntiles && live;
         u = unit_of(a, cid, ncl, ++kq)) {
      live = __shfl_sync(0xffffffffu, sc->abort ? 0 : 1, 0) != 0;
      if (!live) break;
      int rg, ca0, nq, t, pidx;
      bool far;
      cur.seek(a, u, rg, ca0, nq, t, pidx, far);
      const int ra = 2 * rg + rank;
      const uint64_t c0 = (kFar && far) ? a.ctr_f : a.ctr_g;  // this iteration's or the Gram's
      int32_t ar[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ar[i] = draw_row(a.seed, c0 + (uint64_t)(ra * BM + 4 * lane + i), a.m, a.perm_d);
      for (int q = 0; q < nq && live; ++q) {
        const int ca = ca0 + q;
        int32_t br[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          br[i] = draw_row(a.seed, c0 + (uint64_t)(ca * BN + rank * (BN / 2) + 4 * lane + i), a.m,
                           a.perm_d);
        for (int kb = 0; kb < a.nkb; ++kb) {
          int ok = 1;
          if (lane == 0) {
            ok = mbar_wait2(&sc->empty[stage], phase ^ 1u, sc, a) ? 1 : 0;
            if (ok && leader) mbar_expect_tx(&sc->full[stage], 2 * kStageBytes2);  // both CTAs
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            live = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes2);
          const uint32_t sb = sa + kABytes;
          const uint32_t bar = mapa_rank(smem_u32(&sc->full[stage]), 0);
          tma_gather4_pair(sa + lane * 512, &tmY, bar, kb * BK, ar[0], ar[1], ar[2], ar[3]);
          tma_gather4_pair(sb + lane * 512, &tmY, bar, kb * BK, br[0], br[1], br[2], br[3]);
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 0) {
    int stage = 0;
    uint32_t phase = 0;
    if (lane == 0) {
      // -------------------------------------------------------- TMA producer (both CTAs)
      WorkCursor<kFar> cur;
      for (int kq = 0, u = unit_of(a, cid, ncl, 0); u < a.ntiles && !sc->abort;
           u = unit_of(a, cid, ncl, ++kq)) {
        int rg, ca0, nq, t, pidx;
        bool far;
        cur.seek(a, u, rg, ca0, nq, t, pidx, far);
        const int ra = 2 * rg + rank;
        // far tiles read this iteration's rows; the others the Gram's own rows
        const CUtensorMap* map = (kFar && far) ? &tmYf : &tmY;
        for (int q = 0; q < nq && !sc->abort; ++q) {
          const int ca = ca0 + q;
          for (int kb = 0; kb < a.nkb; ++kb) {
            if (!mbar_wait2(&sc->empty[stage], phase ^ 1u, sc, a)) break;
            uint8_t* sa = smem + (size_t)stage * kStageBytes2;
            uint8_t* sb = sa + kABytes;
            if (leader) mbar_expect_tx(&sc->full[stage], 2 * kStageBytes2);  // both CTAs
            const uint32_t bar = mapa_rank(smem_u32(&sc->full[stage]), 0);
            tma_load_2d_pair(smem_u32(sa), map, bar, kb * BK, ra * BM);
            tma_load_2d_pair(smem_u32(sb), map, bar, kb * BK, ca * BN + rank * (BN / 2));
            if (++stage == kSt) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
    if (kFar && kNext && kRecV != 0 && a.ahead_on) {
      __syncwarp();
      const int st0 = __shfl_sync(0xffffffffu, stage, 0);
      const uint32_t ph0 = __shfl_sync(0xffffffffu, phase, 0);
      if (!__shfl_sync(0xffffffffu, sc->abort ? 1 : 0, 0)) {
        if (a.ahead_ldY <= 64)
          gather_ahead_narrow(a, lane);
        else
          gather_ahead<kSt>(a, sc, smem, lane, st0, ph0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // -------------------------------------------------------- MMA issuer (leader)
      WorkCursor<kFar> cur;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tphase[2] = {0, 0};
      int iter = 0;  // tiles issued (accumulator buffer iter & 1)
      bool any = false, ok = true;
      for (int kq = 0, u = unit_of(a, cid, ncl, 0); u < a.ntiles && ok && !sc->abort;
           u = unit_of(a, cid, ncl, ++kq)) {
        int rg, ca0, nq, t, pidx;
        bool far;
        cur.seek(a, u, rg, ca0, nq, t, pidx, far);
        for (int q = 0; q < nq && ok; ++q, ++iter) {
          const int acc = iter & 1;
          if (!mbar_wait2(&sc->tempty[acc], tphase[acc] ^ 1u, sc, a)) { ok = false; break; }
          tphase[acc] ^= 1u;
          tc_fence_after();
          const uint32_t tacc = tmem + (uint32_t)(acc * BN);
          for (int kb = 0; kb < a.nkb; ++kb) {
            if (!mbar_wait2(&sc->full[stage], phase, sc, a)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes2);
            const uint32_t sb = sa + kABytes;
            const uint64_t ad = sdesc_sw128(sa), bd = sdesc_sw128(sb);
            const int krem = a.n - kb * BK;
            const int ksteps = krem >= BK ? BK / 16 : (krem + 15) / 16;
            for (int kk = 0; kk < ksteps; ++kk)
              mma_bf16_pair(tacc, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                            (kb > 0 || kk > 0) ? 1u : 0u);
            any = true;
            mma_commit_pair(&sc->empty[stage], 0x3);
            if (++stage == kSt) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(&sc->tfull[acc], 0x3);
        }
      }
      if (any) {  // drain: every MMA complete before the pair frees TMEM
        mma_commit_pair(&sc->drain, 0x1);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&sc->drain, 0) && globaltimer_ns() - t0 < a.timeout_ns) {
        }
      }
    }
    if (kFar && kNext && kRecV != 0 && !leader && a.nx_on) reset_next_set(a.nx, a.S, cid, ncl, lane);
  } else if (warp < 6) {
    // ---------------------------------------------------------- epilogue (both CTAs)
    // Stored tiles: masked or TMA stores into G, then (recurrence in the same launch,
    // same iteration) the release of the warp's 32-row counter.  Far tiles (kFar): the
    // row's products with alpha_t summed over the unit's tiles into fpart; once a wait
    // for alpha has ended without it, the warp only drains its tiles (the Gram warps
    // always finish their tiles, so every copy and MMA of the launch completes).
    const int quarter = warp & 3;
    uint8_t* stage = out_stage + (warp - 2) * kStageOut;
    float* al_s = reinterpret_cast<float*>(out_stage + kOutBytes + 1024) + (warp - 2) * BN;
    int sbuf = 0;
    WorkCursor<kFar> cur;
    uint32_t tphase[2] = {0, 0};
    int iter = 0;
    bool live = true, dead = false;  // live: the Gram's own waits succeed; dead: alpha gone
    for (int kq = 0, u = unit_of(a, cid, ncl, 0); u < a.ntiles && live;
         u = unit_of(a, cid, ncl, ++kq)) {
      int rg, ca0, nq, t, pidx;
      bool far;
      cur.seek(a, u, rg, ca0, nq, t, pidx, far);
      const int ra = 2 * rg + rank;
      float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // far: alpha of the unit's first column
      const float* al_g = a.alpha + (int64_t)ca0 * BN;
      float4 an0, an1;  // far: the next tile's alpha, loaded ahead
      if (kFar && far && !dead) load_alpha(al_g, lane, an0, an1);
      for (int q = 0; q < nq; ++q, ++iter) {
        const int ca = ca0 + q;
        const int acc = iter & 1;
        if (kFar && far && !dead) {
          dead = !stage_alpha(a, al_g + q * BN, al_s, lane, (ra * BM) / a.b, an0, an1);
          if (!dead && q + 1 < nq) load_alpha(al_g + (q + 1) * BN, lane, an0, an1);
        }
        int ok = 1;
        if (lane == 0) ok = mbar_wait2(&sc->tfull[acc], tphase[acc], sc, a) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          live = false;
          break;
        }
        tphase[acc] ^= 1u;
        tc_fence_after();
        if (kFar && far) {
          if (!dead) {
            if constexpr (kRecV != 1)
              far_tile_dot(tmem, acc, quarter, al_s, a.g_bf16, sum);
            else if (a.g_bf16)
              far_tile_dot<true>(tmem, acc, quarter, al_s, sum);
            else
              far_tile_dot<false>(tmem, acc, quarter, al_s, sum);
          }
        } else {
          if (a.tma_store)
            store_tile_tma(a, tmem, acc, quarter, lane, ra, ca, &tmG, stage, sbuf);
          else
            store_tile_rows(a, tmem, acc, quarter, lane, ra, ca, &tmG, stage, sbuf);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_rank(smem_u32(&sc->tempty[acc]), 0));
        if (kFar && far) continue;
        if (kRecV && !kNext && q == nq - 1) {
          // publish this warp's 32 rows of the unit's tiles: their stores are complete
          // and visible
          if (a.tma_store) {
            if (lane == 0) {
              bulk_wait_all();
              fence_proxy_async_global();
            }
          } else {
            __threadfence();
          }
          __syncwarp();
          if (lane == 0) {
            red_release_add_u32(a.slab + (int64_t)ra * 4 + quarter, (uint32_t)nq);
            red_release_add_u32(&a.q->band_done, (uint32_t)nq);
            stamp_last(rec.trace, 0);
          }
        } else if (kRecV && lane == 0) {
          stamp_last(rec.trace, 0);
        }
      }
      if (kFar && far && live && !dead) {
        const int64_t p = (int64_t)ra * BM + quarter * 32 + lane;
        __stcg(a.fpart + p * a.fs + pidx,
               ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7])));
        if (lane == 0) stamp_last(rec.trace, 1);
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's tensor stores are complete
    __syncwarp();
  } else if (kRecV) {
    // ---------------------------------------------------------- recurrence (warps 6-13)
    // the first C CTAs run chain groups, the others the bulk role
    const int rt = threadIdx.x - kThreads;
    // 1: same iteration, G stored; 2: next iteration's Gram, G complete; 3: same
    // iteration, far sums from the Gram; 4: far sums from the Gram, band complete (the
    // Gram stores the next iteration's band)
    constexpr int kMode = kFar ? (kNext ? 4 : 3) : (kNext ? 2 : 1);
    if ((int)blockIdx.x < rec.C)
      chain_role<kRecV == 1 ? 1 : (kRecV == 2 ? 2 : 3), kRecV == 1 ? 8 : (kRecV == 2 ? 4 : 2),
                 kMode>(rec, blockIdx.x, rt);
    else
      bulk_role<kMode, kGather>(rec, rt, (int)blockIdx.x - rec.C < rec.upd_groups);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs and every copy into either CTA are finished
  tc_fence_after();
  allow_next_grid();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  if (threadIdx.x == 0 && sc->abort) atomicExch(&a.ctrl->abort, 1u);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

bool gram_tc_supported(int64_t S, int64_t n, int b) {
  return S >= 1 && n >= 1 && b >= 1 && S <= kMaxSB && n <= kMaxN;
}

namespace {

struct TcPlan {
  TcArgs a;
  CUtensorMap map, mapG;
};

// Tensor maps and tile counts shared by every variant.  kcl: CTAs per row group.
// gB: layout of G (0 packed block-lower; band_width(b) for the band layout).
cudaError_t plan_tc(const uint16_t* Y, int64_t S, int64_t n, int64_t ldY, int b, int s,
                    uint32_t flags, int kcl, float* G, Ctrl* ctrl, uint32_t timeout_us,
                    TcPlan& P, int gB = 0) {
  const bool diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)n, (cuuint64_t)S};
  const cuuint64_t gstride[1] = {(cuuint64_t)ldY * 2};
  const cuuint32_t box[2] = {BK, BM};
  const cuuint32_t estride[2] = {1, 1};
  memset(&P.map, 0, sizeof(P.map));
  if (Y && enc(&P.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(Y), gdim,
               gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
                   CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  TcArgs& a = P.a;
  a.G = G;
  a.ctrl = ctrl;
  a.q = ctrl;
  a.S = S;
  a.n = (int)n;
  a.b = b;
  a.nkb = (int)((n + BK - 1) / BK);
  a.TR = (int)((S + BM - 1) / BM);
  a.TC = (int)((S + BN - 1) / BN);
  a.diag = diag;
  a.g_bf16 = (flags & CASGD_FLAG_G_BF16) != 0;
  a.timeout_ns = (uint64_t)(timeout_us ? timeout_us : 1000000u) * 1000ull;
  a.slab = nullptr;
  a.fpart = nullptr;
  a.alpha = nullptr;
  a.s = s;
  a.B = band_width(b);
  a.nb = b / 256;
  a.npb = a.uq = 1;
  a.fs = s;
  a.stored_last = false;
  a.n_stored = a.far_head = a.store_tail = 0;
  a.ahead_on = false;
  a.ahead_ldY = 0;
  memset(&a.ahead, 0, sizeof(a.ahead));
  a.nx_on = false;
  memset(&a.nx, 0, sizeof(a.nx));
  a.gB = gB;
  a.seed = a.ctr_g = a.ctr_f = 0;
  a.m = 0;
  a.perm_d = 0;
  a.pc = 0;
  a.wa = a.wb = 1;
  // count the needed tiles on the host with the same rule the kernel walks
  int64_t total = 0;
  for (int g = 0; g * kcl < a.TR; ++g) {
    if (kcl == 2) {
      total += pair_group_tiles(S, b, diag, g);
      continue;
    }
    int last = g * kcl + kcl - 1;
    if (last > a.TR - 1) last = a.TR - 1;
    int64_t lr = (int64_t)last * BM + BM - 1;
    if (lr > S - 1) lr = S - 1;
    const int64_t jmax = lr / b;
    const int64_t lim = (int64_t)b * (diag ? jmax + 1 : jmax);
    int64_t cc = (lim + BN - 1) / BN;
    total += cc < a.TC ? cc : a.TC;
  }
  a.ntiles = (int)total;

  // Output map: G (either layout) viewed as (blocks * b) rows of b FP32 columns; 32x32
  // boxes.
  memset(&P.mapG, 0, sizeof(P.mapG));
  a.tma_store = false;
  const int64_t nblk = g_layout_elems(b, s, diag, gB) / ((int64_t)b * b);
  if (b % 32 == 0 && nblk > 0) {
    const cuuint64_t gdimG[2] = {(cuuint64_t)b, (cuuint64_t)(nblk * b)};
    const cuuint64_t gstrideG[1] = {(cuuint64_t)b * 4};
    const cuuint32_t boxG[2] = {32, 32};
    a.tma_store = enc(&P.mapG, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, G, gdimG, gstrideG, boxG,
                      estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  return cudaSuccess;
}

// The map the row-gathering producer reads X through: X viewed as m rows of n BF16
// columns (pitch ld), a box of 64 columns by one row (tile::gather4 takes four of them),
// 128-byte swizzle, columns from n on read as zeros.  Sets the sampler fields of a.
cudaError_t plan_gather(const RowSource& rs, int64_t n, uint64_t ctr_g, uint64_t ctr_f,
                        TcPlan& P) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)n, (cuuint64_t)rs.m};
  const cuuint64_t gstride[1] = {(cuuint64_t)rs.ld * 2};
  const cuuint32_t box[2] = {BK, 1};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&P.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(rs.X), gdim,
          gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  P.a.seed = rs.seed;
  P.a.ctr_g = ctr_g;
  P.a.ctr_f = ctr_f;
  P.a.m = rs.m;
  P.a.perm_d = rs.perm_d;
  return cudaSuccess;
}

cudaLaunchConfig_t cluster2_config(unsigned threads, size_t smem, cudaStream_t st,
                                   cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_gram_tc(const uint16_t* Y, int64_t S, int64_t n, int64_t ldY, int b, int s,
                           uint32_t flags, int mode, float* G, Ctrl* ctrl, uint32_t timeout_us,
                           Ctx& c) {
  if (S <= 0) return cudaSuccess;
  // mode 0: paired-SM MMA (default); 1: one CTA per tile.  A single row tile always runs
  // on one CTA.
  if ((S + BM - 1) / BM <= 1) mode = 1;
  if (mode != 0 && mode != 1) return cudaErrorInvalidValue;
  const int kcl = mode == 1 ? 1 : 2;
  TcPlan P;
  cudaError_t e = plan_tc(Y, S, n, ldY, b, s, flags, kcl, G, ctrl, timeout_us, P);
  if (e != cudaSuccess) return e;
  TcArgs& a = P.a;
  if (a.ntiles == 0) return cudaSuccess;

  if (mode == 1) {
    e = cudaFuncSetAttribute(gram_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = a.ntiles < c.num_sms ? a.ntiles : c.num_sms;
    gram_tc_kernel<<<grid, kThreads, kSmemBytes, c.stream>>>(P.map, P.mapG, a);
    ++c.launches;
    return cudaGetLastError();
  }
  const void* fn = (const void*)gram_tc2sm_kernel<kStagesPair, 0, false, false>;
  const size_t smem = pair_smem_bytes<kStagesPair>();
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster2_config(kThreads, smem, c.stream, attr);
  cfg.gridDim = dim3(2 * (unsigned)(c.num_sms / 2));
  int max_clusters = 0;
  e = cached_query(c, fn, [&](int& v) {
    cudaError_t r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r != cudaSuccess) return r;
    if (cudaOccupancyMaxActiveClusters(&v, fn, &cfg) != cudaSuccess || v < 1) v = c.num_sms / 2;
    return cudaSuccess;
  }, max_clusters);
  if (e != cudaSuccess) return e;
  const int clusters = a.ntiles < max_clusters ? a.ntiles : max_clusters;
  cfg.gridDim = dim3(2 * (unsigned)clusters);
  RecArgs none;
  memset(&none, 0, sizeof(none));
  e = cudaLaunchKernelEx(&cfg, gram_tc2sm_kernel<kStagesPair, 0, false, false>, P.map, P.mapG,
                         P.map, a, none);
  ++c.launches;
  return e;
}

bool gram_recur_fused_supported(int64_t S, int64_t n, int b) {
  // at least two row tiles (the paired kernel) and one block of G below the diagonal
  return gram_tc_supported(S, n, b) && (S + BM - 1) / BM >= 2 && S / b >= 2;
}

bool far_gram_supported(int64_t S, int64_t n, int b) {
  // whole 256x256 tiles inside one block pair (j, t)
  return gram_recur_fused_supported(S, n, b) && b % 256 == 0;
}

bool ahead_rows_supported(int64_t n, int64_t ldY) {
  // whole 16-byte row copies through the stages, rows of at least 512 bytes that fit a
  // stage; or narrow rows (at most 64 columns) by plain vector loads
  return (n % 8 == 0 && ldY * 2 >= 512 && ldY * 2 <= kStageBytes2) || ldY <= 64;
}

namespace {

// Units of the far-forming order: far (t < j-B) and stored (band, and the diagonal on
// request), nb * npb of each per block pair (j, t).
void far_unit_counts(const TcArgs& a, int64_t& far_units, int64_t& stored_units) {
  int64_t nfar = 0, nst = 0;
  for (int j = 0; j < a.s; ++j) {
    const int nband = j < a.B ? j : a.B;
    nfar += j - nband;
    nst += nband + (a.diag ? 1 : 0);
  }
  far_units = (int64_t)a.nb * a.npb * nfar;
  stored_units = (int64_t)a.nb * a.npb * nst;
}

void set_far_fields(TcArgs& a, int b, int s, float* fpart, const float* alpha) {
  a.fpart = fpart;
  a.alpha = alpha;
  a.npb = far_partials_per_block(b, s);
  a.uq = a.nb / a.npb;
  a.fs = s * a.npb;
}

}  // namespace

cudaError_t launch_gram_band(const uint16_t* Y, float* G, int64_t S, int64_t n, int64_t ldY,
                             int b, int s, uint32_t flags, Ctrl* ctrl, uint32_t timeout_us,
                             const RowSource* rs, uint64_t ctr, Ctx& c) {
  if (!far_gram_supported(S, n, b)) return cudaErrorNotSupported;
  TcPlan P;
  cudaError_t e = plan_tc(rs ? nullptr : Y, S, n, ldY, b, s, flags, 2, G, ctrl, timeout_us, P,
                          band_width(b));
  if (e != cudaSuccess) return e;
  if (rs && (e = plan_gather(*rs, n, ctr, ctr, P)) != cudaSuccess) return e;
  set_far_fields(P.a, b, s, nullptr, nullptr);
  int64_t nfar, nst;
  far_unit_counts(P.a, nfar, nst);
  P.a.n_stored = (int)nst;
  P.a.ntiles = (int)nst;  // the stored units only (they come first)
  if (P.a.ntiles == 0) return cudaSuccess;
  const auto fn = rs ? gram_tc2sm_kernel<kStagesFused, 0, false, true, true>
                     : gram_tc2sm_kernel<kStagesFused, 0, false, true>;
  const size_t smem = pair_smem_bytes<kStagesFused, true>();
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster2_config(kThreads, smem, c.stream, attr);
  cfg.gridDim = dim3(2 * (unsigned)(c.num_sms / 2));
  int max_clusters = 0;
  e = cached_query(c, (const void*)fn, [&](int& v) {
    cudaError_t r = cudaFuncSetAttribute((const void*)fn,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r != cudaSuccess) return r;
    if (cudaOccupancyMaxActiveClusters(&v, (const void*)fn, &cfg) != cudaSuccess || v < 1)
      v = c.num_sms / 2;
    return cudaSuccess;
  }, max_clusters);
  if (e != cudaSuccess) return e;
  const int clusters = P.a.ntiles < max_clusters ? P.a.ntiles : max_clusters;
  cfg.gridDim = dim3(2 * (unsigned)clusters);
  RecArgs none;
  memset(&none, 0, sizeof(none));
  e = cudaLaunchKernelEx(&cfg, fn, P.map, P.mapG, P.map, P.a, none);
  ++c.launches;
  return e;
}

cudaError_t launch_gram_recur(const uint16_t* Yg, float* Gg, bool next, int64_t S, int64_t n,
                              int64_t ldY, int b, int s, float eta, int loss, uint32_t flags,
                              const float* G, const uint16_t* Y, float* r,
                              const float* yY, float* alpha, float* far, uint32_t* slab,
                              float* fpart, float* part, float* w, bool own_margins, Ctrl* ctrl,
                              uint32_t timeout_us, bool g_band, const RowSource* rs,
                              uint64_t ctr_g, uint64_t ctr_f, const AheadRows* ahead, Ctrl* q,
                              uint32_t* cnt, const NextSet* nx, Ctx& c) {
  if (!gram_recur_fused_supported(S, n, b)) return cudaErrorNotSupported;
  const bool far_gram = fpart != nullptr;
  if (far_gram && !far_gram_supported(S, n, b)) return cudaErrorNotSupported;
  if (!far_gram && !Yg) return cudaErrorInvalidValue;
  if (rs && !far_gram) return cudaErrorInvalidValue;  // only the far-forming launch gathers
  const bool gather = rs != nullptr;
  const bool diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  TcPlan P;
  const int gB = (far_gram && g_band) ? band_width(b) : 0;  // layout of Gg and G
  cudaError_t e = plan_tc(gather ? nullptr : (Yg ? Yg : Y), S, n, ldY, b, s, flags, 2, Gg, ctrl,
                          timeout_us, P, gB);
  if (e != cudaSuccess) return e;
  if (gather && (e = plan_gather(*rs, n, ctr_g, ctr_f, P)) != cudaSuccess) return e;
  // far tiles read this iteration's rows (the Gram's own rows unless next; gathering, the
  // same map of X with this iteration's sampler counters)
  CUtensorMap mapYf = P.map;
  if (far_gram && next && !gather) {
    TcPlan Pf;
    e = plan_tc(Y, S, n, ldY, b, s, flags, 2, Gg, ctrl, timeout_us, Pf);
    if (e != cudaSuccess) return e;
    mapYf = Pf.map;
  }
  P.a.slab = next ? nullptr : slab;
  RecArgs rec = make_rec_args(G, r, yY, alpha, far, slab, b, s, eta, loss, flags, timeout_us,
                              ctrl, Y, ldY, n, part, w);
  rec.gB = gB;
  if (q) {  // this iteration's counters (the trace stays in slab's area)
    rec.q = q;
    P.a.q = q;
  }
  if (cnt) {
    rec.upd_chunks = upd_chunk_counters(cnt);
    rec.upd_blocks = upd_block_counters(cnt);
  }
  if (gather) {  // margins and update read this iteration's rows from X
    rec.X = rs->X;
    rec.ldx = rs->ld;
    rec.xseed = rs->seed;
    rec.xctr = ctr_f;
    rec.xm = rs->m;
    rec.xperm = rs->perm_d;
  }
  rec.slab = next ? nullptr : slab;
  if (far_gram) {  // work items: units of uq tiles
    set_far_fields(P.a, b, s, fpart, alpha);
    int64_t nfar, nst;
    far_unit_counts(P.a, nfar, nst);
    // next: the next iteration's band (none without its rows) after one round of far
    // units (far_head is set once the grid is known)
    P.a.stored_last = next;
    if (ahead && next && !gather && ahead_rows_supported(n, ldY)) {
      P.a.ahead_on = true;
      P.a.ahead_ldY = ldY;
      P.a.ahead = *ahead;
    }
    if (nx && next && !gather) {
      P.a.nx_on = true;
      P.a.nx = *nx;
    }
    const bool g_rows = gather ? ctr_g != kNoRows : Yg != nullptr;  // the Gram has rows
    P.a.n_stored = (int)((!next || g_rows) ? nst : 0);
    P.a.ntiles = (int)(nfar + P.a.n_stored);
    P.a.far_head = 0;
    P.a.store_tail = 0;
    rec.fpart = fpart;
    rec.fs = P.a.fs;
    rec.npb = P.a.npb;
    rec.far_gram = true;
    rec.bulk_units = 0;  // no far units: the Gram forms the far sums
    rec.upd_R = upd_row_parts(b, ldY);  // the bulk groups only update: row parts
    rec.upd_units = s * (int)((ldY / 8 + 7) / 8) * rec.upd_R;
    if (own_margins) {  // the bulk groups form the margins first (mG lanes per row, 2 passes)
      int G = 1;
      while (G < ldY / 8 && G < 32) G <<= 1;
      rec.margins = true;
      rec.mG = G;
      rec.mrows = 8 * (32 / G) * 2;
      rec.bulk_units = (int)((S + rec.mrows - 1) / rec.mrows);
      rec.r_w = r;
      rec.wm = w;
      rec.wm_vec = (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
    }
  }
  // what Ctrl::band_done reaches once every stored tile is stored (8 warps per tile)
  if (!next) {
    int64_t total = 0;
    for (int g = 0; (int64_t)g * 256 < S; ++g)
      total += far_gram ? far_gram_stored_tiles(b, diag, g) : pair_group_tiles(S, b, diag, g);
    rec.band_total = (uint32_t)(8 * total);
  }
  const int v = chain_variant(rec);
  using Fn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, TcArgs, RecArgs);
  const Fn table[4][3] = {
      {gram_tc2sm_kernel<kStagesFused, 1, false, false>,
       gram_tc2sm_kernel<kStagesFused, 2, false, false>,
       gram_tc2sm_kernel<kStagesFused, 3, false, false>},
      {gram_tc2sm_kernel<kStagesFused, 1, true, false>,
       gram_tc2sm_kernel<kStagesFused, 2, true, false>,
       gram_tc2sm_kernel<kStagesFused, 3, true, false>},
      {gram_tc2sm_kernel<kStagesFused, 1, false, true>,
       gram_tc2sm_kernel<kStagesFused, 2, false, true>,
       gram_tc2sm_kernel<kStagesFused, 3, false, true>},
      {gram_tc2sm_kernel<kStagesFused, 1, true, true>,
       gram_tc2sm_kernel<kStagesFused, 2, true, true>,
       gram_tc2sm_kernel<kStagesFused, 3, true, true>}};
  const Fn gtable[2][3] = {
      {gram_tc2sm_kernel<kStagesFused, 1, false, true, true>,
       gram_tc2sm_kernel<kStagesFused, 2, false, true, true>,
       gram_tc2sm_kernel<kStagesFused, 3, false, true, true>},
      {gram_tc2sm_kernel<kStagesFused, 1, true, true, true>,
       gram_tc2sm_kernel<kStagesFused, 2, true, true, true>,
       gram_tc2sm_kernel<kStagesFused, 3, true, true, true>}};
  const Fn fn = gather ? gtable[next ? 1 : 0][v - 1]
                       : table[(far_gram ? 2 : 0) + (next ? 1 : 0)][v - 1];
  const size_t smem = far_gram ? pair_smem_bytes<kStagesFused, true>()
                               : pair_smem_bytes<kStagesFused>();
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster2_config(kFusedThreads, smem, c.stream, attr);
  cfg.gridDim = dim3(2 * (unsigned)(c.num_sms / 2));
  int max_clusters = 0;
  e = cached_query(c, (const void*)fn, [&](int& v) {
    cudaError_t r = cudaFuncSetAttribute((const void*)fn,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r != cudaSuccess) return r;
    return cudaOccupancyMaxActiveClusters(&v, (const void*)fn, &cfg);
  }, max_clusters);
  if (e != cudaSuccess) return e;
  // every CTA must be resident at once (the recurrence waits across CTAs); one chain
  // group per 8-row group while at least one bulk group remains
  if (max_clusters < 1) return cudaErrorNotSupported;
  const int grid = 2 * max_clusters;
  rec.C = rec.Uc < grid - 1 ? rec.Uc : grid - 1;
  if (rec.C > grid / 2) rec.C = grid / 2;
  // Far sums from the Gram: the bulk groups only update, so where a chain warp would
  // take more than two rows per phase (b > 8 * grid), chain CTAs may take all but 24 of
  // the CTAs, two row groups each (measured: b = 2048, 180 -> 128-150 us per launch).
  constexpr int kUpdateCtas = 24;
  if (far_gram && rec.Uc > grid && grid > 2 * kUpdateCtas) {
    const int want = (rec.Uc + 1) / 2;
    rec.C = want < grid - kUpdateCtas ? want : grid - kUpdateCtas;
  }
  if (rec.C < 1) return cudaErrorNotSupported;
  rec.upd_groups = rec.margins ? 0 : update_groups(rec, grid - rec.C);
  // the pairs whose CTAs also run the chain (CTAs 0 .. C-1) take fewer Gram items
  P.a.pc = (rec.C + 1) / 2;
  P.a.wa = kChainPairShare;
  P.a.wb = kOtherPairShare;
  if (far_gram && next) {
    const int nfar = P.a.ntiles - P.a.n_stored;
    P.a.far_head = nfar < grid / 2 ? nfar : grid / 2;
    P.a.store_tail = (int)((int64_t)P.a.n_stored * kStoreTailPct / 100);
  }
  cfg.gridDim = dim3((unsigned)grid);
  // Scheduled early behind the gather, a CTA waits in wait_prior_grid() (a hardware
  // wait, no spin) until the gather has completed; the gather blocks are all running
  // by then (they allow this launch only once each has started), so every CTA of this
  // grid is still resident once they leave.
  add_pdl_attr(c, cfg, attr);
  e = cudaLaunchKernelEx(&cfg, fn, P.map, P.mapG, mapYf, P.a, rec);
  ++c.launches;
  return e;
}

}  // namespace casgd
