// Internal declarations shared by the CA-SGD kernels and the C-ABI layer.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract).  Kernel map (steps as numbered in include/casgd.h):
//   k_prep.cu       a1 sampling, a2 gather into Y, a4 BF16 margins; BF16 storage
//   k_gram_simt.cu  a3 Gram on CUDA cores (any n; used for narrow n)
//   k_gram_tc.cu    a3 Gram on tcgen05 tensor cores with TMEM accumulators and TMA
//   k_recur.cu      a6/a7 inner recurrence: persistent chain + bulk CTAs, data-synchronised
//                   (roles in recur_roles.cuh; also run inside the paired-SM Gram launch)
//   k_update.cu     a8 weight update, a9 full-data loss
//   k_sgd.cu        FP32 plain minibatch SGD, the baseline CA-SGD is compared with
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/casgd.h"

namespace casgd {

// Sticky device status bits (workspace word 0).
enum : uint32_t {
  ST_NONFINITE = 1u << 0,
  ST_TIMEOUT = 1u << 1,
  ST_BAD_INDEX = 1u << 2,
};

constexpr int kMaxS = 64;
// alpha slots hold this bit pattern from the gather kernel until the recurrence writes
// their value (a NaN payload no arithmetic produces: computed NaNs are 0x7FFFFFFF), so
// a reader can wait on the values themselves.
constexpr uint32_t kAlphaPending = 0x7FA1FA11u;
constexpr int64_t kMaxSB = 65536;
constexpr int64_t kMaxN = 16384;
constexpr int kLossCtas = 1024;     // upper bound on loss-kernel CTAs (partials)
// per-32-row completion counters of the paired-SM Gram (rows padded to 256-row groups)
constexpr int64_t kMaxSlabs = (kMaxSB + 255) / 256 * 8;
// per-64-column counters of the weight update (the next block whose sum is added to w)
constexpr int64_t kMaxUpdChunks = kMaxN / 64;
// per-(block, 64-column chunk) arrival counters of the update's row parts
constexpr int64_t kMaxUpdBlocks = kMaxS * kMaxUpdChunks;
// The counters area of the workspace: kMaxSlabs row counters, kMaxUpdChunks column
// counters, kMaxUpdBlocks block counters, then the profiling timeline ((kMaxS + 1) x 4
// globaltimer stamps).
__host__ __device__ inline uint32_t* upd_chunk_counters(uint32_t* slab) { return slab + kMaxSlabs; }
__host__ __device__ inline uint32_t* upd_block_counters(uint32_t* slab) {
  return slab + kMaxSlabs + kMaxUpdChunks;
}
__host__ __device__ inline uint64_t* timeline_of(uint32_t* slab) {
  return reinterpret_cast<uint64_t*>(slab + kMaxSlabs + kMaxUpdChunks + kMaxUpdBlocks);
}

// Control block at the start of the workspace (256 bytes, zeroed per step where noted).
struct Ctrl {
  uint32_t status;        // sticky ST_* bits (cleared by casgd_get_status)
  uint32_t abort;         // set by a waiter that timed out; others stop waiting.  The
                          // gather kernel re-arms it each step only while no timeout is
                          // recorded in `status`, so later steps fail fast.
  uint32_t next_unit;     // recurrence work queue (zeroed by the gather kernel)
  uint32_t loss_done;     // loss kernel: CTAs finished (zeroed by the loss kernel's last CTA)
  uint32_t upd_next;      // recurrence: update-unit queue (zeroed by the gather kernel)
  uint32_t diag;          // which wait timed out last: kind << 24 | block << 12 | value seen
  uint32_t band_done;     // Gram in the recurrence's launch: tiles stored x 8 warps, as
                          // released by its epilogue warps (zeroed by the margins step)
  uint32_t ahead_next;    // far-forming launch: chunks of the rows two iterations ahead
                          // taken by its producers (zeroed by the gather kernel)
};
static_assert(sizeof(Ctrl) <= 512, "control block");

// Byte layout of the workspace for one (data, params) pair.
struct Layout {
  int64_t S, ldY, gram_elems;
  int upd_ctas;
  size_t off_idx, off_r, off_yY, off_alpha, off_far, off_Y, off_G, off_upd, off_loss;
  size_t off_Y2, off_G2, off_idx2, off_yY2;  // 0: no second buffers
  size_t off_Y3, off_idx3, off_yY3;  // third row buffers (rows gathered two ahead; 0: none)
  // second recurrence state (with the third row buffers): control block, counters area,
  // margins, alpha, far sums and far partials of the odd iterations of casgd_train
  size_t off_ctrl2, off_cnt2, off_r2, off_alpha2, off_far2, off_fpart2;
  size_t off_fpart;  // far partial sums FP32[S][s * npb] of the far-forming Gram (0: none)
  size_t total;
};

// with_G: false for the feature-sharded calls, whose G lives in the caller's exchange
// buffer
Layout make_layout(int64_t n, int32_t b, int32_t s, uint32_t flags, int num_sms,
                   bool with_G = true);

inline int64_t gram_elems(int64_t b, int64_t s, bool diag) {
  int64_t nblk = diag ? s * (s + 1) / 2 : s * (s - 1) / 2;
  return nblk * b * b;
}

__host__ __device__ inline int64_t packed_offset(int64_t j, int64_t t, int64_t b, bool diag) {
  return (diag ? (j * (j + 1) / 2 + t) : (j * (j - 1) / 2 + t)) * b * b;
}

// Blocks before block row j in the band layout of band width B: sum over j' < j of
// min(j', B), plus one diagonal block per row with diag.
__host__ __device__ inline int64_t band_blocks_before(int64_t j, int64_t B, bool diag) {
  const int64_t lower = j <= B ? j * (j - 1) / 2 : B * (B - 1) / 2 + (j - B) * B;
  return lower + (diag ? j : 0);
}

// Offset (elements) of block (j, t) of G in one of two layouts.  gB = 0: the packed
// block-lower layout (every block t < j, or t <= j with diag; j ascending, then t).
// gB = B > 0: the band layout the far-forming Gram keeps internally -- only the blocks
// the recurrence reads from memory, t = j - min(j, B) .. j-1 ascending, then G_{j,j}
// with diag -- so its buffers grow with s * B instead of s^2 / 2.  Each block b x b,
// row-major.
__host__ __device__ inline int64_t g_block_offset(int64_t j, int64_t t, int64_t b, bool diag,
                                                  int gB) {
  if (gB == 0) return packed_offset(j, t, b, diag);
  const int64_t nb = j < gB ? j : gB;
  return (band_blocks_before(j, gB, diag) + (t - (j - nb))) * b * b;
}

// Floats of G in either layout (gB as above).
inline int64_t g_layout_elems(int64_t b, int64_t s, bool diag, int gB) {
  if (gB == 0) return gram_elems(b, s, diag);
  return band_blocks_before(s, gB, diag) * b * b;
}

// Column tiles (256 wide) that the paired-SM Gram computes for its 256-row group g:
// those holding a needed entry (column block < row block, or <= with the diagonal) of
// the group's last row, which needs the most.
__host__ __device__ inline int pair_group_tiles(int64_t S, int64_t b, bool diag, int g) {
  int64_t last = (int64_t)g * 256 + 255;
  if (last > S - 1) last = S - 1;
  const int64_t jmax = last / b;
  const int64_t lim = b * (diag ? jmax + 1 : jmax);  // columns < lim are needed
  const int64_t tc = (S + 255) / 256;
  const int64_t c = (lim + 255) / 256;
  return (int)(c < tc ? c : tc);
}

// Band width B of the inner recurrence: phase j adds the blocks t = j-B .. j-1 itself
// (their rows of G in a chain lane's registers), the far blocks t < j-B come from
// partial sums formed off the critical path.  As many blocks as a lane holds: 3 for
// b <= 256, 2 for b <= 512, else 1 (and 1 when b is not a multiple of 4).
__host__ __device__ inline int band_width(int64_t b) {
  if (b % 4 != 0) return 1;
  const int64_t nk = (b + 127) / 128;
  return nk <= 2 ? 3 : nk <= 4 ? 2 : 1;
}

// The paired-SM Gram that forms the far sums itself (b a multiple of 256): tiles of
// its 256-row group g that it stores into G -- the band blocks t = j-B .. j-1 and, on
// request, the diagonal block, b/256 column tiles each.
__host__ __device__ inline int far_gram_stored_tiles(int64_t b, bool diag, int g) {
  const int nb = (int)(b / 256);
  const int j = g / nb;
  const int B = band_width(b);
  return nb * ((j < B ? j : B) + (diag ? 1 : 0));
}

// Far partial sums per row and block t of the far-forming Gram: the column tiles of a
// block (b/256) are split into npb groups, each group's tiles summed into one partial
// by one unit of work.  As many groups as keep a row's partials (s-1-B far blocks at
// most) within the 64 a recurrence warp adds (two per lane): finer units spread the
// partials that phase j waits on over more SMs.
__host__ __device__ inline int far_partials_per_block(int64_t b, int s) {
  const int nb = (int)(b / 256);
  int nfb = s - 1 - band_width(b);
  if (nfb < 1) nfb = 1;
  for (int npb = nb; npb > 1; --npb)
    if (nb % npb == 0 && npb * nfb <= 64) return npb;
  return 1;
}

// Row parts of a block in the update fused into the recurrence's launch: units (block,
// 64-column chunk, row part) with at least ~32 units per block (the last block's units
// run after the chain and set the launch's tail; every unit has a fixed latency, so more
// units than the groups clear while the chain runs lengthen it), parts of at least 64
// rows.  Used where the far sums come from the Gram (the bulk groups only update).
__host__ __device__ inline int upd_row_parts(int64_t b, int64_t ldY) {
  const int64_t nchunk = (ldY / 8 + 7) / 8;
  int64_t R = (32 + nchunk - 1) / nchunk;
  const int64_t cap = b / 64 > 1 ? b / 64 : 1;
  if (R > cap) R = cap;
  return (int)(R < 1 ? 1 : R);
}

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// x rounded to the nearest BF16 value (ties to even), as FP32 (CASGD_FLAG_G_BF16)
__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// SplitMix64 output number `counter` of the stream started at state `seed`.
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t counter) {
  uint64_t z = seed + (counter + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ int32_t sample_row(uint64_t seed, uint64_t counter, uint32_t m) {
  uint64_t h = splitmix64_at(seed, counter);
  return (int32_t)(((h >> 32) * (uint64_t)m) >> 32);
}

// Sampling without replacement: counter c is position c mod m of epoch c div m of a
// keyed pseudorandom permutation of [0, m).  The permutation is a four-round balanced
// Feistel network on d-bit values (Luby & Rackoff 1988; d the smallest even width with
// 2^d >= m, at least 2), its round function the low d/2 bits of SplitMix64 output
// number R of the stream started at the round key, the key of epoch e and round r
// being SplitMix64 output number 4e + r of the stream started at seed xor
// 0x6A09E667F3BCC908; values outside [0, m) are walked along their cycle until they
// fall inside (Black & Rogaway 2002), which ends because the start lies on the cycle.
constexpr uint64_t kPermSeedXor = 0x6A09E667F3BCC908ull;
__host__ __device__ inline int perm_width(int64_t m) {
  int d = 2;
  while ((int64_t(1) << d) < m) d += 2;
  return d;
}

__device__ __forceinline__ uint64_t feistel4(uint64_t x, int h, const uint64_t (&key)[4]) {
  const uint64_t mask = (1ull << h) - 1ull;
  uint64_t L = x >> h, R = x & mask;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint64_t t = L ^ (splitmix64_at(key[r], R) & mask);
    L = R;
    R = t;
  }
  return (L << h) | R;
}

// d = perm_width(m)
__device__ __forceinline__ int32_t permuted_row(uint64_t seed, uint64_t counter, uint32_t m,
                                                int d) {
  const uint64_t e = counter / m;
  const uint64_t q = counter - e * m;
  uint64_t key[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) key[r] = splitmix64_at(seed ^ kPermSeedXor, 4ull * e + r);
  uint64_t y = feistel4(q, d / 2, key);
  while (y >= m) y = feistel4(y, d / 2, key);
  return (int32_t)y;
}

// The row of sampler counter `counter`: with replacement (perm_d == 0) or the permuted
// draw (perm_d = perm_width(m)).
__device__ __forceinline__ int32_t draw_row(uint64_t seed, uint64_t counter, uint32_t m,
                                            int perm_d) {
  return perm_d ? permuted_row(seed, counter, m, perm_d) : sample_row(seed, counter, m);
}

// l'(z, y) for the three GLMs, FP32.
__device__ __forceinline__ float loss_deriv(int kind, float z, float y) {
  if (kind == CASGD_LOGISTIC) return -y / (1.0f + expf(y * z));
  if (kind == CASGD_LSQ) return z - y;
  return expf(z) - y;
}

// l(z, y), FP32; the logistic form avoids overflow: log(1+e^{-t}) = max(-t,0) + log1p(e^{-|t|}).
__device__ __forceinline__ float loss_value(int kind, float z, float y) {
  if (kind == CASGD_LOGISTIC) {
    float t = y * z;
    return fmaxf(-t, 0.0f) + log1pf(expf(-fabsf(t)));
  }
  if (kind == CASGD_LSQ) {
    float d = z - y;
    return 0.5f * d * d;
  }
  return expf(z) - y * z;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

// Programmatic dependent launch.  A kernel launched with the programmatic stream
// serialization attribute may be scheduled before the previous kernel of its stream has
// finished; wait_prior_grid() returns once that kernel has completed and its memory
// operations are visible, so it precedes every global access of such a kernel.  For a
// kernel launched without the attribute it returns at once.  allow_next_grid() lets the
// next kernel of the stream be scheduled (it still waits for this one's completion at
// its own wait_prior_grid()); without it that happens when this grid's blocks exit.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ launchers
// Rows of an outer iteration read straight from X (the far-forming launch that gathers
// its own operands): row p of the iteration whose first sampler counter is c0 is row
// draw_row(seed, c0 + p, m, perm_d) of X (pitch ld elements).
struct RowSource {
  const uint16_t* X;
  int64_t ld;
  uint32_t m;
  uint64_t seed;
  int perm_d;
};
// A sampler counter that names no rows (a launch without the next iteration's band).
constexpr uint64_t kNoRows = ~0ull;

// Launch parameters of the kernels one call launches repeatedly (occupancy results, with
// the dynamic shared memory attribute set), found once per call: the queries cost host
// time, and in casgd_train's loop that time would fall between the launches.  Owned by
// the calling C-ABI function, never global.
struct LaunchCache {
  static constexpr int kSlots = 16;
  const void* fn[kSlots] = {};
  int value[kSlots] = {};
  int n = 0;
  bool find(const void* f, int& v) const {
    for (int i = 0; i < n; ++i)
      if (fn[i] == f) {
        v = value[i];
        return true;
      }
    return false;
  }
  void put(const void* f, int v) {
    if (n < kSlots) {
      fn[n] = f;
      value[n] = v;
      ++n;
    }
  }
};

struct Ctx {
  cudaStream_t stream;
  int num_sms;
  int64_t launches;
  LaunchCache* cache = nullptr;
  // launch the gather and the shared launch of an outer iteration (casgd_outer_step,
  // casgd_train) with programmatic stream serialization: each may be scheduled while
  // the one before it ends, and waits for it in wait_prior_grid() before touching memory
  bool pdl = false;
};

// Adds the programmatic stream serialization attribute to cfg when c.pdl (attr must
// have room for one more entry).
inline void add_pdl_attr(const Ctx& c, cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr) {
  if (!c.pdl) return;
  attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  ++cfg.numAttrs;
}

// query(&v) once per kernel `fn` and Ctx cache (every time without a cache).
template <class Query>
cudaError_t cached_query(Ctx& c, const void* fn, Query query, int& v) {
  if (c.cache && c.cache->find(fn, v)) return cudaSuccess;
  const cudaError_t e = query(v);
  if (e == cudaSuccess && c.cache) c.cache->put(fn, v);
  return e;
}

cudaError_t launch_store_bf16(const float* src, int64_t m, int64_t n, int64_t ld_src,
                              uint16_t* dst, int64_t ld_dst, Ctx& c);
// dst[i] = the BF16 bits of src[i] (values already BF16-representable: exact)
cudaError_t launch_bf16_bits(const float* src, int64_t count, uint16_t* dst, Ctx& c);
// dst[i] = src[i] rounded once to BF16 (as FP32), or src[i] itself (fp32): the summed
// partial margins of a feature-sharded outer iteration as the recurrence reads them
cudaError_t launch_sharded_margins(const float* src, int64_t count, bool fp32, float* dst,
                                   Ctx& c);
// permuted: without replacement (per-epoch permutation), else with replacement
cudaError_t launch_sample(int64_t m, int64_t count, uint64_t seed, uint64_t counter0,
                          bool permuted, int32_t* idx, Ctx& c);
// mode: GATHER_AND_MARGINS (sampled rows into Y, labels, indices, BF16 margins and the
// recurrence's reset), GATHER_ONLY (rows, labels, indices), MARGINS_ONLY (margins of
// the rows in Y and the reset).  The margins are bit-identical in every mode.  The reset
// fills alpha, far and (fpart non-null) each row's far partials t < j-B with
// kAlphaPending.  GATHER_ONLY with Y null: the indices and labels only (the rows are read
// from X by the launch that gathers its own operands).
enum { GATHER_AND_MARGINS = 0, GATHER_ONLY = 1, MARGINS_ONLY = 2 };
cudaError_t launch_gather(const casgd_data_t& d, const casgd_params_t& p, const float* w,
                          uint64_t k, const int32_t* idx_in, int32_t* idx, uint16_t* Y,
                          int64_t ldY, float* r, float* yY, float* alpha, float* far,
                          float* fpart, Ctrl* ctrl, uint32_t* slab, int mode, Ctx& c);
// Rows of iteration k_rows (into Yg, yY, idx; skipped without `gather`; Yg null: the
// indices and labels only) and, in the same
// launch, this iteration's recurrence reset without margins (alpha, far, r and the far
// partials pending; counters and queues zeroed): for the far-forming Gram, whose launch
// forms the margins itself.
cudaError_t launch_gather_reset(const casgd_data_t& d, const casgd_params_t& p, uint64_t k_rows,
                                const int32_t* idx_in, int32_t* idx, uint16_t* Yg, float* yY,
                                bool gather, int64_t ldY, float* r, float* alpha, float* far,
                                float* fpart, Ctrl* ctrl, uint32_t* slab, Ctx& c);
// GATHER_ONLY for iteration k_next (into Y_next, yY_next, idx_next) and MARGINS_ONLY for
// the rows in Y, in one launch (the two touch disjoint buffers).
cudaError_t launch_gather_next_margins(const casgd_data_t& d, const casgd_params_t& p,
                                       const float* w, uint64_t k_next, int32_t* idx_next,
                                       uint16_t* Y_next, float* yY_next, const uint16_t* Y,
                                       int64_t ldY, float* r, float* alpha, float* far,
                                       float* fpart, Ctrl* ctrl, uint32_t* slab, Ctx& c);
// g_bf16: every stored entry rounded to BF16 (CASGD_FLAG_G_BF16)
cudaError_t launch_gram_simt(const uint16_t* Y, int64_t S, int64_t n, int64_t ldY, int b,
                             int s, bool diag, bool g_bf16, float* G, Ctx& c);
bool gram_tc_supported(int64_t S, int64_t n, int b);
cudaError_t launch_gram_tc(const uint16_t* Y, int64_t S, int64_t n, int64_t ldY, int b,
                           int s, uint32_t flags, int mode, float* G, Ctrl* ctrl,
                           uint32_t timeout_us, Ctx& c);
// The recurrence with the weight update fused: partial rows part[j * R + rq][:] (ldY
// floats) per block j and row part rq (R = upd_row_parts), added to w (FP32[n]) by the
// last unit of each 64-column chunk.  counters: the workspace's counters area
// (timeline_of).
cudaError_t launch_recur(const float* G, const float* r, const float* yY, float* alpha,
                         float* far, uint32_t* counters, int b, int s, float eta, int loss,
                         uint32_t flags, uint32_t timeout_us, Ctrl* ctrl, const uint16_t* Y,
                         int64_t ldY, int64_t n, float* part, float* w, Ctx& c);
// The paired-SM Gram (of rows Yg into Gg) and the recurrence (with the fused update
// stage, on G and Y) in one launch.  next == false: the same iteration (Yg == Y,
// Gg == G); the Gram's epilogue releases per-32-row counters `slab` (zeroed by the
// margins step) that the recurrence acquires before it reads rows of G.  next == true:
// the Gram is the next iteration's and G is complete.  fpart (b a multiple of 256): the
// Gram forms the far sums itself into fpart FP32[S][s * npb] (npb =
// far_partials_per_block; entries (j-B) * npb of each row of block j filled with
// kAlphaPending by the margins step), which the recurrence adds, from its tiles of this
// iteration (rows Y), and stores only band blocks (and the diagonal on request): with
// next == false this iteration's (Yg == Y, Gg == G), with next == true the next
// iteration's (rows Yg into Gg; Yg null: none) while the recurrence reads this
// iteration's complete band from G.
// cudaErrorNotSupported when the shape does not fit the fused kernel (the caller then
// launches them separately).
bool gram_recur_fused_supported(int64_t S, int64_t n, int b);
bool far_gram_supported(int64_t S, int64_t n, int b);
// The band blocks (and the diagonal on request) of the far-forming Gram alone, from rows
// Y into G (band layout): the band of a run's first iteration.
// rs (non-null): the rows are read from X instead of Y (Y unused), those of the iteration
// whose first sampler counter is ctr.
cudaError_t launch_gram_band(const uint16_t* Y, float* G, int64_t S, int64_t n, int64_t ldY,
                             int b, int s, uint32_t flags, Ctrl* ctrl, uint32_t timeout_us,
                             const RowSource* rs, uint64_t ctr, Ctx& c);
// Rows that a far-forming launch gathers for a later iteration once its own Gram work is
// done (launch_gram_recur's `ahead`): rows ctr .. ctr+S-1 of the sampler (draw_row with
// seed, m, perm_d) of X (pitch ld) into Y (pitch ldY; columns n .. ldY-1 written as
// zeros); n % 8 == 0 for rows wider than 64 columns (ahead_rows_supported).  Their
// labels and indices are gathered separately.
struct AheadRows {
  const uint16_t* X;
  int64_t ld;
  uint32_t m;
  uint64_t seed;
  int perm_d;
  uint64_t ctr;
  uint16_t* Y;
};
// The state of the next outer iteration, which a far-forming launch of casgd_train
// resets while it runs (the loop's launches alternate between two such sets, so no
// launch between them is needed): margins r, alpha and far sums to pending (every row
// p < S), far partials fpart to pending (row p's first ((p / fb) - fB) * fnp of fs),
// the counters of q (next_unit, upd_next, band_done, ahead_next) and the update's
// column and block counters (nchunk and s * nchunk from `counters`) to zero; and the
// indices and labels of the iteration after it (sampler counters ctr .. ctr+S-1 of X's
// m rows into idx and yY; none when yY is null).
struct NextSet {
  float* r;
  float* alpha;
  float* far;
  float* fpart;
  Ctrl* q;
  uint32_t* counters;
  int fs, fb, fB, fnp, nchunk, s;
  const float* y;
  float* yY;
  int32_t* idx;
  uint64_t seed, ctr;
  uint32_t m;
  int perm_d;
};
// Whether launch_gram_recur can gather rows ahead for these shapes.
bool ahead_rows_supported(int64_t n, int64_t ldY);
// own_margins (with fpart): the launch forms the margins itself (r reset to pending by
// launch_gather_reset) from Y and w; w receives the update once the last phase is done.
// g_band (with fpart): Gg and G use the band layout (g_block_offset with gB =
// band_width(b)), else the packed block-lower layout.  rs (non-null, with fpart): every
// row is read from X instead of Yg / Y -- the Gram's own rows those of the iteration
// starting at sampler counter ctr_g, this iteration's (far tiles, margins, update) those
// starting at ctr_f.  ahead (non-null, with fpart and Yg, ahead_rows_supported): the
// launch also gathers those rows (into buffers that none of its other work touches).
// q / cnt (non-null): this iteration's counters and update counters area instead of
// ctrl's and slab's (slab still holds the trace).  nx (non-null, with fpart and Yg): the
// launch also resets that state set.
cudaError_t launch_gram_recur(const uint16_t* Yg, float* Gg, bool next, int64_t S, int64_t n,
                              int64_t ldY, int b, int s, float eta, int loss, uint32_t flags,
                              const float* G, const uint16_t* Y, float* r,
                              const float* yY, float* alpha, float* far, uint32_t* slab,
                              float* fpart, float* part, float* w, bool own_margins, Ctrl* ctrl,
                              uint32_t timeout_us, bool g_band, const RowSource* rs,
                              uint64_t ctr_g, uint64_t ctr_f, const AheadRows* ahead, Ctrl* q,
                              uint32_t* cnt, const NextSet* nx, Ctx& c);
cudaError_t launch_update_reduce(const float* part, int upd_ctas, int64_t n, int64_t ldY,
                                 float* w, Ctrl* ctrl, Ctx& c);
cudaError_t launch_update(const uint16_t* Y, const float* alpha, int64_t S, int64_t n,
                          int64_t ldY, float* w, float* part, int upd_ctas, Ctrl* ctrl,
                          Ctx& c);
int loss_ctas(int num_sms);
// FP32 plain minibatch SGD (k_sgd.cu); ws: sgd_workspace_bytes(b), 256-byte aligned.
size_t sgd_workspace_bytes(int b);
cudaError_t launch_sgd_fp32(const float* X, int64_t m, int64_t n, int64_t ld, const float* y,
                            const casgd_params_t& p, float* w, uint64_t q0, int steps, void* ws,
                            Ctx& c);
cudaError_t launch_loss(const casgd_data_t& d, int loss, const float* w, double* part,
                        double* out_dev, Ctrl* ctrl, Ctx& c);

}  // namespace casgd
