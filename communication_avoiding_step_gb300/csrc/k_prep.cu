// Steps a1 (sampling), a2 (gather) and a4 (BF16 margins), plus the BF16 storage step.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the recipe stores the input matrix and the margin vector in low
// precision; each outer iteration works on s minibatches of b rows.
//
// The gather writes Y (S x ldY BF16, ldY = n rounded up to 64, or to 8 below 128
// columns, zero padded) once per
// outer iteration (in a multi-iteration run, one iteration ahead of its margins).  Y is small next to X and stays L2-resident for the Gram and update
// kernels; it lets the Gram kernel fetch tiles with plain tiled TMA copies.
#include <cuda_bf16.h>

#include "casgd_internal.cuh"
#include "ptx_async.cuh"

namespace casgd {

namespace {

__global__ void store_bf16_kernel(const float* __restrict__ src, int64_t m, int64_t n,
                                  int64_t ld_src, uint16_t* __restrict__ dst, int64_t ld_dst) {
  const int64_t vec_per_row = ld_dst / 8;
  const int64_t total = m * vec_per_row;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = v / vec_per_row;
    const int64_t c0 = (v - row * vec_per_row) * 8;
    const float* s = src + row * ld_src;
    uint32_t packed[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int64_t c = c0 + 2 * h;
      const float a = (c < n) ? s[c] : 0.0f;
      const float b = (c + 1 < n) ? s[c + 1] : 0.0f;
      packed[h] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
    }
    *reinterpret_cast<uint4*>(dst + row * ld_dst + c0) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

__global__ void bf16_bits_kernel(const float* __restrict__ src, int64_t count,
                                 uint16_t* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(src[i]));
}

// The summed margins of a feature-sharded outer iteration (FP32 partial sums, added
// over the ranks) as the recurrence reads them: rounded once to BF16, or kept (fp32).
__global__ void sharded_margins_kernel(const float* __restrict__ src, int64_t count, bool fp32,
                                       float* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = fp32 ? src[i] : round_bf16(src[i]);
}

__global__ void sample_kernel(uint32_t m, int64_t count, uint64_t seed, uint64_t counter0,
                              int perm_d, int32_t* __restrict__ idx) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    idx[i] = draw_row(seed, counter0 + (uint64_t)i, m, perm_d);
}

// One group of G lanes (G a power of two <= 32) per row of Y.  Lane g reads the 16-byte
// vectors g, g+G, ... of the row and accumulates their FP32 dot with w; the group then
// reduces with shuffles and its first lane stores the BF16 margin.  Variants:
//   kCopy && kMargin   gather the sampled rows of X into Y and form the margins (one
//                      outer iteration at a time);
//   kCopy && !kMargin  gather only (Y, labels, indices) for an iteration whose margins
//                      are formed later, once its starting w is known;
//   !kCopy && kMargin  margins of rows already in Y.
// The margin arithmetic is the same in every variant (same lanes, vector order and
// shuffle tree), so a margin does not depend on which variant formed it.  Variants with
// kMargin also prepare the recurrence that follows (queues, counters, pending values).
struct RowArgs {
  const uint16_t* X;
  const float* y;
  int64_t m, n, ld;
  const float* w;
  int64_t S;
  uint64_t seed, counter0;
  const int32_t* idx_in;
  int32_t* idx_out;
  uint16_t* Y;
  int64_t ldY;
  float* r;  // margins: BF16-rounded FP32 values, or the FP32 sums (r_fp32)
  float* yY;
  float* alpha;
  float* far;
  float* fpart;  // far partials [S][fs] of the far-forming Gram (null: not used)
  int fb, fs, fB, fnp;  // b, row stride s * npb, band width, partials per block
  int steps;            // s
  Ctrl* ctrl;
  uint32_t* slab;
  int G;
  int perm_d;  // sampling: 0 with replacement, else perm_width(m) (per-epoch permutation)
  bool r_fp32;  // margins kept in FP32 (CASGD_FLAG_MARGINS_FP32), r then holds floats
};

// The recurrence's per-step reset (one CTA).
__device__ void reset_recurrence(const RowArgs& a) {
  if (threadIdx.x == 0) {
    a.ctrl->next_unit = 0;
    a.ctrl->upd_next = 0;
    a.ctrl->band_done = 0;
    a.ctrl->ahead_next = 0;
    a.ctrl->abort = (a.ctrl->status & ST_TIMEOUT) ? 1u : 0u;  // stays set after a timeout
  }
  const int64_t nslab = (a.S + 255) / 256 * 8;  // the Gram's 32-row counters
  for (int64_t j = threadIdx.x; j < nslab; j += blockDim.x) a.slab[j] = 0;
  const int64_t nchunk = (a.ldY + 63) / 64;
  uint32_t* chunks = upd_chunk_counters(a.slab);  // the update's column counters
  for (int64_t j = threadIdx.x; j < nchunk; j += blockDim.x) chunks[j] = 0;
  uint32_t* blocks = upd_block_counters(a.slab);  // and its (block, chunk) counters
  for (int64_t j = threadIdx.x; j < a.steps * nchunk; j += blockDim.x) blocks[j] = 0;
  uint64_t* summary = timeline_of(a.slab) + (int64_t)kMaxS * 4;  // profiling summary row
  if (threadIdx.x < 4) summary[threadIdx.x] = 0;
}

// The rows of block `blk` (8 warps, 32/G rows per warp).
template <bool kCopy, bool kMargin>
__device__ __forceinline__ void gather_rows(const RowArgs& a, int64_t blk) {
  const int G = a.G;
  const int lane = threadIdx.x & 31;
  const int g = lane & (G - 1);
  const int rows_per_warp = 32 / G;
  const int64_t p = (blk * (blockDim.x >> 5) + (threadIdx.x >> 5)) * rows_per_warp + lane / G;
  const int64_t nvec = a.ldY / 8;
  const bool w_vec = (reinterpret_cast<uintptr_t>(a.w) & 15u) == 0;
  // Every lane of the warp must reach the shuffles, so out-of-range rows only mask.
  const bool live = p < a.S;
  int32_t row = 0;
  bool valid = !kCopy;  // rows already in Y are valid
  if (kCopy && live) {
    if (a.idx_in) {
      row = a.idx_in[p];
      valid = (row >= 0 && (int64_t)row < a.m);
      if (!valid && g == 0) atomicOr(&a.ctrl->status, ST_BAD_INDEX);
    } else {
      row = draw_row(a.seed, a.counter0 + (uint64_t)p, (uint32_t)a.m, a.perm_d);
      valid = true;
    }
  }
  float acc = 0.0f;
  // (a.Y null: the rows are not copied -- the Gram and the units read them from X --
  // only the indices and labels are gathered)
  if (live && a.Y) {
    const uint16_t* xr = kCopy ? a.X + (int64_t)(valid ? row : 0) * a.ld : a.Y + p * a.ldY;
    uint16_t* yr = a.Y + p * a.ldY;
    // kBatch 16-byte loads of the row are issued before any of them is used.
    constexpr int kBatch = 8;
    for (int64_t v0 = g; v0 < nvec; v0 += (int64_t)G * kBatch) {
      uint4 qv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t v = v0 + (int64_t)u * G;
        // vectors past n are never read (X holds only round_up(n, 8) columns of data);
        // Y's padding is written as zeros
        qv[u] = (valid && v < nvec && v * 8 < a.n)
                    ? __ldg(reinterpret_cast<const uint4*>(xr + v * 8))
                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t v = v0 + (int64_t)u * G;
        if (v >= nvec) break;
        const int64_t c0 = v * 8;
        uint32_t parts[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
        float wv[8];
        if (kMargin) {
          if (w_vec && c0 + 8 <= a.n) {
            const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.w + c0));
            const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.w + c0 + 4));
            wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
            wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) wv[e] = c0 + e < a.n ? __ldg(a.w + c0 + e) : 0.0f;
          }
        }
        if (c0 + 8 <= a.n) {  // the whole vector holds features: no masking
          if (kMargin) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              acc = fmaf(__uint_as_float(parts[h] << 16), wv[2 * h], acc);
              acc = fmaf(__uint_as_float(parts[h] & 0xFFFF0000u), wv[2 * h + 1], acc);
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int64_t c = c0 + 2 * h;
            uint32_t lo = parts[h] & 0xFFFFu, hi = parts[h] >> 16;
            if (c >= a.n) lo = 0;
            if (c + 1 >= a.n) hi = 0;
            parts[h] = lo | (hi << 16);
            if (kMargin) {
              if (c < a.n) acc = fmaf(bf16_bits_to_float(lo), wv[2 * h], acc);
              if (c + 1 < a.n) acc = fmaf(bf16_bits_to_float(hi), wv[2 * h + 1], acc);
            }
          }
        }
        if (kCopy)
          *reinterpret_cast<uint4*>(yr + c0) = make_uint4(parts[0], parts[1], parts[2], parts[3]);
      }
    }
  }
  if (kMargin)
    for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
  if (kMargin && live && a.fpart) {  // the row's far partials t < j - B, spread over its lanes
    const int nfar = ((int)(p / a.fb) - a.fB) * a.fnp;
    for (int t = g; t < nfar; t += G) a.fpart[p * a.fs + t] = __uint_as_float(kAlphaPending);
  }
  if (live && g == 0) {
    if (kMargin) {
      a.r[p] = a.r_fp32 ? acc : round_bf16(acc);
      a.alpha[p] = __uint_as_float(kAlphaPending);  // the recurrence waits on these values
      a.far[p] = __uint_as_float(kAlphaPending);
    }
    if (kCopy) {
      a.yY[p] = valid ? __ldg(a.y + row) : 0.0f;
      a.idx_out[p] = row;
    }
  }
}

template <bool kCopy, bool kMargin>
__global__ void __launch_bounds__(256) gather_kernel(RowArgs a) {
  wait_prior_grid();
  allow_next_grid();
  if (kMargin && blockIdx.x == 0) reset_recurrence(a);
  gather_rows<kCopy, kMargin>(a, blockIdx.x);
}

// The recurrence's per-row reset where the margins are formed in the recurrence's launch
// (the far-forming Gram): alpha, far, r and each row's far partials hold kAlphaPending.
// Block `blk` of nr: a grid-stride pass over the S rows, then one warp per row over its
// far-partial slots t < (j-B) * npb, which are contiguous (the stores coalesce).
__device__ void reset_rows(const RowArgs& a, int64_t blk, int64_t nr) {
  const float pend = __uint_as_float(kAlphaPending);
  const int64_t stride = nr * blockDim.x;
  for (int64_t p = blk * blockDim.x + threadIdx.x; p < a.S; p += stride) {
    a.alpha[p] = pend;
    a.far[p] = pend;
    a.r[p] = pend;
  }
  if (!a.fpart) return;
  const int lane = threadIdx.x & 31;
  const int64_t warps = nr * (blockDim.x >> 5);
  for (int64_t p = blk * (blockDim.x >> 5) + (threadIdx.x >> 5); p < a.S; p += warps) {
    const int nfar = ((int)(p / a.fb) - a.fB) * a.fnp;
    float* row = a.fpart + p * a.fs;
    for (int t = lane; t < nfar; t += 32) row[t] = pend;
  }
}

// Wide rows (ldY*2 >= 512 bytes) of block `blk`, RB of them, moved whole by bulk copies:
// the indices and labels first (one thread per row), then one cp.async.bulk per valid
// row from X into shared memory (the row's round_up(n, 8) columns), the columns from n on
// zeroed there (and the whole row for an index outside [0, m)), and one bulk store per
// row into Y.  The bytes in flight cost no registers, so a CTA keeps RB rows moving.
// Every wait is bounded (a timeout records ST_TIMEOUT).
__device__ void gather_rows_bulk(const RowArgs& a, int64_t blk, int RB, uint8_t* sm) {
  __shared__ uint64_t bar;
  __shared__ int32_t s_row[256];
  const int64_t p0 = blk * RB;
  const int nrow = (int)(a.S - p0 < RB ? a.S - p0 : RB);
  const uint32_t pitch = (uint32_t)(a.ldY * 2);            // bytes per row in Y and in sm
  const uint32_t ncopy = (uint32_t)(((a.n + 7) / 8) * 16);  // bytes of data per row
  int32_t row = 0;
  bool valid = false;
  if ((int)threadIdx.x < nrow) {
    const int64_t p = p0 + threadIdx.x;
    if (a.idx_in) {
      row = a.idx_in[p];
      valid = row >= 0 && (int64_t)row < a.m;
      if (!valid) atomicOr(&a.ctrl->status, ST_BAD_INDEX);
    } else {
      row = draw_row(a.seed, a.counter0 + (uint64_t)p, (uint32_t)a.m, a.perm_d);
      valid = true;
    }
    s_row[threadIdx.x] = valid ? row : -1;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // the rows' copies first ...
    uint32_t total = 0;
    for (int i = 0; i < nrow; ++i) total += s_row[i] >= 0 ? ncopy : 0u;
    mbar_expect_tx(&bar, total);
    for (int i = 0; i < nrow; ++i)
      if (s_row[i] >= 0)
        bulk_load(sm + (size_t)i * pitch, a.X + (int64_t)s_row[i] * a.ld, ncopy, &bar);
  }
  if ((int)threadIdx.x < nrow) {  // ... then the labels and indices, while the rows land
    const int64_t p = p0 + threadIdx.x;
    a.yY[p] = valid ? __ldg(a.y + row) : 0.0f;
    a.idx_out[p] = row;
  }
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(&bar, 0)) {
    if (globaltimer_ns() - t0 > 1000000000ull) {  // (copies of this CTA alone: not expected)
      if (threadIdx.x == 0) atomicOr(&a.ctrl->status, ST_TIMEOUT);
      // keep the shared memory until the copies land (bounded), store nothing
      while (!mbar_try_wait(&bar, 0) && globaltimer_ns() - t0 < 2000000000ull) {
      }
      return;
    }
  }
  // zero the columns that are not data: from n on (all of an invalid row)
  for (int i = 0; i < nrow; ++i) {
    uint16_t* r = reinterpret_cast<uint16_t*>(sm + (size_t)i * pitch);
    const int64_t c0 = s_row[i] >= 0 ? a.n : 0;
    for (int64_t cc = c0 + threadIdx.x; cc < a.ldY; cc += blockDim.x) r[cc] = 0;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the bulk stores
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < nrow; ++i)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       reinterpret_cast<uint64_t>(a.Y + (p0 + i) * a.ldY)),
                   "r"(smem_u32(sm + (size_t)i * pitch)), "r"(pitch)
                   : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    // the stores have read shared memory before the CTA leaves (their writes complete
    // with the grid, before the next launch's wait for it returns)
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
}

// The per-row part of the reset for rows [p_lo, p_hi) (as reset_rows).
__device__ void reset_row_range(const RowArgs& a, int64_t p_lo, int64_t p_hi) {
  const float pend = __uint_as_float(kAlphaPending);
  for (int64_t p = p_lo + threadIdx.x; p < p_hi; p += blockDim.x) {
    a.alpha[p] = pend;
    a.far[p] = pend;
    a.r[p] = pend;
  }
  if (!a.fpart) return;
  const int lane = threadIdx.x & 31;
  for (int64_t p = p_lo + (threadIdx.x >> 5); p < p_hi; p += blockDim.x >> 5) {
    const int nfar = ((int)(p / a.fb) - a.fB) * a.fnp;
    float* row = a.fpart + p * a.fs;
    for (int t = lane; t < nfar; t += 32) row[t] = pend;
  }
}

// Wide rows by bulk copies: block `blk` gathers rows [blk*rb, blk*rb + rb) of g and
// resets the same rows of this iteration's recurrence state (mg); block 0 also the
// counters and queues.  Few registers, so several blocks share an SM (their rows'
// bytes in flight add up).
__global__ void __launch_bounds__(256, 4) gather_bulk_reset_kernel(RowArgs g, RowArgs mg, int rb) {
  extern __shared__ __align__(128) uint8_t gather_smem[];
  wait_prior_grid();  // the previous launch reads the buffers this one writes
  allow_next_grid();  // the next launch may take SMs as this one's blocks leave
  const int64_t blk = blockIdx.x;
  if (blk == 0) reset_recurrence(mg);
  const int64_t p_lo = blk * rb;
  reset_row_range(mg, p_lo, p_lo + rb < mg.S ? p_lo + rb : mg.S);
  gather_rows_bulk(g, blk, rb, gather_smem);
}

// Blocks [0, nb_g) gather rows (g: the next iteration's, or this one's for a single
// step), the others reset this iteration's recurrence state (mg).
__global__ void __launch_bounds__(256) gather_reset_kernel(RowArgs g, RowArgs mg, int64_t nb_g) {
  wait_prior_grid();  // the previous launch reads the buffers this one writes
  allow_next_grid();  // the next launch may take SMs as this one's blocks leave
  if ((int64_t)blockIdx.x < nb_g) {
    gather_rows<true, false>(g, blockIdx.x);
  } else {
    const int64_t blk = (int64_t)blockIdx.x - nb_g;
    if (blk == 0) reset_recurrence(mg);
    reset_rows(mg, blk, (int64_t)gridDim.x - nb_g);
  }
}

// Two independent passes in one launch: blocks [0, nb_g) gather the next iteration's
// rows (g), the others form this iteration's margins (mg) from its rows already in Y.
__global__ void __launch_bounds__(256) gather_next_margins_kernel(RowArgs g, RowArgs mg,
                                                                  int64_t nb_g) {
  wait_prior_grid();
  allow_next_grid();
  if ((int64_t)blockIdx.x < nb_g) {
    gather_rows<true, false>(g, blockIdx.x);
  } else {
    if ((int64_t)blockIdx.x == nb_g) reset_recurrence(mg);
    gather_rows<false, true>(mg, (int64_t)blockIdx.x - nb_g);
  }
}

int pow2_at_least(int64_t v, int cap) {
  int g = 1;
  while (g < v && g < cap) g <<= 1;
  return g;
}

}  // namespace

cudaError_t launch_store_bf16(const float* src, int64_t m, int64_t n, int64_t ld_src,
                              uint16_t* dst, int64_t ld_dst, Ctx& c) {
  const int64_t total = m * (ld_dst / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)c.num_sms * 16) blocks = (int64_t)c.num_sms * 16;
  store_bf16_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(src, m, n, ld_src, dst, ld_dst);
  ++c.launches;
  return cudaGetLastError();
}

cudaError_t launch_bf16_bits(const float* src, int64_t count, uint16_t* dst, Ctx& c) {
  if (count == 0) return cudaSuccess;
  int64_t blocks = (count + 255) / 256;
  if (blocks > (int64_t)c.num_sms * 8) blocks = (int64_t)c.num_sms * 8;
  bf16_bits_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(src, count, dst);
  ++c.launches;
  return cudaGetLastError();
}

cudaError_t launch_sharded_margins(const float* src, int64_t count, bool fp32, float* dst,
                                   Ctx& c) {
  if (count == 0) return cudaSuccess;
  int64_t blocks = (count + 255) / 256;
  if (blocks > (int64_t)c.num_sms * 8) blocks = (int64_t)c.num_sms * 8;
  sharded_margins_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(src, count, fp32, dst);
  ++c.launches;
  return cudaGetLastError();
}

cudaError_t launch_sample(int64_t m, int64_t count, uint64_t seed, uint64_t counter0,
                          bool permuted, int32_t* idx, Ctx& c) {
  if (count == 0) return cudaSuccess;
  int64_t blocks = (count + 255) / 256;
  if (blocks > (int64_t)c.num_sms * 8) blocks = (int64_t)c.num_sms * 8;
  sample_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>((uint32_t)m, count, seed, counter0,
                                                        permuted ? perm_width(m) : 0, idx);
  ++c.launches;
  return cudaGetLastError();
}

namespace {

RowArgs row_args(const casgd_data_t& d, const casgd_params_t& p, const float* w, uint64_t k,
                 const int32_t* idx_in, int32_t* idx, uint16_t* Y, int64_t ldY, float* r,
                 float* yY, float* alpha, float* far, float* fpart, Ctrl* ctrl,
                 uint32_t* slab) {
  RowArgs a;
  a.X = static_cast<const uint16_t*>(d.X);
  a.y = d.y;
  a.m = d.m;
  a.n = d.n;
  a.ld = d.ld;
  a.w = w;
  a.S = (int64_t)p.b * p.s;
  a.seed = p.seed;
  a.counter0 = k * (uint64_t)a.S;
  a.idx_in = idx_in;
  a.idx_out = idx;
  a.Y = Y;
  a.ldY = ldY;
  a.r = r;
  a.yY = yY;
  a.alpha = alpha;
  a.far = far;
  a.fpart = fpart;
  a.fb = p.b;
  a.steps = p.s;
  a.fnp = far_partials_per_block(p.b, p.s);
  a.fs = p.s * a.fnp;
  a.fB = band_width(p.b);
  a.ctrl = ctrl;
  a.slab = slab;
  a.G = pow2_at_least(ldY / 8, 32);
  a.perm_d = (p.flags & CASGD_FLAG_SAMPLE_PERMUTED) ? perm_width(d.m) : 0;
  a.r_fp32 = (p.flags & CASGD_FLAG_MARGINS_FP32) != 0;
  return a;
}

// 256-thread blocks on c's stream, with the programmatic serialization attribute when
// c.pdl (attr: room for it)
cudaLaunchConfig_t plain_config(unsigned blocks, const Ctx& c, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  add_pdl_attr(c, cfg, attr);
  return cfg;
}

int64_t row_blocks(const RowArgs& a) {
  const int64_t rows_per_cta = 8 * (32 / a.G);
  return (a.S + rows_per_cta - 1) / rows_per_cta;
}

}  // namespace

cudaError_t launch_gather(const casgd_data_t& d, const casgd_params_t& p, const float* w,
                          uint64_t k, const int32_t* idx_in, int32_t* idx, uint16_t* Y,
                          int64_t ldY, float* r, float* yY, float* alpha, float* far,
                          float* fpart, Ctrl* ctrl, uint32_t* slab, int mode, Ctx& c) {
  RowArgs a = row_args(d, p, w, k, idx_in, idx, Y, ldY, r, yY, alpha, far, fpart, ctrl, slab);
  if (!Y && mode == GATHER_ONLY) a.G = 1;  // indices and labels only: one thread per row
  auto fn = mode == GATHER_AND_MARGINS ? gather_kernel<true, true>
            : mode == GATHER_ONLY      ? gather_kernel<true, false>
                                       : gather_kernel<false, true>;
  fn<<<(unsigned)row_blocks(a), 256, 0, c.stream>>>(a);
  ++c.launches;
  return cudaGetLastError();
}

cudaError_t launch_gather_reset(const casgd_data_t& d, const casgd_params_t& p, uint64_t k_rows,
                                const int32_t* idx_in, int32_t* idx, uint16_t* Yg, float* yY,
                                bool gather, int64_t ldY, float* r, float* alpha, float* far,
                                float* fpart, Ctrl* ctrl, uint32_t* slab, Ctx& c) {
  RowArgs g = row_args(d, p, nullptr, k_rows, idx_in, idx, Yg, ldY, nullptr, yY, nullptr,
                       nullptr, nullptr, ctrl, slab);
  if (!Yg) g.G = 1;  // indices and labels only (the rows are read from X later): one thread per row
  // wide rows move by bulk copies, 32 KB of rows per block (at most 256)
  int rb = 0;
  if (Yg && ldY * 2 >= 512) {
    rb = (int)((32 * 1024) / (ldY * 2));
    if (rb < 1) rb = 1;
    if (rb > 256) rb = 256;
  }
  const RowArgs mg = row_args(d, p, nullptr, 0, nullptr, nullptr, nullptr, ldY, r, nullptr, alpha,
                              far, fpart, ctrl, slab);
  cudaLaunchAttribute attr[1];
  if (gather && rb > 0 && g.S == mg.S) {  // bulk rows; each block resets its own rows
    cudaLaunchConfig_t cfg = plain_config((unsigned)((g.S + rb - 1) / rb), c, attr);
    const size_t smem = (size_t)rb * ldY * 2;
    cfg.dynamicSmemBytes = smem;
    if (smem > 48 * 1024) {
      const cudaError_t ea = cudaFuncSetAttribute(gather_bulk_reset_kernel,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)smem);
      if (ea != cudaSuccess) return ea;
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gather_bulk_reset_kernel, g, mg, rb);
    ++c.launches;
    return e;
  }
  const int64_t nb = gather ? row_blocks(g) : 0;
  const int64_t work = mg.fpart ? mg.S * mg.fs : mg.S;  // reset slots
  int64_t nr = (work + 255) / 256;
  if (nr > (int64_t)c.num_sms * 4) nr = (int64_t)c.num_sms * 4;
  cudaLaunchConfig_t cfg = plain_config((unsigned)(nb + nr), c, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gather_reset_kernel, g, mg, nb);
  ++c.launches;
  return e;
}

cudaError_t launch_gather_next_margins(const casgd_data_t& d, const casgd_params_t& p,
                                       const float* w, uint64_t k_next, int32_t* idx_next,
                                       uint16_t* Y_next, float* yY_next, const uint16_t* Y,
                                       int64_t ldY, float* r, float* alpha, float* far,
                                       float* fpart, Ctrl* ctrl, uint32_t* slab, Ctx& c) {
  const RowArgs g = row_args(d, p, w, k_next, nullptr, idx_next, Y_next, ldY, nullptr, yY_next,
                             nullptr, nullptr, nullptr, ctrl, slab);
  const RowArgs mg = row_args(d, p, w, 0, nullptr, nullptr, const_cast<uint16_t*>(Y), ldY, r,
                              nullptr, alpha, far, fpart, ctrl, slab);
  const int64_t nb = row_blocks(g);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = plain_config((unsigned)(2 * nb), c, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gather_next_margins_kernel, g, mg, nb);
  ++c.launches;
  return e;
}

}  // namespace casgd
