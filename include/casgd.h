/*
 * casgd.h -- C ABI of the GB300 (sm_103a) mixed-precision CA-SGD library (libcasgd.so).
 *
 * Method: "Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
 * GPUs" (abstract).  Communication-avoiding SGD batches s minibatch steps of b rows
 * into one outer iteration whose only cross-process exchange is an sb x sb Gram
 * matrix; the recipe keeps the data matrix and the margins in BF16, forms the Gram
 * matrix from BF16 inputs with FP32 accumulation and runs the inner recurrence and
 * the weight update in FP32.  One outer iteration (S = s*b) does:
 *   a1  sample S row indices (counter-based, reproducible; see casgd_sample_indices)
 *   a2  gather Y = X[idx,:] (S x n, BF16) and y_Y = y[idx]
 *   a3  G = Y Y^T, BF16 products, FP32 accumulation; only blocks G_{j,t}, t < j
 *   a4  r = Y w, FP32 accumulation, rounded once to BF16
 *   a5  (sum of G over processes: absent on one GPU)
 *   a6  for j = 0..s-1: z_j = r_j + sum_{t<j} G_{j,t} alpha_t,
 *       alpha_j = -(eta/b) * l'(z_j, y_j)            (FP32)
 *   a7  l' of the loss: logistic -y/(1+exp(y z)); least squares z-y; Poisson exp(z)-y
 *   a8  w += Y^T alpha                                 (FP32)
 *   a9  (separately) f(w) = (1/m) sum_i l(x_i.w, y_i)
 * In exact arithmetic one outer iteration equals s plain minibatch-SGD steps.
 *
 * Conventions for every call:
 *  - All arrays are allocated by the caller; the library allocates no device or
 *    host memory.  It keeps no state between calls, with one exception: the fixed
 *    scratch array of casgd_update_static (see there).  "device" pointers must be
 *    CUDA device (or managed) memory of the current device; "host" pointers ordinary
 *    memory.
 *  - Flag bits not defined below are rejected with CASGD_ERR_ARG (bit 0x10 named a
 *    Gram variant this build no longer has).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every call is ordered on it; calls documented as "blocks" synchronize it.
 *  - Argument errors are detected on the host before anything is launched and are
 *    returned at once (CASGD_ERR_ARG, CASGD_ERR_WORKSPACE, CASGD_ERR_UNSUPPORTED).
 *    A failed CUDA launch returns CASGD_ERR_CUDA.  Errors found on the device
 *    (CASGD_ERR_NONFINITE, CASGD_ERR_TIMEOUT, CASGD_ERR_BAD_INDEX) are sticky bits in
 *    the workspace, reported by casgd_get_status, casgd_train and casgd_loss.
 *  - Limits: 1 <= m < 2^31; 1 <= n <= 16384; ld % 8 == 0 and ld >= n; X 16-byte
 *    aligned; 1 <= b; 1 <= s <= 64; S = s*b <= 65536.
 *  - The data matrix X is BF16 (raw 16-bit patterns), m x ld row-major; columns
 *    n..ld-1 are never read as data.
 */
#ifndef CASGD_H
#define CASGD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CASGD_ABI_VERSION 1

/* GLM losses (the abstract: logistic, linear and Poisson problems). */
enum { CASGD_LOGISTIC = 0, CASGD_LSQ = 1, CASGD_POISSON = 2 };

/* Return codes. */
enum {
  CASGD_OK = 0,
  CASGD_ERR_ARG = 1,          /* bad pointer, size, alignment or enum            */
  CASGD_ERR_WORKSPACE = 2,    /* workspace missing, misaligned or too small       */
  CASGD_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed             */
  CASGD_ERR_NONFINITE = 4,    /* device: the update produced a NaN or Inf weight  */
  CASGD_ERR_TIMEOUT = 5,      /* device: an inter-CTA wait ran past its bound     */
  CASGD_ERR_BAD_INDEX = 6,    /* device: a caller-given row index outside [0, m)  */
  CASGD_ERR_UNSUPPORTED = 7,  /* valid request this build does not support        */
  CASGD_ERR_SCRATCH_LIMIT = 8, /* too large for casgd_update_static's fixed scratch */
  CASGD_ERR_EXCHANGE = 9       /* the caller's exchange hook returned non-zero      */
};

/* casgd_params_t.flags */
#define CASGD_FLAG_WRITE_DIAG_BLOCKS 0x1u  /* also compute and store G_{j,j} (parity)   */
#define CASGD_FLAG_GRAM_TENSOR       0x2u  /* force the tcgen05 tensor-core Gram kernel */
#define CASGD_FLAG_GRAM_SIMT         0x4u  /* force the CUDA-core Gram kernel          */
#define CASGD_FLAG_GRAM_NO_CLUSTER   0x8u  /* tcgen05 Gram, one CTA per 128x256 tile  */
#define CASGD_FLAG_GRAM_PAIR         0x20u /* tcgen05 Gram, CTA pairs (cta_group::2,
                                              256x256 tiles).  Without a variant flag
                                              the library takes pairs forming the far
                                              sums (FAR_FROM_GRAM) for b a multiple of
                                              256, else pairs; these share their launch
                                              with the recurrence for b <= 512 or
                                              n >= 1024 (with this flag: always), else
                                              run as a launch of their own            */
#define CASGD_FLAG_NO_FUSE           0x40u /* run the paired-SM Gram and the inner
                                              recurrence as two launches.  Otherwise
                                              they share one launch whenever the pair
                                              variant is used (S >= 256, s >= 2): the
                                              recurrence starts on block row j of G as
                                              soon as the Gram has stored it; this
                                              needs every CTA of the launch resident,
                                              so a second fused step running on
                                              another stream at the same time can make
                                              both end with CASGD_ERR_TIMEOUT         */
#define CASGD_FLAG_TRACE_CHAIN       0x100u /* profiling: the recurrence's first chain
                                              warp records four globaltimer stamps per
                                              phase in the workspace (see
                                              casgd_chain_trace); off by default, as
                                              the stamps slow that warp              */
#define CASGD_FLAG_FAR_FROM_GRAM     0x200u /* the paired-SM Gram of the same launch
                                              forms the far sums of the inner
                                              recurrence itself: each tile of G_{j,t}
                                              with t < j-B (B = 3 for b <= 256, 2 for
                                              b <= 512, else 1) is multiplied by
                                              alpha_t in the tile's epilogue, straight
                                              from the tensor-memory accumulator, once
                                              alpha_t is final, and only the band
                                              blocks t = j-B .. j-1 (and G_{j,j} with
                                              WRITE_DIAG_BLOCKS) are stored: G beyond
                                              the band never reaches memory.  Same
                                              sums as the stored-G path in another
                                              order (per row: partials per block t
                                              and column group, then t ascending).
                                              The default wherever it applies (b a
                                              multiple of 256, s >= 2, S >= 256);
                                              this flag forces it: with another
                                              variant flag, FULL_G or a shape it does
                                              not take, CASGD_ERR_UNSUPPORTED          */
#define CASGD_FLAG_FULL_G            0x400u /* store every block G_{j,t}, t < j, and
                                              form the far sums from memory (the
                                              recurrence's bulk groups) even where the
                                              far-forming Gram applies                 */
#define CASGD_FLAG_SAMPLE_PERMUTED   0x800u /* sample without replacement: counter c
                                              draws position c mod m of epoch c div m
                                              of a keyed permutation of the m rows
                                              (casgd_sample_indices_permuted), so each
                                              run of m draws from an epoch boundary
                                              visits every row once.  Also honoured
                                              by casgd_sgd_fp32                       */
#define CASGD_FLAG_MARGINS_FP32      0x1000u /* precision variant: keep the margins r
                                              as their FP32 sums (no rounding to BF16);
                                              the r_out tap then receives S FP32
                                              values (4*S bytes)                      */
#define CASGD_FLAG_G_BF16            0x2000u /* precision variant: round every entry of
                                              G to BF16 (nearest even) after its FP32
                                              accumulation and before the recurrence
                                              uses it, as when G is summed across
                                              processes in BF16; stored blocks (and the
                                              G_out tap) hold the rounded values      */
#define CASGD_FLAG_GATHER_ROWS       0x4000u /* the far-forming launch reads its rows
                                              straight from X: the Gram's producer warp
                                              draws the sampled indices itself and loads
                                              four rows per tile::gather4 TMA copy, and
                                              the margin and update units read X rows
                                              through the same sampler, so the rows are
                                              never gathered into a copy Y (only the
                                              indices and labels are).  Same results bit
                                              for bit; measured 4x slower on GB300 at
                                              n = 2000 (one small TMA copy per four rows
                                              and 64 columns), so off by default.
                                              Ignored where the far-forming Gram does
                                              not apply or indices are given (idx_in)  */
#define CASGD_FLAG_TEST_STALL        0x80000000u /* test only: the recurrence's first
                                              block never signals completion, so every
                                              waiter runs into its time bound and the
                                              step ends with CASGD_ERR_TIMEOUT        */

/* The data set (device pointers). */
typedef struct {
  int64_t m;         /* rows                                                    */
  int64_t n;         /* features                                                */
  int64_t ld;        /* row pitch of X in elements (multiple of 8, >= n)         */
  const void* X;     /* device, BF16 bits, m x ld, 16-byte aligned              */
  const float* y;    /* device, m labels (logistic: +-1; Poisson: counts)        */
} casgd_data_t;

/* Method parameters. */
typedef struct {
  int32_t b;           /* minibatch rows                                       */
  int32_t s;           /* minibatch steps per outer iteration                  */
  float eta;           /* step size; alpha = -(eta/b) l'                        */
  int32_t loss;        /* CASGD_LOGISTIC / CASGD_LSQ / CASGD_POISSON            */
  uint64_t seed;       /* sampling seed                                        */
  uint32_t flags;      /* CASGD_FLAG_*                                         */
  uint32_t timeout_us; /* bound on each inter-CTA wait; 0 = 1,000,000 us        */
} casgd_params_t;

/* Optional taps of one outer iteration (any member may be NULL; device memory). */
typedef struct {
  const int32_t* idx_in; /* S row indices to use instead of sampling; an index
                            outside [0,m) sets CASGD_ERR_BAD_INDEX and its row is
                            treated as zeros                                    */
  int32_t* idx_out;      /* receives the S indices used                         */
  float* G_out;          /* receives G in the packed block-lower layout:
                            blocks (j,t) for t<j (t<=j with WRITE_DIAG_BLOCKS),
                            j ascending then t ascending, each b x b row-major;
                            casgd_gram_elems() floats (with FAR_FROM_GRAM only
                            the band and diagonal blocks are written)           */
  uint16_t* r_out;       /* receives the S BF16 margins (bit patterns); with
                            CASGD_FLAG_MARGINS_FP32 the S FP32 margins (4*S
                            bytes)                                              */
  float* alpha_out;      /* receives the S FP32 step coefficients alpha         */
} casgd_taps_t;

/* Optional instrumentation of casgd_train (host struct). */
typedef struct {
  int64_t launches;      /* out: number of kernels the call launched            */
  void** stage_events;   /* in: NULL, or cudaEvent_t handles; when given, event
                            [it*CASGD_STAGE_EVENTS + e] is recorded on `stream`
                            before stage e of outer iteration it (e = 0 gather,
                            1 Gram, 2 recurrence, 3 update, 4 after update;
                            when the Gram and the recurrence share one launch,
                            events 2 and 3 are both recorded after it); a NULL
                            entry records nothing.  An event between two
                            launches keeps them from overlapping (see
                            casgd_train), so a timed loop with events runs
                            slower than one without                          */
  int32_t n_events;      /* in: length of stage_events                          */
  int32_t gram_kind;     /* out: 1 = tcgen05 Gram kernel used, 2 = CUDA-core,
                            3 = paired-SM tcgen05 Gram and recurrence in one
                            launch, 4 = as 3 with the Gram one outer iteration
                            ahead of the recurrence (casgd_train, iters >= 2),
                            5 = as 3 with the far sums formed by the Gram
                            (CASGD_FLAG_FAR_FROM_GRAM), 6 = as 5 with the
                            next iteration's band stored by the same launch
                            (casgd_train, iters >= 2), 7 = the feature-sharded
                            calls of casgd_train_sharded                        */
} casgd_profile_t;
#define CASGD_STAGE_EVENTS 5

/* Message for a return code (static string; never NULL). */
const char* casgd_strerror(int code);

/* CASGD_ABI_VERSION of the loaded library. */
int casgd_version(void);

/* Number of floats in the packed block-lower G for (b, s, flags); -1 on bad input. */
int64_t casgd_gram_elems(int32_t b, int32_t s, uint32_t flags);

/* Bytes of device workspace casgd_outer_step / casgd_train / casgd_loss need for
 * (data, params); writes *bytes.  Host only, launches nothing.  The workspace must be
 * 256-byte aligned and is owned by the caller; one workspace serves one stream at a
 * time. */
int casgd_workspace_size(const casgd_data_t* data, const casgd_params_t* params,
                         size_t* bytes);

/* Zero the control block of a workspace.  Call once on a fresh workspace (or
 * zero-fill its first 512 bytes) before its first use; the library keeps it
 * consistent afterwards.  Asynchronous. */
int casgd_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Storage step of the recipe (the abstract: the input matrix is stored in low
 * precision).  dst[i*ld_dst + c] = BF16 round-to-nearest-even of src[i*ld_src + c]
 * for c < n, and 0 for n <= c < ld_dst.  src: device FP32 m x ld_src; dst: device
 * BF16 bits m x ld_dst (ld_dst % 8 == 0, 16-byte aligned).  Asynchronous. */
int casgd_store_bf16(const float* src, int64_t m, int64_t n, int64_t ld_src,
                     void* dst, int64_t ld_dst, void* stream);

/* Step a1 on its own.  idx[i] = ((h >> 32) * m) >> 32 where h is output number
 * (counter0 + i) of SplitMix64 started from state `seed` (Steele, Lea & Flood 2014):
 * h = mix(seed + (counter0 + i + 1) * 0x9E3779B97F4A7C15).  Outer iteration k uses
 * counter0 = k*s*b, so plain SGD step q (counters q*b...) sees the same rows.
 * idx: device int32[count].  Asynchronous. */
int casgd_sample_indices(int64_t m, int64_t count, uint64_t seed, uint64_t counter0,
                         int32_t* idx, void* stream);

/* Step a1 without replacement (CASGD_FLAG_SAMPLE_PERMUTED; the abstract leaves the
 * sampling scheme open).  Counter c = counter0 + i draws position q = c mod m of the
 * permutation of epoch e = c div m: d = the smallest even width with 2^d >= m (at
 * least 2); the round keys K_r = SplitMix64 output number 4e + r (r = 0..3) of the
 * stream started at seed ^ 0x6A09E667F3BCC908; the d-bit balanced Feistel network
 * (Luby & Rackoff 1988) maps (L, R) = (x >> d/2, x & mask) four times to
 * (R, L ^ (SplitMix64 output number R of the stream started at K_r) & mask); applied to
 * q and then again while the value is >= m (cycle walking, Black & Rogaway 2002).
 * m in [1, 2^31); idx: device int32[count].  Asynchronous. */
int casgd_sample_indices_permuted(int64_t m, int64_t count, uint64_t seed, uint64_t counter0,
                                  int32_t* idx, void* stream);

/* One outer iteration k (steps a1-a8) on w (device FP32[n], updated in place).
 * ws: device workspace of ws_bytes (casgd_workspace_size).  taps: NULL or optional
 * inputs/outputs for parity checks.  Asynchronous; device errors are sticky in ws. */
int casgd_outer_step(const casgd_data_t* data, const casgd_params_t* params, float* w,
                     uint64_t k, void* ws, size_t ws_bytes, void* stream,
                     const casgd_taps_t* taps);

/* `iters` outer iterations k = k0 .. k0+iters-1.  If loss_every > 0, f(w) is
 * evaluated after every loss_every-th iteration and written to host
 * loss_hist[iters/loss_every].  Blocks at the end (one stream synchronize) and
 * returns the first sticky device error, which it clears.  prof may be NULL.
 * Where the paired-SM Gram shares its launch with the recurrence (see
 * CASGD_FLAG_NO_FUSE) and iters >= 2, the Gram of iteration k+1 runs in the launch
 * of iteration k's recurrence (its rows do not depend on w), on second Y and G
 * buffers that casgd_workspace_size includes for such parameters; with the far-
 * forming Gram (CASGD_FLAG_FAR_FROM_GRAM, the default for b a multiple of 256) the
 * launch of iteration k forms iteration k's far sums and margins and stores the band
 * of iteration k+1, after a launch that gathers iteration k+1's rows.  Where n % 8 == 0
 * with rows of at least 512 bytes, or n <= 64 (not with CASGD_FLAG_GATHER_ROWS), that
 * launch also gathers iteration k+2's rows, indices and labels and resets iteration
 * k+1's recurrence state (third row buffers and a second state in the workspace), so
 * from the second iteration on one launch runs per iteration.  The loop's
 * launches use programmatic dependent launch: each may be scheduled while the one
 * before it ends and waits for that one's completion before it touches memory, so
 * work the caller enqueues on `stream` keeps plain stream order.  Either way the
 * results are bit-identical to iters calls of casgd_outer_step. */
int casgd_train(const casgd_data_t* data, const casgd_params_t* params, float* w,
                uint64_t k0, int32_t iters, void* ws, size_t ws_bytes, void* stream,
                int32_t loss_every, double* loss_hist, casgd_profile_t* prof);

/* casgd_train on inputs that live in host memory: copies X_host (host, data->m rows of
 * data->ld BF16 values, the layout of data->X) into data->X, y_host (host FP32[m]) into
 * data->y and w_host (host FP32[n]) into w_dev on `stream`, runs casgd_train on the device
 * buffers (data, w_dev, ws as there), and copies w_dev back into w_host.  Host buffers
 * should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to run at full
 * rate; pageable memory works but the copies then stage through the driver.  data->X,
 * data->y and w_dev are caller-owned device buffers of those sizes (data->X 16-byte
 * aligned, as for casgd_train).  Blocks until w_host holds the result; returns as
 * casgd_train does, CASGD_ERR_ARG for a null host pointer or w_dev, CASGD_ERR_CUDA when a
 * copy fails. */
int casgd_train_host(const void* X_host, const float* y_host, float* w_host,
                     const casgd_data_t* data, float* w_dev, const casgd_params_t* params,
                     uint64_t k0, int32_t iters, void* ws, size_t ws_bytes, void* stream,
                     int32_t loss_every, double* loss_hist, casgd_profile_t* prof);

/* Step a9: f(w) = (1/m) sum_i l(x_i . w, y_i) with x_i the BF16 rows, each row's
 * dot product and loss in FP32, the sum in FP64.  Writes host *out; blocks. */
int casgd_loss(const casgd_data_t* data, int32_t loss, const float* w, void* ws,
               size_t ws_bytes, void* stream, double* out);

/* Same as casgd_loss but asynchronous: the FP64 result goes to device *out_dev. */
int casgd_loss_async(const casgd_data_t* data, int32_t loss, const float* w, void* ws,
                     size_t ws_bytes, void* stream, double* out_dev);

/* Weight update w += Y^T alpha (step a8) that allocates nothing and takes no
 * workspace.  The paper has no counterpart: this exists for callers that cannot
 * allocate device memory where they apply an update (inside another framework's
 * memory pool that forbids raw cudaMalloc, in loops that must not block on an
 * allocator, or when they only own their input and output buffers).
 *   Y      device BF16 bits, S x ldY row-major (ldY % 8 == 0, ldY >= n), 16-byte aligned
 *   alpha  device FP32[S];  w  device FP32[n], updated in place
 * Its scratch is a fixed array inside the library (4 MiB of partial sums plus a
 * 512-byte control block) that every GPU loading the library holds until exit.  It
 * fits P * ldY <= 1,048,576 floats with P = min(ceil(S/32), 320) (e.g. n <= 3272
 * at P = 320); larger requests return CASGD_ERR_SCRATCH_LIMIT and run nothing.
 * The first call in each CUDA context of a device (the first call on the device, and
 * the first after a cudaDeviceReset) looks up the array's device address; make that
 * call before any stream capture.  Every call shares the array: calls whose
 * work overlaps on the GPU (e.g. on two streams) race and must be serialised by the
 * caller.  Non-finite results are not reported here (inspect w).  Asynchronous. */
int casgd_update_static(const void* Y, int64_t S, int64_t n, int64_t ldY,
                        const float* alpha, float* w, void* stream);

/* ------------------------------------------------------------------------------------
 * Feature-sharded outer iteration: the setting the paper measures.  The abstract's
 * method exists to replace the s AllReduces of s minibatch-SGD steps by a single
 * AllReduce of the sb x sb Gram matrix per outer iteration, communicated in high
 * precision.  With the features split over P processes (process p holds columns
 * c_p .. c_{p+1}-1 of X and the same slice of w), every process draws the same S rows,
 * forms its partial Gram G_p = Y_p Y_p^T and partial margins r_p = Y_p w_p, and the
 * sums G = sum_p G_p, r = sum_p r_p give every process the quantities of the
 * unsharded step (G_{j,t} and r_j are dot products over the features).  The recurrence
 * then runs identically on every process and each updates its own slice of w.
 *
 * An outer iteration is casgd_outer_step_local, then the caller's in-place FP32 sum of
 * the exchange buffer over the processes (for example ncclAllReduce(ncclSum) on
 * `stream`), then casgd_outer_step_finish.  The exchange buffer (caller-owned device
 * FP32, 256-byte aligned, casgd_exchange_elems floats) holds the packed block-lower G
 * (casgd_gram_elems floats, the layout of casgd_taps_t.G_out) followed by the S
 * margins as FP32 partial sums; finish rounds the summed margins once to BF16 (or keeps
 * them in FP32 with CASGD_FLAG_MARGINS_FP32).  With one process the sum is the identity
 * and the result is that of casgd_outer_step with CASGD_FLAG_FULL_G up to FP32
 * summation order.  The far-forming Gram (CASGD_FLAG_FAR_FROM_GRAM) and
 * CASGD_FLAG_G_BF16 are CASGD_ERR_UNSUPPORTED here: the far sums need the summed G, and
 * the buffer is summed in FP32.  Losses need every feature: they are not formed here.
 * ---------------------------------------------------------------------------------- */

/* Floats in the exchange buffer for (b, s, flags): the packed block-lower G
 * (with the diagonal blocks under CASGD_FLAG_WRITE_DIAG_BLOCKS) followed by S = s*b
 * margins; -1 on bad input.  Host only. */
int64_t casgd_exchange_elems(int32_t b, int32_t s, uint32_t flags);

/* Bytes of device workspace the sharded calls need for this process's slice (data->n
 * = its feature count); G is not part of it (it lives in the exchange buffer).  Host
 * only.  Initialise a fresh workspace with casgd_workspace_init. */
int casgd_workspace_size_sharded(const casgd_data_t* data, const casgd_params_t* params,
                                 size_t* bytes);

/* First half of outer iteration k on this process's slice.  data: X_p (m x ld_p BF16,
 * the slice's columns) and the full label vector y (the same on every process); w:
 * device FP32[n_p], this slice of the weights (read only here).  Samples the S rows
 * (the same on every process for the same seed and k), gathers them, and writes G_p and
 * r_p into xbuf (device, 256-byte aligned, casgd_exchange_elems floats).  taps: NULL,
 * or idx_in / idx_out as in casgd_outer_step (other members ignored).  Asynchronous. */
int casgd_outer_step_local(const casgd_data_t* data, const casgd_params_t* params,
                           const float* w, uint64_t k, void* ws, size_t ws_bytes, void* stream,
                           float* xbuf, const casgd_taps_t* taps);

/* Second half, after xbuf holds the sums over the processes: the inner recurrence on
 * the summed G and margins (steps a6, a7) and this slice's update w_p += Y_p^T alpha
 * (a8).  data, params, ws: as for the matching casgd_outer_step_local call, with no
 * other call on ws in between.  taps: NULL, or r_out / alpha_out as in
 * casgd_outer_step (other members ignored).  Asynchronous; device errors are sticky in
 * ws. */
int casgd_outer_step_finish(const casgd_data_t* data, const casgd_params_t* params, float* w,
                            void* ws, size_t ws_bytes, void* stream, const float* xbuf,
                            const casgd_taps_t* taps);

/* The caller's exchange: sum buf[0 .. count-1] (device FP32) in place over the
 * processes, ordered on `stream` (it may enqueue work there and return at once).
 * Returns 0 on success. */
typedef int (*casgd_exchange_fn)(void* ctx, float* buf, int64_t count, void* stream);

/* `iters` sharded outer iterations k = k0 .. k0+iters-1: local, exchange(ctx, xbuf,
 * casgd_exchange_elems(...), stream), finish.  A non-zero exchange return ends the
 * loop with CASGD_ERR_EXCHANGE.  Blocks at the end and returns the first sticky device
 * error, which it clears.  prof may be NULL (stage events: 0 before local, 1 before the
 * exchange, 2 before finish, 3 and 4 after it). */
int casgd_train_sharded(const casgd_data_t* data, const casgd_params_t* params, float* w,
                        uint64_t k0, int32_t iters, void* ws, size_t ws_bytes, void* stream,
                        float* xbuf, casgd_exchange_fn exchange, void* exchange_ctx,
                        casgd_profile_t* prof);

/* Blocks on `stream`, returns the sticky device status of ws (CASGD_OK or the
 * highest-priority CASGD_ERR_* seen) and clears it. */
int casgd_get_status(void* ws, void* stream);

/* Bytes of device workspace casgd_sgd_fp32 needs for minibatch size b (host only). */
int casgd_sgd_workspace_size(int32_t b, size_t* bytes);

/* FP32 plain minibatch SGD, the baseline the paper compares CA-SGD with (its speedup
 * and its final-loss gap are stated against FP32 SGD).  Step q = q0 .. q0+steps-1
 * samples the rows CA-SGD uses for the same minibatch (counters q*b .. q*b+b-1, see
 * casgd_sample_indices) and does, in FP32,
 *     z_i = x_i . w,   alpha_i = -(eta/b) l'(z_i, y_i),   w += sum_i alpha_i x_i.
 *   X   device FP32 m x ld row-major (ld >= n; columns >= n are not read)
 *   y   device FP32[m];  w  device FP32[n], updated in place
 *   params: b, eta, loss, seed, timeout_us and the SAMPLE_PERMUTED flag are used;
 *       s and the other flags are ignored.
 *   ws  device workspace of ws_bytes >= casgd_sgd_workspace_size(b), 256-byte aligned;
 *       device errors are sticky in it (casgd_get_status).
 * One cooperative launch for all steps; asynchronous. */
int casgd_sgd_fp32(const float* X, int64_t m, int64_t n, int64_t ld, const float* y,
                   const casgd_params_t* params, float* w, uint64_t q0, int32_t steps, void* ws,
                   size_t ws_bytes, void* stream);

/* Profiling: copies the chain timeline of the last outer iteration run with
 * CASGD_FLAG_TRACE_CHAIN on ws (data and params as for that call) to host
 * out[4*j + e], j < params->s: globaltimer nanoseconds when the first chain warp
 * started phase j (e = 0), had issued its loads (1), saw alpha_{j-1} and far_j
 * final (2) and had stored its alpha_j (3); then out[4*s + e]: when the last tile
 * of G was stored (e = 0; only when the Gram shares the recurrence's launch), the
 * last far sum (1) and the last fused update partial (2) were stored, 0 where none
 * was; out[4*s + 3] = 0.  out holds 4*s + 4 values.  Blocks on `stream`.  Without
 * the flag the stamps are stale or zero. */
int casgd_chain_trace(const casgd_data_t* data, const casgd_params_t* params, void* ws,
                      size_t ws_bytes, void* stream, uint64_t* out);

#ifdef __cplusplus
}
#endif
#endif /* CASGD_H */
