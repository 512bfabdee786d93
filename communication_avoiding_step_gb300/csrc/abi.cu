// C ABI of libcasgd.so (declared in include/casgd.h): argument checks, workspace
// layout, and the stream-ordered sequence of kernels for one CA-SGD outer iteration.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract).  Step order of one outer iteration: sample and gather the s
// minibatches, form the Gram matrix and the BF16 margins, (sum G across processes --
// absent on one GPU), run the inner recurrence, update the weights.
#include <cstring>

#include "casgd_internal.cuh"

namespace casgd {

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

constexpr int kLossSlots = 64;  // device slots for losses recorded by casgd_train

struct Resolved {
  Layout L;
  Ctrl* ctrl;
  int32_t* idx;
  float* r;  // margins as FP32 values (BF16-representable in the recipe)
  float* yY;
  float* alpha;
  float* far;
  uint32_t* slab;   // the paired-SM Gram's per-32-row completion counters
  uint64_t* trace;  // the recurrence's per-phase timeline
  uint16_t* Y;
  float* G;
  // second buffers of a multi-iteration run whose Gram runs one iteration ahead
  uint16_t* Y2;
  float* G2;
  int32_t* idx2;
  float* yY2;
  // third row buffers: the far-forming launch of iteration k gathers iteration k+2's rows
  uint16_t* Y3;
  int32_t* idx3;
  float* yY3;
  // second recurrence state (odd iterations of a run with the third row buffers)
  Ctrl* ctrl2;
  uint32_t* cnt2;
  float* r2;
  float* alpha2;
  float* far2;
  float* fpart2;
  float* fpart;  // far partial sums of the far-forming Gram (null: not laid out)
  float* upd;
  double* loss_part;
  double* loss_slots;
};

bool check_data(const casgd_data_t* d) {
  if (!d || !d->X || !d->y) return false;
  if (d->m < 1 || d->m >= (int64_t(1) << 31)) return false;
  if (d->n < 1 || d->n > kMaxN) return false;
  if (d->ld < d->n || (d->ld % 8) != 0) return false;
  if ((reinterpret_cast<uintptr_t>(d->X) & 15u) != 0) return false;
  return true;
}

constexpr uint32_t kKnownFlags =
    CASGD_FLAG_WRITE_DIAG_BLOCKS | CASGD_FLAG_GRAM_TENSOR | CASGD_FLAG_GRAM_SIMT |
    CASGD_FLAG_GRAM_NO_CLUSTER | CASGD_FLAG_GRAM_PAIR | CASGD_FLAG_NO_FUSE |
    CASGD_FLAG_TRACE_CHAIN | CASGD_FLAG_FAR_FROM_GRAM | CASGD_FLAG_FULL_G |
    CASGD_FLAG_SAMPLE_PERMUTED | CASGD_FLAG_MARGINS_FP32 | CASGD_FLAG_G_BF16 |
    CASGD_FLAG_GATHER_ROWS | CASGD_FLAG_TEST_STALL;

bool check_params(const casgd_params_t* p) {
  if (!p) return false;
  if (p->flags & ~kKnownFlags) return false;
  if (p->b < 1 || p->s < 1 || p->s > kMaxS) return false;
  if ((int64_t)p->b * p->s > kMaxSB) return false;
  if (p->loss < CASGD_LOGISTIC || p->loss > CASGD_POISSON) return false;
  if (!(p->eta == p->eta)) return false;  // NaN
  return true;
}

int device_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CASGD_ERR_CUDA;
  if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CASGD_ERR_CUDA;
  return CASGD_OK;
}

Resolved resolve(void* ws, const Layout& L) {
  char* base = static_cast<char*>(ws);
  Resolved R;
  R.L = L;
  R.ctrl = reinterpret_cast<Ctrl*>(base);
  R.idx = reinterpret_cast<int32_t*>(base + L.off_idx);
  R.r = reinterpret_cast<float*>(base + L.off_r);
  R.yY = reinterpret_cast<float*>(base + L.off_yY);
  R.alpha = reinterpret_cast<float*>(base + L.off_alpha);
  R.far = reinterpret_cast<float*>(base + L.off_far);
  R.slab = reinterpret_cast<uint32_t*>(base + L.off_far + align_up((size_t)L.S * sizeof(float)));
  R.trace = timeline_of(R.slab);
  R.Y = reinterpret_cast<uint16_t*>(base + L.off_Y);
  R.G = reinterpret_cast<float*>(base + L.off_G);
  R.Y2 = L.off_Y2 ? reinterpret_cast<uint16_t*>(base + L.off_Y2) : nullptr;
  R.G2 = L.off_G2 ? reinterpret_cast<float*>(base + L.off_G2) : nullptr;
  R.idx2 = L.off_idx2 ? reinterpret_cast<int32_t*>(base + L.off_idx2) : nullptr;
  R.yY2 = L.off_yY2 ? reinterpret_cast<float*>(base + L.off_yY2) : nullptr;
  R.Y3 = L.off_Y3 ? reinterpret_cast<uint16_t*>(base + L.off_Y3) : nullptr;
  R.idx3 = L.off_idx3 ? reinterpret_cast<int32_t*>(base + L.off_idx3) : nullptr;
  R.yY3 = L.off_yY3 ? reinterpret_cast<float*>(base + L.off_yY3) : nullptr;
  R.ctrl2 = L.off_ctrl2 ? reinterpret_cast<Ctrl*>(base + L.off_ctrl2) : nullptr;
  R.cnt2 = L.off_cnt2 ? reinterpret_cast<uint32_t*>(base + L.off_cnt2) : nullptr;
  R.r2 = L.off_r2 ? reinterpret_cast<float*>(base + L.off_r2) : nullptr;
  R.alpha2 = L.off_alpha2 ? reinterpret_cast<float*>(base + L.off_alpha2) : nullptr;
  R.far2 = L.off_far2 ? reinterpret_cast<float*>(base + L.off_far2) : nullptr;
  R.fpart2 = L.off_fpart2 ? reinterpret_cast<float*>(base + L.off_fpart2) : nullptr;
  R.fpart = L.off_fpart ? reinterpret_cast<float*>(base + L.off_fpart) : nullptr;
  R.upd = reinterpret_cast<float*>(base + L.off_upd);
  R.loss_part = reinterpret_cast<double*>(base + L.off_loss);
  R.loss_slots = R.loss_part + kLossCtas;
  return R;
}

int check_ws(void* ws, size_t ws_bytes, const Layout& L) {
  if (!ws) return CASGD_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return CASGD_ERR_WORKSPACE;
  if (ws_bytes < L.total) return CASGD_ERR_WORKSPACE;
  return CASGD_OK;
}

// Layout for the loss alone (control block + partials), used when no params are known.
size_t loss_only_bytes() {
  return align_up(sizeof(Ctrl)) + align_up((size_t)(kLossCtas + kLossSlots) * sizeof(double));
}

int gram_choice(const casgd_params_t* p, int64_t S, int64_t n) {
  const bool tc_ok = gram_tc_supported(S, n, p->b);
  if (p->flags & CASGD_FLAG_GRAM_TENSOR) return tc_ok ? 1 : -1;
  if (p->flags & CASGD_FLAG_GRAM_SIMT) return 2;
  // Default: tensor cores (measured faster than the CUDA-core kernel for every feature
  // count here, n = 18 .. 2000, because writing G dominates for narrow n).
  return tc_ok ? 1 : 2;
}

// Tensor-core variant (forced by a flag; else CTA pairs forming the far sums in the
// recurrence's launch for b a multiple of 256; else CTA pairs, sharing their launch with
// the recurrence while the chain's rows fit one warp each on half the SMs, b <= 512) and
// whether the recurrence shares its launch.
struct GramPlan {
  int choice;  // 1 tensor cores, 2 CUDA cores, -1 unsupported
  int mode;    // tensor cores: 0 pairs, 1 single CTA
  bool fused;  // pairs sharing their launch with the recurrence
  bool far;    // ... and forming the far sums (CASGD_FLAG_FAR_FROM_GRAM)
};

GramPlan gram_plan(int64_t n, int32_t b, int32_t s, uint32_t flags) {
  casgd_params_t p{};
  p.b = b;
  p.s = s;
  p.flags = flags;
  const int64_t S = (int64_t)b * s;
  GramPlan g;
  g.choice = gram_choice(&p, S, n);
  g.mode = (flags & CASGD_FLAG_GRAM_NO_CLUSTER) ? 1 : 0;
  // Without a variant flag the recurrence shares the pairs' launch for b <= 512 or deep K
  // (n >= 1024); wide blocks over shallow K run the Gram and the recurrence as two
  // launches (measured faster there: writing G bounds the Gram).
  const bool fuse_shape = b <= 512 || n >= 1024 || (flags & CASGD_FLAG_GRAM_PAIR);
  g.fused = g.choice == 1 && g.mode == 0 && !(flags & CASGD_FLAG_NO_FUSE) && fuse_shape &&
            gram_recur_fused_supported(S, n, b);
  // The far-forming Gram (pairs in the recurrence's launch, b % 256 == 0): the default
  // wherever it applies (measured faster than storing G on all five workloads), forced
  // by FAR_FROM_GRAM (which fails where it cannot apply), off with FULL_G or another
  // variant flag.
  const uint32_t other = CASGD_FLAG_GRAM_SIMT | CASGD_FLAG_GRAM_NO_CLUSTER |
                         CASGD_FLAG_NO_FUSE | CASGD_FLAG_FULL_G;
  const bool far_ok = g.choice == 1 && !(flags & other) && far_gram_supported(S, n, b);
  g.far = far_ok;
  if (g.far) {
    g.mode = 0;
    g.fused = true;
  } else if (flags & CASGD_FLAG_FAR_FROM_GRAM) {
    g.choice = -1;
  }
  return g;
}

int record(casgd_profile_t* prof, int64_t it, int e, cudaStream_t st) {
  if (!prof || !prof->stage_events) return CASGD_OK;
  const int64_t i = it * CASGD_STAGE_EVENTS + e;
  if (i >= prof->n_events || !prof->stage_events[i]) return CASGD_OK;  // (null: none here)
  if (cudaEventRecord(static_cast<cudaEvent_t>(prof->stage_events[i]), st) != cudaSuccess)
    return CASGD_ERR_CUDA;
  return CASGD_OK;
}

#define CK(expr)                                  \
  do {                                            \
    if ((expr) != cudaSuccess) return CASGD_ERR_CUDA; \
  } while (0)

// The sampled rows of the data set as the gathering launch reads them.
RowSource row_source(const casgd_data_t* d, const casgd_params_t* p) {
  RowSource rs;
  rs.X = static_cast<const uint16_t*>(d->X);
  rs.ld = d->ld;
  rs.m = (uint32_t)d->m;
  rs.seed = p->seed;
  rs.perm_d = (p->flags & CASGD_FLAG_SAMPLE_PERMUTED) ? perm_width(d->m) : 0;
  return rs;
}

int outer_step_impl(const casgd_data_t* d, const casgd_params_t* p, float* w, uint64_t k,
                    void* ws, size_t ws_bytes, cudaStream_t st, const casgd_taps_t* taps,
                    Ctx& c, casgd_profile_t* prof, int64_t it) {
  const Layout L = make_layout(d->n, p->b, p->s, p->flags, c.num_sms);
  int rc = check_ws(ws, ws_bytes, L);
  if (rc != CASGD_OK) return rc;
  Resolved R = resolve(ws, L);
  const GramPlan gp = gram_plan(d->n, p->b, p->s, p->flags);
  const int choice = gp.choice;
  if (choice < 0) return CASGD_ERR_UNSUPPORTED;
  const bool diag = (p->flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  float* G = (taps && taps->G_out) ? taps->G_out : R.G;
  const int32_t* idx_in = taps ? taps->idx_in : nullptr;
  if (prof) prof->gram_kind = choice;

  // the shared launch may be scheduled while the gather ends (programmatic dependent
  // launch; it waits for the gather's completion before it touches memory)
  c.pdl = true;
  if ((rc = record(prof, it, 0, st)) != CASGD_OK) return rc;
  // With CASGD_FLAG_GATHER_ROWS the far-forming launch reads its rows straight from X
  // (drawing the sampled indices itself), unless the caller gives the indices; otherwise
  // the rows are gathered into Y first.
  const bool gather = gp.far && !idx_in && (p->flags & CASGD_FLAG_GATHER_ROWS);
  const RowSource rs = row_source(d, p);
  const uint64_t ctr = k * (uint64_t)L.S;
  if (gp.far)  // the indices and labels (rows into Y only with given indices) and the
               // reset; the margins are formed in the shared launch
    CK(launch_gather_reset(*d, *p, k, idx_in, R.idx, gather ? nullptr : R.Y, R.yY, true, L.ldY,
                           R.r, R.alpha, R.far, R.fpart, R.ctrl, R.slab, c));
  else
    CK(launch_gather(*d, *p, w, k, idx_in, R.idx, R.Y, L.ldY, R.r, R.yY, R.alpha, R.far,
                     nullptr, R.ctrl, R.slab, GATHER_AND_MARGINS, c));
  if ((rc = record(prof, it, 1, st)) != CASGD_OK) return rc;
  // The update's first stage rides in the recurrence (one partial row per block,
  // s <= 64 <= upd_ctas rows of the partial buffer); the reduce adds the s rows to w.
  const int mode = gp.mode;
  const bool fused = gp.fused;
  if (fused) {
    // Gram and recurrence in one launch.  (The sum of G over processes would split it:
    // on one GPU it is the identity.)
    CK(launch_gram_recur(R.Y, G, false, L.S, d->n, L.ldY, p->b, p->s, p->eta, p->loss, p->flags,
                         G, R.Y, R.r, R.yY, R.alpha, R.far, R.slab, gp.far ? R.fpart : nullptr,
                         R.upd, w, gp.far, R.ctrl, p->timeout_us,
                         /*g_band=*/G == R.G, gather ? &rs : nullptr, ctr, ctr, nullptr,
                         nullptr, nullptr, nullptr, c));
    if ((rc = record(prof, it, 2, st)) != CASGD_OK) return rc;
  } else {
    if (choice == 1)
      CK(launch_gram_tc(R.Y, L.S, d->n, L.ldY, p->b, p->s, p->flags, mode, G, R.ctrl,
                        p->timeout_us, c));
    else
      CK(launch_gram_simt(R.Y, L.S, d->n, L.ldY, p->b, p->s, diag,
                          (p->flags & CASGD_FLAG_G_BF16) != 0, G, c));
    // (The sum of G over processes would sit here; on one GPU it is the identity.)
    if ((rc = record(prof, it, 2, st)) != CASGD_OK) return rc;
    CK(launch_recur(G, R.r, R.yY, R.alpha, R.far, R.slab, p->b, p->s, p->eta, p->loss,
                    p->flags, p->timeout_us, R.ctrl, R.Y, L.ldY, d->n, R.upd, w, c));
  }
  if (prof) prof->gram_kind = gp.far ? 5 : fused ? 3 : choice;
  // the update (a8) finished inside the recurrence's launch
  if ((rc = record(prof, it, 3, st)) != CASGD_OK) return rc;
  if ((rc = record(prof, it, 4, st)) != CASGD_OK) return rc;

  if (taps) {
    if (taps->idx_out)
      CK(cudaMemcpyAsync(taps->idx_out, R.idx, L.S * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    if (taps->r_out) {
      if (p->flags & CASGD_FLAG_MARGINS_FP32)
        CK(cudaMemcpyAsync(taps->r_out, R.r, L.S * sizeof(float), cudaMemcpyDeviceToDevice, st));
      else  // the BF16 bit patterns of the (BF16-valued) margins
        CK(launch_bf16_bits(R.r, L.S, taps->r_out, c));
    }
    if (taps->alpha_out)
      CK(cudaMemcpyAsync(taps->alpha_out, R.alpha, L.S * sizeof(float), cudaMemcpyDeviceToDevice, st));
  }
  return CASGD_OK;
}

// casgd_train with the paired-SM Gram sharing the recurrence's launch: the Gram of
// iteration k+1 (whose rows are sampled ahead: only the margins need the current w)
// runs in the launch of iteration k's recurrence, on double-buffered Y and G.  With the
// far-forming Gram (far) the launch of iteration k forms iteration k's far sums (they
// need this iteration's alpha), its margins and update, and stores the band of iteration
// k+1, so the recurrence starts on a complete band; the first iteration's band comes
// from a prologue launch.  Every value is computed as in outer_step_impl (same kernels'
// arithmetic), only the order of independent work changes.  The loop's gather and
// shared launches use programmatic dependent launch (Ctx::pdl).  Stage events per
// iteration: 0 before the gather of the next iteration's rows (with the stored-G Gram
// also this iteration's margins), 1 before the shared launch, 2, 3 and 4 after it (it
// ends with the update).
int train_pipelined(const casgd_data_t* d, const casgd_params_t* p, float* w, uint64_t k0,
                    int32_t iters, const Layout& L, const Resolved& R, Ctx& c,
                    casgd_profile_t* prof, int32_t loss_every, int& slot, int& flushed,
                    double* loss_hist, bool far) {
  uint16_t* Yb[2] = {R.Y, R.Y2};
  float* Gb[2] = {R.G, R.G2};
  int32_t* Ib[2] = {R.idx, R.idx2};
  float* yb[2] = {R.yY, R.yY2};
  const cudaStream_t st = c.stream;
  int rc;
  float* fpart = far ? R.fpart : nullptr;
  // with CASGD_FLAG_GATHER_ROWS the far-forming loop reads every row straight from X (no
  // Y); its launches draw the sampled indices themselves, the gather launches only the
  // indices and labels
  const RowSource rs = row_source(d, p);
  const bool gather = far && (p->flags & CASGD_FLAG_GATHER_ROWS);
  const RowSource* rsp = gather ? &rs : nullptr;
  if (prof) prof->gram_kind = far ? 6 : 4;
  // the gather launches and the shared launches of the loop overlap each other's start
  // and end (programmatic dependent launch); each waits for its predecessor's completion
  // before it touches memory, so the results are those of plain stream order
  c.pdl = true;
  // With third row buffers (far-forming, not gathering, rows ahead_rows_supported) the
  // launch of iteration k also gathers iteration k+2's rows (its producers, once their
  // Gram work is done), its indices and labels, and resets the recurrence state of
  // iteration k+1, which alternates between two sets; from the second iteration on
  // nothing runs between two such launches.  The row buffers rotate over three sets,
  // the G buffers over two.
  const bool ahead = far && !gather && R.Y3 != nullptr;
  uint16_t* Yr[3] = {R.Y, R.Y2, R.Y3};
  int32_t* Ir[3] = {R.idx, R.idx2, R.idx3};
  float* yr[3] = {R.yY, R.yY2, R.yY3};
  float* rS[2] = {R.r, R.r2};
  float* aS[2] = {R.alpha, R.alpha2};
  float* fS[2] = {R.far, R.far2};
  float* fpS[2] = {fpart, R.fpart2};
  Ctrl* qS[2] = {R.ctrl, R.ctrl2};
  uint32_t* cS[2] = {R.slab, R.cnt2};
  for (int32_t it = 0; it < iters; ++it) {
    const int cur = it & 1, nxt = cur ^ 1;
    const uint64_t k = k0 + (uint64_t)it;
    // rows, labels and indices of this iteration (c) and the next (n)
    uint16_t* Yc = ahead ? Yr[it % 3] : Yb[cur];
    uint16_t* Yn = ahead ? Yr[(it + 1) % 3] : Yb[nxt];
    int32_t* Ic = ahead ? Ir[it % 3] : Ib[cur];
    int32_t* In = ahead ? Ir[(it + 1) % 3] : Ib[nxt];
    float* yc = ahead ? yr[it % 3] : yb[cur];
    float* yn = ahead ? yr[(it + 1) % 3] : yb[nxt];
    if ((rc = record(prof, it, 0, st)) != CASGD_OK) return rc;
    if (it == 0) {  // prologue: this iteration's rows and its Gram (far: its band)
      CK(launch_gather(*d, *p, w, k, nullptr, Ic, gather ? nullptr : Yc, L.ldY, R.r, yc,
                       R.alpha, R.far, nullptr, R.ctrl, R.slab, GATHER_ONLY, c));
      if (far)
        CK(launch_gram_band(gather ? nullptr : Yc, Gb[cur], L.S, d->n, L.ldY, p->b, p->s,
                            p->flags, R.ctrl, p->timeout_us, rsp, k * (uint64_t)L.S, c));
      else
        CK(launch_gram_tc(Yc, L.S, d->n, L.ldY, p->b, p->s, p->flags, 0, Gb[cur], R.ctrl,
                          p->timeout_us, c));
    }
    const int cs = ahead ? (it & 1) : 0;  // this iteration's state set
    if (far) {
      // next iteration's rows (gathering: its indices and labels only) and this
      // iteration's reset; with rows gathered ahead only in the first iteration (after
      // it, rows, indices, labels and state come with the launches before)
      if (!ahead || it == 0)
        CK(launch_gather_reset(*d, *p, k + 1, nullptr, In, gather ? nullptr : Yn, yn,
                               it + 1 < iters, L.ldY, R.r, R.alpha, R.far, fpart, R.ctrl,
                               R.slab, c));
    } else if (it + 1 < iters) {  // next iteration's rows (into the buffers the last launch
                                  // freed) and this iteration's margins, in one launch
      CK(launch_gather_next_margins(*d, *p, w, k + 1, In, Yn, yn, Yc, L.ldY, R.r, R.alpha,
                                    R.far, fpart, R.ctrl, R.slab, c));
    } else {
      CK(launch_gather(*d, *p, w, k, nullptr, Ic, Yc, L.ldY, R.r, yc, R.alpha, R.far, fpart,
                       R.ctrl, R.slab, MARGINS_ONLY, c));
    }
    if ((rc = record(prof, it, 1, st)) != CASGD_OK) return rc;
    // (The sum of G over processes would sit before this launch; on one GPU it is the
    // identity.)
    if (far) {  // this iteration's far sums; the next iteration's band (if any) into Gb[nxt]
      AheadRows ah{};
      NextSet nx{};
      const bool two = it + 2 < iters;
      if (ahead && two)
        ah = AheadRows{rs.X, rs.ld, rs.m, rs.seed, rs.perm_d, (k + 2) * (uint64_t)L.S,
                       Yr[(it + 2) % 3]};
      if (ahead && it + 1 < iters) {  // the next iteration's state; iteration k+2's labels
        const int ns = cs ^ 1;
        const int npb = far_partials_per_block(p->b, p->s);
        nx = NextSet{rS[ns], aS[ns], fS[ns], fpS[ns], qS[ns], cS[ns], p->s * npb, p->b,
                     band_width(p->b), npb, (int)((L.ldY + 63) / 64), p->s, d->y,
                     two ? yr[(it + 2) % 3] : nullptr, two ? Ir[(it + 2) % 3] : nullptr,
                     rs.seed, (k + 2) * (uint64_t)L.S, rs.m, rs.perm_d};
      }
      CK(launch_gram_recur(gather ? nullptr : (it + 1 < iters ? Yn : nullptr), Gb[nxt], true,
                           L.S, d->n, L.ldY, p->b, p->s, p->eta, p->loss, p->flags, Gb[cur],
                           gather ? nullptr : Yc, rS[cs], yc, aS[cs], fS[cs], R.slab, fpS[cs],
                           R.upd, w, true, R.ctrl, p->timeout_us, /*g_band=*/true, rsp,
                           it + 1 < iters ? (k + 1) * (uint64_t)L.S : kNoRows,
                           k * (uint64_t)L.S, ah.Y ? &ah : nullptr, qS[cs], cS[cs],
                           nx.r ? &nx : nullptr, c));
    } else if (it + 1 < iters) {
      CK(launch_gram_recur(Yn, Gb[nxt], true, L.S, d->n, L.ldY, p->b, p->s, p->eta, p->loss,
                           p->flags, Gb[cur], Yc, R.r, yc, R.alpha, R.far, R.slab, nullptr,
                           R.upd, w, false, R.ctrl, p->timeout_us, false, nullptr, 0, 0,
                           nullptr, nullptr, nullptr, nullptr, c));
    } else {
      CK(launch_recur(Gb[cur], R.r, yc, R.alpha, R.far, R.slab, p->b, p->s, p->eta, p->loss,
                      p->flags, p->timeout_us, R.ctrl, Yc, L.ldY, d->n, R.upd, w, c));
    }
    // the update (a8) finished inside that launch
    if ((rc = record(prof, it, 2, st)) != CASGD_OK) return rc;
    if ((rc = record(prof, it, 3, st)) != CASGD_OK) return rc;
    if ((rc = record(prof, it, 4, st)) != CASGD_OK) return rc;
    if (loss_every > 0 && (it + 1) % loss_every == 0) {
      CK(launch_loss(*d, p->loss, w, R.loss_part, R.loss_slots + slot, R.ctrl, c));
      if (++slot == kLossSlots) {
        CK(cudaMemcpyAsync(loss_hist + flushed, R.loss_slots, slot * sizeof(double),
                           cudaMemcpyDeviceToHost, st));
        CK(cudaStreamSynchronize(st));
        flushed += slot;
        slot = 0;
      }
    }
  }
  return CASGD_OK;
}

int status_to_code(uint32_t st) {
  if (st & ST_TIMEOUT) return CASGD_ERR_TIMEOUT;
  if (st & ST_BAD_INDEX) return CASGD_ERR_BAD_INDEX;
  if (st & ST_NONFINITE) return CASGD_ERR_NONFINITE;
  return CASGD_OK;
}

int read_and_clear_status(Ctrl* ctrl, cudaStream_t st) {
  uint32_t v = 0;
  CK(cudaMemcpyAsync(&v, &ctrl->status, sizeof(v), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  if (v != 0) {
    CK(cudaMemsetAsync(&ctrl->status, 0, sizeof(uint32_t), st));
    CK(cudaStreamSynchronize(st));
  }
  return status_to_code(v);
}

// ---------------------------------------------------- feature-sharded outer iteration
// The abstract's distributed setting: each process holds a slice of the features
// (columns of X and of w), every process draws the same rows, and the only exchange of
// an outer iteration is one sum over the processes of the sb x sb Gram matrix (with the
// margins), in FP32.  The far sums of the recurrence need the summed G, so these calls
// store G (the packed block-lower layout) into the caller's exchange buffer, followed
// by the S partial margins as FP32 sums (rounded once to BF16 only after the sum).
constexpr uint32_t kShardedUnsupported = CASGD_FLAG_FAR_FROM_GRAM | CASGD_FLAG_G_BF16;

uint32_t sharded_flags(uint32_t f) { return f | CASGD_FLAG_FULL_G | CASGD_FLAG_NO_FUSE; }

Layout sharded_layout(int64_t n, const casgd_params_t* p) {
  return make_layout(n, p->b, p->s, sharded_flags(p->flags), 0, false);
}

int64_t exchange_elems_of(const casgd_params_t* p) {
  return gram_elems(p->b, p->s, (p->flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0) +
         (int64_t)p->b * p->s;
}

int check_xbuf(const float* xbuf) {
  if (!xbuf || (reinterpret_cast<uintptr_t>(xbuf) % kAlign) != 0) return CASGD_ERR_ARG;
  return CASGD_OK;
}

int sharded_local_impl(const casgd_data_t* d, const casgd_params_t* p, const float* w,
                       uint64_t k, void* ws, size_t ws_bytes, float* xbuf,
                       const casgd_taps_t* taps, Ctx& c) {
  if (p->flags & kShardedUnsupported) return CASGD_ERR_UNSUPPORTED;
  const Layout L = sharded_layout(d->n, p);
  int rc = check_ws(ws, ws_bytes, L);
  if (rc != CASGD_OK) return rc;
  if ((rc = check_xbuf(xbuf)) != CASGD_OK) return rc;
  const Resolved R = resolve(ws, L);
  casgd_params_t q = *p;
  q.flags = sharded_flags(p->flags) | CASGD_FLAG_MARGINS_FP32;  // partial margins: FP32 sums
  const GramPlan gp = gram_plan(d->n, p->b, p->s, q.flags);
  if (gp.choice < 0) return CASGD_ERR_UNSUPPORTED;
  float* G = xbuf;
  float* r_part = xbuf + L.gram_elems;
  c.pdl = false;
  // rows, labels, indices, this slice's partial margins and the recurrence's reset
  CK(launch_gather(*d, q, w, k, taps ? taps->idx_in : nullptr, R.idx, R.Y, L.ldY, r_part, R.yY,
                   R.alpha, R.far, nullptr, R.ctrl, R.slab, GATHER_AND_MARGINS, c));
  if (gp.choice == 1)
    CK(launch_gram_tc(R.Y, L.S, d->n, L.ldY, p->b, p->s, q.flags, gp.mode, G, R.ctrl,
                      p->timeout_us, c));
  else
    CK(launch_gram_simt(R.Y, L.S, d->n, L.ldY, p->b, p->s,
                        (p->flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0, false, G, c));
  if (taps && taps->idx_out)
    CK(cudaMemcpyAsync(taps->idx_out, R.idx, L.S * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                       c.stream));
  return CASGD_OK;
}

int sharded_finish_impl(const casgd_data_t* d, const casgd_params_t* p, float* w, void* ws,
                        size_t ws_bytes, const float* xbuf, const casgd_taps_t* taps, Ctx& c) {
  if (p->flags & kShardedUnsupported) return CASGD_ERR_UNSUPPORTED;
  const Layout L = sharded_layout(d->n, p);
  int rc = check_ws(ws, ws_bytes, L);
  if (rc != CASGD_OK) return rc;
  if ((rc = check_xbuf(xbuf)) != CASGD_OK) return rc;
  const Resolved R = resolve(ws, L);
  const uint32_t flags = sharded_flags(p->flags);
  const bool r_fp32 = (p->flags & CASGD_FLAG_MARGINS_FP32) != 0;
  c.pdl = false;
  // the summed margins, rounded once (the recipe) or kept in FP32 (MARGINS_FP32)
  CK(launch_sharded_margins(xbuf + L.gram_elems, L.S, r_fp32, R.r, c));
  // recurrence on the summed G (identical on every process), then this slice's update
  CK(launch_recur(xbuf, R.r, R.yY, R.alpha, R.far, R.slab, p->b, p->s, p->eta, p->loss, flags,
                  p->timeout_us, R.ctrl, R.Y, L.ldY, d->n, R.upd, w, c));
  if (taps) {
    if (taps->r_out) {
      if (r_fp32)
        CK(cudaMemcpyAsync(taps->r_out, R.r, L.S * sizeof(float), cudaMemcpyDeviceToDevice,
                           c.stream));
      else
        CK(launch_bf16_bits(R.r, L.S, taps->r_out, c));
    }
    if (taps->alpha_out)
      CK(cudaMemcpyAsync(taps->alpha_out, R.alpha, L.S * sizeof(float),
                         cudaMemcpyDeviceToDevice, c.stream));
  }
  return CASGD_OK;
}

}  // namespace

Layout make_layout(int64_t n, int32_t b, int32_t s, uint32_t flags, int num_sms, bool with_G) {
  (void)num_sms;
  Layout L;
  L.S = (int64_t)b * s;
  // Y's pitch: whole 128-byte lines for wide rows (the Gram's TMA reads of a row segment
  // then touch one L2 line instead of two: measured 132 -> 128 us per shared launch at
  // n = 2000), 16-byte vectors for narrow ones
  L.ldY = n >= 128 ? (n + 63) / 64 * 64 : (n + 7) / 8 * 8;
  const bool diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  const GramPlan gp = gram_plan(n, b, s, flags);
  // the far-forming Gram keeps only the band blocks (band layout); the others store
  // every block of the packed block-lower G
  L.gram_elems = g_layout_elems(b, s, diag, gp.far ? band_width(b) : 0);
  int64_t u = (L.S + 31) / 32;
  L.upd_ctas = (int)(u > 320 ? 320 : u);
  size_t off = align_up(sizeof(Ctrl));
  L.off_loss = off;
  off += align_up((size_t)(kLossCtas + kLossSlots) * sizeof(double));
  L.off_idx = off;
  off += align_up((size_t)L.S * sizeof(int32_t));
  L.off_r = off;  // margins FP32[S] (BF16 values, or FP32 sums with MARGINS_FP32)
  off += align_up((size_t)L.S * sizeof(float));
  L.off_yY = off;
  off += align_up((size_t)L.S * sizeof(float));
  L.off_alpha = off;
  off += align_up((size_t)L.S * sizeof(float));
  L.off_far = off;  // far sums FP32[S]; the counters area (see timeline_of)
  off += align_up((size_t)L.S * sizeof(float)) +
         align_up((kMaxSlabs + kMaxUpdChunks + kMaxUpdBlocks) * sizeof(uint32_t) +
                  (kMaxS + 1) * 4 * sizeof(uint64_t));
  L.off_Y = off;
  off += align_up((size_t)L.S * L.ldY * sizeof(uint16_t));
  L.off_upd = off;
  // partial rows: upd_ctas for the two-kernel update, s * R for the update fused into
  // the recurrence (one row per block and row part)
  const int64_t upd_fused = (int64_t)s * upd_row_parts(b, L.ldY);
  const int64_t upd_rows = L.upd_ctas > upd_fused ? L.upd_ctas : upd_fused;
  off += align_up((size_t)upd_rows * L.ldY * sizeof(float));
  L.off_G = with_G ? off : 0;
  if (with_G) off += align_up((size_t)L.gram_elems * sizeof(float));
  L.off_Y2 = L.off_G2 = L.off_idx2 = L.off_yY2 = L.off_fpart = 0;
  L.off_Y3 = L.off_idx3 = L.off_yY3 = 0;
  L.off_ctrl2 = L.off_cnt2 = L.off_r2 = L.off_alpha2 = L.off_far2 = L.off_fpart2 = 0;
  if (gp.fused) {  // casgd_train gathers the rows (and runs the Gram) one iteration ahead
    L.off_idx2 = off;
    off += align_up((size_t)L.S * sizeof(int32_t));
    L.off_yY2 = off;
    off += align_up((size_t)L.S * sizeof(float));
    if (!(gp.far && (flags & CASGD_FLAG_GATHER_ROWS))) {  // (gathering from X: no second Y)
      L.off_Y2 = off;
      off += align_up((size_t)L.S * L.ldY * sizeof(uint16_t));
    }
    L.off_G2 = off;  // the far-forming Gram stores the next iteration's band into it
    off += align_up((size_t)L.gram_elems * sizeof(float));
  }
  if (gp.far) {
    L.off_fpart = off;
    off += align_up((size_t)L.S * s * far_partials_per_block(b, s) * sizeof(float));
  }
  if (gp.fused && gp.far && !(flags & CASGD_FLAG_GATHER_ROWS) && ahead_rows_supported(n, L.ldY)) {
    L.off_idx3 = off;
    off += align_up((size_t)L.S * sizeof(int32_t));
    L.off_yY3 = off;
    off += align_up((size_t)L.S * sizeof(float));
    L.off_Y3 = off;
    off += align_up((size_t)L.S * L.ldY * sizeof(uint16_t));
    L.off_ctrl2 = off;
    off += align_up(sizeof(Ctrl));
    L.off_cnt2 = off;
    off += align_up((kMaxSlabs + kMaxUpdChunks + kMaxUpdBlocks) * sizeof(uint32_t) +
                    (kMaxS + 1) * 4 * sizeof(uint64_t));
    L.off_r2 = off;
    off += align_up((size_t)L.S * sizeof(float));
    L.off_alpha2 = off;
    off += align_up((size_t)L.S * sizeof(float));
    L.off_far2 = off;
    off += align_up((size_t)L.S * sizeof(float));
    L.off_fpart2 = off;
    off += align_up((size_t)L.S * s * far_partials_per_block(b, s) * sizeof(float));
  }
  L.total = off;
  return L;
}

}  // namespace casgd

using namespace casgd;

extern "C" {

const char* casgd_strerror(int code) {
  switch (code) {
    case CASGD_OK: return "ok";
    case CASGD_ERR_ARG: return "invalid argument";
    case CASGD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CASGD_ERR_CUDA: return "CUDA runtime error";
    case CASGD_ERR_NONFINITE: return "non-finite weight produced on the device";
    case CASGD_ERR_TIMEOUT: return "an inter-CTA wait on the device exceeded its time bound";
    case CASGD_ERR_BAD_INDEX: return "a given row index is outside [0, m)";
    case CASGD_ERR_UNSUPPORTED: return "request not supported by this build";
    case CASGD_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of casgd_update_static";
    case CASGD_ERR_EXCHANGE: return "the caller's exchange (sum over processes) reported a failure";
    default: return "unknown casgd status";
  }
}

int casgd_version(void) { return CASGD_ABI_VERSION; }

int64_t casgd_gram_elems(int32_t b, int32_t s, uint32_t flags) {
  if (b < 1 || s < 1 || s > kMaxS || (int64_t)b * s > kMaxSB) return -1;
  return gram_elems(b, s, (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0);
}

int casgd_workspace_size(const casgd_data_t* data, const casgd_params_t* params,
                         size_t* bytes) {
  if (!bytes || !check_params(params)) return CASGD_ERR_ARG;
  if (!data || data->n < 1 || data->n > kMaxN) return CASGD_ERR_ARG;
  *bytes = make_layout(data->n, params->b, params->s, params->flags, 0).total;
  return CASGD_OK;
}

int casgd_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < sizeof(Ctrl))
    return CASGD_ERR_WORKSPACE;
  if (cudaMemsetAsync(ws, 0, sizeof(Ctrl), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CASGD_ERR_CUDA;
  return CASGD_OK;
}

int casgd_store_bf16(const float* src, int64_t m, int64_t n, int64_t ld_src, void* dst,
                     int64_t ld_dst, void* stream) {
  if (!src || !dst || m < 0 || n < 1 || ld_src < n || ld_dst < n || (ld_dst % 8) != 0)
    return CASGD_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0) return CASGD_ERR_ARG;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  return launch_store_bf16(src, m, n, ld_src, static_cast<uint16_t*>(dst), ld_dst, c) ==
                 cudaSuccess ? CASGD_OK : CASGD_ERR_CUDA;
}

int casgd_sample_indices(int64_t m, int64_t count, uint64_t seed, uint64_t counter0,
                         int32_t* idx, void* stream) {
  if (m < 1 || m >= (int64_t(1) << 31) || count < 0 || (count > 0 && !idx)) return CASGD_ERR_ARG;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  return launch_sample(m, count, seed, counter0, false, idx, c) == cudaSuccess
             ? CASGD_OK
             : CASGD_ERR_CUDA;
}

int casgd_sample_indices_permuted(int64_t m, int64_t count, uint64_t seed, uint64_t counter0,
                                  int32_t* idx, void* stream) {
  if (m < 1 || m >= (int64_t(1) << 31) || count < 0 || (count > 0 && !idx)) return CASGD_ERR_ARG;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  return launch_sample(m, count, seed, counter0, true, idx, c) == cudaSuccess
             ? CASGD_OK
             : CASGD_ERR_CUDA;
}

int casgd_outer_step(const casgd_data_t* data, const casgd_params_t* params, float* w,
                     uint64_t k, void* ws, size_t ws_bytes, void* stream,
                     const casgd_taps_t* taps) {
  if (!check_data(data) || !check_params(params) || !w) return CASGD_ERR_ARG;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  return outer_step_impl(data, params, w, k, ws, ws_bytes, c.stream, taps, c, nullptr, 0);
}

int casgd_loss_async(const casgd_data_t* data, int32_t loss, const float* w, void* ws,
                     size_t ws_bytes, void* stream, double* out_dev) {
  if (!check_data(data) || !w || !out_dev || loss < CASGD_LOGISTIC || loss > CASGD_POISSON)
    return CASGD_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < loss_only_bytes())
    return CASGD_ERR_WORKSPACE;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  Layout L = make_layout(data->n, 1, 1, 0, c.num_sms);
  Resolved R = resolve(ws, L);
  return launch_loss(*data, loss, w, R.loss_part, out_dev, R.ctrl, c) == cudaSuccess
             ? CASGD_OK : CASGD_ERR_CUDA;
}

int casgd_loss(const casgd_data_t* data, int32_t loss, const float* w, void* ws,
               size_t ws_bytes, void* stream, double* out) {
  if (!out) return CASGD_ERR_ARG;
  if (!check_data(data) || !w || loss < CASGD_LOGISTIC || loss > CASGD_POISSON)
    return CASGD_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < loss_only_bytes())
    return CASGD_ERR_WORKSPACE;
  Layout L = make_layout(data->n, 1, 1, 0, 0);
  Resolved R = resolve(ws, L);
  int rc = casgd_loss_async(data, loss, w, ws, ws_bytes, stream, R.loss_slots);
  if (rc != CASGD_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(out, R.loss_slots, sizeof(double), cudaMemcpyDeviceToHost, st));
  return read_and_clear_status(R.ctrl, st);
}

int casgd_train_host(const void* X_host, const float* y_host, float* w_host,
                     const casgd_data_t* data, float* w_dev, const casgd_params_t* params,
                     uint64_t k0, int32_t iters, void* ws, size_t ws_bytes, void* stream,
                     int32_t loss_every, double* loss_hist, casgd_profile_t* prof) {
  if (!X_host || !y_host || !w_host || !w_dev || !check_data(data)) return CASGD_ERR_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xbytes = (size_t)data->m * (size_t)data->ld * sizeof(uint16_t);
  if (cudaMemcpyAsync(const_cast<void*>(data->X), X_host, xbytes, cudaMemcpyHostToDevice,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(const_cast<float*>(data->y), y_host, (size_t)data->m * sizeof(float),
                      cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(w_dev, w_host, (size_t)data->n * sizeof(float), cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return CASGD_ERR_CUDA;
  const int rc = casgd_train(data, params, w_dev, k0, iters, ws, ws_bytes, stream, loss_every,
                             loss_hist, prof);
  if (rc != CASGD_OK) return rc;
  if (cudaMemcpyAsync(w_host, w_dev, (size_t)data->n * sizeof(float), cudaMemcpyDeviceToHost,
                      st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return CASGD_ERR_CUDA;
  return CASGD_OK;
}

int casgd_train(const casgd_data_t* data, const casgd_params_t* params, float* w,
                uint64_t k0, int32_t iters, void* ws, size_t ws_bytes, void* stream,
                int32_t loss_every, double* loss_hist, casgd_profile_t* prof) {
  if (!check_data(data) || !check_params(params) || !w || iters < 0 || loss_every < 0)
    return CASGD_ERR_ARG;
  if (loss_every > 0 && iters / loss_every > 0 && !loss_hist) return CASGD_ERR_ARG;
  LaunchCache cache;  // occupancy of the kernels the loop repeats, found once per call
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0, &cache};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  const Layout L = make_layout(data->n, params->b, params->s, params->flags, c.num_sms);
  int rc = check_ws(ws, ws_bytes, L);
  if (rc != CASGD_OK) return rc;
  Resolved R = resolve(ws, L);
  int slot = 0, flushed = 0;
  if (iters >= 2 && L.off_G2 != 0) {  // the second buffers of the pipelined loop exist
    rc = train_pipelined(data, params, w, k0, iters, L, R, c, prof, loss_every, slot, flushed,
                         loss_hist, L.off_fpart != 0);
    if (rc != CASGD_OK) return rc;
    iters = 0;  // done
  }
  for (int32_t it = 0; it < iters; ++it) {
    rc = outer_step_impl(data, params, w, k0 + (uint64_t)it, ws, ws_bytes, c.stream, nullptr,
                         c, prof, it);
    if (rc != CASGD_OK) return rc;
    if (loss_every > 0 && (it + 1) % loss_every == 0) {
      CK(launch_loss(*data, params->loss, w, R.loss_part, R.loss_slots + slot, R.ctrl, c));
      if (++slot == kLossSlots) {
        CK(cudaMemcpyAsync(loss_hist + flushed, R.loss_slots, slot * sizeof(double),
                           cudaMemcpyDeviceToHost, c.stream));
        CK(cudaStreamSynchronize(c.stream));
        flushed += slot;
        slot = 0;
      }
    }
  }
  if (slot > 0)
    CK(cudaMemcpyAsync(loss_hist + flushed, R.loss_slots, slot * sizeof(double),
                       cudaMemcpyDeviceToHost, c.stream));
  if (prof) prof->launches = c.launches;
  return read_and_clear_status(R.ctrl, c.stream);
}

int64_t casgd_exchange_elems(int32_t b, int32_t s, uint32_t flags) {
  casgd_params_t p{};
  p.b = b;
  p.s = s;
  p.flags = flags;
  p.eta = 0.0f;
  if (!check_params(&p)) return -1;
  return exchange_elems_of(&p);
}

int casgd_workspace_size_sharded(const casgd_data_t* data, const casgd_params_t* params,
                                 size_t* bytes) {
  if (!bytes || !check_params(params)) return CASGD_ERR_ARG;
  if (!data || data->n < 1 || data->n > kMaxN) return CASGD_ERR_ARG;
  if (params->flags & kShardedUnsupported) return CASGD_ERR_UNSUPPORTED;
  *bytes = sharded_layout(data->n, params).total;
  return CASGD_OK;
}

int casgd_outer_step_local(const casgd_data_t* data, const casgd_params_t* params,
                           const float* w, uint64_t k, void* ws, size_t ws_bytes, void* stream,
                           float* xbuf, const casgd_taps_t* taps) {
  if (!check_data(data) || !check_params(params) || !w) return CASGD_ERR_ARG;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  return sharded_local_impl(data, params, w, k, ws, ws_bytes, xbuf, taps, c);
}

int casgd_outer_step_finish(const casgd_data_t* data, const casgd_params_t* params, float* w,
                            void* ws, size_t ws_bytes, void* stream, const float* xbuf,
                            const casgd_taps_t* taps) {
  if (!check_data(data) || !check_params(params) || !w) return CASGD_ERR_ARG;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  return sharded_finish_impl(data, params, w, ws, ws_bytes, xbuf, taps, c);
}

int casgd_train_sharded(const casgd_data_t* data, const casgd_params_t* params, float* w,
                        uint64_t k0, int32_t iters, void* ws, size_t ws_bytes, void* stream,
                        float* xbuf, casgd_exchange_fn exchange, void* exchange_ctx,
                        casgd_profile_t* prof) {
  if (!check_data(data) || !check_params(params) || !w || iters < 0 || !exchange)
    return CASGD_ERR_ARG;
  LaunchCache cache;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0, &cache};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  const int64_t count = exchange_elems_of(params);
  if (params->flags & kShardedUnsupported) return CASGD_ERR_UNSUPPORTED;
  int rc = check_ws(ws, ws_bytes, sharded_layout(data->n, params));
  if (rc != CASGD_OK) return rc;
  if ((rc = check_xbuf(xbuf)) != CASGD_OK) return rc;
  for (int32_t it = 0; it < iters; ++it) {
    if ((rc = record(prof, it, 0, c.stream)) != CASGD_OK) return rc;
    rc = sharded_local_impl(data, params, w, k0 + (uint64_t)it, ws, ws_bytes, xbuf, nullptr, c);
    if (rc != CASGD_OK) return rc;
    if ((rc = record(prof, it, 1, c.stream)) != CASGD_OK) return rc;
    // the one exchange of the outer iteration, issued by the caller on `stream`
    if (exchange(exchange_ctx, xbuf, count, stream) != 0) return CASGD_ERR_EXCHANGE;
    if ((rc = record(prof, it, 2, c.stream)) != CASGD_OK) return rc;
    rc = sharded_finish_impl(data, params, w, ws, ws_bytes, xbuf, nullptr, c);
    if (rc != CASGD_OK) return rc;
    if ((rc = record(prof, it, 3, c.stream)) != CASGD_OK) return rc;
    if ((rc = record(prof, it, 4, c.stream)) != CASGD_OK) return rc;
  }
  if (prof) {
    prof->launches = c.launches;
    prof->gram_kind = 7;
  }
  return read_and_clear_status(static_cast<Ctrl*>(ws), c.stream);
}

int casgd_get_status(void* ws, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return CASGD_ERR_WORKSPACE;
  return read_and_clear_status(static_cast<Ctrl*>(ws), static_cast<cudaStream_t>(stream));
}

int casgd_sgd_workspace_size(int32_t b, size_t* bytes) {
  if (!bytes || b < 1 || b > (1 << 20)) return CASGD_ERR_ARG;
  *bytes = sgd_workspace_bytes(b);
  return CASGD_OK;
}

int casgd_sgd_fp32(const float* X, int64_t m, int64_t n, int64_t ld, const float* y,
                   const casgd_params_t* params, float* w, uint64_t q0, int32_t steps, void* ws,
                   size_t ws_bytes, void* stream) {
  if (!X || !y || !w || !params || m < 1 || m >= (int64_t(1) << 31) || n < 1 || n > kMaxN ||
      ld < n || steps < 0)
    return CASGD_ERR_ARG;
  if (params->b < 1 || params->b > (1 << 20) || params->loss < CASGD_LOGISTIC ||
      params->loss > CASGD_POISSON || !(params->eta == params->eta))
    return CASGD_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 ||
      ws_bytes < sgd_workspace_bytes(params->b))
    return CASGD_ERR_WORKSPACE;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  if (device_sms(&c.num_sms) != CASGD_OK) return CASGD_ERR_CUDA;
  CK(launch_sgd_fp32(X, m, n, ld, y, *params, w, q0, steps, ws, c));
  return CASGD_OK;
}

int casgd_chain_trace(const casgd_data_t* data, const casgd_params_t* params, void* ws,
                      size_t ws_bytes, void* stream, uint64_t* out) {
  if (!out || !check_params(params) || !data || data->n < 1 || data->n > kMaxN)
    return CASGD_ERR_ARG;
  const Layout L = make_layout(data->n, params->b, params->s, params->flags, 0);
  int rc = check_ws(ws, ws_bytes, L);
  if (rc != CASGD_OK) return rc;
  Resolved R = resolve(ws, L);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(out, R.trace, (size_t)params->s * 4 * sizeof(uint64_t),
                     cudaMemcpyDeviceToHost, st));
  CK(cudaMemcpyAsync(out + (size_t)params->s * 4, R.trace + (size_t)kMaxS * 4,
                     4 * sizeof(uint64_t), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  return CASGD_OK;
}

}  // extern "C"
