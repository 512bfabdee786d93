// Steps a6/a7 (and the first stage of a8) as a stand-alone persistent launch, for Gram
// variants that run as their own kernel.  The roles (chain and bulk groups, fused update
// units, data-synchronised waits) are described in recur_roles.cuh.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the inner recurrence runs in high precision.
//
// One cooperative launch (all CTAs co-resident): the first C CTAs run the chain role,
// the others the bulk role, each CTA being one 256-thread role group.
#include "recur_roles.cuh"

namespace casgd {

namespace {

template <int kB, int kKB>
__global__ void __launch_bounds__(kRecThreads) recur_kernel(RecArgs a) {
  if ((int)blockIdx.x < a.C)
    chain_role<kB, kKB, 0>(a, blockIdx.x, threadIdx.x);
  else
    bulk_role<0>(a, threadIdx.x, (int)blockIdx.x - a.C < a.upd_groups);
}

}  // namespace

RecArgs make_rec_args(const float* G, const float* r, const float* yY, float* alpha,
                      float* far, uint32_t* counters, int b, int s, float eta, int loss,
                      uint32_t flags, uint32_t timeout_us, Ctrl* ctrl, const uint16_t* Y,
                      int64_t ldY, int64_t n, float* part, float* w) {
  RecArgs a;
  a.G = G;
  a.gB = 0;  // packed block-lower G (the far-forming launch sets the band layout)
  a.X = nullptr;  // rows from Y (the far-forming launch may read them from X instead)
  a.ldx = 0;
  a.xseed = a.xctr = 0;
  a.xm = 0;
  a.xperm = 0;
  a.r = r;
  a.yY = yY;
  a.alpha = alpha;
  a.far = far;
  a.trace = (flags & CASGD_FLAG_TRACE_CHAIN) ? timeline_of(counters) : nullptr;
  a.upd_chunks = upd_chunk_counters(counters);
  a.upd_blocks = upd_block_counters(counters);
  a.w = w;
  a.n = n;
  a.ctrl = ctrl;
  a.q = ctrl;
  a.timeout_ns = (uint64_t)(timeout_us ? timeout_us : 1000000u) * 1000ull;
  a.b = b;
  a.s = s;
  a.S = (int64_t)b * s;
  a.loss = loss;
  a.U = (b + kRecRows - 1) / kRecRows;
  a.Uc = (b + kChainRows - 1) / kChainRows;
  a.vec4 = (b % 4) == 0;
  a.B = band_width(b);  // as many blocks as a chain lane holds in registers
  a.bulk_units = 0;  // far units: (block, chunk of kT blocks) pairs x row units
  for (int j = a.B + 1; j < s; ++j) a.bulk_units += a.U;
  a.coef = -(eta / (float)b);
  a.Y = Y;
  a.part = part;
  a.ldY = ldY;
  // update units: s blocks x ceil(ldY / 64) column chunks (x R row parts where the far
  // sums come from the Gram: launch_gram_recur)
  a.upd_R = 1;
  a.upd_units = s * (int)((ldY / 8 + 7) / 8);
  a.slab = nullptr;
  a.fpart = nullptr;
  a.fs = a.npb = 0;
  a.band_total = 0;
  a.margins = a.wm_vec = false;
  a.r_fp32 = (flags & CASGD_FLAG_MARGINS_FP32) != 0;
  a.mrows = a.mG = 0;
  a.r_w = nullptr;
  a.wm = nullptr;
  a.far_gram = false;
  a.C = 0;
  a.upd_groups = 0;
  a.diag = (flags & CASGD_FLAG_WRITE_DIAG_BLOCKS) != 0;
  a.stall_test = (flags & CASGD_FLAG_TEST_STALL) != 0;
  return a;
}

cudaError_t launch_recur(const float* G, const float* r, const float* yY, float* alpha,
                         float* far, uint32_t* counters, int b, int s, float eta, int loss,
                         uint32_t flags, uint32_t timeout_us, Ctrl* ctrl, const uint16_t* Y,
                         int64_t ldY, int64_t n, float* part, float* w, Ctx& c) {
  RecArgs a = make_rec_args(G, r, yY, alpha, far, counters, b, s, eta, loss, flags, timeout_us,
                            ctrl, Y, ldY, n, part, w);
  const int v = chain_variant(a);
  const void* fn = v == 3   ? (const void*)recur_kernel<3, 2>
                   : v == 2 ? (const void*)recur_kernel<2, 4>
                            : (const void*)recur_kernel<1, 8>;
  int per_sm = 0;
  cudaError_t e = cached_query(c, fn, [&](int& v) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, kRecThreads, 0);
  }, per_sm);
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
  a.upd_groups = update_groups(a, (int)(grid - a.C));
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel(fn, dim3((unsigned)grid), dim3(kRecThreads), args, 0, c.stream);
  ++c.launches;
  return e;
}

}  // namespace casgd
