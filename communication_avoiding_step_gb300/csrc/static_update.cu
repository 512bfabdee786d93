// casgd_update_static: the weight update w += Y^T alpha without any caller-provided
// workspace and without allocating device memory.
//
// Some callers cannot allocate device memory at the point where they want to apply an
// update: code running inside another framework's memory pool that forbids raw
// cudaMalloc, real-time loops that must not block on the allocator, or embedders that
// hand this library only the buffers they already own.  This entry point serves them:
// the scratch it needs (one FP32 partial row per CTA of the update, and a status word)
// lives in a fixed array compiled into the library, held by every GPU that loads it
// until the process exits.
//
// The array has room for 1,048,576 partial floats (4 MiB) plus a 512-byte control
// block.  The update uses P = min(ceil(S/32), 320) partial rows of ldY floats, so
// P * ldY must be at most 1,048,576 (for example n <= 3272 at the largest P);
// larger requests are refused with CASGD_ERR_SCRATCH_LIMIT before anything runs.
//
// All calls share the one array and it keeps whatever the previous call left.  The
// partial rows are overwritten completely on every call; the status word is cleared
// at the start of each call.  Calls whose kernels overlap on the GPU (for instance on
// two streams at once) race on the array and must be serialised by the caller.
#include <cuda.h>

#include <mutex>

#include "casgd_internal.cuh"

namespace casgd {
namespace {

constexpr int64_t kStaticPartials = int64_t(1) << 20;  // floats of partial rows
constexpr int64_t kStaticCtrlFloats = 128;             // 512 bytes for the control block
constexpr int kMaxDevices = 64;

// The fixed scratch: a control block followed by the partial rows.
static __device__ __align__(256) float g_static_update_scratch[kStaticCtrlFloats + kStaticPartials];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};  // context the address belongs to

// Unique id (over the process's life) of the calling thread's current context, from the
// driver API through the runtime's entry-point lookup; 0 if it cannot be found.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_cur || !get_id) {
    void* p1 = nullptr;
    void* p2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 12000, cudaEnableDefault,
                                         &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return 0;
    get_cur = reinterpret_cast<CtxGetCurrentFn>(p1);
    get_id = reinterpret_cast<CtxGetIdFn>(p2);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch on the current device.  Host code only sees a host-side
// stand-in under the array's name, so the address is looked up with that device current
// (cudaGetSymbolAddress) the first time a call runs in a context of that device, and
// kept with the context's unique id: a device reset (cudaDeviceReset) or a new primary
// context in this process gives a new id, so the address is looked up again instead of
// pointing into the old context's memory.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CASGD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CASGD_ERR_UNSUPPORTED;
  const unsigned long long id = current_context_id();  // 0: no context bound yet
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_addr[dev] || id == 0 || g_ctx_id[dev] != id) {
    void* p = nullptr;
    // (binds the device's primary context first if the thread had none)
    if (cudaGetSymbolAddress(&p, g_static_update_scratch) != cudaSuccess || !p)
      return CASGD_ERR_CUDA;
    g_addr[dev] = p;
    g_ctx_id[dev] = id ? id : current_context_id();
  }
  *out = g_addr[dev];
  return CASGD_OK;
}

}  // namespace
}  // namespace casgd

using namespace casgd;

extern "C" int casgd_update_static(const void* Y, int64_t S, int64_t n, int64_t ldY,
                                   const float* alpha, float* w, void* stream) {
  if (!Y || !alpha || !w) return CASGD_ERR_ARG;
  if (S < 1 || S > kMaxSB || n < 1 || n > kMaxN || ldY < n || (ldY % 8) != 0)
    return CASGD_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(Y) & 15u) != 0) return CASGD_ERR_ARG;
  const int64_t u = (S + 31) / 32;
  const int upd_ctas = (int)(u > 320 ? 320 : u);  // the same split the outer step uses
  if ((int64_t)upd_ctas * ldY > kStaticPartials) return CASGD_ERR_SCRATCH_LIMIT;

  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc != CASGD_OK) return rc;
  Ctx c{static_cast<cudaStream_t>(stream), 0, 0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CASGD_ERR_CUDA;
  Ctrl* ctrl = static_cast<Ctrl*>(base);
  float* part = static_cast<float*>(base) + kStaticCtrlFloats;
  if (cudaMemsetAsync(&ctrl->status, 0, sizeof(uint32_t), c.stream) != cudaSuccess)
    return CASGD_ERR_CUDA;
  return launch_update(static_cast<const uint16_t*>(Y), alpha, S, n, ldY, w, part, upd_ctas,
                       ctrl, c) == cudaSuccess
             ? CASGD_OK
             : CASGD_ERR_CUDA;
}
