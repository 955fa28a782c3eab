// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.  The pages describe nothing like it; it exists for integration.
//
// fa_bwd needs a caller-provided workspace (the row statistic D and the fp32
// dQ accumulator).  Some callers have no way to provide one: a plugin inside
// another runtime that is handed only its input and output tensors, or code
// on a path where a device allocation is not allowed (cudaMalloc can
// synchronise the device and can fail under memory pressure).  For them this
// entry point takes its scratch from a fixed array in the library's own
// device memory instead.
//
// Rules that follow from sharing one static array:
//  * The array holds kNoAllocScratchBytes (32 MiB) on every GPU that loads
//    the library, until the process exits.  Problems whose workspace
//    (fa_bwd_workspace_size) exceeds it are rejected with FA_ERR_WORKSPACE
//    before anything is launched.
//  * Every call uses the same array and the array keeps the last call's
//    contents; the backward preprocess step rewrites D and zeroes the dQ
//    accumulator at the start of every call, so nothing stale is read.
//  * Calls that overlap on the GPU (different streams, or different host
//    threads without ordering) race on the array.  Order them on one stream.
//  * The first call on a device resolves the array's device address with
//    cudaGetSymbolAddress, with that device current; make that first call
//    before any stream capture.  The address is kept together with the
//    driver context it belongs to: after cudaDeviceReset (or under another
//    context on the same device) the library's module is loaded afresh, so
//    a call made under a context other than the recorded one looks the
//    address up again instead of reusing a stale one.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "fa_host.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (the library links
// the static runtime and not libcuda directly), resolved once.
CtxGetCurrentFn resolve_ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

std::mutex g_scratch_mu;
struct ScratchAddr {
  CUcontext ctx;
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// The kernels of this library exist for sm_103 only: on any other device the
// symbol lookup below would fail for want of a code image.
fa_status check_current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return FA_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess)
    return FA_ERR_UNSUPPORTED;
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  if (*dev < 0 || *dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Device address of g_noalloc_scratch for the current device and context
// (looked up once per device and context).  In host code the array's name is
// only a host-side handle, never a device address, so kernels receive this
// pointer instead.
fa_status scratch_for_current_device(void** out) {
  int dev = 0;
  fa_status st = check_current_device(&dev);
  if (st != FA_OK) return st;
  CtxGetCurrentFn get_ctx = resolve_ctx_get_current();
  CUcontext ctx = nullptr;
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& e = g_scratch[dev];
  if (e.ptr == nullptr || e.ctx != ctx || ctx == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear the failed lookup's error so that no later call reports it
      e.ptr = nullptr;
      return FA_ERR_LAUNCH;
    }
    // The runtime makes the primary context current during the lookup when
    // none was: record the context the address now belongs to.
    CUcontext now = nullptr;
    if (get_ctx(&now) != CUDA_SUCCESS) return FA_ERR_LAUNCH;
    e.ctx = now;
    e.ptr = p;
  }
  *out = e.ptr;
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    int causal, float scale, void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  // need == 0 only for sizes fa_bwd rejects: its checks name the error (they
  // run before it looks at the workspace).
  if (need == 0) return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, nullptr, 0, B, H, N, d, causal, scale, stream);
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const fa_status st = scratch_for_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, N, d, causal, scale, stream);
}
