// fused_linear_residual_rmsnorm_fp8_noalloc: the residual + RMSNorm + FP8
// entry point for callers that cannot allocate device memory.
//
// Who needs this: code that must never reach the CUDA allocator while it runs,
// for example a serving step with a hard latency budget (cudaMalloc can
// synchronise the device and take milliseconds), or a plugin inside a host
// framework that owns all device memory and gives the plugin none of it.  Such
// callers cannot hand us a workspace.
//
// Instead of a caller-provided workspace, this entry point uses one fixed
// scratch array compiled into the library (kNoAllocScratchBytes, 8 MiB).  Every
// GPU that loads the library holds that array until the process exits.  The
// array is shared by all calls: calls that may overlap on the GPU (different
// streams without ordering between them) race on it and must not be issued.
// Every check of the workspace entry point runs first; only a call that passes
// them all enqueues anything: the clear of the counters the kernels wait on
// (an asynchronous memset on the caller's stream, so a call that timed out
// leaves no stale counts behind), then the kernel.  No cudaMalloc, cudaFree or
// allocating library routine is called.
#include <mutex>

#include "host_common.h"

namespace fl {
namespace {

constexpr size_t kNoAllocScratchBytes = FL_NOALLOC_SCRATCH_BYTES;
// Scratch for the no-allocation entry point; zero-filled when the module loads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev];

// Device address of the scratch array for `device` (the current device).  The
// name g_noalloc_scratch is only a host-side handle in host code; the kernels
// must be given this address.  Looked up once per device (the first call on
// that device), with the device current; the address then stays valid for the
// life of the process's CUDA context on that device.
void* scratch_address(int device) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (device < 0 || device >= kMaxDev) return nullptr;
  if (g_noalloc_ptr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[device] = p;
  }
  return g_noalloc_ptr[device];
}

}  // namespace
}  // namespace fl

extern "C" int fused_linear_residual_rmsnorm_fp8_noalloc(const void* X, const void* W, const void* b,
                                                         const void* Z, const void* gamma, float eps, void* Yq,
                                                         float* row_scale, int M, int N, int K, int64_t ldx,
                                                         int64_t ldw, int64_t ldz, int64_t ldq, void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0 || !(eps >= 0.f)) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  DeviceInfo di;
  const int st = current_device(&di);
  if (st != FL_OK) return st;
  void* scratch = scratch_address(di.device);
  if (scratch == nullptr) return FL_ERR_CUDA;
  // A shape whose workspace exceeds the scratch array fails with FL_ERR_WORKSPACE, like a
  // workspace that is too small.
  return rmsnorm_fp8_enqueue(X, W, b, Z, gamma, eps, Yq, row_scale, nullptr, M, N, K, ldx, ldw, ldz, ldq, scratch,
                             kNoAllocScratchBytes, static_cast<cudaStream_t>(stream), true);
}
