// fused_linear_residual_rmsnorm_fp8_noalloc: the residual + RMSNorm + FP8
// entry point for callers that cannot allocate device memory.
//
// Who needs this: code that must never reach the CUDA allocator while it runs,
// for example a decode loop being recorded into a CUDA graph (an allocation
// inside a capture breaks the capture), a serving step with a hard latency
// budget (cudaMalloc can synchronise the device and take milliseconds), or a
// plugin inside a host framework that owns all device memory and gives the
// plugin none of it.  Such callers cannot hand us a workspace.
//
// Instead of a caller-provided workspace, this entry point uses one fixed
// scratch array compiled into the library (kNoAllocScratchBytes, 8 MiB).  Every
// GPU that loads the library holds that array until the process exits.  The
// array is shared by all calls: calls that may overlap on the GPU (different
// streams without ordering between them) race on it and must not be issued.
// The counters the kernels wait on are cleared with an asynchronous memset on
// the caller's stream before every launch, so a call that timed out leaves no
// stale state behind.  No cudaMalloc, cudaFree or allocating library routine
// is called.
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
// must be given this address.  Looked up once per device.
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
  // Argument checks come first so that a rejected call enqueues nothing, not
  // even the counter clear below.
  if (M < 0 || N < 0 || K < 0 || !(eps >= 0.f)) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Z == nullptr || gamma == nullptr || Yq == nullptr || row_scale == nullptr ||
      (K > 0 && (X == nullptr || W == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldz < N || ldq < N || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(b) || !aligned16(Z) || !aligned16(gamma) || !aligned16(Yq) ||
      !aligned16(row_scale))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldz, 2) || !pitch_ok(ldq, 1) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2))))
    return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  const int st = current_device(&di);
  if (st != FL_OK) return st;
  const size_t need = fl_rmsnorm_fp8_workspace_bytes(M, N, K);
  if (need > kNoAllocScratchBytes) return FL_ERR_WORKSPACE;  // shape too large for the static scratch
  void* scratch = scratch_address(di.device);
  if (scratch == nullptr) return FL_ERR_CUDA;
  // The arrival counters sit at the start of the scratch layout and must start
  // at zero: decode (M <= 32, K > 0) keeps N/128 + 2 of them, prefill 2 per
  // 128-row block; the region is padded to 256 bytes.
  const size_t counters = (M <= 32 && K > 0) ? static_cast<size_t>(cdiv(N, 128) + 2) * sizeof(unsigned)
                                             : static_cast<size_t>(2 * cdiv(M, kBM)) * sizeof(unsigned);
  const size_t clear = (counters + 255) / 256 * 256;
  if (cudaMemsetAsync(scratch, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FL_ERR_CUDA;
  return fused_linear_residual_rmsnorm_fp8(X, W, b, Z, gamma, eps, Yq, row_scale, M, N, K, ldx, ldw, ldz, ldq,
                                           scratch, kNoAllocScratchBytes, stream);
}
