// Host-side helpers shared by the entry points: device query, the device
// status word, tensor-map encoding, argument checks and kernel launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "fused_linear.h"
#include "gemm_kernel.cuh"

namespace fl {

struct DeviceInfo {
  int device;
  int num_sms;
  int cc;  // major * 10 + minor
};

// Current device, its SM count and compute capability; FL_ERR_ARCH unless sm_103.
int current_device(DeviceInfo* out);
// Device address of this library's status word on the current device.
int* device_status_ptr(int device);
uint64_t wait_timeout_ns();
int max_ctas_override();
// Makes sure the kernel may use `smem_bytes` of dynamic shared memory on `device`.
bool ensure_smem_attr(const void* kernel, int device, int smem_bytes);

// 2-D tiled tensor map over a row-major [outer, inner] matrix with row pitch
// `ld_elems` elements of `elem_bytes` bytes each.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
               uint64_t outer, uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool pitch_ok(int64_t ld, int elem_bytes) { return ((ld * elem_bytes) & 15) == 0; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Fills the launch-independent parts of GemmParams.
inline void init_params(GemmParams& p, int M, int N, int K, int n_per_tile) {
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m_blocks = cdiv(M, kBM);
  p.num_n_blocks = cdiv(N, n_per_tile);
  p.num_k_blocks = cdiv(K, kBK);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  p.group_m = 16;
  p.timeout_ns = wait_timeout_ns();
}

// Launches fused_gemm_kernel<EPI> persistently: one CTA per SM (capped by the
// tile count and the test override, but never below `min_grid`).  With
// `cooperative` the launch fails instead of starting if not every CTA can be
// resident at once (needed when CTAs wait on one another).
template <int EPI>
int launch_gemm(GemmParams& p, const DeviceInfo& di, cudaStream_t stream, bool cooperative, int min_grid) {
  using T = EpiTraits<EPI>;
  const void* kfn = reinterpret_cast<const void*>(&fused_gemm_kernel<EPI>);
  if (!ensure_smem_attr(kfn, di.device, T::kSmemBytes)) return FL_ERR_CUDA;
  p.status = device_status_ptr(di.device);
  if (p.status == nullptr) return FL_ERR_CUDA;
  int grid = di.num_sms < p.num_tiles ? di.num_sms : p.num_tiles;
  const int cap = max_ctas_override();
  if (cap > 0 && cap < grid) grid = cap;
  if (grid < min_grid) grid = min_grid;
  if (grid > di.num_sms) return FL_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = T::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = cooperative ? attr : nullptr;
  cfg.numAttrs = cooperative ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_gemm_kernel<EPI>, p);
  return e == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

}  // namespace fl
