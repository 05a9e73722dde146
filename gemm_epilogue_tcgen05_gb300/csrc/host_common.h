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
// 1 (default): kernels whose CTAs wait on one another launch with the cooperative attribute;
// 0: without it (fl_set_cooperative_launch).
int cooperative_launch_mode();
// Makes sure the kernel may use `smem_bytes` of dynamic shared memory on `device`.
bool ensure_smem_attr(const void* kernel, int device, int smem_bytes);

// 2-D tiled tensor map over a row-major [outer, inner] matrix with row pitch
// `ld_elems` elements of `elem_bytes` bytes each.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
               uint64_t outer, uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every workspace the library takes starts with its status record: kWsStatusBytes bytes, of
// which the first ST_WORDS ints are written by a kernel that gives up a bounded wait and read
// back by fl_check_device_status.  The layout proper follows it.
constexpr size_t kWsStatusBytes = 256;

// Device memory to clear (cudaMemsetAsync on the launch stream) right before the kernel is
// enqueued, once every check has passed; bytes == 0: nothing.  Cleared at most once.
struct PreLaunchClear {
  void* ptr = nullptr;
  size_t bytes = 0;
  bool done = false;
};
inline int run_clear(PreLaunchClear* c, cudaStream_t s) {
  if (c == nullptr || c->bytes == 0 || c->done) return FL_OK;
  if (cudaMemsetAsync(c->ptr, 0, c->bytes, s) != cudaSuccess) return FL_ERR_CUDA;
  c->done = true;
  return FL_OK;
}
inline bool pitch_ok(int64_t ld, int elem_bytes) { return ((ld * elem_bytes) & 15) == 0; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Process-wide switch for the two-CTA (cta_group::2) mainloop: 1 = use it when
// M spans at least two 128-row blocks (default), 0 = always one CTA per tile.
int cta_pairing_mode();
int linear_decode_mode();  // 1: M <= 32 calls of GELU, SwiGLU, QKV + RoPE (both forms), the block-scaled
                           // write-back and both chain steps run the decode kernels
// Decode-shaped (M <= 32) GELU, SwiGLU, QKV + RoPE and block-scaled write-back (k_linear_decode_*.cu).  Returns FL_OK, an
// error, or kDecodeNotTaken when the call should run on the GEMM kernel instead.
constexpr int kDecodeNotTaken = -2;
int linear_decode_gelu(const void* X, const void* W, const void* b, void* Y, int M, int N, int K, int64_t ldx,
                       int64_t ldw, int64_t ldy, int mode, const DeviceInfo& di, cudaStream_t s);
int linear_decode_swiglu(const void* X, const void* Wg, const void* Wu, const void* bg, const void* bu, void* Y, int M,
                         int N, int K, int64_t ldx, int64_t ldw, int64_t ldy, const DeviceInfo& di, cudaStream_t s);
int linear_decode_qkv(const void* X, const void* Wqkv, const void* bqkv, void* const outs[3], const int32_t* positions,
                      int M, int K, int d_model, int seq_len, float theta, int64_t ldx, int64_t ldw, int64_t ldo,
                      const DeviceInfo& di, cudaStream_t s);
// The decode launch plan of a call with num_f W-row tiles and num_kb k blocks (see fl_linear_decode_shape).
void linear_decode_plan_gelu(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                             int* launches);
void linear_decode_plan_swiglu(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                               int* launches);
void linear_decode_plan_qkv(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                            int* launches);
void linear_decode_plan_qkv_fp8kv(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                                  int* launches);
void linear_decode_plan_quant(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                              int* launches);
int linear_decode_quant(const void* X, const void* W, const void* b, const float* inv_smooth, void* Yq, void* scales,
                        int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldq, int64_t lds, int fmt,
                        const DeviceInfo& di, cudaStream_t s);
int linear_decode_resgamma(const void* X, const void* W, const void* b, const void* Z, const void* gamma, void* H2,
                           void* H1, float* rms_partials, int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldz,
                           int64_t ldh, const DeviceInfo& di, cudaStream_t s);
int linear_decode_rowscale(const void* H2, const void* W1, const void* b1, const float* rms_partials, int n_norm,
                           float eps, void* Y, int M, int N, int K, int64_t ldh, int64_t ldw, int64_t ldy,
                           const DeviceInfo& di, cudaStream_t s);
void linear_decode_plan_resgamma(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                                 int* launches);
void linear_decode_plan_rowscale(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                                 int* launches);
int linear_decode_qkv_fp8kv(const void* X, const void* Wqkv, const void* bqkv, void* Q, void* Kq, void* Vq,
                            float* k_scale, float* v_scale, const int32_t* positions, int M, int K, int d_model,
                            int kv_width, int seq_len, float theta, int64_t ldx, int64_t ldw, int64_t ldq, int64_t ldkv,
                            int64_t lds, const DeviceInfo& di, cudaStream_t s);
// CTAs per cluster for a problem with M rows.
inline int choose_cg(int M) { return (cta_pairing_mode() != 0 && M > kBM) ? 2 : 1; }

// Fills the launch-independent parts of GemmParams for tiles of `cg` x 128 rows.
inline void init_params(GemmParams& p, int M, int N, int K, int n_per_tile, int cg) {
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m_blocks = cdiv(M, kBM);
  p.num_n_blocks = cdiv(N, n_per_tile);
  p.num_k_blocks = cdiv(K, kBK);
  p.num_m_tiles = cdiv(p.num_m_blocks, cg);
  p.num_tiles = p.num_m_tiles * p.num_n_blocks;
  p.group_m = 32 / cg;  // raster groups of 32 row blocks
  p.timeout_ns = wait_timeout_ns();
}

// Internal: the pair (cluster) launch was refused; the caller retries with one CTA per tile.
constexpr int kRetryUnpaired = -1;

// Launches fused_gemm_kernel<EPI, CG> persistently: as many CTAs (CG = 1) or
// CTA pairs (CG = 2) as can be resident, capped by the tile count and the test
// override, but never fewer than `min_units` (tiles that must run at once).
// With `cooperative` the launch fails instead of starting if not every CTA can
// be resident at once (needed when CTAs wait on one another).
// p.status: where a timed-out wait is recorded; null selects the device-wide status word.
template <int EPI, int CG>
int launch_gemm_cg(GemmParams& p, const DeviceInfo& di, cudaStream_t stream, bool cooperative, int min_units,
                   PreLaunchClear* clear) {
  using T = EpiTraits<EPI, CG>;
  const void* kfn = reinterpret_cast<const void*>(&fused_gemm_kernel<EPI, CG>);
  if (!ensure_smem_attr(kfn, di.device, T::kSmemBytes)) return CG == 2 ? kRetryUnpaired : FL_ERR_CUDA;
  if (p.status == nullptr) p.status = device_status_ptr(di.device);
  if (p.status == nullptr) return FL_ERR_CUDA;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = T::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  int max_units = di.num_sms;
  if (CG == 2) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = 2;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
    cfg.gridDim = dim3(2 * (di.num_sms / 2));
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fused_gemm_kernel<EPI, CG>, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      return kRetryUnpaired;
    }
    max_units = clusters;
  }
  int units = max_units < p.num_tiles ? max_units : p.num_tiles;
  const int cap = max_ctas_override() / CG;
  if (max_ctas_override() > 0 && cap < units) units = cap > 0 ? cap : 1;
  if (units < min_units) units = min_units;
  if (units > max_units) return CG == 2 ? kRetryUnpaired : FL_ERR_UNSUPPORTED;
  cfg.gridDim = dim3(CG * units);
  // The grid never exceeds what can be resident at once (computed above); the cooperative
  // attribute makes the driver guarantee it.  fl_set_cooperative_launch(0) drops the attribute
  // for tools that refuse cooperative launches of clusters (a profiler serialising the device).
  if (cooperative && cooperative_launch_mode() != 0) {
    attr[nattr].id = cudaLaunchAttributeCooperative;
    attr[nattr].val.cooperative = 1;
    ++nattr;
  }
  cfg.attrs = nattr ? attr : nullptr;
  cfg.numAttrs = nattr;
  if (run_clear(clear, stream) != FL_OK) return FL_ERR_CUDA;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_gemm_kernel<EPI, CG>, p);
  if (e == cudaSuccess) return FL_OK;
  if (CG == 2) {
    cudaGetLastError();
    return kRetryUnpaired;
  }
  return FL_ERR_CUDA;
}

// Runs `setup(cg, params)` (which fills the tensor maps and epilogue fields for
// tiles of cg x 128 rows) and launches; a refused pair launch is retried with
// one CTA per tile.  `clear`, if given, is enqueued right before the first launch.
template <int EPI, class Setup>
int run_gemm(int M, Setup&& setup, const DeviceInfo& di, cudaStream_t stream, bool cooperative,
             int min_units, PreLaunchClear* clear = nullptr) {
  GemmParams p;
  int cg = choose_cg(M);
  if (cg == 2) {
    if (!setup(2, p)) return FL_ERR_CUDA;
    const int st = launch_gemm_cg<EPI, 2>(p, di, stream, cooperative, min_units, clear);
    if (st != kRetryUnpaired) return st;
  }
  if (!setup(1, p)) return FL_ERR_CUDA;
  return launch_gemm_cg<EPI, 1>(p, di, stream, cooperative, min_units, clear);
}

// fused_linear_residual_rmsnorm_fp8 after its argument checks, over a given workspace
// (k_rmsnorm.cu).  scratch_mode (the no-allocation entry point): failures go to the device-wide
// status word instead of the workspace's record, and the workspace's counters are cleared on
// `s` right before the launch, after every check has passed.
int rmsnorm_fp8_enqueue(const void* X, const void* W, const void* b, const void* Z, const void* gamma, float eps,
                        void* Yq, float* row_scale, void* h_out, int M, int N, int K, int64_t ldx, int64_t ldw,
                        int64_t ldz, int64_t ldq, void* workspace, size_t workspace_bytes, cudaStream_t s,
                        bool scratch_mode);

}  // namespace fl
