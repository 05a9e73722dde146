// Decode-shaped (M <= 32 tokens) GELU, SwiGLU, QKV + RoPE and its FP8 K/V form: parameters, cluster size and launch of
// linear_decode_kernel (decode_linear_kernel.cuh).  The entry points in k_gelu.cu, k_swiglu.cu and
// k_qkv.cu call these first; kDecodeNotTaken sends the call to the GEMM kernel instead.
#include <cmath>
#include <mutex>

#include "decode_linear_kernel.cuh"
#include "host_common.h"

namespace fl {
namespace {

template <int C, int KIND>
void ld_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t s) {
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kLdSmemBytes;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the weight prefetch may overlap the preceding kernel's tail
  // (everything the kernel reads or writes besides W waits in griddepcontrol.wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
}

// Clusters of C CTAs of this kernel the device holds at once (cached per device).
template <int C, int KIND>
int ld_fit(const DeviceInfo& di) {
  static std::mutex mu;
  static int cache[64];
  static bool known[64];
  if (di.device < 0 || di.device >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[di.device]) {
    int n = 0;
    const void* kfn = reinterpret_cast<const void*>(&linear_decode_kernel<C, KIND>);
    if (ensure_smem_attr(kfn, di.device, kLdSmemBytes)) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      ld_config<C, KIND>(cfg, attr, C * (di.num_sms / C), nullptr);
      cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
      if (cudaOccupancyMaxActiveClusters(&n, kfn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    }
    cache[di.device] = n;
    known[di.device] = true;
  }
  return cache[di.device];
}

template <int C, int KIND>
int ld_launch(const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s) {
  const void* kfn = reinterpret_cast<const void*>(&linear_decode_kernel<C, KIND>);
  if (!ensure_smem_attr(kfn, di.device, kLdSmemBytes)) return kDecodeNotTaken;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  ld_config<C, KIND>(cfg, attr, p.num_f * C, s);
  if (cudaLaunchKernelEx(&cfg, linear_decode_kernel<C, KIND>, p) != cudaSuccess) {
    cudaGetLastError();  // a refused launch configuration: the GEMM kernel takes the call
    return kDecodeNotTaken;
  }
  return FL_OK;
}

// Cluster size: the largest C (8, 4, 2) that splits K into at least one k block per CTA and keeps
// every tile's cluster resident at once on the SMs the grid may use; else one CTA per tile.  With
// more tiles than SMs the stream would run in two uneven waves (measured: SwiGLU 32 x 14336 x 4096,
// 224 tiles, 45.0 us against 42.9 us on the GEMM kernel), so the GEMM kernel takes those calls.
template <int KIND>
int ld_run(const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s) {
  const int cap = max_ctas_override();
  const int sms = cap > 0 && cap < di.num_sms ? cap : di.num_sms;
  if (p.num_f > sms) return kDecodeNotTaken;
  auto fits = [&](int c, int fit) { return c <= p.num_kb && static_cast<long long>(p.num_f) * c <= sms && fit >= p.num_f; };
  if (fits(8, 8 <= p.num_kb ? ld_fit<8, KIND>(di) : 0)) return ld_launch<8, KIND>(p, di, s);
  if (fits(4, 4 <= p.num_kb ? ld_fit<4, KIND>(di) : 0)) return ld_launch<4, KIND>(p, di, s);
  if (fits(2, 2 <= p.num_kb ? ld_fit<2, KIND>(di) : 0)) return ld_launch<2, KIND>(p, di, s);
  return ld_launch<1, KIND>(p, di, s);
}

bool ld_common(LinearDecodeParams& p, const void* X, int M, int K, int64_t ldx, const DeviceInfo& di) {
  std::memset(&p, 0, sizeof(p));
  if (!encode_2d(&p.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kLdTokens,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  p.M = M;
  p.K = K;
  p.num_kb = cdiv(K, kBK);
  p.status = device_status_ptr(di.device);
  p.timeout_ns = wait_timeout_ns();
  return p.status != nullptr;
}

bool ld_taken(int M, int K) { return linear_decode_mode() != 0 && M > 0 && M <= kLdTokens && K > 0; }

}  // namespace

int linear_decode_gelu(const void* X, const void* W, const void* b, void* Y, int M, int N, int K, int64_t ldx,
                       int64_t ldw, int64_t ldy, int mode, const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K)) return kDecodeNotTaken;
  LinearDecodeParams p;
  if (!ld_common(p, X, M, K, ldx, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = N;
  p.num_f = cdiv(N, 128);
  p.bias = static_cast<const __nv_bfloat16*>(b);
  p.out[0] = static_cast<__nv_bfloat16*>(Y);
  p.ldo = ldy;
  return mode == FL_GELU_TANH ? ld_run<LD_GELU_TANH>(p, di, s) : ld_run<LD_GELU_ERF>(p, di, s);
}

int linear_decode_swiglu(const void* X, const void* Wg, const void* Wu, const void* bg, const void* bu, void* Y, int M,
                         int N, int K, int64_t ldx, int64_t ldw, int64_t ldy, const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K)) return kDecodeNotTaken;
  LinearDecodeParams p;
  if (!ld_common(p, X, M, K, ldx, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wg, K, N, ldw, kBK, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&p.map_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wu, K, N, ldw, kBK, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = N;
  p.num_f = cdiv(N, 64);
  p.bias = static_cast<const __nv_bfloat16*>(bg);
  p.bias2 = static_cast<const __nv_bfloat16*>(bu);
  p.out[0] = static_cast<__nv_bfloat16*>(Y);
  p.ldo = ldy;
  return ld_run<LD_SWIGLU>(p, di, s);
}

int linear_decode_qkv(const void* X, const void* Wqkv, const void* bqkv, void* const outs[3], const int32_t* positions,
                      int M, int K, int d_model, int seq_len, float theta, int64_t ldx, int64_t ldw, int64_t ldo,
                      const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K) || d_model % 128 != 0) return kDecodeNotTaken;
  LinearDecodeParams p;
  if (!ld_common(p, X, M, K, ldx, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wqkv, K, 3 * d_model, ldw, kBK, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = d_model;
  p.kv_width = d_model;
  p.num_f = 3 * d_model / 128;  // one head of one section per tile
  p.bias = static_cast<const __nv_bfloat16*>(bqkv);
  for (int i = 0; i < 3; ++i) p.out[i] = static_cast<__nv_bfloat16*>(outs[i]);
  p.ldo = ldo;
  p.positions = positions;
  p.seq_len = seq_len;
  p.log2_theta = std::log2(static_cast<double>(theta));
  return ld_run<LD_QKV_ROPE>(p, di, s);
}

int linear_decode_qkv_fp8kv(const void* X, const void* Wqkv, const void* bqkv, void* Q, void* Kq, void* Vq,
                            float* k_scale, float* v_scale, const int32_t* positions, int M, int K, int d_model,
                            int kv_width, int seq_len, float theta, int64_t ldx, int64_t ldw, int64_t ldq, int64_t ldkv,
                            int64_t lds, const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K) || d_model % 128 != 0 || kv_width % 128 != 0) return kDecodeNotTaken;
  const int rows = d_model + 2 * kv_width;
  LinearDecodeParams p;
  if (!ld_common(p, X, M, K, ldx, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wqkv, K, rows, ldw, kBK, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = d_model;
  p.kv_width = kv_width;
  p.num_f = rows / 128;  // one head of one section per tile
  p.bias = static_cast<const __nv_bfloat16*>(bqkv);
  p.out[0] = static_cast<__nv_bfloat16*>(Q);
  p.ldo = ldq;
  p.out_kv[0] = static_cast<uint8_t*>(Kq);
  p.out_kv[1] = static_cast<uint8_t*>(Vq);
  p.ldkv = ldkv;
  p.kv_scale[0] = k_scale;
  p.kv_scale[1] = v_scale;
  p.lds = lds;
  p.positions = positions;
  p.seq_len = seq_len;
  p.log2_theta = std::log2(static_cast<double>(theta));
  return ld_run<LD_QKV_FP8KV>(p, di, s);
}

}  // namespace fl
