// fused_qkv_rope: fused QKV projection, split write-back and RoPE on Q and K.
//   "Triton 算子融合: Linear 与 Attention" (aiqz.cc), §QKV投影融合;
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 B, §累加器布局 and §用形状与步长把约定钉死.
// fused_qkv_rope_fp8kv: the same with grouped-query widths and the K/V cache entry
// written in FP8 by the epilogue ("GEMM Epilogue 完全拆解", §一个瓦片的字节账).
// A 256-column output tile covers two heads of one section (Q, K or V), so the
// section, and with it the output tensor and whether to rotate, is uniform per tile.
#include <cmath>

#include "host_common.h"

namespace fl {
namespace {

// Shared checks of the QKV entry points: sizes, RoPE parameters and section widths.
int check_qkv(int M, int K, int n_heads, int n_kv_heads, int head_dim, int seq_len, float theta,
              const int32_t* positions, int* d_model, int* kv_width) {
  if (M < 0 || K < 0 || n_heads < 0 || n_kv_heads < 0 || head_dim < 0) return FL_ERR_INVALID_ARG;
  if (positions == nullptr && seq_len <= 0) return FL_ERR_INVALID_ARG;
  if (!(theta > 0.f) || !std::isfinite(theta)) return FL_ERR_INVALID_ARG;
  const long long q_ll = static_cast<long long>(n_heads) * head_dim;
  const long long kv_ll = static_cast<long long>(n_kv_heads) * head_dim;
  if (q_ll + 2 * kv_ll > (1 << 28)) return FL_ERR_INVALID_ARG;
  *d_model = static_cast<int>(q_ll);
  *kv_width = static_cast<int>(kv_ll);
  return FL_OK;
}

template <int EPI>
int launch_qkv(const void* X, const void* Wqkv, const void* bqkv, void* const outs[3], const int32_t* positions,
               int M, int K, int d_model, int kv_width, int head_dim, int seq_len, float theta, int64_t ldx,
               int64_t ldw, int64_t ldq, int64_t ldkv, float* kscale, float* vscale, int64_t lds,
               cudaStream_t stream) {
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  const int width = d_model + 2 * kv_width;
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, width, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wqkv, K, width, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, outs[0], d_model, M, ldq, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    for (int i = 1; i < 3; ++i) {
      const bool ok = EPI == EPI_QKV_FP8KV
                          ? encode_2d(&p.map_out[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, outs[i], kv_width, M, ldkv,
                                      128, 32, CU_TENSOR_MAP_SWIZZLE_128B)
                          : encode_2d(&p.map_out[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, outs[i], kv_width, M,
                                      ldkv, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
      if (!ok) return false;
    }
    p.bias = static_cast<const __nv_bfloat16*>(bqkv);
    p.positions = positions;
    p.seq_len = seq_len > 0 ? seq_len : 1;
    p.head_dim = head_dim;
    p.d_model = d_model;
    p.kv_width = kv_width;
    p.log2_theta = std::log2(static_cast<double>(theta));  // double: the float overload is too coarse
    p.kscale = kscale;
    p.vscale = vscale;
    p.lds = lds;
    return true;
  };
  return run_gemm<EPI>(M, setup, di, stream, false, 1);
}

}  // namespace
}  // namespace fl

extern "C" int fused_qkv_rope(const void* X, const void* Wqkv, const void* bqkv, void* Q, void* Kout, void* V,
                              const int32_t* positions, int M, int K, int n_heads, int head_dim, int seq_len,
                              float theta, int64_t ldx, int64_t ldw, int64_t ldo, void* stream) {
  using namespace fl;
  int d_model = 0, kv_width = 0;
  int st = check_qkv(M, K, n_heads, n_heads, head_dim, seq_len, theta, positions, &d_model, &kv_width);
  if (st != FL_OK) return st;
  if (M == 0 || d_model == 0) return FL_OK;
  if (head_dim != 128 || d_model % 256 != 0) return FL_ERR_UNSUPPORTED;
  if (Q == nullptr || Kout == nullptr || V == nullptr || (K > 0 && (X == nullptr || Wqkv == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldo < d_model || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wqkv) || !aligned16(bqkv) || !aligned16(Q) || !aligned16(Kout) ||
      !aligned16(V))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldo, 2) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2)))) return FL_ERR_ALIGNMENT;
  void* const outs[3] = {Q, Kout, V};
  DeviceInfo di;
  st = current_device(&di);
  if (st != FL_OK) return st;
  // a few tokens: the swap-AB decode kernel streams W instead of padding a 256-row tile
  st = linear_decode_qkv(X, Wqkv, bqkv, outs, positions, M, K, d_model, seq_len, theta, ldx, ldw, ldo, di,
                         static_cast<cudaStream_t>(stream));
  if (st != kDecodeNotTaken) return st;
  return launch_qkv<EPI_QKV_ROPE>(X, Wqkv, bqkv, outs, positions, M, K, d_model, kv_width, head_dim, seq_len,
                                  theta, ldx, ldw, ldo, ldo, nullptr, nullptr, 0, static_cast<cudaStream_t>(stream));
}

extern "C" int fused_qkv_rope_fp8kv(const void* X, const void* Wqkv, const void* bqkv, void* Q, void* Kq, void* Vq,
                                    float* k_scale, float* v_scale, const int32_t* positions, int M, int K,
                                    int n_heads, int n_kv_heads, int head_dim, int seq_len, float theta, int64_t ldx,
                                    int64_t ldw, int64_t ldq, int64_t ldkv, int64_t lds, void* stream) {
  using namespace fl;
  int d_model = 0, kv_width = 0;
  int st = check_qkv(M, K, n_heads, n_kv_heads, head_dim, seq_len, theta, positions, &d_model, &kv_width);
  if (st != FL_OK) return st;
  if (M == 0 || d_model + kv_width == 0) return FL_OK;
  if (head_dim != 128 || d_model == 0 || kv_width == 0 || d_model % 256 != 0 || kv_width % 256 != 0)
    return FL_ERR_UNSUPPORTED;
  if (Q == nullptr || Kq == nullptr || Vq == nullptr || k_scale == nullptr ||
      v_scale == nullptr || (K > 0 && (X == nullptr || Wqkv == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldq < d_model || ldkv < kv_width || lds < n_kv_heads || (K > 0 && (ldx < K || ldw < K)))
    return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wqkv) || !aligned16(bqkv) || !aligned16(Q) || !aligned16(Kq) ||
      !aligned16(Vq))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldq, 2) || !pitch_ok(ldkv, 1) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2))))
    return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  st = current_device(&di);
  if (st != FL_OK) return st;
  // a few tokens: the swap-AB decode kernel streams W instead of padding a 256-row tile
  st = linear_decode_qkv_fp8kv(X, Wqkv, bqkv, Q, Kq, Vq, k_scale, v_scale, positions, M, K, d_model, kv_width,
                               seq_len, theta, ldx, ldw, ldq, ldkv, lds, di, static_cast<cudaStream_t>(stream));
  if (st != kDecodeNotTaken) return st;
  void* const outs[3] = {Q, Kq, Vq};
  return launch_qkv<EPI_QKV_FP8KV>(X, Wqkv, bqkv, outs, positions, M, K, d_model, kv_width, head_dim, seq_len,
                                   theta, ldx, ldw, ldq, ldkv, k_scale, v_scale, lds,
                                   static_cast<cudaStream_t>(stream));
}
