// fused_qkv_rope: fused QKV projection, split write-back and RoPE on Q and K.
//   "Triton 算子融合: Linear 与 Attention" (aiqz.cc), §QKV投影融合;
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 B, §累加器布局 and §用形状与步长把约定钉死.
// A 256-column output tile covers two heads of one section (Q, K or V), so the
// section, and with it the output tensor and whether to rotate, is uniform per tile.
#include <cmath>

#include "host_common.h"

extern "C" int fused_qkv_rope(const void* X, const void* Wqkv, const void* bqkv, void* Q, void* Kout, void* V,
                              const int32_t* positions, int M, int K, int n_heads, int head_dim, int seq_len,
                              float theta, int64_t ldx, int64_t ldw, int64_t ldo, void* stream) {
  using namespace fl;
  if (M < 0 || K < 0 || n_heads < 0 || head_dim < 0) return FL_ERR_INVALID_ARG;
  if (positions == nullptr && seq_len <= 0) return FL_ERR_INVALID_ARG;
  if (!(theta > 0.f) || !std::isfinite(theta)) return FL_ERR_INVALID_ARG;
  const long long d_model_ll = static_cast<long long>(n_heads) * head_dim;
  if (d_model_ll > (1 << 28)) return FL_ERR_INVALID_ARG;
  const int d_model = static_cast<int>(d_model_ll);
  if (M == 0 || d_model == 0) return FL_OK;
  if (head_dim != 128 || d_model % 256 != 0) return FL_ERR_UNSUPPORTED;
  if (Q == nullptr || Kout == nullptr || V == nullptr || (K > 0 && (X == nullptr || Wqkv == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldo < d_model || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wqkv) || !aligned16(bqkv) || !aligned16(Q) || !aligned16(Kout) ||
      !aligned16(V))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldo, 2) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2)))) return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;

  void* outs[3] = {Q, Kout, V};
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, 3 * d_model, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wqkv, K, 3 * d_model, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    for (int i = 0; i < 3; ++i)
      if (!encode_2d(&p.map_out[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, outs[i], d_model, M, ldo, 64, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    p.bias = static_cast<const __nv_bfloat16*>(bqkv);
    p.positions = positions;
    p.seq_len = seq_len > 0 ? seq_len : 1;
    p.head_dim = head_dim;
    p.d_model = d_model;
    p.log2_theta = std::log2(theta);
    return true;
  };
  return run_gemm<EPI_QKV_ROPE>(M, setup, di, static_cast<cudaStream_t>(stream), false, 1);
}
