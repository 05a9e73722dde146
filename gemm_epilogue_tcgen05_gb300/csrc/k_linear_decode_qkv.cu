// Decode-shaped (M <= 32) fused_qkv_rope: the decode kernel's QKV + RoPE kind.
#include "linear_decode_host.cuh"

namespace fl {

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

void linear_decode_plan_qkv(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                         int* launches) {
  ld_plan_out<LD_QKV_ROPE>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

}  // namespace fl
