// Decode-shaped (M <= 32) fused_qkv_rope_fp8kv: the decode kernel's QKV + RoPE kind with the
// K/V cache entry in FP8.
#include "linear_decode_host.cuh"

namespace fl {

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

void linear_decode_plan_qkv_fp8kv(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                         int* launches) {
  ld_plan_out<LD_QKV_FP8KV>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

}  // namespace fl
