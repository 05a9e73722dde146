// Decode-shaped (M <= 32) fused_linear_gelu, bf16: the decode kernel's GELU kinds.
#include "linear_decode_host.cuh"

namespace fl {

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

void linear_decode_plan_gelu(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                         int* launches) {
  ld_plan_out<LD_GELU_TANH>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

}  // namespace fl
