// Decode-shaped (M <= 32) fused_swiglu: the decode kernel's SwiGLU kind.
#include "linear_decode_host.cuh"

namespace fl {

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

void linear_decode_plan_swiglu(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                         int* launches) {
  ld_plan_out<LD_SWIGLU>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

}  // namespace fl
