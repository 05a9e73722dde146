// Decode-shaped (M <= 32) steps of the deferred-scale chain (fused_linear_residual_gamma and
// fused_linear_rms_rowscale): the decode kernel's chain kinds.
#include "linear_decode_host.cuh"

namespace fl {

int linear_decode_resgamma(const void* X, const void* W, const void* b, const void* Z, const void* gamma, void* H2,
                           void* H1, float* rms_partials, int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldz,
                           int64_t ldh, const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K)) return kDecodeNotTaken;
  const int num_f = cdiv(N, 128);
  if (ld_plan<LD_RESGAMMA>(num_f, cdiv(K, kBK), di).launches == 0) return kDecodeNotTaken;
  LinearDecodeParams p;
  if (!ld_common(p, X, M, K, ldx, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = N;
  p.num_f = num_f;
  p.bias = static_cast<const __nv_bfloat16*>(b);
  p.out[0] = static_cast<__nv_bfloat16*>(H2);
  p.out[1] = static_cast<__nv_bfloat16*>(H1);
  p.ldo = ldh;
  p.resid = static_cast<const __nv_bfloat16*>(Z);
  p.ldz = ldz;
  p.gamma = static_cast<const __nv_bfloat16*>(gamma);
  p.partials = rms_partials;
  // each 256-column entry receives the sums of its two 128-feature tiles by atomic adds onto zero
  const size_t pbytes = static_cast<size_t>(cdiv(N, 256)) * static_cast<size_t>(M) * sizeof(float);
  if (cudaMemsetAsync(rms_partials, 0, pbytes, s) != cudaSuccess) return FL_ERR_CUDA;
  return ld_run<LD_RESGAMMA>(p, di, s);
}

int linear_decode_rowscale(const void* H2, const void* W1, const void* b1, const float* rms_partials, int n_norm,
                           float eps, void* Y, int M, int N, int K, int64_t ldh, int64_t ldw, int64_t ldy,
                           const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K)) return kDecodeNotTaken;
  LinearDecodeParams p;
  if (!ld_common(p, H2, M, K, ldh, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W1, K, N, ldw, kBK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = N;
  p.num_f = cdiv(N, 128);
  p.bias = static_cast<const __nv_bfloat16*>(b1);
  p.out[0] = static_cast<__nv_bfloat16*>(Y);
  p.ldo = ldy;
  p.partials = const_cast<float*>(rms_partials);
  p.n_partials = cdiv(n_norm, 256);
  p.n_norm = n_norm;
  p.eps = eps;
  return ld_run<LD_ROWSCALE>(p, di, s);
}

void linear_decode_plan_resgamma(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                                 int* launches) {
  ld_plan_out<LD_RESGAMMA>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

void linear_decode_plan_rowscale(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                                 int* launches) {
  ld_plan_out<LD_ROWSCALE>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

}  // namespace fl
