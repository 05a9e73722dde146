// Decode-shaped (M <= 32) fused_linear_quant: the decode kernel's block-scaled kind.
#include "linear_decode_host.cuh"

namespace fl {

int linear_decode_quant(const void* X, const void* W, const void* b, const float* inv_smooth, void* Yq, void* scales,
                        int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldq, int64_t lds, int fmt,
                        const DeviceInfo& di, cudaStream_t s) {
  if (!ld_taken(M, K)) return kDecodeNotTaken;
  LinearDecodeParams p;
  if (!ld_common(p, X, M, K, ldx, di) ||
      !encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return FL_ERR_CUDA;
  p.n_out = N;
  p.num_f = cdiv(N, 128);  // a tile of 128 features holds whole blocks of every format
  p.bias = static_cast<const __nv_bfloat16*>(b);
  p.qout = static_cast<uint8_t*>(Yq);
  p.ldq = ldq;
  p.qscale = scales;
  p.qlds = lds;
  p.smooth = inv_smooth;
  p.qfmt = fmt;
  return ld_run<LD_QUANT>(p, di, s);
}

void linear_decode_plan_quant(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm,
                              int* launches) {
  ld_plan_out<LD_QUANT>(num_f, num_kb, di, cluster, ctas_per_sm, launches);
}

}  // namespace fl
