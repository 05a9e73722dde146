// fused_linear_quant: Linear (+ bias) with a block-scaled quantised write-back.
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §仿射量化与尾声的五步: optionally the
//   output is first multiplied per column by an inverse smoothing factor (step 3, for a
//   layer fed by SmoothQuant/QuaRot-style smoothing), then per block the maximum gives the
//   scale, the values are rounded to the target format, packed compactly (two 4-bit codes
//   per byte) and the scale array is written by the same epilogue.
#include "host_common.h"

extern "C" int fused_linear_quant(const void* X, const void* W, const void* b, const float* inv_smooth, void* Yq,
                                  void* scales, int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldq,
                                  int64_t lds, int fmt, void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (fmt != FL_QUANT_FP8_1X128 && fmt != FL_QUANT_INT4_G32 && fmt != FL_QUANT_NVFP4_G16) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (fmt != FL_QUANT_FP8_1X128 && (N & 1)) return FL_ERR_UNSUPPORTED;
  if (Yq == nullptr || scales == nullptr || (K > 0 && (X == nullptr || W == nullptr))) return FL_ERR_INVALID_ARG;
  const int block = fmt == FL_QUANT_FP8_1X128 ? 128 : (fmt == FL_QUANT_INT4_G32 ? 32 : 16);
  const int64_t qbytes = fmt == FL_QUANT_FP8_1X128 ? N : N / 2;
  if (ldq < qbytes || lds < cdiv(N, block) || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(b) || !aligned16(inv_smooth) || !aligned16(Yq) ||
      !aligned16(scales))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldq, 1) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2)))) return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  // a few tokens: the swap-AB decode kernel streams W instead of padding a 256-row tile
  st = linear_decode_quant(X, W, b, inv_smooth, Yq, scales, M, N, K, ldx, ldw, ldq, lds, fmt, di,
                           static_cast<cudaStream_t>(stream));
  if (st != kDecodeNotTaken) return st;
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, N, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Yq, qbytes, M, ldq, 128, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.bias = static_cast<const __nv_bfloat16*>(b);
    p.smooth = inv_smooth;
    p.quant_fmt = fmt;
    p.qscale = scales;
    p.lds = lds;
    return true;
  };
  return run_gemm<EPI_QUANT>(M, setup, di, static_cast<cudaStream_t>(stream), false, 1);
}
