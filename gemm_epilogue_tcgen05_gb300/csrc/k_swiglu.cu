// fused_swiglu: Y = SiLU(X Wgate^T + bgate) * (X Wup^T + bup).
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 B and §末尾布局调整.
// Each shared-memory B stage holds the 128 gate rows and the 128 up rows of the
// same output features, so one 128x256 accumulator holds both halves of every
// pair and the epilogue multiplies them in registers.
#include "host_common.h"

extern "C" int fused_swiglu(const void* X, const void* Wgate, const void* Wup, const void* bgate, const void* bup,
                            void* Y, int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldy, void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Y == nullptr || (K > 0 && (X == nullptr || Wgate == nullptr || Wup == nullptr))) return FL_ERR_INVALID_ARG;
  if (ldy < N || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wgate) || !aligned16(Wup) || !aligned16(bgate) || !aligned16(bup) ||
      !aligned16(Y))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldy, 2) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2)))) return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  // a few tokens: the swap-AB decode kernel streams W instead of padding a 256-row tile
  st = linear_decode_swiglu(X, Wgate, Wup, bgate, bup, Y, M, N, K, ldx, ldw, ldy, di,
                            static_cast<cudaStream_t>(stream));
  if (st != kDecodeNotTaken) return st;

  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, N, K, 128, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wgate, K, N, ldw, kBK, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wup, K, N, ldw, kBK, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, ldy, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.bias = static_cast<const __nv_bfloat16*>(bgate);
    p.bias2 = static_cast<const __nv_bfloat16*>(bup);
    return true;
  };
  return run_gemm<EPI_SWIGLU>(M, setup, di, static_cast<cudaStream_t>(stream), false, 1);
}
