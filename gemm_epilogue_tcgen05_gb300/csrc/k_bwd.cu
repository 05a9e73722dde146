// Backward epilogues on the dgrad GEMM.
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 D: the gradient w.r.t. a block's
//   input is a GEMM with the weight, and f'(h) is applied in that GEMM's epilogue;
//   §末尾布局调整 (SwiGLU 反向): one upstream value becomes a (gate, up) pair, written at
//   twice the width.
// W is taken as stored by the forward layer ([n_out, n_in], n_in contiguous), so the
// contraction runs over its rows and the B operand reaches the tensor cores MN-major.
#include "host_common.h"

namespace fl {
namespace {

// Checks shared by both entry points: dZ [M,K] (K = n_out), W [K,N], saved [M,N], out [M, out_w].
int check_dgrad(const void* dZ, const void* W, const void* s0, const void* s1, const void* out, int M, int N, int K,
                int64_t ldz, int64_t ldw, int64_t lds, int64_t ldo, int out_w) {
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (out == nullptr || s0 == nullptr || (K > 0 && (dZ == nullptr || W == nullptr))) return FL_ERR_INVALID_ARG;
  if (ldo < out_w || lds < N || (K > 0 && (ldz < K || ldw < N))) return FL_ERR_INVALID_ARG;
  if (!aligned16(dZ) || !aligned16(W) || !aligned16(s0) || !aligned16(s1) || !aligned16(out))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldo, 2) || !pitch_ok(lds, 2) || (K > 0 && (!pitch_ok(ldz, 2) || !pitch_ok(ldw, 2))))
    return FL_ERR_ALIGNMENT;
  return FL_OK;
}

template <int EPI>
int launch_dgrad(const void* dZ, const void* W, const void* s0, const void* s1, void* out, int M, int N, int K,
                 int64_t ldz, int64_t ldw, int64_t lds, int64_t ldo, int out_w, cudaStream_t stream) {
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, N, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dZ, K, M, ldz, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         // W [K, N], N contiguous: boxes of 64 columns x 64 rows (K)
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, N, K, ldw, 64, kBK,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, out_w, M, ldo, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.saved0 = static_cast<const __nv_bfloat16*>(s0);
    p.saved1 = static_cast<const __nv_bfloat16*>(s1);
    p.ld_saved = lds;
    // saved activations [M, N]: boxes of 32 columns x 32 rows (one epilogue warp's unit)
    if (!encode_2d(&p.map_saved[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s0, N, M, lds, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B) ||
        (s1 != nullptr && !encode_2d(&p.map_saved[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s1, N, M, lds, 32, 32,
                                     CU_TENSOR_MAP_SWIZZLE_64B)))
      return false;
    return true;
  };
  return run_gemm<EPI>(M, setup, di, stream, false, 1);
}

}  // namespace
}  // namespace fl

extern "C" int fused_dgrad_gelu(const void* dZ, const void* W, const void* H, void* dH, int M, int N, int K,
                                int64_t ldz, int64_t ldw, int64_t ldh, int64_t ldo, int mode, void* stream) {
  using namespace fl;
  if (mode != FL_GELU_ERF && mode != FL_GELU_TANH) return FL_ERR_INVALID_ARG;
  const int st = check_dgrad(dZ, W, H, nullptr, dH, M, N, K, ldz, ldw, ldh, ldo, N);
  if (st != FL_OK || M == 0 || N == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return mode == FL_GELU_TANH
             ? launch_dgrad<EPI_GELU_BWD_TANH>(dZ, W, H, nullptr, dH, M, N, K, ldz, ldw, ldh, ldo, N, s)
             : launch_dgrad<EPI_GELU_BWD_ERF>(dZ, W, H, nullptr, dH, M, N, K, ldz, ldw, ldh, ldo, N, s);
}

extern "C" int fused_swiglu_bwd(const void* dO, const void* Wd, const void* G, const void* U, void* dGU, int M, int N,
                                int K, int64_t ldo_in, int64_t ldw, int64_t ldgu, int64_t ldout, void* stream) {
  using namespace fl;
  if (N > (1 << 29)) return FL_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && U == nullptr) return FL_ERR_INVALID_ARG;
  const int st = check_dgrad(dO, Wd, G, U, dGU, M, N, K, ldo_in, ldw, ldgu, ldout, 2 * N);
  if (st != FL_OK || M == 0 || N == 0) return st;
  return launch_dgrad<EPI_SWIGLU_BWD>(dO, Wd, G, U, dGU, M, N, K, ldo_in, ldw, ldgu, ldout, 2 * N,
                                      static_cast<cudaStream_t>(stream));
}
