// GEMM -> residual -> RMSNorm -> GEMM with the row scale deferred into the second GEMM.
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 A: y = RMSNorm(x W0 + z, gamma) W1
//   = r (.) ((x W0 + z) (.) gamma) W1 with r one scalar per row.  Epilogue 1 writes
//   h1 = x W0 + z, h2 = h1 (.) gamma and per-tile partial sums of h1^2; the partials of
//   a row are merged and r applied in epilogue 2 (no separate reduction launch, no
//   wait between the two GEMMs beyond stream order).
#include "host_common.h"

extern "C" int fl_rms_partials_per_row(int n_norm) { return n_norm <= 0 ? 0 : fl::cdiv(n_norm, 256); }

extern "C" int fused_linear_residual_gamma(const void* X, const void* W, const void* b, const void* Z,
                                           const void* gamma, void* H2, void* H1, float* rms_partials, int M,
                                           int N, int K, int64_t ldx, int64_t ldw, int64_t ldz, int64_t ldh,
                                           void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Z == nullptr || gamma == nullptr || H2 == nullptr || rms_partials == nullptr ||
      (K > 0 && (X == nullptr || W == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldz < N || ldh < N || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(b) || !aligned16(Z) || !aligned16(gamma) || !aligned16(H2) ||
      !aligned16(H1) || !aligned16(rms_partials))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldz, 2) || !pitch_ok(ldh, 2) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2))))
    return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  // a few tokens: the swap-AB decode kernel streams W instead of padding a 256-row tile (it adds the
  // sums of two 128-feature tiles per 256-column entry, after zeroing the entries on the stream)
  st = linear_decode_resgamma(X, W, b, Z, gamma, H2, H1, rms_partials, M, N, K, ldx, ldw, ldz, ldh, di,
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
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H2, N, M, ldh, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    if (H1 != nullptr && !encode_2d(&p.map_out[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H1, N, M, ldh, 64, 32,
                                    CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.store_h1 = H1 != nullptr;
    p.bias = static_cast<const __nv_bfloat16*>(b);
    p.resid = static_cast<const __nv_bfloat16*>(Z);
    p.ldz = ldz;
    p.gamma = static_cast<const __nv_bfloat16*>(gamma);
    p.rms_partials = rms_partials;
    return true;
  };
  return run_gemm<EPI_RESID_GAMMA>(M, setup, di, static_cast<cudaStream_t>(stream), false, 1);
}

extern "C" int fused_linear_rms_rowscale(const void* H2, const void* W1, const void* b1, const float* rms_partials,
                                         int n_norm, float eps, void* Y, int M, int N, int K, int64_t ldh,
                                         int64_t ldw, int64_t ldy, void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0 || n_norm <= 0 || !(eps >= 0.f)) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Y == nullptr || rms_partials == nullptr || (K > 0 && (H2 == nullptr || W1 == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldy < N || (K > 0 && (ldh < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(H2) || !aligned16(W1) || !aligned16(b1) || !aligned16(Y)) return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldy, 2) || (K > 0 && (!pitch_ok(ldh, 2) || !pitch_ok(ldw, 2)))) return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  st = linear_decode_rowscale(H2, W1, b1, rms_partials, n_norm, eps, Y, M, N, K, ldh, ldw, ldy, di,
                              static_cast<cudaStream_t>(stream));
  if (st != kDecodeNotTaken) return st;
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, N, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H2, K, M, ldh, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W1, K, N, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, ldy, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.bias = static_cast<const __nv_bfloat16*>(b1);
    p.rms_partials = const_cast<float*>(rms_partials);
    p.n_partials = cdiv(n_norm, 256);
    p.n_norm = n_norm;
    p.eps = eps;
    return true;
  };
  return run_gemm<EPI_ROWSCALE>(M, setup, di, static_cast<cudaStream_t>(stream), false, 1);
}
