// fused_linear_gelu: Linear + bias + GELU (erf or tanh form).
//   "Triton 算子融合: Linear 与 Attention" (aiqz.cc), §Linear算子剖析 and §GELU激活融合.
// bf16 operands run on the persistent tcgen05 kernel; fp32 operands run on a
// CUDA-core fp32-FMA kernel (tensor-core TF32 would not meet fp32 accuracy).
#include "host_common.h"

namespace fl {

// fp32 path: 64x64 output tile per block, 16x16 threads, 4x4 outputs per thread.
constexpr int kSimtTile = 64;
constexpr int kSimtK = 16;

__global__ void __launch_bounds__(256) linear_gelu_f32_kernel(const float* __restrict__ X,
                                                              const float* __restrict__ W,
                                                              const float* __restrict__ b, float* __restrict__ Y,
                                                              int M, int N, int K, long long ldx, long long ldw,
                                                              long long ldy, int mode) {
  __shared__ float xs[kSimtK][kSimtTile + 1];
  __shared__ float ws[kSimtK][kSimtTile + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * 16 + tx;
  const int m0 = blockIdx.y * kSimtTile, n0 = blockIdx.x * kSimtTile;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += kSimtK) {
    for (int e = tid; e < kSimtTile * kSimtK; e += 256) {
      const int r = e / kSimtK, kk = e % kSimtK;
      const int k = k0 + kk;
      xs[kk][r] = (m0 + r < M && k < K) ? X[(m0 + r) * ldx + k] : 0.f;
      ws[kk][r] = (n0 + r < N && k < K) ? W[(n0 + r) * ldw + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = ws[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      const float v = acc[i][j] + (b ? b[n] : 0.f);
      float y;
      if (mode == FL_GELU_ERF) {
        y = 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
      } else {
        y = 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
      }
      Y[m * ldy + n] = y;
    }
  }
}

}  // namespace fl

extern "C" int fused_linear_gelu(const void* X, const void* W, const void* b, void* Y, int M, int N, int K,
                                 int64_t ldx, int64_t ldw, int64_t ldy, int dtype, int mode, void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (dtype != FL_F32 && dtype != FL_BF16) return FL_ERR_INVALID_ARG;
  if (mode != FL_GELU_ERF && mode != FL_GELU_TANH) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Y == nullptr || (K > 0 && (X == nullptr || W == nullptr))) return FL_ERR_INVALID_ARG;
  if (ldy < N || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  const int es = dtype == FL_F32 ? 4 : 2;
  if (!aligned16(X) || !aligned16(W) || !aligned16(b) || !aligned16(Y)) return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldy, es) || (K > 0 && (!pitch_ok(ldx, es) || !pitch_ok(ldw, es)))) return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (dtype == FL_F32) {
    dim3 grid(cdiv(N, kSimtTile), cdiv(M, kSimtTile));
    linear_gelu_f32_kernel<<<grid, dim3(16, 16), 0, s>>>(
        static_cast<const float*>(X), static_cast<const float*>(W), static_cast<const float*>(b),
        static_cast<float*>(Y), M, N, K, ldx, ldw, ldy, mode);
    return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
  }

  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, N, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, ldy, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.bias = static_cast<const __nv_bfloat16*>(b);
    return true;
  };
  return mode == FL_GELU_TANH ? run_gemm<EPI_GELU_TANH>(M, setup, di, s, false, 1)
                              : run_gemm<EPI_GELU_ERF>(M, setup, di, s, false, 1);
}
