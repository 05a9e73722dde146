// fused_linear_gelu: Linear + bias + GELU (erf or tanh form).
//   "Triton 算子融合: Linear 与 Attention" (aiqz.cc), §Linear算子剖析 and §GELU激活融合.
// bf16 operands run on the persistent tcgen05 kernel.  fp32 operands run on tcgen05 too, as
// three TF32 products per term (below): one TF32 product alone would miss fp32 accuracy.
#include "host_common.h"

namespace fl {

// ---------------------------------------------------------------- fp32: 3 x TF32 on tcgen05
// x = hi + lo with hi = x with the low 13 mantissa bits cleared (exactly representable in
// TF32, so the tensor core's conversion leaves it unchanged) and lo = x - hi (exact in fp32).
// A B^T ~ A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T; the dropped A_lo B_lo^T term and the TF32
// rounding of lo are ~2^-21 of each product, accumulated in fp32 in TMEM.  One CTA computes
// one 128 x 256 output tile; a two-stage TMA ring holds the fp32 tiles (32 K per 128-byte
// swizzled row), split in place into hi and a lo copy at the same swizzled offsets.
constexpr int kTfBK = 32;
constexpr int kTfABytes = 128 * kTfBK * 4;                  // 16 KB
constexpr int kTfBBytes = 256 * kTfBK * 4;                  // 32 KB
constexpr int kTfHalf = kTfABytes + kTfBBytes;              // operands as loaded (then hi)
constexpr int kTfStageBytes = 2 * kTfHalf;                  // + lo copies
constexpr int kTfStages = 2;
constexpr int kTfThreads = 128;
constexpr int kTfSmemBytes = kTfStages * kTfStageBytes + 1024 /*bars*/ + 1024 /*align*/;

struct alignas(128) Tf32Params {
  CUtensorMap map_a;  // X [M, K] fp32, box {32, 128}
  CUtensorMap map_b;  // W [N, K] fp32, box {32, 256}
  const float* bias;
  float* y;
  long long ldy;
  int M, N, K, mode;
  int* status;
  unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(kTfThreads, 1) linear_gelu_tf32x3_kernel(const __grid_constant__ Tf32Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kTfStages * kTfStageBytes);  // [2] tiles landed
  uint64_t* mdone_bar = full_bar + kTfStages;                                          // [2] MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone_bar + kTfStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = static_cast<int>(blockIdx.y) * 128, n0 = static_cast<int>(blockIdx.x) * 256;
  const int num_kb = (p.K + kTfBK - 1) / kTfBK;
  const WaitCtx wctx{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTfStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&mdone_bar[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto issue = [&](int kb) {
    uint8_t* st = smem + (kb % kTfStages) * kTfStageBytes;
    mbar_arrive_expect_tx(&full_bar[kb % kTfStages], kTfHalf);
    tma_load_2d(&p.map_a, &full_bar[kb % kTfStages], st, kb * kTfBK, m0);
    tma_load_2d(&p.map_b, &full_bar[kb % kTfStages], st + kTfABytes, kb * kTfBK, n0);
  };
  if (threadIdx.x == 0)
    for (int kb = 0; kb < num_kb && kb < kTfStages; ++kb) issue(kb);
  constexpr uint32_t idesc = idesc_tf32_f32(128, 256);
  int issued = num_kb < kTfStages ? num_kb : kTfStages;  // k blocks whose tiles were requested
  int committed = 0;                                       // k blocks whose MMAs were issued
  bool ok = true;
  for (int kb = 0; kb < num_kb; ++kb) {
    const int s = kb % kTfStages;
    const uint32_t ph = static_cast<uint32_t>(kb / kTfStages) & 1u;
    ok = __syncthreads_and(ok && mbar_wait(&full_bar[s], ph, wctx, W_MMA_FULL)) != 0;
    if (!ok) break;
    // split into hi (in place) and lo (second half of the stage), 16 bytes at a time
    uint4* v = reinterpret_cast<uint4*>(smem + s * kTfStageBytes);
    uint4* lo = reinterpret_cast<uint4*>(smem + s * kTfStageBytes + kTfHalf);
    for (int i = threadIdx.x; i < kTfHalf / 16; i += kTfThreads) {
      const uint4 x = v[i];
      const uint4 h = make_uint4(x.x & 0xFFFFE000u, x.y & 0xFFFFE000u, x.z & 0xFFFFE000u, x.w & 0xFFFFE000u);
      v[i] = h;
      lo[i] = make_uint4(__float_as_uint(__uint_as_float(x.x) - __uint_as_float(h.x)),
                         __float_as_uint(__uint_as_float(x.y) - __uint_as_float(h.y)),
                         __float_as_uint(__uint_as_float(x.z) - __uint_as_float(h.z)),
                         __float_as_uint(__uint_as_float(x.w) - __uint_as_float(h.w)));
    }
    fence_async_smem();  // the tensor core reads what the threads wrote
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t base = smem_u32(smem + s * kTfStageBytes);
      const uint64_t a_hi = sdesc_k_sw128(base), b_hi = sdesc_k_sw128(base + kTfABytes);
      const uint64_t a_lo = sdesc_k_sw128(base + kTfHalf), b_lo = sdesc_k_sw128(base + kTfHalf + kTfABytes);
#pragma unroll
      for (int k = 0; k < kTfBK / 8; ++k) {  // 8 TF32 = 32 bytes per instruction: +2 in the descriptors
        mma_tf32(tmem_base, a_hi + 2 * k, b_hi + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
        mma_tf32(tmem_base, a_hi + 2 * k, b_lo + 2 * k, idesc, 1u);
        mma_tf32(tmem_base, a_lo + 2 * k, b_hi + 2 * k, idesc, 1u);
      }
      mma_commit(&mdone_bar[s]);
      committed = kb + 1;
      if (kb + kTfStages < num_kb) {
        // the stage is refilled once its MMAs have read it
        if (mbar_wait(&mdone_bar[s], ph, wctx, W_MMA_TMEM_EMPTY)) {
          issue(kb + kTfStages);
          ++issued;
        } else {
          ok = false;
        }
      }
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
  }
  if (threadIdx.x == 0) {
    if (ok && num_kb > 0) {
      const int last = num_kb - 1;
      ok = mbar_wait(&mdone_bar[last % kTfStages], static_cast<uint32_t>(last / kTfStages) & 1u, wctx, W_DRAIN);
    }
    if (!ok) {
      // leave no copy in flight and no MMA running before the CTA frees its memory: wait for
      // each stage's most recent load and for the last commit (it covers every earlier MMA)
      for (int kb = issued > kTfStages ? issued - kTfStages : 0; kb < issued; ++kb)
        mbar_wait_quiet(&full_bar[kb % kTfStages], static_cast<uint32_t>(kb / kTfStages) & 1u, p.timeout_ns);
      if (committed > 0)
        mbar_wait_quiet(&mdone_bar[(committed - 1) % kTfStages],
                        static_cast<uint32_t>((committed - 1) / kTfStages) & 1u, p.timeout_ns);
    }
  }
  ok = __syncthreads_and(ok) != 0;
  if (ok) {
    tc_fence_after();
    const int m = m0 + warp * 32 + lane;
    const bool row_ok = m < p.M;
    float* yrow = p.y + static_cast<long long>(row_ok ? m : 0) * p.ldy;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float v[32];
      if (num_kb > 0) {
        uint32_t r[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      const int col0 = n0 + c * 32;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = col0 + j;
        const float x = v[j] + (p.bias != nullptr && n < p.N ? __ldg(p.bias + n) : 0.f);
        v[j] = p.mode == FL_GELU_ERF ? 0.5f * x * (1.f + erff(x * 0.70710678118654752f))
                                     : 0.5f * x * (1.f + tanhf(0.7978845608028654f * (x + 0.044715f * x * x * x)));
      }
      if (!row_ok) continue;
      if (col0 + 32 <= p.N) {  // 16-byte aligned: ldy % 4 == 0, col0 % 32 == 0
#pragma unroll
        for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(yrow + col0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < p.N) yrow[col0 + j] = v[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
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
  if (dtype == FL_BF16) {
    // a few tokens: the swap-AB decode kernel streams W instead of padding a 256-row tile
    st = linear_decode_gelu(X, W, b, Y, M, N, K, ldx, ldw, ldy, mode, di, s);
    if (st != kDecodeNotTaken) return st;
  }

  if (dtype == FL_F32) {
    Tf32Params p;
    std::memset(&p, 0, sizeof(p));
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, X, K, M, ldx, kTfBK, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, W, K, N, ldw, kTfBK, 256,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return FL_ERR_CUDA;
    p.bias = static_cast<const float*>(b);
    p.y = static_cast<float*>(Y);
    p.ldy = ldy;
    p.M = M;
    p.N = N;
    p.K = K;
    p.mode = mode;
    p.status = device_status_ptr(di.device);
    p.timeout_ns = wait_timeout_ns();
    if (p.status == nullptr) return FL_ERR_CUDA;
    const void* kfn = reinterpret_cast<const void*>(&linear_gelu_tf32x3_kernel);
    if (!ensure_smem_attr(kfn, di.device, kTfSmemBytes)) return FL_ERR_CUDA;
    dim3 grid(cdiv(N, 256), cdiv(M, 128));
    linear_gelu_tf32x3_kernel<<<grid, kTfThreads, kTfSmemBytes, s>>>(p);
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
