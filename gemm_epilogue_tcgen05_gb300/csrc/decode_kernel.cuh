// Decode-shaped (M <= 32 tokens) down projection + residual + RMSNorm + FP8.
//
// With a few dozen tokens the GEMM degenerates into a stream over W, so the
// kernel is organised around reading W once at full HBM bandwidth and keeping
// launches to one ("GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §边界五: when the
// mainloop is short, saving a launch matters more than hiding the epilogue).
//
//   * swap-AB: D^T[128 features x 32 tokens] = W_tile[128 x K] * X[32 x K]^T on
//     tcgen05 (M = 128 output features, N = 32 tokens, fp32 in TMEM);
//   * split-K over every SM: the (feature tile, 64-wide k block) units are cut
//     into one contiguous range per CTA, so each CTA streams the same number of
//     W bytes;
//   * the CTA whose partial completes a feature tile (counted with an atomic)
//     adds bias and residual, and emits per-token partial sum of squares and
//     max |h * gamma| over its 128 features (the tile-local half of the
//     two-level row reduction, §模式 A);
//   * after a grid-wide count of finished feature tiles (bounded spin, all CTAs
//     co-resident by cooperative launch) the finishers merge the per-token
//     partials and write the E4M3 codes and the per-token scale
//     (§仿射量化与尾声的五步).
#pragma once
#include "gemm_kernel.cuh"

namespace fl {

constexpr int kDecTokens = 32;
constexpr int kDecStages = 8;
constexpr int kDecABytes = 128 * kBK * 2;  // W tile
constexpr int kDecBBytes = kDecTokens * kBK * 2;  // X tile
constexpr int kDecStageBytes = kDecABytes + kDecBBytes;
constexpr int kDecMaxSeg = 32;
constexpr int kDecSmemBytes = kDecStages * kDecStageBytes + 32 * 129 * 4 + 128 * 4 + 1024 + 1024;

struct alignas(128) DecodeParams {
  CUtensorMap map_w;  // W [N, K] bf16, box {64, 128}
  CUtensorMap map_x;  // X [M, K] bf16, box {64, 32}
  int M, N, K;
  int num_f;          // feature tiles of 128
  int num_kb;         // k blocks of 64
  long long units;    // num_f * num_kb
  int seg_max;        // segment slots per CTA in `partials`
  const __nv_bfloat16* bias;
  const __nv_bfloat16* resid;
  long long ldz;
  const __nv_bfloat16* gamma;
  float eps;
  uint8_t* yq;
  long long ldq;
  float* row_scale;
  float* partials;    // [grid][seg_max][128 features][32 tokens]
  float* hbuf;        // [num_f][32 tokens][128 features]
  float2* stats;      // [num_f][32 tokens]
  unsigned* counters; // [num_f] k-block arrivals, then finished tiles, then finishers that left
  int* status;
  unsigned long long timeout_ns;
};

__host__ __device__ inline long long dec_unit_begin(long long c, long long units, long long grid) {
  return c * units / grid;
}
// CTA whose unit range contains unit u.
__host__ __device__ inline int dec_cta_of(long long u, long long units, long long grid) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}

__device__ __forceinline__ bool spin_until(const unsigned* ctr, unsigned need, const int* status,
                                           unsigned long long timeout_ns, int* status_w, int where, int detail) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_u32(ctr) == need) return true;  // exact count: reset to 0 after use
    if ((i & 15u) == 15u) {
      if (*reinterpret_cast<const volatile int*>(status + ST_CODE) != 0) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        record_failure(status_w, where, detail);
        return false;
      }
    }
    __nanosleep(64);
  }
}

__global__ void __launch_bounds__(kThreads, 1) rmsnorm_fp8_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_mem = smem;
  float* hT = reinterpret_cast<float*>(smem + kDecStages * kDecStageBytes);  // [32][129]
  float* gs = hT + 32 * 129;                                                   // [128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gs + 128);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + kDecStages;
  uint64_t* tfull_bar = bars + 2 * kDecStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* fin_count = abort_flag + 1;
  volatile int* epi_stop = abort_flag + 2;  // written by the epilogue leader only
  volatile int* fin_list = abort_flag + 4;  // [kDecMaxSeg]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wctx{abort_flag, p.status, p.timeout_ns};
  const long long G = gridDim.x;
  const long long u_begin = dec_unit_begin(blockIdx.x, p.units, G);
  const long long u_end = dec_unit_begin(blockIdx.x + 1, p.units, G);
  const int f_first = static_cast<int>(u_begin / p.num_kb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *fin_count = 0;
    *epi_stop = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_w);
    tma_prefetch_desc(&p.map_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer: W and X tiles per unit
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
      bool ok = true;
      for (long long u = u_begin; u < u_end; ++u) {
        const int f = static_cast<int>(u / p.num_kb);
        const int kb = static_cast<int>(u - static_cast<long long>(f) * p.num_kb);
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wctx, W_PRODUCER_EMPTY)) { ok = false; break; }
        uint8_t* a_dst = stage_mem + stage * kDecStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kDecStageBytes);
        tma_load_2d(&p.map_w, &full_bar[stage], a_dst, kb * kBK, f * 128);
        tma_load_2d(&p.map_x, &full_bar[stage], a_dst + kDecABytes, kb * kBK, 0);
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kDecStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok)
        for (int s = 0; s < kDecStages; ++s)
          if (issued_mask & (1u << s)) mbar_wait_quiet(&full_bar[s], (issued_phase >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA: one accumulator per segment
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kDecTokens);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int ls = 0;
      for (long long u = u_begin; u < u_end && ok; ++ls) {
        const int f = static_cast<int>(u / p.num_kb);
        const long long seg_begin = u;
        const long long seg_end = min(u_end, static_cast<long long>(f + 1) * p.num_kb);
        const int abuf = ls & 1;
        const uint32_t use = static_cast<uint32_t>(ls >> 1);
        if (!mbar_wait(&tempty_bar[abuf], (use & 1u) ^ 1u, wctx, W_MMA_TMEM_EMPTY)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + abuf * kDecTokens;
        for (; u < seg_end; ++u) {
          if (!mbar_wait(&full_bar[stage], phase, wctx, W_MMA_FULL)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_mem + stage * kDecStageBytes);
          const uint64_t adesc = sdesc_k_sw128(a_addr);
          const uint64_t bdesc = sdesc_k_sw128(a_addr + kDecABytes);
          const bool first = u == seg_begin;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (!first || k > 0) ? 1u : 0u);
          mma_commit(&empty_bar[stage]);
          if (++stage == kDecStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[abuf]);
      }
      mma_commit(drain_bar);
      mbar_wait_quiet(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;
    const int r = q * 32 + lane;  // feature row of the tile owned by this thread
    const int ti = threadIdx.x - 64;  // 0..127
    const bool leader = ti == 0;
    // Phase 1: drain each segment's partial accumulator to global scratch and count k blocks.
    int ls = 0;
    for (long long u = u_begin; u < u_end; ++ls) {
      const int f = static_cast<int>(u / p.num_kb);
      const long long seg_begin = u;
      const long long seg_end = min(u_end, static_cast<long long>(f + 1) * p.num_kb);
      u = seg_end;
      const int abuf = ls & 1;
      const uint32_t use = static_cast<uint32_t>(ls >> 1);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull_bar[abuf], use & 1u, wctx, W_EPI_TMEM_FULL));
      if (ok) {
        tc_fence_after();
        uint32_t acc[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf * kDecTokens, acc);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&tempty_bar[abuf]);
        float4* dst = reinterpret_cast<float4*>(
            p.partials + ((static_cast<size_t>(blockIdx.x) * p.seg_max + (f - f_first)) * 128 + r) * kDecTokens);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          __stcg(dst + i, make_float4(__uint_as_float(acc[4 * i]), __uint_as_float(acc[4 * i + 1]),
                                      __uint_as_float(acc[4 * i + 2]), __uint_as_float(acc[4 * i + 3])));
      }
      __threadfence();
      named_bar_sync(1, kEpiThreads);
      if (leader) {
        const int stop = *abort_flag;
        if (!stop) {
          __threadfence();
          const unsigned add = static_cast<unsigned>(seg_end - seg_begin);
          const unsigned old = atomicAdd(p.counters + f, add);
          if (old + add == static_cast<unsigned>(p.num_kb)) fin_list[(*fin_count)++] = f;
        }
        *epi_stop = stop;
      }
      named_bar_sync(1, kEpiThreads);
      if (*epi_stop) break;  // uniform: only the leader writes it, between the two barriers
    }
    const int nfin = *epi_stop ? 0 : *fin_count;
    // Phase 2: finish the feature tiles this CTA completed: h = sum of partials + b + z.
    for (int i = 0; i < nfin; ++i) {
      const int f = fin_list[i];
      const int n = f * 128 + r;
      const bool n_ok = n < p.N;
      float h[kDecTokens];
#pragma unroll
      for (int t = 0; t < kDecTokens; ++t) h[t] = 0.f;
      const int c_lo = dec_cta_of(static_cast<long long>(f) * p.num_kb, p.units, G);
      const int c_hi = dec_cta_of(static_cast<long long>(f + 1) * p.num_kb - 1, p.units, G);
      for (int c = c_lo; c <= c_hi; ++c) {
        const int cf_first = static_cast<int>(dec_unit_begin(c, p.units, G) / p.num_kb);
        const float4* src = reinterpret_cast<const float4*>(
            p.partials + ((static_cast<size_t>(c) * p.seg_max + (f - cf_first)) * 128 + r) * kDecTokens);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 w = __ldcg(src + j);
          h[4 * j] += w.x; h[4 * j + 1] += w.y; h[4 * j + 2] += w.z; h[4 * j + 3] += w.w;
        }
      }
      const float bn = (p.bias && n_ok) ? __bfloat162float(p.bias[n]) : 0.f;
#pragma unroll
      for (int t = 0; t < kDecTokens; ++t) {
        const float z = (t < p.M && n_ok) ? __bfloat162float(p.resid[t * p.ldz + n]) : 0.f;
        hT[t * 129 + r] = h[t] + bn + z;
      }
      gs[r] = n_ok ? __bfloat162float(p.gamma[n]) : 0.f;
      named_bar_sync(1, kEpiThreads);
      {
        // token t, quarter part of the 128 features
        const int t = ti >> 2, part = ti & 3;
        float ss = 0.f, am = 0.f;
        float* hrow = p.hbuf + (static_cast<size_t>(f) * kDecTokens + t) * 128 + part * 32;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 w;
          w.x = hT[t * 129 + part * 32 + j];
          w.y = hT[t * 129 + part * 32 + j + 1];
          w.z = hT[t * 129 + part * 32 + j + 2];
          w.w = hT[t * 129 + part * 32 + j + 3];
          ss = fmaf(w.x, w.x, fmaf(w.y, w.y, fmaf(w.z, w.z, fmaf(w.w, w.w, ss))));
          am = fmaxf(am, fmaxf(fmaxf(fabsf(w.x * gs[part * 32 + j]), fabsf(w.y * gs[part * 32 + j + 1])),
                               fmaxf(fabsf(w.z * gs[part * 32 + j + 2]), fabsf(w.w * gs[part * 32 + j + 3]))));
          __stcg(reinterpret_cast<float4*>(hrow + j), w);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        if (part == 0) __stcg(p.stats + static_cast<size_t>(f) * kDecTokens + t, make_float2(ss, am));
      }
      named_bar_sync(1, kEpiThreads);
      if (leader) p.counters[f] = 0u;  // every contributor has arrived; ready for the next call
    }
    // Phase 3: wait until every feature tile has published its per-token partials.
    __threadfence();
    named_bar_sync(1, kEpiThreads);
    if (leader) {
      int stop = *epi_stop || *abort_flag;
      if (!stop && nfin > 0) {
        __threadfence();
        atomicAdd(p.counters + p.num_f, static_cast<unsigned>(nfin));
        if (!spin_until(p.counters + p.num_f, static_cast<unsigned>(p.num_f), p.status, p.timeout_ns, p.status,
                        W_DECODE_ROWS, p.num_f)) {
          stop = 1;
          *abort_flag = 1;
        }
      }
      *epi_stop = stop;
    }
    named_bar_sync(1, kEpiThreads);
    const bool finish = !*epi_stop && nfin > 0;
    if (finish) {
      // Phase 4: merge per-token statistics over all feature tiles, quantise, store.
      const int t = ti >> 2, part = ti & 3;
      float SS = 0.f, A = 0.f;
      for (int f2 = 0; f2 < p.num_f; ++f2) {
        const float2 w = __ldcg(p.stats + static_cast<size_t>(f2) * kDecTokens + t);
        SS += w.x;
        A = fmaxf(A, w.y);
      }
      const float qs = A > 0.f ? 448.f / A : 0.f;
      for (int i = 0; i < nfin; ++i) {
        const int f = fin_list[i];
        if (f == 0 && part == 0 && t < p.M) p.row_scale[t] = rsqrtf(SS / static_cast<float>(p.N) + p.eps) * A * (1.f / 448.f);
        if (t >= p.M) continue;
        const float* hrow = p.hbuf + (static_cast<size_t>(f) * kDecTokens + t) * 128 + part * 32;
        const int n0 = f * 128 + part * 32;
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 hv = __ldcg(reinterpret_cast<const float4*>(hrow + j));
          const float g0 = n0 + j < p.N ? __bfloat162float(p.gamma[n0 + j]) : 0.f;
          const float g1 = n0 + j + 1 < p.N ? __bfloat162float(p.gamma[n0 + j + 1]) : 0.f;
          const float g2 = n0 + j + 2 < p.N ? __bfloat162float(p.gamma[n0 + j + 2]) : 0.f;
          const float g3 = n0 + j + 3 < p.N ? __bfloat162float(p.gamma[n0 + j + 3]) : 0.f;
          w[j / 4] = f32x2_to_e4m3x2(hv.x * g0 * qs, hv.y * g1 * qs) |
                     (f32x2_to_e4m3x2(hv.z * g2 * qs, hv.w * g3 * qs) << 16);
        }
        uint8_t* dst = p.yq + static_cast<size_t>(t) * p.ldq + n0;
        if (n0 + 32 <= p.N) {
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          for (int j = 0; j < 32 && n0 + j < p.N; ++j) dst[j] = static_cast<uint8_t>(w[j / 4] >> (8 * (j % 4)));
        }
      }
    }
    named_bar_sync(1, kEpiThreads);
    if (leader && finish) {
      // The last finisher to leave resets the grid-wide counters for the next call.
      const unsigned old = atomicAdd(p.counters + p.num_f + 1, static_cast<unsigned>(nfin));
      if (old + nfin == static_cast<unsigned>(p.num_f)) {
        p.counters[p.num_f] = 0u;
        p.counters[p.num_f + 1] = 0u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 64);
  }
}

}  // namespace fl
