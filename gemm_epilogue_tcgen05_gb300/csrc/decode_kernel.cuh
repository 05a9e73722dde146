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
constexpr int kDecStages = 10;
constexpr int kDecABytes = 128 * kBK * 2;  // W tile
constexpr int kDecBBytes = kDecTokens * kBK * 2;  // X tile
constexpr int kDecStageBytes = kDecABytes + kDecBBytes;
constexpr int kDecMaxSeg = 32;
// After the weight stream the stage ring is idle; finishing reuses it: up to kDecGatherSlots
// contributors' 16 KB partial tiles are gathered there (cp.async), and the h tiles of the
// first kDecHoldTiles finished feature tiles wait there for the grid-wide statistics.
constexpr int kDecGatherSlots = 10;
constexpr int kDecHoldTiles = 2;
// W units (16 KB each) of its range that a CTA pulls into L2 before waiting for the
// preceding kernel on the stream (programmatic dependent launch).
constexpr int kDecL2PrefetchUnits = 24;
constexpr int kDecSmemBytes = kDecStages * kDecStageBytes + 32 * 129 * 4 + 128 * 4 + 1024 + 1024;

struct alignas(128) DecodeParams {
  CUtensorMap map_w;  // W [N, K] bf16, box {64, 128}
  CUtensorMap map_x;  // X [M, K] bf16, box {64, 32}
  int M, N, K;
  int num_f;          // feature tiles of 128
  int num_kb;         // k blocks of 64
  int units;          // num_f * num_kb (the host keeps units * (grid + 1) < 2^31)
  int seg_max;        // segment slots per CTA in `partials`
  const __nv_bfloat16* bias;
  const __nv_bfloat16* resid;
  long long ldz;
  const __nv_bfloat16* gamma;
  float eps;
  uint8_t* yq;
  long long ldq;
  float* row_scale;
  __nv_bfloat16* hout;  // nullable [M][ldh]: h = X W^T + b + z in bf16 (the residual stream after the add)
  long long ldh;
  float* partials;    // [grid][seg_max][128 features][32 tokens]
  float* hbuf;        // [num_f][32 tokens][128 features]
  float2* stats;      // [num_f][32 tokens] (flat kernel)
  unsigned* counters; // [num_f] k-block arrivals, then finished tiles, then finishers that left
  // Cluster kernel: per (feature tile, token) the tile's sum of h^2 and max |h * gamma|, each in a
  // 64-bit word whose high half is the call's epoch ([num_f][32 tokens][2]), and the workspace's
  // epoch word (the previous call's epoch; this call's is one more).
  unsigned long long* recs;
  unsigned* epoch;
  int* status;
  unsigned long long timeout_ns;
};

// First unit of CTA c: units are cut into `grid` contiguous ranges of near-equal size.
// 32-bit arithmetic on purpose (64-bit division is a long instruction sequence).
__host__ __device__ inline int dec_unit_begin(int c, int units, int grid) {
  return static_cast<int>(static_cast<unsigned>(c) * static_cast<unsigned>(units) / static_cast<unsigned>(grid));
}
// CTA whose unit range contains unit u.
__host__ __device__ inline int dec_cta_of(int u, int units, int grid) {
  return static_cast<int>((static_cast<unsigned>(u + 1) * static_cast<unsigned>(grid) - 1u) /
                          static_cast<unsigned>(units));
}

// h[n .. n+3] of one token's row as bf16 (one 8-byte store when all four lie below `limit`;
// the row is 16-byte aligned and n a multiple of 4).
__device__ __forceinline__ void store_h4(__nv_bfloat16* row, int n, int limit, const float4& h) {
  if (n + 4 <= limit) {
    *reinterpret_cast<uint2*>(row + n) = make_uint2(pack_bf16x2(h.x, h.y), pack_bf16x2(h.z, h.w));
  } else {
    const float e[4] = {h.x, h.y, h.z, h.w};
    for (int j = 0; j < 4 && n + j < limit; ++j) row[n + j] = __float2bfloat16_rn(e[j]);
  }
}

// Bounded spin until *ctr == need.  Gives up when `status` already holds a failure (the count can
// then never complete) or after timeout_ns, recording the failure in status_w.
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
  const int G = static_cast<int>(gridDim.x);
  const int u_begin = dec_unit_begin(blockIdx.x, p.units, G);
  const int u_end = dec_unit_begin(blockIdx.x + 1, p.units, G);
  const int f_first = u_begin / p.num_kb;  // the loops below walk units without dividing

  // The next kernel on the stream may be scheduled now: it only runs on SMs this grid has
  // left, and waits for this grid's completion before touching anything it writes.
  griddep_launch_dependents();
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
    // The weight stream does not depend on earlier work on the stream: start pulling the
    // first units of this CTA's range into L2 while that work may still be finishing (an L2
    // prefetch is coherent with any write, so this is safe whatever precedes).
    int f = f_first, kb = u_begin - f_first * p.num_kb;
    for (int u = u_begin; u < u_end && u < u_begin + kDecL2PrefetchUnits; ++u, ++kb) {
      if (kb == p.num_kb) {
        kb = 0;
        ++f;
      }
      tma_prefetch_l2_2d(&p.map_w, kb * kBK, f * 128);
    }
  }
  if (warp == 2 && u_end > u_begin) {
    // (An epilogue warp, idle until the first partial, so the weight stream starts at once.)
    // Any CTA covering a feature tile may finish it: pull that tile's residual
    // columns (one 256-byte run per token) and gamma / bias into L2 now.
    const int f_last = (u_end - 1) / p.num_kb;
    for (int f = f_first; f <= f_last; ++f) {
      const int n0 = f * 128;
      const uint32_t bytes = static_cast<uint32_t>(min(128, p.N - n0) * 2) & ~15u;
      if (bytes == 0) continue;
      for (int t = lane; t < p.M + 2; t += 32) {
        const __nv_bfloat16* src = t < p.M ? p.resid + static_cast<size_t>(t) * p.ldz + n0
                                           : (t == p.M ? p.gamma + n0 : p.bias + n0);
        if (t == p.M + 1 && p.bias == nullptr) continue;
        bulk_prefetch_l2(src, bytes);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // X, Z, gamma, b and the workspace may be written by the preceding kernel.
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer: W and X tiles per unit
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
      bool ok = true;
      // W is read exactly once: keep it from evicting the partials, statistics
      // and residual columns the finishing phases read back from L2.
      const uint64_t w_policy = l2_policy_evict_first();
      int f = f_first, kb = u_begin - f_first * p.num_kb;
      for (int u = u_begin; u < u_end; ++u, ++kb) {
        if (kb == p.num_kb) {
          kb = 0;
          ++f;
        }
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wctx, W_PRODUCER_EMPTY)) { ok = false; break; }
        uint8_t* a_dst = stage_mem + stage * kDecStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kDecStageBytes);
        tma_load_2d_hint(&p.map_w, &full_bar[stage], a_dst, kb * kBK, f * 128, w_policy);
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
      int u = u_begin;
      for (int f = f_first; u < u_end && ok; ++ls, ++f) {
        const int seg_begin = u;
        const int seg_end = min(u_end, (f + 1) * p.num_kb);
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
    // Global traffic of every phase is laid out so that a warp touches
    // contiguous memory: partial tiles go through shared memory on the way out,
    // and the finishing passes walk the tile token-major (one warp = one token,
    // 4 features per lane).
    const int q = warp & 3;
    const int ti = threadIdx.x - 64;  // 0..127
    const bool leader = ti == 0;
    const int fq = ti & 31;           // feature quad (features 4*fq .. 4*fq+3 of a tile) in the finishing passes
    uint8_t* stage_w = reinterpret_cast<uint8_t*>(hT) + q * 4096;  // this warp's 32 x 128-byte staging rows
    // Residual, bias and gamma of a feature tile in the layout of the token-major pass
    // (token (ti/32) + 4k, features 4*fq .. 4*fq+3 of the tile).
    float z[8][4], b4[4], g4[4];
    int side_tile = -1;
    auto load_side = [&](int ft) {
      const int n = ft * 128 + fq * 4;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = (ti >> 5) + 4 * k;
        load_bf16x4(p.resid + static_cast<size_t>(t) * p.ldz, n, t < p.M ? p.N : 0, z[k]);
      }
      load_bf16x4(p.bias, n, p.bias ? p.N : 0, b4);
      load_bf16x4(p.gamma, n, p.N, g4);
      side_tile = ft;
    };
    // Phase 1: drain each segment's partial accumulator to global scratch and count k blocks.
    int ls = 0;
    int f = f_first;
    for (int u = u_begin; u < u_end; ++ls, ++f) {
      const int seg_begin = u;
      const int seg_end = min(u_end, (f + 1) * p.num_kb);
      u = seg_end;
      const int abuf = ls & 1;
      const uint32_t use = static_cast<uint32_t>(ls >> 1);
      // The last segment's tile is the likeliest one for this CTA to finish: fetch its side
      // operands now, while its last MMAs are still running.
      if (seg_end == u_end) load_side(f);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull_bar[abuf], use & 1u, wctx, W_EPI_TMEM_FULL));
      if (ok) {
        tc_fence_after();
        uint32_t acc[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf * kDecTokens, acc);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&tempty_bar[abuf]);
        // lane = feature row (32 tokens, 128 bytes): stage rows with 16-byte chunks XOR-swizzled by row
        const uint32_t srow = smem_u32(stage_w) + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(srow + ((c ^ (lane & 7)) << 4), acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
        __syncwarp();
        // this warp's 32 rows are 4 KB of the slot [128 rows][32 tokens]; write them contiguously
        float4* dst = reinterpret_cast<float4*>(p.partials) +
                      (static_cast<size_t>(blockIdx.x) * p.seg_max + (f - f_first)) * 1024 + q * 256;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int idx = lane + 32 * k, row = idx >> 3, chunk = idx & 7;
          const float4 v = *reinterpret_cast<const float4*>(stage_w + row * 128 + ((chunk ^ (row & 7)) << 4));
          __stcg(dst + idx, v);
        }
        __syncwarp();
      }
      __threadfence();
      named_bar_sync(1, kEpiThreads);
      if (leader) {
        const int stop = *abort_flag;
        if (!stop) {
          __threadfence();
          const unsigned add = static_cast<unsigned>(seg_end - seg_begin);
          const unsigned old = atomicAdd(p.counters + f, add);
          if (old + add == static_cast<unsigned>(p.num_kb)) {
            __threadfence();  // acquire: the other contributors' partials are visible from here on
            fin_list[(*fin_count)++] = f;
          }
        }
        *epi_stop = stop;
      }
      named_bar_sync(1, kEpiThreads);
      if (*epi_stop) break;  // uniform: only the leader writes it, between the two barriers
    }
    const int nfin = *epi_stop ? 0 : *fin_count;
    // Phase 2: finish the feature tiles this CTA completed: h = sum of partials + b + z,
    // then per-token partial sum of h^2 and max |h * gamma| over the tile's 128 features.
    for (int i = 0; i < nfin; ++i) {
      const int f = fin_list[i];
      if (side_tile != f) load_side(f);
      // contributors' partials, read contiguously: float4 number (ti + 128 k) of each slot is
      // feature row ti/8 + 16 k, tokens 4*(ti%8) .. 4*(ti%8)+3
      float4 acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int c_lo = dec_cta_of(f * p.num_kb, p.units, G);
      const int c_hi = dec_cta_of((f + 1) * p.num_kb - 1, p.units, G);
      const int ncontrib = c_hi - c_lo + 1;
      if (ncontrib <= kDecGatherSlots) {
        // One round trip: every thread copies the 8 float4 it will sum from each contributor's
        // 16 KB partial tile into the idle stage ring (cp.async, all in flight at once).
        for (int j = 0; j < ncontrib; ++j) {
          const int c = c_lo + j;
          const int cf_first = dec_unit_begin(c, p.units, G) / p.num_kb;
          const float4* src = reinterpret_cast<const float4*>(p.partials) +
                              (static_cast<size_t>(c) * p.seg_max + (f - cf_first)) * 1024 + ti;
          const uint32_t dst = smem_u32(stage_mem + j * 16384) + ti * 16;
#pragma unroll
          for (int k = 0; k < 8; ++k) cp_async_16(dst + k * 2048, src + 128 * k);
        }
        cp_async_wait_all();
        for (int j = 0; j < ncontrib; ++j) {
          const float4* slot = reinterpret_cast<const float4*>(stage_mem + j * 16384) + ti;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 w = slot[128 * k];
            acc[k].x += w.x; acc[k].y += w.y; acc[k].z += w.z; acc[k].w += w.w;
          }
        }
      } else {
        for (int c0 = c_lo; c0 <= c_hi; c0 += 4) {
          float4 w[4][8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = c0 + j;
            if (c <= c_hi) {
              const int cf_first = dec_unit_begin(c, p.units, G) / p.num_kb;
              const float4* src = reinterpret_cast<const float4*>(p.partials) +
                                  (static_cast<size_t>(c) * p.seg_max + (f - cf_first)) * 1024 + ti;
#pragma unroll
              for (int k = 0; k < 8; ++k) w[j][k] = __ldcg(src + 128 * k);
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) w[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              acc[k].x += w[j][k].x; acc[k].y += w[j][k].y; acc[k].z += w[j][k].z; acc[k].w += w[j][k].w;
            }
        }
      }
      // transpose through shared memory: hT[token][feature row]
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int row = (ti >> 3) + 16 * k, t0 = 4 * (ti & 7);
        hT[(t0 + 0) * 129 + row] = acc[k].x;
        hT[(t0 + 1) * 129 + row] = acc[k].y;
        hT[(t0 + 2) * 129 + row] = acc[k].z;
        hT[(t0 + 3) * 129 + row] = acc[k].w;
      }
      named_bar_sync(1, kEpiThreads);
      // token-major pass: warp w handles tokens w, w+4, ...; each lane 4 features
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = (ti >> 5) + 4 * k;
        float4 hv;
        hv.x = hT[t * 129 + fq * 4 + 0] + b4[0] + z[k][0];
        hv.y = hT[t * 129 + fq * 4 + 1] + b4[1] + z[k][1];
        hv.z = hT[t * 129 + fq * 4 + 2] + b4[2] + z[k][2];
        hv.w = hT[t * 129 + fq * 4 + 3] + b4[3] + z[k][3];
        if (i < kDecHoldTiles) {
          reinterpret_cast<float4*>(stage_mem + (kDecGatherSlots + i) * 16384)[t * 32 + fq] = hv;
        } else {
          __stcg(reinterpret_cast<float4*>(p.hbuf + (static_cast<size_t>(f) * kDecTokens + t) * 128) + fq, hv);
        }
        float ss = hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w;
        float am = fmaxf(fmaxf(fabsf(hv.x * g4[0]), fabsf(hv.y * g4[1])), fmaxf(fabsf(hv.z * g4[2]), fabsf(hv.w * g4[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ss += __shfl_xor_sync(0xffffffffu, ss, o);
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        }
        if (lane == 0) __stcg(p.stats + static_cast<size_t>(f) * kDecTokens + t, make_float2(ss, am));
        if (p.hout != nullptr && t < p.M) store_h4(p.hout + static_cast<size_t>(t) * p.ldh, f * 128 + fq * 4, p.N, hv);
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
      // Phase 4: merge per-token statistics over all feature tiles (one lane per token),
      // then quantise this CTA's finished tiles token-major and store the codes.
      float* qs_s = gs;  // [32] 448 / max|h * gamma| per token
      if (ti < 32) {
        const int t = ti;
        float SS = 0.f, A = 0.f;
        for (int f0 = 0; f0 < p.num_f; f0 += 32) {
          float2 w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            w[j] = f0 + j < p.num_f ? __ldcg(p.stats + static_cast<size_t>(f0 + j) * kDecTokens + t)
                                    : make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            SS += w[j].x;
            A = fmaxf(A, w[j].y);
          }
        }
        qs_s[t] = A > 0.f ? 448.f / A : 0.f;
        bool has_tile0 = false;
        for (int i = 0; i < nfin; ++i) has_tile0 |= fin_list[i] == 0;
        if (has_tile0 && t < p.M) p.row_scale[t] = rsqrtf(SS / static_cast<float>(p.N) + p.eps) * A * (1.f / 448.f);
      }
      named_bar_sync(1, kEpiThreads);
      for (int i = 0; i < nfin; ++i) {
        const int f = fin_list[i];
        const int n = f * 128 + fq * 4;
        float g4[4];
        load_bf16x4(p.gamma, n, p.N, g4);
        float4 hv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = (ti >> 5) + 4 * k;
          hv[k] = i < kDecHoldTiles
                      ? reinterpret_cast<const float4*>(stage_mem + (kDecGatherSlots + i) * 16384)[t * 32 + fq]
                      : __ldcg(reinterpret_cast<const float4*>(p.hbuf + (static_cast<size_t>(f) * kDecTokens + t) * 128) + fq);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = (ti >> 5) + 4 * k;
          if (t >= p.M) continue;
          const float qs = qs_s[t];
          // + 0: a zero row codes as +0 whatever the sign of gamma
          const uint32_t w = f32x2_to_e4m3x2(fmaf(hv[k].x * g4[0], qs, 0.f), fmaf(hv[k].y * g4[1], qs, 0.f)) |
                             (f32x2_to_e4m3x2(fmaf(hv[k].z * g4[2], qs, 0.f), fmaf(hv[k].w * g4[3], qs, 0.f)) << 16);
          uint8_t* dst = p.yq + static_cast<size_t>(t) * p.ldq + n;
          if (n + 4 <= p.N) {
            *reinterpret_cast<uint32_t*>(dst) = w;
          } else {
            for (int j = 0; j < 4 && n + j < p.N; ++j) dst[j] = static_cast<uint8_t>(w >> (8 * j));
          }
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
