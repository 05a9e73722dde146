// Decode-shaped (M <= 32 tokens) down projection + residual + RMSNorm + FP8, one thread-block
// cluster per 128-feature tile.
//
// The same computation as rmsnorm_fp8_decode_kernel, organised so that no partial result
// leaves the chip before the row statistics:
//   * cluster f (C CTAs) owns features [128 f, 128 f + 128); CTA r of the cluster streams the
//     k blocks [r K/C, (r+1) K/C) of that W tile (swap-AB on tcgen05: D^T[128 x 32 tokens]
//     in TMEM), so every CTA reads the same number of W bytes;
//   * the C partial tiles are summed through distributed shared memory, in rank order (so the
//     result is deterministic), each CTA reducing 128/C of the features and adding bias and
//     residual; the resulting h and the per-token partial sums of h^2 and max |h * gamma| go
//     to the cluster leader's shared memory, and every other CTA of the cluster leaves, so
//     the SMs free up for the next kernel on the stream;
//   * the leaders publish their cluster's per-token partials ("GEMM Epilogue 完全拆解",
//     §模式 A: the tile-local half of the two-level row reduction), each value in a 64-bit word
//     tagged with the call's epoch, and count themselves on a grid-wide counter; every leader
//     polls all num_f partials of its tokens and the count at once (bounded; every cluster is
//     resident, the host checks) until each carries this call's epoch and the count is exactly
//     num_f, so the wait and the loads are one round trip, then merges them per token in a fixed
//     order and writes the E4M3 codes and the per-token scale (§仿射量化与尾声的五步).
//     The tag alone tells a value of this call from one of an earlier, completed call.  The count
//     gives the wait a condition that lives in the workspace where the host can see it: a count
//     that can never be exactly num_f (a workspace not zero-filled as the contract asks, or one a
//     failure test has set) makes the wait run out and report FL_ERR_TIMEOUT rather than finish.
//     It is a relaxed add, not a release: the tags already make each record self-validating, and a
//     release fence in front of the add cost about 0.2 us per call.
// Every CTA passes the cluster barriers it shares with its peers whatever happens (errors only
// skip work), so a timed-out wait can never leave a peer blocked at a barrier.
#pragma once
#include "decode_kernel.cuh"

namespace fl {

constexpr int kDcStages = 10;
// W tiles (16 KB) of its k range that a CTA pulls into L2 before waiting for the preceding
// kernel (measured back to back: 0 -> 28.6 us per call, 8 -> 27.5, 16 -> 26.9, 32 -> 29.4).
constexpr int kDcL2PrefetchUnits = 16;
constexpr int kDcSmallBytes = 8192;  // per-token partials of the ranks (Sall), flags
constexpr int kDcSmemBytes = kDcStages * kDecStageBytes + kDcSmallBytes + 1024 /*bars*/ + 1024 /*align*/;

template <int C>
__global__ void __launch_bounds__(kThreads, 1) rmsnorm_fp8_decode_cluster_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(C == 1 || C == 2 || C == 4 || C == 8, "cluster size");
  constexpr int kRows = 128 / C;          // feature rows this CTA reduces
  constexpr int kGroups = kRows / 8;      // groups of 8 features per token
  constexpr int kItems = 32 * kGroups;    // (token, group) items
  constexpr int kIpt = (kItems + 127) / 128;  // items per epilogue thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_mem = smem;
  float* P = reinterpret_cast<float*>(stage_mem);  // [32 tokens][128 features] after the stream
  uint8_t* small = smem + kDcStages * kDecStageBytes;
  float2* Sall = reinterpret_cast<float2*>(small);         // [8][32] the ranks' per-token partials (leader)
  volatile int* flags = reinterpret_cast<volatile int*>(Sall + 8 * 32);  // [0] ok, [1] grid count reached
  uint64_t* bars = reinterpret_cast<uint64_t*>(small + kDcSmallBytes);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + kDcStages;
  uint64_t* tfull_bar = bars + 2 * kDcStages;
  uint64_t* drain_bar = tfull_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wctx{abort_flag, p.status, p.timeout_ns};
  const uint32_t rank = C > 1 ? cluster_ctarank() : 0u;
  const int f = static_cast<int>(blockIdx.x) / C;  // feature tile of this cluster
  const int kb0 = static_cast<int>(rank) * p.num_kb / C;
  const int kb1 = (static_cast<int>(rank) + 1) * p.num_kb / C;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDcStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    flags[0] = 1;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_w);
    tma_prefetch_desc(&p.map_x);
    // The weights do not depend on earlier work on the stream: pull the first tiles into L2 now,
    // before the wait below (an L2 prefetch is coherent with any write).  Measured: issuing them
    // here, ahead of the producer's own loads of the same tiles, beats issuing them from another
    // warp while the producer starts (25.4 vs 27.7 us per call back to back).
    for (int kb = kb0; kb < kb1 && kb < kb0 + kDcL2PrefetchUnits; ++kb) tma_prefetch_l2_2d(&p.map_w, kb * kBK, f * 128);
  }
  if (warp == 2) {
    // residual rows, gamma and bias of this cluster's features into L2 (one 256-byte run each)
    const int n0 = f * 128;
    const uint32_t bytes = static_cast<uint32_t>(min(128, p.N - n0) * 2) & ~15u;
    if (bytes != 0)
      for (int t = lane; t < p.M + 2; t += 32) {
        if (t == p.M + 1 && p.bias == nullptr) continue;
        const __nv_bfloat16* src = t < p.M ? p.resid + static_cast<size_t>(t) * p.ldz + n0
                                           : (t == p.M ? p.gamma + n0 : p.bias + n0);
        bulk_prefetch_l2(src, bytes);
      }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // X, Z, gamma, b and the workspace may be written by the preceding kernel
  // this call's epoch (leaders): one more than the previous call's, which the last leader of that
  // call stored after every leader had read it
  const unsigned epoch = rank == 0 && threadIdx.x >= 32 ? ld_relaxed_u32(p.epoch) + 1u : 0u;

  // Residual, bias and gamma of the epilogue threads' reduce items (phase 2): loaded by the
  // epilogue warps while the weights stream, so none of their latency is left for the tail.
  const int ti = static_cast<int>(threadIdx.x) - 64;  // epilogue thread 0..127, or negative
  float zs[kIpt][8], bs[kIpt][8], gs[kIpt][8];

  // ---------------------------------------------------------------- phase 1: stream W, partial tile
  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
      bool ok = true;
      const uint64_t w_policy = l2_policy_evict_first();
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wctx, W_PRODUCER_EMPTY)) { ok = false; break; }
        uint8_t* a_dst = stage_mem + stage * kDecStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kDecStageBytes);
        tma_load_2d_hint(&p.map_w, &full_bar[stage], a_dst, kb * kBK, f * 128, w_policy);
        tma_load_2d(&p.map_x, &full_bar[stage], a_dst + kDecABytes, kb * kBK, 0);
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kDcStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) {
        flags[0] = 0;
        for (int s = 0; s < kDcStages; ++s)
          if (issued_mask & (1u << s)) mbar_wait_quiet(&full_bar[s], (issued_phase >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kDecTokens);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, wctx, W_MMA_FULL)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stage_mem + stage * kDecStageBytes);
        const uint64_t adesc = sdesc_k_sw128(a_addr);
        const uint64_t bdesc = sdesc_k_sw128(a_addr + kDecABytes);
#pragma unroll
        for (int k = 0; k < kBK / kUmmaK; ++k)
          mma_bf16(tmem_base, adesc + 2 * k, bdesc + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        mma_commit(&empty_bar[stage]);
        if (++stage == kDcStages) { stage = 0; phase ^= 1u; }
      }
      if (ok) mma_commit(tfull_bar);
      else flags[0] = 0;
      mma_commit(drain_bar);
      mbar_wait_quiet(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // TMEM lane quarter q = feature rows 32 q .. 32 q + 31; each thread one row, 32 tokens.
    const int q = warp & 3;
#pragma unroll
    for (int it = 0; it < kIpt; ++it) {
      const int item = ti + 128 * it;
      const int t = item / kGroups, g = item % kGroups;
      const int n = f * 128 + static_cast<int>(rank) * kRows + g * 8;
      const bool in = item < kItems;
      const __nv_bfloat16* zr = p.resid + static_cast<size_t>(in && t < p.M ? t : 0) * p.ldz;
      const int zl = in && t < p.M ? p.N : 0, bl = in && p.bias ? p.N : 0, gl = in ? p.N : 0;
      load_bf16x4(zr, n, zl, *reinterpret_cast<float(*)[4]>(zs[it]));
      load_bf16x4(zr, n + 4, zl, *reinterpret_cast<float(*)[4]>(zs[it] + 4));
      load_bf16x4(p.bias, n, bl, *reinterpret_cast<float(*)[4]>(bs[it]));
      load_bf16x4(p.bias, n + 4, bl, *reinterpret_cast<float(*)[4]>(bs[it] + 4));
      load_bf16x4(p.gamma, n, gl, *reinterpret_cast<float(*)[4]>(gs[it]));
      load_bf16x4(p.gamma, n + 4, gl, *reinterpret_cast<float(*)[4]>(gs[it] + 4));
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar, 0, wctx, W_EPI_TMEM_FULL));
    if (ok) {
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16), acc);
      tmem_ld_wait();
      // P[t][n]: for a fixed token the warp writes 32 consecutive floats (no bank conflict)
      const int n = q * 32 + lane;
#pragma unroll
      for (int t = 0; t < 32; ++t) P[t * 128 + n] = __uint_as_float(acc[t]);
    } else if (lane == 0) {
      flags[0] = 0;
    }
  }
  // Cluster barrier A: every CTA of the cluster has its partial tile in P (each thread's arrive
  // releases its own writes, so the CTA needs no barrier of its own in front of it).
  __syncwarp();
  if (C > 1) cluster_sync_all();
  else __syncthreads();

  // ---------------------------------------------------------------- phase 2: cluster reduce, h, statistics
  // In the leader's shared memory: H [32 tokens][128 features] fp32 right after P, and the
  // ranks' per-token partials Sall [C][32].
  float* H = P + 32 * 128;
  // The ranks' ok flags and partial tiles are all loaded at once (reading a peer's P is safe
  // whatever its flag says: the partials are used only when every flag is set).
  int fv[C];
  float4 xa[kIpt][C], xb[kIpt][C];
  if constexpr (C > 1) {
#pragma unroll
    for (int j = 0; j < C; ++j)
      fv[j] = ld_dsmem_s32(mapa_shared(smem_u32(const_cast<int*>(flags)), static_cast<uint32_t>(j)));
  } else {
    fv[0] = flags[0];
  }
  if (ti >= 0) {
#pragma unroll
    for (int it = 0; it < kIpt; ++it) {
      const int item = ti + 128 * it;
      if (item >= kItems) continue;
      const int t = item / kGroups, g = item % kGroups;
      const int row = static_cast<int>(rank) * kRows + g * 8;
      const uint32_t local = smem_u32(P + t * 128 + row);
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if constexpr (C > 1) {
          const uint32_t ra = mapa_shared(local, static_cast<uint32_t>(j));
          xa[it][j] = ld_dsmem_f4(ra);
          xb[it][j] = ld_dsmem_f4(ra + 16);
        } else {
          xa[it][j] = *reinterpret_cast<const float4*>(P + t * 128 + row);
          xb[it][j] = *reinterpret_cast<const float4*>(P + t * 128 + row + 4);
        }
      }
    }
  }
  int all = 1;
#pragma unroll
  for (int j = 0; j < C; ++j) all &= fv[j] != 0 ? 1 : 0;
  const bool cl_ok = all != 0;
  if (ti >= 0 && cl_ok) {
#pragma unroll
    for (int it = 0; it < kIpt; ++it) {
      // The groups of one token sit in kGroups consecutive lanes; kItems is a multiple of 32, so
      // whether a thread has an item is the same across its warp.
      const int item = ti + 128 * it;
      const bool has = item < kItems;
      const int t = item / kGroups, g = item % kGroups;
      const int row = static_cast<int>(rank) * kRows + g * 8;  // first feature row within the tile
      float ss = 0.f, am = 0.f;
      if (has) {
        float4 a = xa[it][0], b = xb[it][0];
#pragma unroll
        for (int j = 1; j < C; ++j) {  // rank order: deterministic
          a.x += xa[it][j].x; a.y += xa[it][j].y; a.z += xa[it][j].z; a.w += xa[it][j].w;
          b.x += xb[it][j].x; b.y += xb[it][j].y; b.z += xb[it][j].z; b.w += xb[it][j].w;
        }
        const float s8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float hv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          hv[e] = s8[e] + bs[it][e] + zs[it][e];  // features past N: W rows, b and z are zero there
          ss += hv[e] * hv[e];
          am = fmaxf(am, fabsf(hv[e] * gs[it][e]));
        }
        if (p.hout != nullptr && t < p.M) {  // h leaves in bf16 as well (the residual stream after the add)
          __nv_bfloat16* hrow = p.hout + static_cast<size_t>(t) * p.ldh;
          store_h4(hrow, f * 128 + row, p.N, make_float4(hv[0], hv[1], hv[2], hv[3]));
          store_h4(hrow, f * 128 + row + 4, p.N, make_float4(hv[4], hv[5], hv[6], hv[7]));
        }
        // h to the leader's H[t][row ..]
        const uint32_t hl = smem_u32(H + t * 128 + row);
        if constexpr (C > 1) {
          const uint32_t hr = mapa_shared(hl, 0u);
          st_dsmem_f4(hr, make_float4(hv[0], hv[1], hv[2], hv[3]));
          st_dsmem_f4(hr + 16, make_float4(hv[4], hv[5], hv[6], hv[7]));
        } else {
          *reinterpret_cast<float4*>(H + t * 128 + row) = make_float4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<float4*>(H + t * 128 + row + 4) = make_float4(hv[4], hv[5], hv[6], hv[7]);
        }
      }
      // this rank's per-token partial over its kRows features: a butterfly over the token's lanes
      // (every lane ends with the same bits, whatever the run)
#pragma unroll
      for (int o = kGroups / 2; o > 0; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      }
      if (has && g == 0) {
        const uint32_t sl = smem_u32(Sall + rank * 32 + t);
        if constexpr (C > 1) st_dsmem_f2(mapa_shared(sl, 0u), make_float2(ss, am));
        else Sall[t] = make_float2(ss, am);
      }
    }
  }
  // Cluster barrier B: every read of a peer's P and every write into the leader's H and Sall is
  // done; the other CTAs of the cluster then leave, freeing their SMs for the next kernel.
  __syncwarp();
  if (C > 1) cluster_sync_all();
  else __syncthreads();

  if (rank == 0) {
    // ---------------------------------------------------------------- phase 3: publish, grid-wide count (leader)
    // this thread's quantisation slice: token tq, features 32 (ti % 4) .. + 31 of the tile; its
    // gamma is loaded before the grid-wide wait
    const int tq = ti >> 2, c0 = (ti & 3) * 32;
    const int n = f * 128 + c0;
    float gq[32];
    if (ti >= 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) load_bf16x4(p.gamma, n + 4 * k, p.N, *reinterpret_cast<float(*)[4]>(gq + 4 * k));
    }
    const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
    if (warp == 1 && cl_ok) {
      // the MMA warp is idle now: it merges the ranks' partials (lane = token) and publishes
      // them, each value with the epoch in the same 64-bit word, then counts the cluster, while the
      // epilogue warps load gamma
      float ss = 0.f, am = 0.f;
      for (int j = 0; j < C; ++j) {  // rank order: deterministic
        const float2 v = Sall[j * 32 + lane];
        ss += v.x;
        am = fmaxf(am, v.y);
      }
      unsigned long long* rec = p.recs + (static_cast<size_t>(f) * kDecTokens + lane) * 2;
      st_relaxed_u64x2(rec, tag | __float_as_uint(ss), tag | __float_as_uint(am));
      __syncwarp();
      if (lane == 0) red_relaxed_add_u32(p.counters + p.num_f, 1u);
    }

    // ---------------------------------------------------------------- phase 4: merge statistics, quantise (leader)
    // The four threads of token tq each merge every fourth cluster's partial (fixed order), then
    // combine by a butterfly, so all four hold the same bits.  Each group of 8 partials, and the
    // count, is polled until all carry this call's epoch and the count is exactly num_f (a cluster
    // that failed publishes nothing, and every wait gives up once a failure is recorded).  A
    // record's two words are read in one 16-byte load (each word is single-copy atomic and carries
    // its own tag) and the poll spins without a sleep: both together measured 0.06 us faster per
    // call back to back, 0.08 us with another kernel between calls (5 alternating runs on one box,
    // every run faster).
    float SS = 0.f, A = 0.f;
    bool ready = true;
    if (ti >= 0) {
      ready = cl_ok;
      const uint64_t t0 = global_timer_ns();
      for (int cb = ti & 3; cb < p.num_f && ready; cb += 32) {
        for (uint32_t i = 0;; ++i) {
          unsigned long long w[8][2];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = cb + 4 * j;
            const unsigned long long* rec = p.recs + (static_cast<size_t>(c) * kDecTokens + tq) * 2;
            if (c < p.num_f) {
              ld_relaxed_u64x2(rec, w[j][0], w[j][1]);
            } else {
              w[j][0] = tag;
              w[j][1] = tag;
            }
          }
          bool all = ld_relaxed_u32(p.counters + p.num_f) == static_cast<unsigned>(p.num_f);
#pragma unroll
          for (int j = 0; j < 8; ++j) all = all && (w[j][0] >> 32) == epoch && (w[j][1] >> 32) == epoch;
          if (all) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (cb + 4 * j >= p.num_f) continue;  // past the last tile: contributes nothing
              SS += __uint_as_float(static_cast<uint32_t>(w[j][0]));
              A = fmaxf(A, __uint_as_float(static_cast<uint32_t>(w[j][1])));
            }
            break;
          }
          if ((i & 15u) == 15u) {
            if (*reinterpret_cast<const volatile int*>(p.status + ST_CODE) != 0) {
              ready = false;
              break;
            }
            if (global_timer_ns() - t0 > p.timeout_ns) {
              record_failure(p.status, W_DECODE_ROWS, p.num_f);
              ready = false;
              break;
            }
          }
        }
      }
    }
    const bool finish = __syncthreads_and(ready ? 1 : 0) != 0;
    if (finish && ti >= 0) {
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        SS += __shfl_xor_sync(0xffffffffu, SS, o);
        A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, o));
      }
      const float qs = A > 0.f ? 448.f / A : 0.f;
      if (f == 0 && (ti & 3) == 0 && tq < p.M)
        p.row_scale[tq] = rsqrtf(SS / static_cast<float>(p.N) + p.eps) * A * (1.f / 448.f);
      if (tq < p.M && n < p.N) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 hv = *reinterpret_cast<const float4*>(H + tq * 128 + c0 + 4 * k);
          const float* gg = gq + 4 * k;
          // + 0: a zero row codes as +0 whatever the sign of gamma
          w[k] = f32x2_to_e4m3x2(fmaf(hv.x * gg[0], qs, 0.f), fmaf(hv.y * gg[1], qs, 0.f)) |
                 (f32x2_to_e4m3x2(fmaf(hv.z * gg[2], qs, 0.f), fmaf(hv.w * gg[3], qs, 0.f)) << 16);
        }
        uint8_t* dst = p.yq + static_cast<size_t>(tq) * p.ldq + n;
        if (n + 32 <= p.N) {  // 16-byte aligned: ldq % 16 == 0, n % 32 == 0
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < p.N) dst[j] = static_cast<uint8_t>(w[j >> 2] >> (8 * (j & 3)));
        }
      }
    }
    if (threadIdx.x == 64 && finish) {
      // the last leader to leave resets the counters for the next call and stores this call's
      // epoch (every leader has read the count and the previous epoch once the leavers are complete)
      const unsigned old = atomicAdd(p.counters + p.num_f + 1, 1u);
      if (old + 1u == static_cast<unsigned>(p.num_f)) {
        p.counters[p.num_f] = 0u;
        p.counters[p.num_f + 1] = 0u;
        *p.epoch = epoch;
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace fl
