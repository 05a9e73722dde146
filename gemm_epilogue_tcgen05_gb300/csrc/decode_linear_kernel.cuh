// Decode-shaped (M <= 32 tokens) Linear layers with element-wise epilogues: bias + GELU, SwiGLU,
// the fused QKV projection with RoPE, and its grouped-query form with the K/V cache entry in FP8.
//
// With a few dozen tokens the GEMM is a stream over W ("GEMM Epilogue 完全拆解"
// (pinghaoyang.com.cn), §边界五), and a 256-row output tile would spend its tensor-core time on
// rows that do not exist.  The kernel therefore swaps the operands like the RMSNorm decode
// kernel: D^T[128 W rows x 32 tokens] = W_tile * X^T on tcgen05 (MMA M = 128, N = 32), one
// thread-block cluster of C CTAs per tile of W rows, CTA r streaming the k blocks
// [r K/C, (r+1) K/C).  No row statistic couples the tiles, so the tail stays inside the cluster:
// the C partial tiles are summed through distributed shared memory in rank order (deterministic),
// each CTA finishing its share of the tile's outputs: bias, then GELU (§GELU激活融合 of "Triton
// 算子融合: Linear 与 Attention"), SiLU(g) u (§模式 B of the epilogue page), or the rotation of
// adjacent feature pairs of Q and K (§QKV投影融合 of the Triton page; §模式 B), written as bf16
// with 16-byte stores.
//
// A tile of W rows is
//   GELU:   128 output features;
//   QKV:    one head (128 rows) of the Q, K or V section of the stacked W_qkv (the FP8 K/V form:
//           K rotated, then K and V as E4M3 with one scale per token and head, max|.|/448 over the
//           head's 128 values; there each CTA finishes whole tokens, all 128 features of the head,
//           so the maximum is a shuffle inside the CTA and needs no exchange between the CTAs);
//   SwiGLU: 64 gate rows and the 64 up rows of the same 64 output features (two TMA boxes), so the
//           gate and up values of a feature sit in the same tile.
//   block-scaled write-back: 128 output features, finished like the FP8 K/V form by whole tokens,
//           so every block of 128, 32 or 16 columns of a token lies inside one CTA.
//   the deferred-scale chain: 128 output features; step 1 (h1 = XW^T + b + Z, h2 = h1 * gamma and
//           each token's sum of h1^2) is finished by whole tokens, step 2 (r * (H2 W1^T) + b1) by
//           features like GELU.
// Every CTA passes both cluster barriers whatever happens (errors only skip work).
#pragma once
#include "gemm_kernel.cuh"

namespace fl {

enum LinearDecodeKind : int {
  LD_GELU_TANH = 0, LD_GELU_ERF = 1, LD_SWIGLU = 2, LD_QKV_ROPE = 3, LD_QKV_FP8KV = 4, LD_QUANT = 5,
  LD_RESGAMMA = 6,  // step 1 of the deferred-scale chain: h1 = XW^T + b + Z, h1 * gamma, sums of h1^2
  LD_ROWSCALE = 7   // step 2: y = r * (H2 W1^T) + b1 with r merged from the step-1 sums
};

constexpr int kLdTokens = 32;                   // MMA N: the tokens
constexpr int kLdStages = 10;
constexpr int kLdABytes = 128 * kBK * 2;        // W rows of the tile
constexpr int kLdStageBytes = kLdABytes + kLdTokens * kBK * 2;
// W k blocks a CTA pulls into L2 before griddepcontrol.wait.  Measured per call (3 alternating runs on
// one box, us; back to back in a graph / interleaved with another kernel / single launch), window 8
// against 16: QKV + FP8 K/V 32 x 6144 x 4096 12.15 / 12.88 / 20.1 against 12.02 / 13.72 / 20.8, QKV
// 32 x 12288 x 4096 18.4 / 20.6 / 29.1 against 19.0 / 22.5 / 30.4, GELU 32 x 16384 x 4096 22.6 / 23.3
// / 31.4 against 22.3 / 23.8 / 31.7, SwiGLU 32 x 14336 x 4096 35.6 / 38.7 / 48.1 against 37.4 / 39.8 /
// 48.5.  A deep window competes with the call's own stream when no earlier call is left to overlap.
constexpr int kLdL2PrefetchUnits = 8;

struct alignas(128) LinearDecodeParams {
  CUtensorMap map_w;   // W [rows, K] bf16, box {64, 128}; SwiGLU: W_gate, box {64, 64}
  CUtensorMap map_w2;  // SwiGLU: W_up, box {64, 64}
  CUtensorMap map_x;   // X [M, K] bf16, box {64, 32}
  int M, K;
  int n_out;           // output features: GELU N, SwiGLU d_ff, QKV d_model (the Q section)
  int kv_width;        // QKV: width of the K and V sections (= n_out for the plain QKV)
  int num_f, num_kb;   // W-row tiles, 64-wide k blocks
  int f0;              // first tile of this launch (a call with more tiles than fit at once takes several)
  const __nv_bfloat16* bias;   // [W rows] or null (SwiGLU: b_gate [d_ff])
  const __nv_bfloat16* bias2;  // SwiGLU: b_up [d_ff] or null
  __nv_bfloat16* out[3];       // GELU, SwiGLU: out[0]; QKV: Q, K, V (FP8 K/V form: Q only)
  long long ldo;
  uint8_t* out_kv[2];          // FP8 K/V form: K and V codes [M, kv_width]
  long long ldkv;
  float* kv_scale[2];          // FP8 K/V form: K and V scales [M][lds], one per head
  long long lds;
  uint8_t* qout;               // block-scaled form: codes [M, n_out] (FP8) or [M, n_out / 2] (4-bit), row pitch ldq
  long long ldq;
  void* qscale;                // its scales [M][qlds]: fp32 (FP8, INT4) or E4M3 bytes (NVFP4)
  long long qlds;
  const float* smooth;         // its optional inverse smoothing factors [n_out]
  int qfmt;                    // QF_FP8_1X128, QF_INT4_G32 or QF_NVFP4_G16
  // the deferred-scale chain (out[0] = H2 or Y, out[1] = H1 or null, both with row pitch ldo)
  const __nv_bfloat16* resid;  // step 1: Z [M, n_out], row pitch ldz
  long long ldz;
  const __nv_bfloat16* gamma;  // step 1: gamma [n_out]
  float* partials;             // [n_partials][M] sums of h1^2 per 256 columns: step 1 adds, step 2 reads
  int n_partials, n_norm;      // step 2: entries per row and the normalised width
  float eps;
  const int* positions;        // QKV: token positions [M], or null for m % seq_len
  int seq_len;
  double log2_theta;
  int* status;
  unsigned long long timeout_ns;
};

constexpr int kLdSmallBytes = 1024;  // RoPE frequencies (128 floats), per-token maxima (32), flags
// S stages of 20 KB: 10 with one CTA per SM, 5 with two (for more clusters than SMs hold singly)
__host__ __device__ constexpr int ld_smem_bytes(int S) {
  return S * kLdStageBytes + kLdSmallBytes + 1024 /*bars*/ + 1024 /*align*/;
}
constexpr int kLdStagesPair = 5;
__host__ __device__ constexpr int ld_pow2_at_least(int x) { return x <= 1 ? 1 : 2 * ld_pow2_at_least((x + 1) / 2); }

// C CTAs per cluster (1 to 8) split K; the tile's groups of 8 output features are shared out
// as evenly as 8-feature groups allow (rank r finishes groups [r G / C, (r + 1) G / C)), except in
// the FP8 K/V form, where rank r finishes tokens [32 r / C, 32 (r + 1) / C) over every group.
template <int C, int KIND, int S>
__global__ void __launch_bounds__(kThreads, S == kLdStages ? 1 : 2)
    linear_decode_kernel(const __grid_constant__ LinearDecodeParams p) {
  static_assert(C >= 1 && C <= 8, "cluster size");
  static_assert(S == kLdStages || S == kLdStagesPair, "stages");
  constexpr bool kSwiglu = KIND == LD_SWIGLU;
  constexpr int kOut = kSwiglu ? 64 : 128;    // output features per tile
  constexpr int kG = kOut / 8;                // groups of 8 features per tile
  constexpr int kGmax = (kG + C - 1) / C;     // groups per CTA, at most
  constexpr int kP2 = ld_pow2_at_least(kGmax);  // lanes per token: a power of two for the butterflies
  // FP8 K/V form: (token, group) items of this rank's tokens, a token's 16 groups in 16 lanes
  constexpr bool kTokSplit = KIND == LD_QKV_FP8KV || KIND == LD_QUANT || KIND == LD_RESGAMMA;
  constexpr int kTokMax = (32 + C - 1) / C;   // tokens per CTA, at most
  constexpr int kItems = kTokSplit ? kTokMax * kG : 32 * kP2;  // (token, group slot) items
  constexpr int kIpt = (kItems + 127) / 128;  // items per epilogue thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_mem = smem;
  float* P = reinterpret_cast<float*>(stage_mem);  // [32 tokens][128 W rows] after the stream
  uint8_t* small = smem + S * kLdStageBytes;
  float* inv_freq = reinterpret_cast<float*>(small);            // QKV: [64] hi, [64] lo
  volatile int* flags = reinterpret_cast<volatile int*>(inv_freq + 160);  // [0] this CTA ok
  uint64_t* bars = reinterpret_cast<uint64_t*>(small + kLdSmallBytes);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + S;
  uint64_t* tfull_bar = bars + 2 * S;
  uint64_t* drain_bar = tfull_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wctx{abort_flag, p.status, p.timeout_ns};
  const uint32_t rank = C > 1 ? cluster_ctarank() : 0u;
  const int f = p.f0 + static_cast<int>(blockIdx.x) / C;  // W-row tile of this cluster
  const int kb0 = static_cast<int>(rank) * p.num_kb / C;
  const int kb1 = (static_cast<int>(rank) + 1) * p.num_kb / C;
  // this CTA's groups of 8 output features in the tile: [g0, g0 + ng) (token split: all of them)
  const int g0 = kTokSplit ? 0 : static_cast<int>(rank) * kG / C;
  const int ng = kTokSplit ? kG : (static_cast<int>(rank) + 1) * kG / C - g0;
  // this CTA's tokens (token split): [tk0, tk1)
  const int tk0 = kTokSplit ? static_cast<int>(rank) * 32 / C : 0;
  const int tk1 = kTokSplit ? (static_cast<int>(rank) + 1) * 32 / C : 32;
  // first W row of the tile (SwiGLU: of its gate half, and of its up half in W_up)
  const int wrow = f * (kSwiglu ? 64 : 128);

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    flags[0] = 1;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_w);
    tma_prefetch_desc(&p.map_x);
    if (kSwiglu) tma_prefetch_desc(&p.map_w2);
    // the weights do not depend on earlier work on the stream: first tiles into L2 before the wait
    for (int kb = kb0; kb < kb1 && kb < kb0 + kLdL2PrefetchUnits; ++kb) {
      tma_prefetch_l2_2d(&p.map_w, kb * kBK, wrow);
      if (kSwiglu) tma_prefetch_l2_2d(&p.map_w2, kb * kBK, wrow);
    }
  }
  constexpr bool kQkv = KIND == LD_QKV_ROPE || KIND == LD_QKV_FP8KV;
  if (kQkv && threadIdx.x >= 64 && threadIdx.x < 128) {
    const int i = threadIdx.x - 64;  // pair index within the head
    const double fr = exp2(-(2.0 * i / 128.0) * p.log2_theta);  // theta^(-2i/128)
    const float hi = static_cast<float>(fr);
    inv_freq[i] = hi;
    inv_freq[64 + i] = static_cast<float>(fr - static_cast<double>(hi));
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // X, the biases and the positions may be written by the preceding kernel

  // this thread's items: token t = item / kP2, output features 8 (g0 + gl) .. + 7 of the tile for slot
  // gl = item % kP2 < ng; token split: token tk0 + item / kG, features 8 (item % kG) .. + 7
  const int ti = static_cast<int>(threadIdx.x) - 64;  // epilogue thread 0..127, or negative
  auto item_tg = [&](int item, int& t, int& gl) {
    if (kTokSplit) {
      t = tk0 + item / kG;
      gl = item % kG;
    } else {
      t = item / kP2;
      gl = item % kP2;
    }
  };
  // item < kItems, the token inside this CTA's range, a feature group inside its share; the same
  // across a warp's lanes of one token (kG and kP2 are powers of two dividing 32)
  auto item_has = [&](int item, int t, int gl) { return item < kItems && t < tk1 && gl < ng; };
  float bs[kIpt][8], b2s[kIpt][8];  // bias (and SwiGLU's up bias, or the chain's residual)
  float gs[kIpt][8], rr[kIpt];      // the chain: gamma (step 1), the token's row scale (step 2)

  // ---------------------------------------------------------------- phase 1: stream W, partial tile
  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
      bool ok = true;
      const uint64_t w_policy = l2_policy_evict_first();
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wctx, W_PRODUCER_EMPTY)) { ok = false; break; }
        uint8_t* a_dst = stage_mem + stage * kLdStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kLdStageBytes);
        if (kSwiglu) {
          // gate rows 0..63, up rows 64..127 of the A tile (8 KB each in the 128-byte swizzle)
          tma_load_2d_hint(&p.map_w, &full_bar[stage], a_dst, kb * kBK, wrow, w_policy);
          tma_load_2d_hint(&p.map_w2, &full_bar[stage], a_dst + 64 * kBK * 2, kb * kBK, wrow, w_policy);
        } else {
          tma_load_2d_hint(&p.map_w, &full_bar[stage], a_dst, kb * kBK, wrow, w_policy);
        }
        tma_load_2d(&p.map_x, &full_bar[stage], a_dst + kLdABytes, kb * kBK, 0);
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) {
        flags[0] = 0;
        for (int s = 0; s < S; ++s)
          if (issued_mask & (1u << s)) mbar_wait_quiet(&full_bar[s], (issued_phase >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kLdTokens);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, wctx, W_MMA_FULL)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stage_mem + stage * kLdStageBytes);
        const uint64_t adesc = sdesc_k_sw128(a_addr);
        const uint64_t bdesc = sdesc_k_sw128(a_addr + kLdABytes);
#pragma unroll
        for (int k = 0; k < kBK / kUmmaK; ++k)
          mma_bf16(tmem_base, adesc + 2 * k, bdesc + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        mma_commit(&empty_bar[stage]);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (ok) mma_commit(tfull_bar);
      else flags[0] = 0;
      mma_commit(drain_bar);
      mbar_wait_quiet(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // The biases of this thread's items, loaded while the weights stream.
#pragma unroll
    for (int it = 0; it < kIpt; ++it) {
      const int item = ti + 128 * it;
      int t, gl;
      item_tg(item, t, gl);
      const bool in = item_has(item, t, gl);
      const int j = (g0 + (gl < ng ? gl : 0)) * 8;  // feature within the tile
      const int n = (kSwiglu ? f * 64 : f * 128) + j;        // W row (SwiGLU: output feature)
      const int lim = kQkv ? p.num_f * 128 : p.n_out;  // entries of the bias vectors
      const int bl = in && p.bias ? lim : 0, b2l = in && p.bias2 ? lim : 0;
      load_bf16x4(p.bias, n, bl, *reinterpret_cast<float(*)[4]>(bs[it]));
      load_bf16x4(p.bias, n + 4, bl, *reinterpret_cast<float(*)[4]>(bs[it] + 4));
      if (kSwiglu) {
        load_bf16x4(p.bias2, n, b2l, *reinterpret_cast<float(*)[4]>(b2s[it]));
        load_bf16x4(p.bias2, n + 4, b2l, *reinterpret_cast<float(*)[4]>(b2s[it] + 4));
      }
      if constexpr (KIND == LD_RESGAMMA) {  // the residual row and gamma of this item
        const bool zin = in && t < p.M;
        const __nv_bfloat16* zr = p.resid + static_cast<size_t>(zin ? t : 0) * p.ldz;
        load_bf16x4(zr, n, zin ? p.n_out : 0, *reinterpret_cast<float(*)[4]>(b2s[it]));
        load_bf16x4(zr, n + 4, zin ? p.n_out : 0, *reinterpret_cast<float(*)[4]>(b2s[it] + 4));
        load_bf16x4(p.gamma, n, in ? p.n_out : 0, *reinterpret_cast<float(*)[4]>(gs[it]));
        load_bf16x4(p.gamma, n + 4, in ? p.n_out : 0, *reinterpret_cast<float(*)[4]>(gs[it] + 4));
      }
      if constexpr (KIND == LD_ROWSCALE) {  // r of the item's token, from the step-1 sums (in order)
        float ssum = 0.f;
        if (in && t < p.M)
          for (int q = 0; q < p.n_partials; ++q) ssum += __ldg(p.partials + static_cast<size_t>(q) * p.M + t);
        rr[it] = rsqrtf(ssum / static_cast<float>(p.n_norm) + p.eps);
      }
    }
    // TMEM lane quarter q = W rows 32 q .. 32 q + 31 of the tile; each thread one row, 32 tokens.
    const int q = warp & 3;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar, 0, wctx, W_EPI_TMEM_FULL));
    if (ok) {
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16), acc);
      tmem_ld_wait();
      const int r = q * 32 + lane;
#pragma unroll
      for (int t = 0; t < 32; ++t) P[t * 128 + r] = __uint_as_float(acc[t]);
    } else if (lane == 0) {
      flags[0] = 0;
    }
  }
  // Cluster barrier A: every CTA of the cluster has its partial tile in P.
  __syncwarp();
  if (C > 1) cluster_sync_all();
  else __syncthreads();

  // ---------------------------------------------------------------- phase 2: reduce, epilogue, store
  int fv[C];
  if constexpr (C > 1) {
#pragma unroll
    for (int j = 0; j < C; ++j)
      fv[j] = ld_dsmem_s32(mapa_shared(smem_u32(const_cast<int*>(flags)), static_cast<uint32_t>(j)));
  } else {
    fv[0] = flags[0];
  }
  // QKV: section (0 Q, 1 K, 2 V) of the tile (a tile is one head of one section) and its first column
  const int sec = !kQkv ? 0 : (f * 128 < p.n_out ? 0 : (f * 128 < p.n_out + p.kv_width ? 1 : 2));
  const int col_base = !kQkv ? f * kOut : f * 128 - (sec == 0 ? 0 : (sec == 1 ? p.n_out : p.n_out + p.kv_width));
  const int width = !kQkv || sec == 0 ? p.n_out : p.kv_width;
  const bool fp8 = KIND == LD_QKV_FP8KV && sec > 0;  // the same for every CTA of the cluster
  // The C partials of item `it` (token t, features j..j+7 of the tile) from every rank's P, in
  // flight at once (SwiGLU: the gate rows j.., and the up rows 64 + j..).
  constexpr int kCu = kSwiglu ? C : 1;
  float4 xa[kIpt][C], xb[kIpt][C], ya[kIpt][kCu], yb[kIpt][kCu];
  auto load_item = [&](int it, int t, int j) {
    const uint32_t la = smem_u32(P + t * 128 + j);
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const uint32_t ra = C > 1 ? mapa_shared(la, static_cast<uint32_t>(c)) : la;
      xa[it][c] = C > 1 ? ld_dsmem_f4(ra) : *reinterpret_cast<const float4*>(P + t * 128 + j);
      xb[it][c] = C > 1 ? ld_dsmem_f4(ra + 16) : *reinterpret_cast<const float4*>(P + t * 128 + j + 4);
      if constexpr (kSwiglu) {
        ya[it][c] = C > 1 ? ld_dsmem_f4(ra + 256) : *reinterpret_cast<const float4*>(P + t * 128 + 64 + j);
        yb[it][c] = C > 1 ? ld_dsmem_f4(ra + 272) : *reinterpret_cast<const float4*>(P + t * 128 + 68 + j);
      }
    }
  };
  // FP8 K/V form: cluster barrier B is split.  Every item's partials are loaded first; the
  // barrier's first half then says this CTA has read everything it needs from its peers' P (the
  // loads have returned before the release), and its second half, before the CTA leaves, keeps
  // its own P alive until every peer has read it, with the epilogue and the stores in between.
  // The other kinds load their first item's partials with the flags and each later item's just
  // before its epilogue, and keep the whole barrier at the end.  (Measured, 20 back-to-back calls, 5 alternating runs on one box: FP8 K/V
  // 32 x 6144 x 4096 12.06 us against 12.60 with the feature split and one barrier more; QKV
  // 32 x 12288 x 4096 is slower split, 21.0 against 19.4, and 19.3 against 19.0 with the loads
  // of both its items ahead of the epilogue.)
  constexpr bool kSplitB = kTokSplit && C > 1;
  // The partials are loaded together with the flags, not after them: reading a peer's P is safe
  // whatever its flag says (the values are used only when every flag is set), and the tail loses
  // one distributed-shared-memory round trip (measured, 3 alternating runs on one box: FP8 K/V
  // 32 x 6144 x 4096 interleaved 12.88 -> 12.73 us, one launch 20.15 -> 19.80 us, back to back
  // unchanged at 12.2 us; QKV 32 x 12288 x 4096 back to back 18.40 -> 18.26 us).
  if constexpr (kSplitB) {
    if (ti >= 0) {
#pragma unroll
      for (int it = 0; it < kIpt; ++it) {
        const int item = ti + 128 * it;
        int t, gl;
        item_tg(item, t, gl);
        if (item_has(item, t, gl)) load_item(it, t, (g0 + gl) * 8);
      }
    }
    __syncwarp();
    cluster_arrive_release();
  } else if (ti >= 0) {
    int t, gl;
    item_tg(ti, t, gl);
    if (item_has(ti, t, gl)) load_item(0, t, (g0 + gl) * 8);  // the first item's; the others in the loop
  }
  int all = 1;
#pragma unroll
  for (int j = 0; j < C; ++j) all &= fv[j] != 0 ? 1 : 0;
  const bool ok = all != 0;

  // Sums in rank order, epilogue, stores.
  float y[kIpt][8];
  float h1v[kIpt][8];  // the chain's step 1: h1 itself
  if (ti >= 0) {
#pragma unroll
    for (int it = 0; it < kIpt; ++it) {
      const int item = ti + 128 * it;
      int t, gl;
      item_tg(item, t, gl);
      const bool has = item_has(item, t, gl);
      const int j = (g0 + (gl < ng ? gl : 0)) * 8;  // first output feature within the tile
#pragma unroll
      for (int e = 0; e < 8; ++e) y[it][e] = h1v[it][e] = 0.f;
      if (has && ok) {
        if constexpr (!kSplitB) {
          if (it > 0) load_item(it, t, j);
        }
        float s[8], s2[8];
        float4 a = xa[it][0], b = xb[it][0], u = make_float4(0.f, 0.f, 0.f, 0.f), v = u;
        if constexpr (kSwiglu) {
          u = ya[it][0];
          v = yb[it][0];
        }
#pragma unroll
        for (int c = 1; c < C; ++c) {
          a.x += xa[it][c].x; a.y += xa[it][c].y; a.z += xa[it][c].z; a.w += xa[it][c].w;
          b.x += xb[it][c].x; b.y += xb[it][c].y; b.z += xb[it][c].z; b.w += xb[it][c].w;
          if constexpr (kSwiglu) {
            u.x += ya[it][c].x; u.y += ya[it][c].y; u.z += ya[it][c].z; u.w += ya[it][c].w;
            v.x += yb[it][c].x; v.y += yb[it][c].y; v.z += yb[it][c].z; v.w += yb[it][c].w;
          }
        }
        s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w; s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
        s2[0] = u.x; s2[1] = u.y; s2[2] = u.z; s2[3] = u.w; s2[4] = v.x; s2[5] = v.y; s2[6] = v.z; s2[7] = v.w;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float h = s[e] + bs[it][e];
          if (KIND == LD_GELU_TANH) y[it][e] = gelu_tanh_f(h);
          else if (KIND == LD_GELU_ERF) y[it][e] = gelu_erf_f(h);
          else if (KIND == LD_SWIGLU) y[it][e] = silu_f(h) * (s2[e] + b2s[it][e]);
          else if (KIND == LD_ROWSCALE) y[it][e] = fmaf(rr[it], s[e], bs[it][e]);  // r (H2 W1^T) + b1
          else if (KIND == LD_RESGAMMA) {
            h1v[it][e] = s[e] + (bs[it][e] + b2s[it][e]);  // h1 = X W^T + (b + z), as the GEMM epilogue
            y[it][e] = gs[it][e] * h1v[it][e];            // h2 = gamma (.) h1 feeds step 2 unscaled
          }
          else y[it][e] = h;
        }
        if (kQkv && sec < 2) {
          // adjacent pairs (2i, 2i + 1) of the head: i = (j + e) / 2
          const float pos = static_cast<float>(p.positions != nullptr ? (t < p.M ? p.positions[t] : 0)
                                                                       : t % p.seq_len);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int i = (j + e) >> 1;
            float sn, cs;
            rope_sincos(pos, inv_freq[i], inv_freq[64 + i], sn, cs);
            const float x0 = y[it][e], x1 = y[it][e + 1];
            y[it][e] = x0 * cs - x1 * sn;
            y[it][e + 1] = x0 * sn + x1 * cs;
          }
        }
      }
      if constexpr (KIND == LD_RESGAMMA) {
        // the tile's sum of h1^2 for token t: this item's 8 values, then a butterfly over the token's
        // 16 lanes (lanes without an item hold zeros); the two 128-feature tiles of a 256-column entry
        // both add to it, and the host has zeroed it, so 0 + a + b gives the same bits in either order
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(h1v[it][e], h1v[it][e], ss);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const int col = col_base + j;
        if (has && ok && t < p.M) {
          if (gl == 0) atomicAdd(p.partials + static_cast<size_t>(f >> 1) * p.M + t, ss);
          if (p.out[1] != nullptr && col < width) {  // h1 itself, the residual stream
            __nv_bfloat16* dst = p.out[1] + static_cast<size_t>(t) * p.ldo + col;
            if (col + 8 <= width) {  // 16-byte aligned: ldo % 8 == 0, col % 8 == 0
              uint4 w;
              w.x = pack_bf16x2(h1v[it][0], h1v[it][1]);
              w.y = pack_bf16x2(h1v[it][2], h1v[it][3]);
              w.z = pack_bf16x2(h1v[it][4], h1v[it][5]);
              w.w = pack_bf16x2(h1v[it][6], h1v[it][7]);
              *reinterpret_cast<uint4*>(dst) = w;
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (col + e < width) dst[e] = __float2bfloat16_rn(h1v[it][e]);
            }
          }
        }
      }
      if constexpr (KIND == LD_QUANT) {
        // Block-scaled write-back ("GEMM Epilogue 完全拆解", §仿射量化与尾声的五步): y times the optional
        // inverse smoothing factor (step 3), then per block of 128 (FP8), 32 (INT4) or 16 (NVFP4)
        // columns the maximum, the scale and the codes, with the arithmetic of the GEMM kernel's
        // epilogue.  A token's 16 groups of 8 features sit in 16 consecutive lanes, so a block's
        // maximum is a butterfly over its 16, 4 or 2 lanes (lanes without an item hold zeros).
        const int col = col_base + j;
        if (p.smooth != nullptr) {
          float sm[8];
          if (col + 8 <= width) {  // 32-byte aligned: smooth is 16-byte aligned, col % 8 == 0
            const float4 s0 = *reinterpret_cast<const float4*>(p.smooth + col);
            const float4 s1 = *reinterpret_cast<const float4*>(p.smooth + col + 4);
            sm[0] = s0.x; sm[1] = s0.y; sm[2] = s0.z; sm[3] = s0.w;
            sm[4] = s1.x; sm[5] = s1.y; sm[6] = s1.z; sm[7] = s1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) sm[e] = col + e < width ? p.smooth[col + e] : 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) y[it][e] *= sm[e];
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[it][e]));
        const int lanes = p.qfmt == QF_FP8_1X128 ? 16 : (p.qfmt == QF_INT4_G32 ? 4 : 2);  // the same in every lane
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
          if (o < lanes) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const bool wr = has && ok && t < p.M && col < width;
        uint8_t* qrow = p.qout + static_cast<size_t>(wr ? t : 0) * p.ldq;
        if (p.qfmt == QF_FP8_1X128) {
          const float qs = amax > 0.f ? 448.f / amax : 0.f;
          uint32_t w[2];
#pragma unroll
          for (int k = 0; k < 2; ++k)  // + 0: a zero block codes as +0
            w[k] = f32x2_to_e4m3x2(fmaf(y[it][4 * k], qs, 0.f), fmaf(y[it][4 * k + 1], qs, 0.f)) |
                   (f32x2_to_e4m3x2(fmaf(y[it][4 * k + 2], qs, 0.f), fmaf(y[it][4 * k + 3], qs, 0.f)) << 16);
          if (wr) {
            if (gl == 0) static_cast<float*>(p.qscale)[static_cast<size_t>(t) * p.qlds + col / 128] = amax * (1.f / 448.f);
            if (col + 8 <= width) {  // 8-byte aligned: ldq % 16 == 0, col % 8 == 0
              *reinterpret_cast<uint2*>(qrow + col) = make_uint2(w[0], w[1]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (col + e < width) qrow[col + e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
            }
          }
        } else {
          uint32_t word = 0, sc = 0;
          if (p.qfmt == QF_INT4_G32) {
            const float inv = amax > 0.f ? 7.f / amax : 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              int qv = __float2int_rn(y[it][e] * inv);  // round half to even
              qv = max(-7, min(7, qv));
              word |= (static_cast<uint32_t>(qv) & 15u) << (4 * e);
            }
          } else {
            const float s = round_to_e4m3(amax * (1.f / 6.f), sc);
            const float inv = s > 0.f ? 1.f / s : 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e)  // + 0 as above
              word |= f32x2_to_e2m1x2(fmaf(y[it][2 * e], inv, 0.f), fmaf(y[it][2 * e + 1], inv, 0.f)) << (8 * e);
          }
          if (wr) {
            if (p.qfmt == QF_INT4_G32) {
              if ((gl & 3) == 0) static_cast<float*>(p.qscale)[static_cast<size_t>(t) * p.qlds + col / 32] = amax * (1.f / 7.f);
            } else if ((gl & 1) == 0) {
              static_cast<uint8_t*>(p.qscale)[static_cast<size_t>(t) * p.qlds + col / 16] = static_cast<uint8_t>(sc);
            }
            uint8_t* dst = qrow + col / 2;  // two codes per byte, column 2i in the low nibble of byte i
            if (col + 8 <= width) {  // 4-byte aligned: ldq % 16 == 0, col % 8 == 0
              *reinterpret_cast<uint32_t*>(dst) = word;
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (col + 2 * i < width) dst[i] = static_cast<uint8_t>(word >> (8 * i));
            }
          }
        }
      }
      if (fp8) {
        // the head's max |y| of token t: a butterfly over the token's kG lanes, which hold all 128
        // features of the head (lanes without an item hold zeros); then scale and codes
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[it][e]));
#pragma unroll
        for (int o = kG / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float qs = amax > 0.f ? 448.f / amax : 0.f;
        const int col = col_base + j;
        if (has && ok && t < p.M) {
          if (gl == 0) p.kv_scale[sec - 1][static_cast<size_t>(t) * p.lds + col_base / 128] = amax * (1.f / 448.f);
          if (col < width) {
            uint32_t w[2];
#pragma unroll
            for (int k = 0; k < 2; ++k)
              w[k] = f32x2_to_e4m3x2(fmaf(y[it][4 * k], qs, 0.f), fmaf(y[it][4 * k + 1], qs, 0.f)) |
                     (f32x2_to_e4m3x2(fmaf(y[it][4 * k + 2], qs, 0.f), fmaf(y[it][4 * k + 3], qs, 0.f)) << 16);
            uint8_t* dst = p.out_kv[sec - 1] + static_cast<size_t>(t) * p.ldkv + col;
            if (col + 8 <= width) {  // 8-byte aligned: ldkv % 16 == 0, col % 8 == 0
              *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (col + e < width) dst[e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
            }
          }
        }
      }
      if (KIND != LD_QUANT && !fp8 && has && ok) {
        const int col = col_base + j;
        __nv_bfloat16* out = p.out[sec];
        if (t < p.M && col < width) {
          __nv_bfloat16* dst = out + static_cast<size_t>(t) * p.ldo + col;
          if (col + 8 <= width) {  // 16-byte aligned: ldo % 8 == 0, col % 8 == 0
            uint4 w;
            w.x = pack_bf16x2(y[it][0], y[it][1]);
            w.y = pack_bf16x2(y[it][2], y[it][3]);
            w.z = pack_bf16x2(y[it][4], y[it][5]);
            w.w = pack_bf16x2(y[it][6], y[it][7]);
            *reinterpret_cast<uint4*>(dst) = w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (col + e < width) dst[e] = __float2bfloat16_rn(y[it][e]);
          }
        }
      }
    }
  }
  // Cluster barrier B (its second half in the FP8 K/V form): every peer has read this CTA's P
  // before it leaves.
  __syncwarp();
  if (kSplitB) cluster_wait_acquire();
  else if (C > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace fl
