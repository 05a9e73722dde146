// Persistent, warp-specialised tcgen05 GEMM with the epilogue applied to the
// accumulator tile while it sits in tensor memory.
//
// The two-phase structure (mainloop produces an accumulator tile, the epilogue
// transforms it before the only write to global memory) and its overlap with
// the next tile's mainloop follow "GEMM Epilogue 完全拆解: 推理内核的最后一公里"
// (pinghaoyang.com.cn), §主循环与尾声 and §Blackwell 的张量内存.
//
// One CTA per SM, 192 threads:
//   warp 0      TMA producer: X and W tiles into a ring of shared-memory stages
//   warp 1      owns tensor memory; one thread issues tcgen05.mma into one of
//               two accumulator buffers (double-buffered TMEM)
//   warps 2..5  epilogue: tcgen05.ld -> registers -> tile function -> smem ->
//               TMA store; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31,
//               i.e. tile rows 32*(w%4)+lane, one row per thread.
// CG = 2 (the default): two CTAs on neighbouring SMs form a cluster and compute a
// 256-row tile with tcgen05.mma.cta_group::2; each loads its 128 rows of X and half
// of the W tile, the leader issues the MMAs and multicasts its commits.  CG = 1:
// one CTA per 128-row tile.  B is K-major (W stored [N, K]) or, for the dgrad
// epilogues, MN-major (W stored [K, N]).
// Tiles are walked in a static persistent order (tile = blockIdx.x / CG + i * clusters)
// with grouped rasterisation so that concurrently running CTAs share X and W
// panels in L2; the RMSNorm epilogue walks them row-major (raster groups of one row block).
#pragma once
#include "ptx.cuh"

namespace fl {

constexpr int kBM = 128;          // rows per tile (MMA M)
constexpr int kBK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kStagingBytes = 4096;  // one 32-row x 128-byte TMA store box per buffer
constexpr int kSavedBoxBytes = 2048;  // one 32-row x 32-column bf16 box of a saved activation

enum EpiKind : int {
  EPI_GELU_TANH = 0, EPI_GELU_ERF = 1, EPI_QKV_ROPE = 2, EPI_SWIGLU = 3, EPI_RMSNORM_FP8 = 4,
  EPI_RESID_GAMMA = 5,  // h1 = acc + b + z; stores h1 (optional) and h1 * gamma; per-row partial sum h1^2
  EPI_ROWSCALE = 6,     // y = r * acc + b with r = 1/sqrt(sum of the row's partials / n + eps)
  EPI_CE = 7,           // per-row online log-sum-exp state + label logit; last tile of a row block merges
  EPI_QUANT = 8,        // block-scaled quantised write-back: FP8 1x128, INT4 g32 or NVFP4 g16 + scales
  EPI_QKV_FP8KV = 9,    // QKV + RoPE, Q in bf16, K and V as E4M3 with one scale per token and kv head
  EPI_GELU_BWD_TANH = 10,  // dgrad (B = W as stored, MN-major) times GELU'(saved pre-activation), tanh form
  EPI_SWIGLU_BWD = 11,     // dgrad of the down projection -> interleaved (dg, du) pairs, double width
  EPI_GELU_BWD_ERF = 12    // as EPI_GELU_BWD_TANH with the erf form's derivative
};
enum QuantFmt : int { QF_FP8_1X128 = 0, QF_INT4_G32 = 1, QF_NVFP4_G16 = 2 };

struct alignas(128) GemmParams {
  CUtensorMap map_a;       // X [M, K] bf16, box {64, 128}
  CUtensorMap map_b;       // W [N, K] bf16, box {64, 256}; SwiGLU: W_gate, box {64, 128}
  CUtensorMap map_b2;      // SwiGLU: W_up, box {64, 128}
  CUtensorMap map_out[3];  // outputs; box {64 bf16 | 128 fp8 columns, 32 rows}; QKV: Q, K, V
  int M, N, K;             // N: logical output features (QKV: 3*d_model, SwiGLU: d_ff)
  int num_m_blocks, num_n_blocks, num_k_blocks;
  int num_m_tiles, num_tiles;  // tiles of (CTAs per cluster) x 128 rows; one tile per cluster
  int group_m;             // m-tiles per raster group (1 = row-major tile order)
  const __nv_bfloat16* bias;
  const __nv_bfloat16* bias2;  // SwiGLU: b_up
  // QKV + RoPE
  const int* positions;
  int seq_len, head_dim, d_model;
  double log2_theta;
  // residual + RMSNorm + FP8
  const __nv_bfloat16* resid;
  long long ldz;
  const __nv_bfloat16* gamma;
  float eps;
  float* row_scale;
  float2* partials;        // [num_m_blocks][num_n_blocks][128] (sum h^2, max |h*gamma|)
  float* rms_partials;     // [ceil(n/256)][M] per-row partial sums of squares (GEMM -> RMSNorm -> GEMM chain)
  int n_partials, n_norm;
  int store_h1;            // RESID_GAMMA and RMSNORM_FP8: also store h (bf16) through map_out[1]
  // LM-head cross-entropy
  const int* labels;       // [M]; negative = ignored row
  float* loss;             // [M]
  float2* ce_partials;     // [num_n_blocks][M] (running max, sum of exp(h - max)) per tile
  float* label_logit;      // [M]
  int store_logits;
  // block-scaled quantised write-back
  int quant_fmt;
  void* qscale;            // fp32 [M][lds] (FP8, INT4) or E4M3 bytes [M][lds] (NVFP4)
  long long lds;
  const float* smooth;     // nullable fp32 [N]: inverse smoothing factor per output column
  // QKV with an FP8 K/V cache: K/V section width (n_kv_heads * head_dim) and their scales [M][lds]
  int kv_width;
  float* kscale;
  float* vscale;
  // backward epilogues: saved activations [M][ld_saved] (GELU: the pre-activation H;
  // SwiGLU: the gate G and up U)
  const __nv_bfloat16* saved0;
  const __nv_bfloat16* saved1;
  long long ld_saved;
  CUtensorMap map_saved[2];  // the same, box {32 columns, 32 rows}, 64-byte swizzle
  unsigned* counters;      // [2][num_m_blocks]: arrivals, finished readers
  int* status;
  unsigned long long timeout_ns;
};

// CG = CTAs per cluster sharing one MMA: 1 (tcgen05 cta_group::1, 128-row tile per CTA) or
// 2 (cta_group::2: the pair computes a 256-row tile; each CTA loads its 128 rows of X and half
// of the W tile, so a stage is 32 KB instead of 48 KB and six stages fit).
template <int EPI, int CG>
struct EpiTraits {
  static constexpr int kMmaN = 256;                               // accumulator columns per tile
  static constexpr int kOutN = (EPI == EPI_SWIGLU) ? 128 : 256;   // output columns per tile
  static constexpr bool kFp8 = (EPI == EPI_RMSNORM_FP8);
  // B operand MN-major (W as stored [K, N], N contiguous): TMA boxes of 64 columns x kBK rows
  static constexpr bool kBMn = (EPI == EPI_GELU_BWD_TANH || EPI == EPI_GELU_BWD_ERF || EPI == EPI_SWIGLU_BWD);
  static constexpr int kBChunkBytes = 64 * kBK * 2;
  // saved activations the backward epilogues read (GELU: H; SwiGLU: G and U), staged per warp
  static constexpr int kNSaved = EPI == EPI_SWIGLU_BWD ? 2 : (kBMn ? 1 : 0);
  static constexpr int kSavedBytes = 4 * 2 * kNSaved * kSavedBoxBytes;  // 4 warps x 2 buffers
  // the backward kernels give one stage to the saved-activation buffers (measured: 5 stages run
  // the pair mainloop as fast as 6)
  static constexpr int kStages = CG == 2 ? (kBMn ? 5 : 6) : (kBMn ? 3 : 4);
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBRows = kMmaN / CG;                       // W rows this CTA loads per stage
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * kMmaN;
  static constexpr int kSmemBytes = kStages * kStageBytes + 4 * 2 * kStagingBytes + kSavedBytes +
                                    1024 /*bars*/ + 1024 /*alignment slack*/;
};

__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
  const int per_group = p.group_m * p.num_n_blocks;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gsize = min(p.num_m_tiles - first_m, p.group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

// 32 bf16 values [col0, col0+32) of a vector (bias, gamma) as fp32; zeros past n_limit.
__device__ __forceinline__ void load_vec32(const __nv_bfloat16* ptr, int col0, int n_limit, float (&v)[32]) {
  if (ptr == nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
    return;
  }
  if (col0 + 32 <= n_limit) {
    const uint4* q = reinterpret_cast<const uint4*>(ptr + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w = __ldg(q + i);
      v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
      v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
      v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
      v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (col0 + j < n_limit) ? __bfloat162float(ptr[col0 + j]) : 0.f;
  }
}

// 32 fp32 values [col0, col0+32) of a vector (the inverse smoothing factors); zeros past n_limit.
// `ptr` is 16-byte aligned and col0 a multiple of 32.
__device__ __forceinline__ void load_f32x32(const float* ptr, int col0, int n_limit, float (&v)[32]) {
  if (col0 + 32 <= n_limit) {
    const float4* q = reinterpret_cast<const float4*>(ptr + col0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 w = __ldg(q + i);
      v[4 * i + 0] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (col0 + j < n_limit) ? __ldg(ptr + col0 + j) : 0.f;
  }
}

// 32 bf16 values of one row of a matrix (the residual): row-pointer based.
__device__ __forceinline__ void load_row32(const __nv_bfloat16* row, bool row_ok, int col0, int n_limit,
                                           float (&v)[32]) {
  if (!row_ok) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
    return;
  }
  load_vec32(row, col0, n_limit, v);
}

// 32 bf16 values of a row as raw 16-byte words (zero outside the row or past n_limit), so a
// load can be issued one unit ahead of its use and unpacked later.
__device__ __forceinline__ void load_raw32(const __nv_bfloat16* row, bool row_ok, int col0, int n_limit,
                                           uint4 (&w)[4]) {
  if (row_ok && col0 + 32 <= n_limit) {
    const uint4* q = reinterpret_cast<const uint4*>(row + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = __ldg(q + i);
    return;
  }
  const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
  uint32_t e[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int c = col0 + 2 * k;
    const uint32_t lo = (row_ok && c < n_limit) ? __ldg(r + c) : 0u;
    const uint32_t hi = (row_ok && c + 1 < n_limit) ? __ldg(r + c + 1) : 0u;
    e[k] = lo | (hi << 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = make_uint4(e[4 * i], e[4 * i + 1], e[4 * i + 2], e[4 * i + 3]);
}
__device__ __forceinline__ void unpack32(const uint4 (&w)[4], float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[8 * i + 0] = bf16_lo(w[i].x); v[8 * i + 1] = bf16_hi(w[i].x);
    v[8 * i + 2] = bf16_lo(w[i].y); v[8 * i + 3] = bf16_hi(w[i].y);
    v[8 * i + 4] = bf16_lo(w[i].z); v[8 * i + 5] = bf16_hi(w[i].z);
    v[8 * i + 6] = bf16_lo(w[i].w); v[8 * i + 7] = bf16_hi(w[i].w);
  }
}

// Four bf16 values base[n .. n + 3] as floats; entries at or past `limit` read as zero.
__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16* base, int n, int limit, float (&v)[4]) {
  if (n + 4 <= limit) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(base + n));
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = n + j < limit ? __bfloat162float(base[n + j]) : 0.f;
  }
}

__device__ __forceinline__ void tmem_load32f(uint32_t taddr, bool zero, float (&v)[32]) {
  if (zero) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
    return;
  }
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// sin and cos of the RoPE angle pos * f for an integer-valued position (exact in fp32) and a
// frequency held as two floats f = hi + lo.  The product is carried exactly (FMA residual),
// reduced modulo 2 pi by Cody and Waite's method (2 pi split into two floats, one FMA per
// part) and only the reduced angle is rounded, so large positions keep the angle accurate
// to a few fp32 ulps instead of pos * 2^-24.
__device__ __forceinline__ void rope_sincos(float pos, float hi, float lo, float& sn, float& cs) {
  const float p = pos * hi;
  const float e = fmaf(pos, hi, -p);     // pos * hi - p, exactly
  const float t = fmaf(pos, lo, e);      // the small part of the angle
  const float k = rintf(p * 0.159154943091895336f);  // nearest multiple of 2 pi
  float r = fmaf(-k, 6.28318548202514648f, p);         // 2 pi rounded to fp32 ...
  r = fmaf(-k, -1.74845553146951657e-07f, r);          // ... and the remainder 2 pi - that
  sincosf(r + t, &sn, &cs);
}

__device__ __forceinline__ float gelu_tanh_f(float v) {
  // 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
  const float u = v * fmaf(0.0356774081363f, v * v, 0.7978845608028654f);
  const float hv = 0.5f * v;
  return fmaf(hv, tanh_approx(u), hv);
}
__device__ __forceinline__ float gelu_erf_f(float v) { return 0.5f * v * (1.f + erff(v * 0.70710678118654752f)); }
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }
// GELU'(h) of the tanh form: 0.5 (1 + t) + 0.5 h (1 - t^2) c (1 + 3 a h^2), t = tanh(c (h + a h^3)),
// c = sqrt(2/pi), a = 0.044715.
__device__ __forceinline__ float gelu_tanh_grad_f(float h) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  const float h2 = h * h;
  const float t = tanh_approx(c * h * fmaf(a, h2, 1.f));
  return fmaf(0.5f * h * (1.f - t * t), c * fmaf(3.f * a, h2, 1.f), 0.5f * (1.f + t));
}
// GELU'(h) of the erf form: Phi(h) + h phi(h).
__device__ __forceinline__ float gelu_erf_grad_f(float h) {
  return fmaf(h * 0.3989422804014327f, __expf(-0.5f * h * h), 0.5f * (1.f + erff(h * 0.70710678118654752f)));
}

// Writes 32 bf16 values (one row segment) into a 128B-swizzled staging row:
// `unit` (0 or 1) selects which half of the 128-byte row they fill.
__device__ __forceinline__ void stage_bf16_32(uint32_t buf, int lane, int unit, const float (&v)[32]) {
  const uint32_t row = buf + lane * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int chunk = unit * 4 + c;
    st_shared_v4(row + ((chunk ^ (lane & 7)) << 4), pack_bf16x2(v[8 * c + 0], v[8 * c + 1]),
                 pack_bf16x2(v[8 * c + 2], v[8 * c + 3]), pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                 pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
  }
}
// Writes 32 E4M3 codes (32 bytes) into a 128B-swizzled staging row; `unit` 0..3.
__device__ __forceinline__ void stage_fp8_32(uint32_t buf, int lane, int unit, const float (&v)[32]) {
  const uint32_t row = buf + lane * 128;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 16 * c + 4 * i;
      w[i] = f32x2_to_e4m3x2(v[j], v[j + 1]) | (f32x2_to_e4m3x2(v[j + 2], v[j + 3]) << 16);
    }
    const int chunk = unit * 2 + c;
    st_shared_v4(row + ((chunk ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
  }
}

// Saved activations of the backward epilogues, one 32-column unit at a time: the warp's lane 0
// TMA-loads the 32 x 32 box of each saved tensor for its 32 rows into the warp's double buffer
// (64-byte swizzle; L2 evict-first, since each saved value is read once and should not push the
// operand panels out of L2), and every thread reads its own row back from shared memory,
// conflict-free.  Ragged edges come from the TMA zero fill.  Units are numbered across the warp's
// tiles, and the loads run two units ahead.  (Measured against per-thread 16-byte row loads from
// global memory: as fast without the hint, about 1 % faster with it.)
template <int NS>
struct SavedRing {
  uint32_t base;      // this warp's buffers [2][NS] x kSavedBoxBytes (shared-memory address)
  uint64_t* bar;      // this warp's two barriers
  uint32_t issued;    // units whose loads were issued
  uint32_t consumed;  // units read
  __device__ __forceinline__ uint32_t box(uint32_t unit, int t) const {
    return base + ((unit & 1u) * NS + t) * kSavedBoxBytes;
  }
  // lane 0: the boxes of unit `issued`, at column x and row y of every saved tensor.  The
  // buffer was last read two units ago; the caller has passed a warp barrier since.
  __device__ __forceinline__ void issue(const CUtensorMap* maps, int x, int y) {
    const uint32_t b = issued & 1u;
    fence_async_smem();  // the warp's reads of this buffer come before the copy's writes
    mbar_arrive_expect_tx(&bar[b], NS * kSavedBoxBytes);
    const uint64_t pol = l2_policy_evict_first();
#pragma unroll
    for (int t = 0; t < NS; ++t) tma_load_2d_to_hint(&maps[t], &bar[b], box(issued, t), x, y, pol);
    ++issued;
  }
  // Waits for unit `consumed`; false if the wait ran out.
  __device__ __forceinline__ bool wait(const WaitCtx& w) {
    return mbar_wait(&bar[consumed & 1u], (consumed >> 1) & 1u, w, W_EPI_SAVED);
  }
  // This thread's row (32 bf16) of saved tensor t in unit `consumed`.
  __device__ __forceinline__ void row(int t, int lane, uint4 (&q)[4]) const {
    const uint32_t r = box(consumed, t) + lane * 64;  // 64-byte rows; 16-byte chunk c at c ^ ((lane >> 1) & 3)
#pragma unroll
    for (int c = 0; c < 4; ++c) q[c] = ld_shared_v4(r + ((c ^ ((lane >> 1) & 3)) << 4));
  }
  // Lets every copy still in flight land (teardown after an error: nothing may write into
  // shared memory once the CTA has left).
  __device__ __forceinline__ void drain(uint64_t timeout_ns) {
    for (; consumed < issued; ++consumed) mbar_wait_quiet(&bar[consumed & 1u], (consumed >> 1) & 1u, timeout_ns);
  }
};

// Per-warp double-buffered TMA store of 32-row x 128-byte boxes.
struct StoreRing {
  uint32_t base;  // this warp's two staging buffers (shared-memory address)
  int count;
  // Returns a staging buffer whose previous store has finished reading it.
  __device__ __forceinline__ uint32_t acquire(int lane) {
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    return base + (count & 1) * kStagingBytes;
  }
  // Both staging buffers at once (every earlier store has finished reading them); the
  // caller commits the first, then the second.
  __device__ __forceinline__ void acquire_pair(int lane, uint32_t& first, uint32_t& second) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    first = base + (count & 1) * kStagingBytes;
    second = base + ((count + 1) & 1) * kStagingBytes;
  }
  // Publishes the staged box to the async proxy and stores it at (x, y).
  __device__ __forceinline__ void commit(const CUtensorMap* map, uint32_t buf, int lane, int x, int y) {
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      // outputs are written once: evict-first keeps the operand panels in L2
      tma_store_2d_u32_hint(map, buf, x, y, l2_policy_evict_first());
      bulk_commit();
    }
    ++count;
  }
};

// Bounded spin until all `need` tiles of a row block have published their
// partial row statistics.  Returns false on timeout or if another CTA has
// already recorded a failure (then the exchange can never complete).
__device__ __forceinline__ bool wait_row_block(const GemmParams& p, int mb, unsigned need) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_u32(p.counters + mb) == need) return true;  // exact count: reset to 0 after use
    if ((i & 15u) == 15u) {
      if (*reinterpret_cast<volatile int*>(p.status + ST_CODE) != 0) return false;
      if (global_timer_ns() - t0 > p.timeout_ns) {
        record_failure(p.status, W_ROW_EXCHANGE, mb);
        return false;
      }
    }
    __nanosleep(100);
  }
}

template <int EPI, int CG>
__global__ void __launch_bounds__(kThreads, 1) fused_gemm_kernel(const __grid_constant__ GemmParams p) {
  using T = EpiTraits<EPI, CG>;
  constexpr int kStages = T::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_mem = smem;
  uint8_t* staging = smem + kStages * T::kStageBytes;
  uint8_t* saved_mem = staging + 4 * 2 * kStagingBytes;  // backward epilogues: [4 warps][2][kNSaved] boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(saved_mem + T::kSavedBytes);
  uint64_t* full_bar = bars;                 // [kStages]  TMA landed
  uint64_t* empty_bar = bars + kStages;      // [kStages]  MMAs reading the stage finished
  uint64_t* tfull_bar = bars + 2 * kStages;  // [2]        accumulator buffer complete
  uint64_t* tempty_bar = tfull_bar + 2;      // [2]        epilogue done reading the buffer
  uint64_t* drain_bar = tempty_bar + 2;      // [1]        all MMAs complete (teardown)
  uint64_t* saved_bar = drain_bar + 1;       // [4][2]     saved-activation boxes landed (backward)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(saved_bar + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_stop = reinterpret_cast<volatile int*>(tmem_slot + 2);  // written by the epilogue leader only
  volatile int* ce_last = reinterpret_cast<volatile int*>(tmem_slot + 3);   // idem: this tile merges its row block
  // QKV only: RoPE frequency of pair i as two floats, inv_freq[i] + inv_freq[64 + i]
  float* inv_freq = reinterpret_cast<float*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wctx{abort_flag, p.status, p.timeout_ns};
  // Cluster bookkeeping: rank 0 of a pair (the leader) issues the MMAs for both CTAs.
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool mma_cta = rank == 0;
  const int tile0 = static_cast<int>(blockIdx.x) / CG;
  const int tstride = static_cast<int>(gridDim.x) / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 4 * CG);  // one arrival per epilogue warp of every CTA in the cluster
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&saved_bar[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0 && p.num_k_blocks > 0) {
    tma_prefetch_desc(&p.map_a);
    tma_prefetch_desc(&p.map_b);
    if (EPI == EPI_SWIGLU) tma_prefetch_desc(&p.map_b2);
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_slot, T::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, T::kTmemCols);
      tmem_relinquish();
    }
  }
  if ((EPI == EPI_QKV_ROPE || EPI == EPI_QKV_FP8KV) && threadIdx.x >= 64 && threadIdx.x < 128) {
    const int i = threadIdx.x - 64;  // pair index within a head (head_dim 128 -> 64 pairs)
    const double f = exp2(-(2.0 * i / p.head_dim) * p.log2_theta);  // theta^(-2i/head_dim)
    const float hi = static_cast<float>(f);
    inv_freq[i] = hi;
    inv_freq[64 + i] = static_cast<float>(f - static_cast<double>(hi));
  }
  tc_fence_before();
  if constexpr (CG == 2) {
    cluster_sync_all();  // both CTAs' barriers and tensor memory exist before any cross-CTA use
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;  // per stage: ever issued / parity of the last issue
      bool ok = true;
      for (int t = tile0; t < p.num_tiles && ok; t += tstride) {
        int mt, nb;
        tile_coords(p, t, mt, nb);
        const int mb = mt * CG + static_cast<int>(rank);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          const bool got = CG == 2 ? mbar_wait_cl(&empty_bar[stage], phase ^ 1u, wctx, W_PRODUCER_EMPTY)
                                   : mbar_wait(&empty_bar[stage], phase ^ 1u, wctx, W_PRODUCER_EMPTY);
          if (!got) { ok = false; break; }
          uint8_t* a_dst = stage_mem + stage * T::kStageBytes;
          uint8_t* b_dst = a_dst + T::kABytes;
          if constexpr (CG == 2) {
            // Both CTAs' copies complete on the leader's barrier, which expects the bytes of the pair.
            if (mma_cta) mbar_arrive_expect_tx(&full_bar[stage], 2 * T::kStageBytes);
            const uint32_t full_cl = mapa_shared(smem_u32(&full_bar[stage]), 0);
            tma_load_2d_pair(&p.map_a, full_cl, a_dst, kb * kBK, mb * kBM);
            if (EPI == EPI_SWIGLU) {
              // the leader holds the 128 gate rows, the peer the 128 up rows of the same features
              tma_load_2d_pair(rank == 0 ? &p.map_b : &p.map_b2, full_cl, b_dst, kb * kBK, nb * 128);
            } else if (T::kBMn) {
              // this CTA's 128 columns of the W tile as two 64-column chunks, rows = this K block
              for (int c = 0; c < 2; ++c)
                tma_load_2d_pair(&p.map_b, full_cl, b_dst + c * T::kBChunkBytes,
                                 nb * T::kMmaN + static_cast<int>(rank) * 128 + c * 64, kb * kBK);
            } else {
              tma_load_2d_pair(&p.map_b, full_cl, b_dst, kb * kBK, nb * T::kMmaN + static_cast<int>(rank) * 128);
            }
          } else {
            mbar_arrive_expect_tx(&full_bar[stage], T::kStageBytes);
            tma_load_2d(&p.map_a, &full_bar[stage], a_dst, kb * kBK, mb * kBM);
            if (EPI == EPI_SWIGLU) {
              // gate rows and up rows of the same 128 output features, stacked in one B stage
              tma_load_2d(&p.map_b, &full_bar[stage], b_dst, kb * kBK, nb * 128);
              tma_load_2d(&p.map_b2, &full_bar[stage], b_dst + 128 * kBK * 2, kb * kBK, nb * 128);
            } else if (T::kBMn) {
              for (int c = 0; c < 4; ++c)
                tma_load_2d(&p.map_b, &full_bar[stage], b_dst + c * T::kBChunkBytes, nb * T::kMmaN + c * 64,
                            kb * kBK);
            } else {
              tma_load_2d(&p.map_b, &full_bar[stage], b_dst, kb * kBK, nb * T::kMmaN);
            }
          }
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && mma_cta) {
        // Do not leave copies landing in shared memory after the CTA exits (the leader's barriers
        // also count the peer's copies; the peer waits for the leader at the final cluster barrier).
        const uint64_t deadline = global_timer_ns() + p.timeout_ns;
        for (int s = 0; s < kStages; ++s) {
          const uint64_t now = global_timer_ns();
          if (issued_mask & (1u << s))
            mbar_wait_quiet(&full_bar[s], (issued_phase >> s) & 1u, now < deadline ? deadline - now : 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && mma_cta) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM * CG, T::kMmaN, T::kBMn);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = tile0; t < p.num_tiles && ok; t += tstride, ++local) {
        const int abuf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        const bool free_acc = CG == 2 ? mbar_wait_cl(&tempty_bar[abuf], (use & 1u) ^ 1u, wctx, W_MMA_TMEM_EMPTY)
                                      : mbar_wait(&tempty_bar[abuf], (use & 1u) ^ 1u, wctx, W_MMA_TMEM_EMPTY);
        if (!free_acc) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + abuf * T::kMmaN;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          const bool got = CG == 2 ? mbar_wait_cl(&full_bar[stage], phase, wctx, W_MMA_FULL)
                                   : mbar_wait(&full_bar[stage], phase, wctx, W_MMA_FULL);
          if (!got) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_mem + stage * T::kStageBytes);
          const uint64_t adesc = sdesc_k_sw128(a_addr);
          const uint64_t bdesc = T::kBMn ? sdesc_mn_sw128(a_addr + T::kABytes, T::kBChunkBytes)
                                         : sdesc_k_sw128(a_addr + T::kABytes);
          // per K step of 16: A (K-major) +32 bytes inside its 128-byte swizzled rows; B +32 bytes
          // likewise, or, MN-major, +16 rows of 128 bytes (>> 4 in the descriptor)
          constexpr uint64_t kBStep = T::kBMn ? (16 * 128) >> 4 : 2;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            if constexpr (CG == 2) {
              mma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + kBStep * k, idesc, (kb | k) != 0 ? 1u : 0u);
            } else {
              mma_bf16(d_tmem, adesc + 2 * k, bdesc + kBStep * k, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          if constexpr (CG == 2) {
            mma_commit_pair_mc(&empty_bar[stage], 0x3);  // frees the stage in both CTAs
          } else {
            mma_commit(&empty_bar[stage]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if constexpr (CG == 2) {
          mma_commit_pair_mc(&tfull_bar[abuf], 0x3);  // both CTAs' epilogues may read their halves
        } else {
          mma_commit(&tfull_bar[abuf]);
        }
      }
      // Every MMA issued by this thread must be complete before TMEM is freed.
      if constexpr (CG == 2) {
        mma_commit_pair(drain_bar);
      } else {
        mma_commit(drain_bar);
      }
      mbar_wait_quiet(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;  // TMEM lane quarter owned by this warp
    const int row_in_tile = q * 32 + lane;
    StoreRing ring{smem_u32(staging) + (warp - 2) * 2 * kStagingBytes, 0};
    const bool k_empty = p.num_k_blocks == 0;
    int local = 0;
    // Backward epilogues: the saved activations of this warp's rows, 32-column units numbered
    // across the warp's tiles (8 per tile), loaded two units ahead by lane 0.
    SavedRing<T::kNSaved> sring{smem_u32(saved_mem) + static_cast<uint32_t>(q * 2 * T::kNSaved * kSavedBoxBytes),
                                saved_bar + 2 * q, 0u, 0u};
    bool saved_issue = true;  // lane 0: false after a failed wait (no further copies)
    auto issue_saved = [&]() {  // lane 0: the next unit, if the warp has one
      const int t = tile0 + static_cast<int>(sring.issued >> 3) * tstride;
      if (!saved_issue || t >= p.num_tiles) return;
      int smt, snb;
      tile_coords(p, t, smt, snb);
      const int smb = smt * CG + static_cast<int>(rank);
      sring.issue(p.map_saved, snb * 256 + static_cast<int>(sring.issued & 7u) * 32, smb * kBM + q * 32);
    };
    // This thread's row of the next unit of every saved tensor (zero if its wait ran out); then
    // the warp frees the buffer and lane 0 refills it two units ahead.
    auto take_saved = [&](float (&a)[32], float (&b)[32]) {
      const bool got = sring.wait(wctx);
      uint4 qa[4], qb[4];
      sring.row(0, lane, qa);
      if constexpr (T::kNSaved == 2) sring.row(1, lane, qb);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (!got) qa[i] = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (T::kNSaved == 2) {
          if (!got) qb[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      unpack32(qa, a);  // uses every loaded word: the reads are complete before the warp barrier
      if constexpr (T::kNSaved == 2) unpack32(qb, b);
      __syncwarp();
      ++sring.consumed;
      if (lane == 0) {
        if (!got) saved_issue = false;
        issue_saved();
      }
    };
    if constexpr (T::kNSaved > 0) {
      if (lane == 0) {
        issue_saved();
        issue_saved();
      }
    }
    // Releases accumulator buffer `a`: one arrival per warp on the leader's barrier.
    auto release_acc = [&](int a) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) {
          mbar_arrive_remote(mapa_shared(smem_u32(&tempty_bar[a]), 0));
        } else {
          mbar_arrive(&tempty_bar[a]);
        }
      }
    };
    for (int t = tile0; t < p.num_tiles; t += tstride, ++local) {
      int mt, nb;
      tile_coords(p, t, mt, nb);
      const int mb = mt * CG + static_cast<int>(rank);
      const int abuf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      const int m = mb * kBM + row_in_tile;
      const bool row_ok = m < p.M;
      const int y_box = mb * kBM + q * 32;
      // warp-uniform: tcgen05.ld below is a warp-collective instruction
      const bool ok = __all_sync(0xffffffffu, CG == 2 ? mbar_wait_cl(&tfull_bar[abuf], use & 1u, wctx, W_EPI_TMEM_FULL)
                                                       : mbar_wait(&tfull_bar[abuf], use & 1u, wctx, W_EPI_TMEM_FULL));
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf * T::kMmaN;

      if constexpr (EPI == EPI_GELU_TANH || EPI == EPI_GELU_ERF || EPI == EPI_QKV_ROPE || EPI == EPI_QKV_FP8KV) {
        if (!ok) break;
        constexpr bool kQkv = EPI == EPI_QKV_ROPE || EPI == EPI_QKV_FP8KV;
        int n0 = nb * T::kOutN;  // first output column of the tile
        int sec = 0, base = 0;
        float pos = 0.f;
        if constexpr (kQkv) {
          // 0 = Q, 1 = K, 2 = V (a tile never straddles two sections)
          if (n0 >= p.d_model) {
            sec = 1;
            base = p.d_model;
            if (n0 >= p.d_model + p.kv_width) {
              sec = 2;
              base += p.kv_width;
            }
          }
          n0 -= base;
          const int pi = row_ok ? (p.positions ? __ldg(p.positions + m) : m % p.seq_len) : 0;
          pos = static_cast<float>(pi);
        }
        const int n_limit = kQkv ? (sec == 0 ? p.d_model : p.kv_width) : p.N;
        const __nv_bfloat16* bias = p.bias ? p.bias + base : nullptr;
        if constexpr (kQkv) {
          if (sec == 0 || (EPI == EPI_QKV_ROPE && sec == 1)) {
            // Rotated bf16 section: the tile's two heads share their angles (same row, same pair
            // index), so each group of 16 angles is computed once and applied to both heads,
            // which are staged side by side in the two buffers of the ring.
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {
              uint32_t buf0, buf1;
              ring.acquire_pair(lane, buf0, buf1);
#pragma unroll 1
              for (int gg = 0; gg < 2; ++gg) {
                const int g = c2 * 2 + gg;  // 16-pair group within a head
                float sn[16], cs[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  rope_sincos(pos, inv_freq[g * 16 + i], inv_freq[64 + g * 16 + i], sn[i], cs[i]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  float v[32], b[32];
                  tmem_load32f(tacc + h * 128 + g * 32, k_empty, v);
                  load_vec32(bias, n0 + h * 128 + g * 32, n_limit, b);
#pragma unroll
                  for (int j = 0; j < 32; j += 2) {
                    const float x0 = v[j] + b[j], x1 = v[j + 1] + b[j + 1];
                    v[j] = x0 * cs[j >> 1] - x1 * sn[j >> 1];
                    v[j + 1] = x0 * sn[j >> 1] + x1 * cs[j >> 1];
                  }
                  stage_bf16_32(h == 0 ? buf0 : buf1, lane, gg, v);
                }
              }
              ring.commit(&p.map_out[sec], buf0, lane, n0 + c2 * 64, y_box);
              ring.commit(&p.map_out[sec], buf1, lane, n0 + 128 + c2 * 64, y_box);
            }
            release_acc(abuf);
            continue;
          }
        }
        if constexpr (EPI == EPI_QKV_FP8KV) {
          if (sec > 0) {
            // K/V cache entry in FP8 ("GEMM Epilogue 完全拆解", §一个瓦片的字节账): per head of
            // head_dim (= 128) values of this row, K is rotated, scale = max|.|/448 over the
            // head, and the codes are stored with it.  The two heads of a tile share their
            // rotation angles (same row, same pair index), so each group of 16 angles serves
            // both heads: pass 1 takes the heads' maxima, pass 2 reloads the accumulator from
            // TMEM, rotates again and quantises into one staging buffer per head.  The group
            // loops stay rolled to keep the kernel's code small.
            float amax0 = 0.f, amax1 = 0.f;
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
              float sn[16], cs[16];
              if (sec == 1) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  rope_sincos(pos, inv_freq[g * 16 + i], inv_freq[64 + g * 16 + i], sn[i], cs[i]);
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float v[32], b[32];
                tmem_load32f(tacc + h * 128 + g * 32, k_empty, v);
                load_vec32(bias, n0 + h * 128 + g * 32, n_limit, b);
                float am = 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                  float x0 = v[j] + b[j], x1 = v[j + 1] + b[j + 1];
                  if (sec == 1) {
                    const float r0 = x0 * cs[j >> 1] - x1 * sn[j >> 1];
                    x1 = x0 * sn[j >> 1] + x1 * cs[j >> 1];
                    x0 = r0;
                  }
                  am = fmaxf(am, fmaxf(fabsf(x0), fabsf(x1)));
                }
                if (h == 0) amax0 = fmaxf(amax0, am);
                else amax1 = fmaxf(amax1, am);
              }
            }
            const float qs0 = amax0 > 0.f ? 448.f / amax0 : 0.f;
            const float qs1 = amax1 > 0.f ? 448.f / amax1 : 0.f;
            if (row_ok) {
              float* sp = (sec == 1 ? p.kscale : p.vscale) + static_cast<long long>(m) * p.lds + (n0 >> 7);
              if (n0 < n_limit) sp[0] = amax0 * (1.f / 448.f);
              if (n0 + 128 < n_limit) sp[1] = amax1 * (1.f / 448.f);
            }
            uint32_t buf0, buf1;
            ring.acquire_pair(lane, buf0, buf1);
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
              float sn[16], cs[16];
              if (sec == 1) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  rope_sincos(pos, inv_freq[g * 16 + i], inv_freq[64 + g * 16 + i], sn[i], cs[i]);
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float v[32], b[32];
                tmem_load32f(tacc + h * 128 + g * 32, k_empty, v);
                load_vec32(bias, n0 + h * 128 + g * 32, n_limit, b);
                const float qs = h == 0 ? qs0 : qs1;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                  float x0 = v[j] + b[j], x1 = v[j + 1] + b[j + 1];
                  if (sec == 1) {
                    const float r0 = x0 * cs[j >> 1] - x1 * sn[j >> 1];
                    x1 = x0 * sn[j >> 1] + x1 * cs[j >> 1];
                    x0 = r0;
                  }
                  v[j] = fmaf(x0, qs, 0.f);  // + 0: a rotated -0 codes as 0
                  v[j + 1] = fmaf(x1, qs, 0.f);
                }
                stage_fp8_32(h == 0 ? buf0 : buf1, lane, g, v);
              }
            }
            ring.commit(&p.map_out[sec], buf0, lane, n0, y_box);
            ring.commit(&p.map_out[sec], buf1, lane, n0 + 128, y_box);
            release_acc(abuf);
            continue;
          }
        }
        // GELU: the bias of the next 32-column unit is loaded while this one is computed
        // (measured +1 % on the GELU kernels; the QKV kernels keep plain loads, -1 % otherwise)
        constexpr bool kBiasAhead = EPI == EPI_GELU_TANH || EPI == EPI_GELU_ERF;
        const bool has_bias = bias != nullptr;
        uint4 bq[4];
        if constexpr (kBiasAhead) load_raw32(bias, has_bias, n0, n_limit, bq);
#pragma unroll 1
        for (int c = 0; c < T::kOutN / 64; ++c) {
          const uint32_t buf = ring.acquire(lane);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col0 = n0 + c * 64 + u * 32;
            float v[32], b[32];
            if constexpr (kBiasAhead) {
              unpack32(bq, b);
              if (c * 2 + u + 1 < T::kOutN / 32) load_raw32(bias, has_bias, col0 + 32, n_limit, bq);
            } else {
              load_vec32(bias, col0, n_limit, b);
            }
            tmem_load32f(tacc + c * 64 + u * 32, k_empty, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += b[j];
            if constexpr (EPI == EPI_GELU_TANH) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = gelu_tanh_f(v[j]);
            } else if constexpr (EPI == EPI_GELU_ERF) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = gelu_erf_f(v[j]);

            }  // QKV: only the unrotated V section reaches this loop
            stage_bf16_32(buf, lane, u, v);
          }
          ring.commit(&p.map_out[sec], buf, lane, n0 + c * 64, y_box);
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_SWIGLU) {
        if (!ok) break;
        const int n0 = nb * 128;  // accumulator columns [0,128) = gate, [128,256) = up
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const uint32_t buf = ring.acquire(lane);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col0 = n0 + c * 64 + u * 32;
            float g[32], v[32], b[32];
            tmem_load32f(tacc + c * 64 + u * 32, k_empty, g);
            load_vec32(p.bias, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = silu_f(g[j] + b[j]);
            tmem_load32f(tacc + 128 + c * 64 + u * 32, k_empty, v);
            load_vec32(p.bias2, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = g[j] * (v[j] + b[j]);
            stage_bf16_32(buf, lane, u, v);
          }
          ring.commit(&p.map_out[0], buf, lane, n0 + c * 64, y_box);
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_RESID_GAMMA) {
        // Epilogue 1 of the chain: h1 = acc + b + z (the residual stream), h2 = h1 (.) gamma feeds the
        // next GEMM unscaled, and the tile's partial sum of h1^2 per row goes to the partials array.
        if (!ok) break;
        const int n0 = nb * 256;
        const __nv_bfloat16* zrow = p.resid + static_cast<long long>(row_ok ? m : 0) * p.ldz;
        float ss = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float h[2][32];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col0 = n0 + c * 64 + u * 32;
            float z[32], b[32];
            tmem_load32f(tacc + c * 64 + u * 32, k_empty, h[u]);
            load_row32(zrow, row_ok, col0, p.N, z);
            load_vec32(p.bias, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              h[u][j] += b[j] + z[j];
              ss = fmaf(h[u][j], h[u][j], ss);
            }
          }
          if (p.store_h1) {
            const uint32_t buf = ring.acquire(lane);
            stage_bf16_32(buf, lane, 0, h[0]);
            stage_bf16_32(buf, lane, 1, h[1]);
            ring.commit(&p.map_out[1], buf, lane, n0 + c * 64, y_box);
          }
          const uint32_t buf = ring.acquire(lane);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float g[32];
            load_vec32(p.gamma, n0 + c * 64 + u * 32, p.N, g);
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] *= h[u][j];
            stage_bf16_32(buf, lane, u, g);
          }
          ring.commit(&p.map_out[0], buf, lane, n0 + c * 64, y_box);
        }
        if (row_ok) p.rms_partials[static_cast<size_t>(nb) * p.M + m] = ss;
        release_acc(abuf);
      } else if constexpr (EPI == EPI_ROWSCALE) {
        // Epilogue 2 of the chain: the row scale r, deferred past this GEMM (it is one scalar per
        // row, so (r v) W = r (v W)), is merged from the row's partials and applied here.
        if (!ok) break;
        float ssum = 0.f;
        if (row_ok)
          for (int j = 0; j < p.n_partials; ++j) ssum += __ldg(p.rms_partials + static_cast<size_t>(j) * p.M + m);
        const float r = rsqrtf(ssum / static_cast<float>(p.n_norm) + p.eps);
        const int n0 = nb * 256;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const uint32_t buf = ring.acquire(lane);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col0 = n0 + c * 64 + u * 32;
            float v[32], b[32];
            tmem_load32f(tacc + c * 64 + u * 32, k_empty, v);
            load_vec32(p.bias, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaf(r, v[j], b[j]);
            stage_bf16_32(buf, lane, u, v);
          }
          ring.commit(&p.map_out[0], buf, lane, n0 + c * 64, y_box);
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_CE) {
        // Stateful epilogue ("GEMM Epilogue 完全拆解", §模式 C): each tile keeps, per row, the running
        // maximum m and s = sum exp(h - m) over its columns and picks the label's logit; the last
        // tile of a 128-row block to finish (an atomic count, no waiting) merges the row's states in
        // column-tile order into loss = m + log s - h[label].  Like the RMSNorm exchange, the
        // 128 threads take the same named barriers and leave together right after one.
        if (mb >= p.num_m_blocks) {
          if (!ok) break;
          release_acc(abuf);
          continue;
        }
        const int n0 = nb * 256;
        const int label = row_ok ? __ldg(p.labels + m) : -1;
        if (ok) {
          float mx = -INFINITY, se = 0.f, hl = 0.f;
          bool has_label = false;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t buf = 0;
            if (p.store_logits) buf = ring.acquire(lane);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int col0 = n0 + c * 64 + u * 32;
              float v[32], b[32];
              tmem_load32f(tacc + c * 64 + u * 32, k_empty, v);
              load_vec32(p.bias, col0, p.N, b);
              float um = -INFINITY;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                v[j] = col0 + j < p.N ? v[j] + b[j] : -INFINITY;  // columns past the vocabulary count for nothing
                um = fmaxf(um, v[j]);
                if (col0 + j == label) {
                  hl = v[j];
                  has_label = true;
                }
              }
              const float nm = fmaxf(mx, um);
              if (nm > -INFINITY) {
                float add = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) add += __expf(v[j] - nm);
                se = (mx > -INFINITY ? se * __expf(mx - nm) : 0.f) + add;
                mx = nm;
              }
              if (p.store_logits) stage_bf16_32(buf, lane, u, v);
            }
            if (p.store_logits) ring.commit(&p.map_out[0], buf, lane, n0 + c * 64, y_box);
          }
          if (row_ok) {
            p.ce_partials[static_cast<size_t>(nb) * p.M + m] = make_float2(mx, se);
            if (has_label) p.label_logit[m] = hl;
          }
        }
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (threadIdx.x == 64) {
          const int stop = *abort_flag;
          int last = 0;
          if (!stop) {
            __threadfence();
            last = atomicAdd(p.counters + mb, 1u) == static_cast<unsigned>(p.num_n_blocks) - 1u;
            if (last) __threadfence();  // acquire: every tile's state for this row block is visible
          }
          *epi_stop = stop;
          *ce_last = last;
        }
        named_bar_sync(1, kEpiThreads);
        if (*epi_stop) break;  // uniform: only the leader writes it, between the two barriers
        if (*ce_last) {
          if (row_ok) {
            float M_ = -INFINITY, S_ = 0.f;
            for (int j0 = 0; j0 < p.num_n_blocks; j0 += 16) {
              float2 w[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[j] = j0 + j < p.num_n_blocks ? __ldcg(p.ce_partials + static_cast<size_t>(j0 + j) * p.M + m)
                                               : make_float2(-INFINITY, 0.f);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float nm = fmaxf(M_, w[j].x);
                if (nm > -INFINITY) {
                  S_ = (M_ > -INFINITY ? S_ * __expf(M_ - nm) : 0.f) + (w[j].x > -INFINITY ? w[j].y * __expf(w[j].x - nm) : 0.f);
                  M_ = nm;
                }
              }
            }
            float l;
            if (label < 0) {
              l = 0.f;
            } else if (label >= p.N) {
              l = __int_as_float(0x7fc00000);  // NaN: label outside the vocabulary
            } else {
              l = M_ + __logf(S_) - __ldcg(p.label_logit + m);
            }
            p.loss[m] = l;
          }
          if (threadIdx.x == 64) p.counters[mb] = 0u;  // every tile of this row block has arrived
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_GELU_BWD_TANH || EPI == EPI_GELU_BWD_ERF) {
        // "GEMM Epilogue 完全拆解", §模式 D: the dgrad GEMM's epilogue multiplies by f'(h), with the
        // saved pre-activation h from the warp's saved-activation ring.
        if (!ok) break;
        const int n0 = nb * 256;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const uint32_t buf = ring.acquire(lane);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float h[32], v[32];
            take_saved(h, h);
            tmem_load32f(tacc + c * 64 + u * 32, k_empty, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] *= EPI == EPI_GELU_BWD_TANH ? gelu_tanh_grad_f(h[j]) : gelu_erf_grad_f(h[j]);
            stage_bf16_32(buf, lane, u, v);
          }
          ring.commit(&p.map_out[0], buf, lane, n0 + c * 64, y_box);
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_SWIGLU_BWD) {
        // "GEMM Epilogue 完全拆解", §末尾布局调整 (SwiGLU 反向): one upstream value dy of feature n
        // gives (dg, du) = (dy u SiLU'(g), dy SiLU(g)); the pair is packed into one 32-bit word
        // and the row is written at twice the width (columns 2n and 2n + 1).  The saved gate and
        // up values come from the warp's saved-activation ring.
        if (!ok) break;
        const int n0 = nb * 256;
#pragma unroll 1
        for (int u = 0; u < 8; ++u) {
          const int col0 = n0 + u * 32;
          float g[32], up[32], dy[32];
          take_saved(g, up);
          tmem_load32f(tacc + u * 32, k_empty, dy);
          const uint32_t buf = ring.acquire(lane);
          const uint32_t srow_s = buf + lane * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 4 * c + i;
              const float s = __fdividef(1.f, 1.f + __expf(-g[j]));  // sigmoid; 0 when e^{-g} overflows
              const float dg = dy[j] * up[j] * (s * fmaf(g[j], 1.f - s, 1.f));
              const float du = dy[j] * (g[j] * s);
              w[i] = pack_bf16x2(dg, du);
            }
            st_shared_v4(srow_s + ((c ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
          ring.commit(&p.map_out[0], buf, lane, 2 * col0, y_box);
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_QUANT) {
        // "GEMM Epilogue 完全拆解", §仿射量化与尾声的五步: block maximum -> scale -> codes -> compact
        // layout, scales written beside the codes in the same epilogue.  Blocks are row segments
        // of one thread, so no cross-thread reduction is needed.
        if (!ok) break;
        const int n0 = nb * 256;
        // Step 3 (optional scale-factor correction): the output of a smoothed layer is multiplied
        // per column by the inverse smoothing factor before the block maximum and the rounding.
        const bool has_sm = p.smooth != nullptr;
        if (p.quant_fmt == QF_FP8_1X128) {
#pragma unroll 1
          for (int blk = 0; blk < 2; ++blk) {
            float amax = 0.f;
#pragma unroll 1
            for (int u = 0; u < 4; ++u) {
              float v[32], b[32];
              tmem_load32f(tacc + blk * 128 + u * 32, k_empty, v);
              load_vec32(p.bias, n0 + blk * 128 + u * 32, p.N, b);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += b[j];
              if (has_sm) {
                load_f32x32(p.smooth, n0 + blk * 128 + u * 32, p.N, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= b[j];
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
            }
            const float qs = amax > 0.f ? 448.f / amax : 0.f;
            if (row_ok && n0 + blk * 128 < p.N)
              static_cast<float*>(p.qscale)[static_cast<long long>(m) * p.lds + nb * 2 + blk] = amax * (1.f / 448.f);
            const uint32_t buf = ring.acquire(lane);
#pragma unroll 1
            for (int u = 0; u < 4; ++u) {
              float v[32], b[32];
              tmem_load32f(tacc + blk * 128 + u * 32, k_empty, v);
              load_vec32(p.bias, n0 + blk * 128 + u * 32, p.N, b);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += b[j];
              if (has_sm) {
                load_f32x32(p.smooth, n0 + blk * 128 + u * 32, p.N, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= b[j];
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = fmaf(v[j], qs, 0.f);  // + 0: a zero block codes as +0
              stage_fp8_32(buf, lane, u, v);
            }
            ring.commit(&p.map_out[0], buf, lane, n0 + blk * 128, y_box);
          }
        } else {
          // INT4 / NVFP4: 4 bits per value, a 256-column tile is one 128-byte row of codes
          const uint32_t buf = ring.acquire(lane);
          const uint32_t srow = buf + lane * 128;
#pragma unroll 1
          for (int u = 0; u < 8; ++u) {
            const int col0 = n0 + u * 32;
            float v[32], b[32];
            tmem_load32f(tacc + u * 32, k_empty, v);
            load_vec32(p.bias, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += b[j];
            if (has_sm) {
              load_f32x32(p.smooth, col0, p.N, b);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] *= b[j];
            }
            uint32_t w[4];
            if (p.quant_fmt == QF_INT4_G32) {
              float amax = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
              const float inv = amax > 0.f ? 7.f / amax : 0.f;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t word = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  int qv = __float2int_rn(v[8 * i + e] * inv);  // round half to even
                  qv = max(-7, min(7, qv));
                  word |= (static_cast<uint32_t>(qv) & 15u) << (4 * e);
                }
                w[i] = word;
              }
              if (row_ok && col0 < p.N)
                static_cast<float*>(p.qscale)[static_cast<long long>(m) * p.lds + nb * 8 + u] = amax * (1.f / 7.f);
            } else {
              uint32_t codes[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[16 * h + j]));
                uint32_t sc;
                const float s = round_to_e4m3(amax * (1.f / 6.f), sc);
                codes[h] = sc;
                const float inv = s > 0.f ? 1.f / s : 0.f;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  uint32_t word = 0;
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int j = 16 * h + 8 * i + 2 * e;
                    word |= f32x2_to_e2m1x2(fmaf(v[j], inv, 0.f), fmaf(v[j + 1], inv, 0.f)) << (8 * e);  // +0 as above
                  }
                  w[2 * h + i] = word;
                }
              }
              if (row_ok && col0 < p.N) {
                uint8_t* sp = static_cast<uint8_t*>(p.qscale) + static_cast<long long>(m) * p.lds + nb * 16 + u * 2;
                sp[0] = static_cast<uint8_t>(codes[0]);
                if (col0 + 16 < p.N) sp[1] = static_cast<uint8_t>(codes[1]);
              }
            }
            st_shared_v4(srow + ((u ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
          ring.commit(&p.map_out[0], buf, lane, n0 / 2, y_box);
        }
        release_acc(abuf);
      } else if constexpr (EPI == EPI_RMSNORM_FP8) {
        // The 128 epilogue threads take the same named barriers in every
        // iteration and leave the loop together, right after a barrier.
        if (mb >= p.num_m_blocks) {  // the pair's second row block lies past M: no rows, no exchange
          if (!ok) break;
          release_acc(abuf);
          continue;
        }
        const int n0 = nb * 256;
        const __nv_bfloat16* zrow = p.resid + static_cast<long long>(row_ok ? m : 0) * p.ldz;
        // Pass 1: h = acc + b + z; partial sum of h^2 and partial max |h * gamma| over this tile's columns.
        // With h_out, h also leaves in bf16 (the residual stream after the add, [E] §模式 A), two
        // 32-column units per staging buffer, while the row exchange is still ahead.
        float ss = 0.f, am = 0.f;
        if (ok) {
          uint32_t hbuf = 0;
#pragma unroll 1
          for (int u = 0; u < 8; ++u) {
            const int col0 = n0 + u * 32;
            float v[32], z[32], g[32], b[32];
            tmem_load32f(tacc + u * 32, k_empty, v);
            load_row32(zrow, row_ok, col0, p.N, z);
            load_vec32(p.gamma, col0, p.N, g);
            load_vec32(p.bias, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float h = v[j] + b[j] + z[j];
              ss = fmaf(h, h, ss);
              am = fmaxf(am, fabsf(h * g[j]));
              v[j] = h;
            }
            if (p.store_h1) {
              if ((u & 1) == 0) hbuf = ring.acquire(lane);
              stage_bf16_32(hbuf, lane, u & 1, v);
              if (u & 1) ring.commit(&p.map_out[1], hbuf, lane, n0 + (u >> 1) * 64, y_box);
            }
          }
          p.partials[static_cast<size_t>(mb * p.num_n_blocks + nb) * kBM + row_in_tile] = make_float2(ss, am);
        }
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (threadIdx.x == 64) {
          int stop = *abort_flag;
          if (!stop) {
            __threadfence();
            atomicAdd(p.counters + mb, 1u);
            if (!wait_row_block(p, mb, static_cast<unsigned>(p.num_n_blocks))) {
              stop = 1;
              *abort_flag = 1;
            }
          }
          *epi_stop = stop;
        }
        named_bar_sync(1, kEpiThreads);
        if (*epi_stop) break;  // uniform: only the leader writes it, between the two barriers
        // Merge the partials of every tile of this row block (fixed order: deterministic).
        float SS = 0.f, A = 0.f;
        const float2* prow = p.partials + static_cast<size_t>(mb) * p.num_n_blocks * kBM + row_in_tile;
        for (int j = 0; j < p.num_n_blocks; ++j) {
          const float2 w = __ldcg(prow + static_cast<size_t>(j) * kBM);
          SS += w.x;
          A = fmaxf(A, w.y);
        }
        named_bar_sync(1, kEpiThreads);
        if (threadIdx.x == 64) {
          // The last tile of the row block to finish reading resets the counters for the next call.
          const unsigned old = atomicAdd(p.counters + p.num_m_blocks + mb, 1u);
          if (old == static_cast<unsigned>(p.num_n_blocks) - 1u) {
            p.counters[mb] = 0u;
            p.counters[p.num_m_blocks + mb] = 0u;
          }
        }
        const float r = rsqrtf(SS / static_cast<float>(p.N) + p.eps);
        const float qs = A > 0.f ? 448.f / A : 0.f;  // y / scale = h * gamma * 448 / max|h * gamma|
        if (nb == 0 && row_ok) p.row_scale[m] = r * A * (1.f / 448.f);
        // Pass 2: codes.
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const uint32_t buf = ring.acquire(lane);
#pragma unroll 1
          for (int u = 0; u < 4; ++u) {
            const int col0 = n0 + c * 128 + u * 32;
            float v[32], z[32], g[32], b[32];
            tmem_load32f(tacc + c * 128 + u * 32, k_empty, v);
            load_row32(zrow, row_ok, col0, p.N, z);
            load_vec32(p.gamma, col0, p.N, g);
            load_vec32(p.bias, col0, p.N, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaf((v[j] + b[j] + z[j]) * g[j], qs, 0.f);  // + 0: a zero row codes as +0
            stage_fp8_32(buf, lane, u, v);
          }
          ring.commit(&p.map_out[0], buf, lane, n0 + c * 128, y_box);
        }
        release_acc(abuf);
      }
    }
    if (lane == 0) {
      bulk_wait_all();
      if constexpr (T::kNSaved > 0) sring.drain(p.timeout_ns);  // copies still in flight after an error
    }
  }

  if constexpr (CG == 2) {
    cluster_sync_all();  // neither CTA leaves while the other may still touch its memory
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2) {
      tmem_dealloc_pair(tmem_base, T::kTmemCols);
    } else {
      tmem_dealloc(tmem_base, T::kTmemCols);
    }
  }
}

}  // namespace fl
