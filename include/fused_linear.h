/* fused_linear.h — C ABI of the GB300 (sm_103a) fused Linear + epilogue library.
 *
 * Every entry point computes a Linear layer Y = X W^T (+ b) on the tcgen05
 * tensor cores, keeps the fp32 accumulator tile in tensor memory, and applies
 * the memory-bound tail ("epilogue") to that tile before anything is written
 * to HBM; no intermediate tensor is materialised.
 *
 * Conventions shared by all entry points
 *   - Matrices are row-major.  X is [M, K] with leading dimension ldx (in
 *     elements), W is [N, K] (one row per output feature, the PyTorch Linear
 *     layout) with leading dimension ldw, outputs are [M, N_out] with their own
 *     leading dimension.  All leading dimensions are in elements.
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them.  Except where stated, bf16 means IEEE
 *     bfloat16 stored as 16-bit words.
 *   - Calls are asynchronous: they validate the arguments on the host, enqueue
 *     their work on `stream` (a cudaStream_t; NULL = legacy default stream:
 *     normally one kernel; the exceptions are stated with each call) and
 *     return.  Device-side failures (a bounded wait that ran out) are recorded
 *     in the status record at the start of the call's workspace (calls that take
 *     one: fl_check_device_status(workspace, stream)) or else in a device-wide
 *     status word (fl_device_status(stream)).
 *   - Alignment (a requirement of the tensor-memory-access copies): every base
 *     pointer must be 16-byte aligned and every leading dimension times the
 *     element size must be a multiple of 16 bytes.
 *   - M, N or K equal to 0 is allowed; M == 0 or N == 0 enqueues nothing, and
 *     K == 0 treats X W^T as zero.
 *   - Return value: an fl_status code (FL_OK = 0).  A call rejected by its
 *     checks (every code but FL_ERR_CUDA) enqueues nothing.  FL_ERR_CUDA after
 *     a call's first launch (a decode call that runs as several launches, the
 *     host-buffer pipeline) can leave the launches before it enqueued.
 *
 * Page citations name the page title and its section:
 *   "Triton 算子融合: Linear 与 Attention" (aiqz.cc, triton-operator-fusion-linear-attention)
 *   "GEMM Epilogue 完全拆解: 推理内核的最后一公里" (pinghaoyang.com.cn, gemm-epilogue-fusion)
 */
#ifndef FUSED_LINEAR_H
#define FUSED_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FL_API __attribute__((visibility("default")))
#else
#define FL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fl_status {
    FL_OK = 0,
    FL_ERR_INVALID_ARG = 1,   /* null pointer, negative size, leading dim below the row width */
    FL_ERR_UNSUPPORTED = 2,   /* a shape or option this build does not implement */
    FL_ERR_ALIGNMENT = 3,     /* pointer or row pitch not 16-byte aligned */
    FL_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    FL_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    FL_ERR_TIMEOUT = 6,       /* a device-side bounded wait ran out (see fl_device_status) */
    FL_ERR_ARCH = 7           /* the current device is not sm_103 */
} fl_status;

enum { FL_F32 = 0, FL_BF16 = 1 };
enum { FL_GELU_ERF = 0, FL_GELU_TANH = 1 };

/* Linear + bias + GELU.
 *   "Triton 算子融合: Linear 与 Attention", §Linear算子剖析 (Y[m,n] = sum_k X[m,k] W[n,k] + b[n])
 *   and §GELU激活融合 (erf form 0.5 v (1 + erf(v / sqrt 2)); tanh form
 *   0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))).
 * X [M,K], W [N,K], b [N] (nullable: no bias), Y [M,N].  X, W, b and Y all have
 * dtype `dtype`: FL_BF16 (tcgen05 bf16 MMA, fp32 accumulate, one bf16 rounding
 * at the store) or FL_F32 (fp32 operands and output; on the tensor cores as three
 * TF32 products per term, hi*hi + hi*lo + lo*hi with x = hi + lo split exactly, fp32
 * accumulate: within ~2^-21 of each product, where one TF32 product would miss fp32 accuracy).
 * mode: FL_GELU_ERF or FL_GELU_TANH.  Y must not alias X, W or b.
 * bf16 with M <= 32 runs the decode kernel (fl_set_linear_decode): one launch, or several
 * when its W-row tiles do not all fit on the GPU at once (fl_linear_decode_shape reports which).
 */
FL_API int fused_linear_gelu(const void* X, const void* W, const void* b, void* Y,
                      int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldy,
                      int dtype, int mode, void* stream);

/* Fused QKV projection + RoPE with split write-back.
 *   "Triton 算子融合: Linear 与 Attention", §QKV投影融合: [Q|K|V] = X Wqkv^T + bqkv with
 *   Q, K, V the first, middle and last d = n_heads * head_dim output columns.
 *   "GEMM Epilogue 完全拆解", §模式 B and §累加器布局 (RoPE rotates each adjacent
 *   feature pair (2i, 2i+1) of a head by pos * theta^(-2i/head_dim)), and
 *   §用形状与步长把约定钉死 (layout contract).
 * Layout contract: Q, Kout and V are three separate row-major bf16 [M, d] tensors
 * with the same leading dimension ldo.  Q and Kout are written ALREADY ROTATED;
 * downstream code must not rotate them again.  V is not rotated.  Order: bias,
 * then rotation, then one bf16 rounding.
 * X [M,K] bf16, Wqkv [3d, K] bf16 (W_q, W_k, W_v stacked by rows), bqkv [3d] bf16
 * (nullable).  positions: nullable device int32 [M]; when NULL row m has
 * position m % seq_len (rows are sequences of seq_len tokens laid end to end).
 * Positions must lie in [0, 2^24).  head_dim must be 128 and d a multiple of 256.
 * M <= 32 runs the decode kernel, one head per W-row tile (fl_set_linear_decode).
 */
FL_API int fused_qkv_rope(const void* X, const void* Wqkv, const void* bqkv,
                   void* Q, void* Kout, void* V, const int32_t* positions,
                   int M, int K, int n_heads, int head_dim, int seq_len, float theta,
                   int64_t ldx, int64_t ldw, int64_t ldo, void* stream);

/* QKV projection + RoPE whose epilogue writes the K/V cache entry in FP8.
 *   "GEMM Epilogue 完全拆解", §一个瓦片的字节账 (the K/V write-back quantised to FP8 in
 *   the epilogue, half the bytes of bf16) with the scale of §仿射量化与尾声的五步 taken
 *   over one head of one token: s = max|y| / 448 over its head_dim values, codes
 *   E4M3(y / s) (round to nearest even, saturating); a head whose maximum is 0 gets
 *   s = 0 and zero codes.
 * Grouped-query widths: Wqkv [(n_heads + 2 n_kv_heads) * head_dim, K] bf16 with rows
 * [Q | K | V]; bqkv nullable.  Q [M, n_heads*head_dim] bf16 (rotated, pitch ldq elements);
 * Kq, Vq [M, n_kv_heads*head_dim] E4M3 bytes (K rotated, V not; pitch ldkv bytes, a
 * multiple of 16); k_scale, v_scale [M, lds] fp32, one per (token, kv head).
 * Positions as in fused_qkv_rope.  head_dim must be 128 and n_heads, n_kv_heads even
 * and non-zero (FL_ERR_UNSUPPORTED otherwise).  M <= 32 runs the decode kernel, whose
 * clusters exchange each head's per-token maximum in distributed shared memory. */
FL_API int fused_qkv_rope_fp8kv(const void* X, const void* Wqkv, const void* bqkv, void* Q, void* Kq, void* Vq,
                                float* k_scale, float* v_scale, const int32_t* positions, int M, int K,
                                int n_heads, int n_kv_heads, int head_dim, int seq_len, float theta,
                                int64_t ldx, int64_t ldw, int64_t ldq, int64_t ldkv, int64_t lds, void* stream);

/* SwiGLU up-projection: Y = SiLU(X Wgate^T + bgate) * (X Wup^T + bup).
 *   "GEMM Epilogue 完全拆解", §模式 B and §末尾布局调整 (a gate/value pair gives one
 *   value; the output has half the width of the [gate|up] product).
 * X [M,K] bf16; Wgate and Wup [N,K] bf16 with the same leading dimension ldw;
 * bgate, bup [N] bf16 (each nullable); Y [M,N] bf16.  The gate and up rows
 * that feed the same output columns are loaded side by side into one
 * shared-memory stage, so no host-side repacking of the weights is needed.
 * M <= 32 runs the decode kernel: 64 gate and the 64 matching up rows per W-row tile.
 */
FL_API int fused_swiglu(const void* X, const void* Wgate, const void* Wup,
                 const void* bgate, const void* bup, void* Y,
                 int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldy, void* stream);

/* Down projection + residual + RMSNorm + per-row FP8 E4M3 quantised write-back.
 *   "GEMM Epilogue 完全拆解", §模式 A: h = X W^T (+ b) + Z, r = 1/sqrt(mean_n h^2 + eps)
 *   (one scalar per row), y = r * h (.) gamma; §仿射量化与尾声的五步 steps 1, 2 and 5
 *   with one block per row: scale = max_n |y| / 448, Yq = e4m3(y / scale) rounded
 *   to nearest even and saturated to +-448, scale written beside Yq.
 * The row statistics span all N columns, which several output tiles share: each
 * tile emits per-row partial sums of squares and partial maxima, which are merged
 * inside the same kernel through `workspace` (the two-level reduction of §模式 A).
 * X [M,K] bf16, W [N,K] bf16, b [N] bf16 (nullable), Z [M,N] bf16 residual with
 * leading dimension ldz, gamma [N] bf16.  Yq [M,N] E4M3 bytes (leading dimension
 * ldq, a multiple of 16), row_scale [M] fp32 (dequantise with Yq * row_scale).
 * A row whose maximum is 0 gets scale 0 and zero codes.
 * h_out: nullable bf16 [M,N] with the residual's leading dimension ldz: when given,
 * h = X W^T + b + Z (the residual stream after the add, which the next block of a
 * model reads) is also written, rounded once to bf16; NULL writes nothing extra.
 * h_out must not overlap Z (FL_ERR_INVALID_ARG).
 * workspace: device memory of at least fl_rmsnorm_fp8_workspace_bytes(M, N, K)
 * bytes, 256-byte aligned and ZERO-FILLED before its first use.  Its first 256 bytes
 * are this call's status record: a device-side wait that runs out is recorded there
 * (read and clear it with fl_check_device_status(workspace, stream)).  The kernels
 * reset the counters they keep there before they return, so the same workspace
 * serves later calls on the same stream without clearing; after FL_ERR_TIMEOUT
 * it must be zero-filled again.  Calls that may run concurrently must not share
 * a workspace.  M <= 32 with K > 0 runs a split-K decode kernel: one thread-block
 * cluster per 128-feature tile, its CTAs each streaming an equal share of K, when
 * every cluster fits on the GPU at once, else one CTA per SM each streaming an equal
 * share of all of W; larger M runs the persistent prefill kernel.  All keep every
 * CTA resident at once (the prefill kernel launches cooperatively) and fail with
 * FL_ERR_CUDA if that is impossible.
 * N must not exceed 256 * (number of SMs) on the prefill path.
 */
FL_API int fused_linear_residual_rmsnorm_fp8(const void* X, const void* W, const void* b,
                                      const void* Z, const void* gamma, float eps,
                                      void* Yq, float* row_scale, void* h_out,
                                      int M, int N, int K,
                                      int64_t ldx, int64_t ldw, int64_t ldz, int64_t ldq,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* Same computation as fused_linear_residual_rmsnorm_fp8 (without h_out), for callers
 * that cannot allocate device memory and so cannot supply a workspace: a serving loop
 * that must not stall in the allocator (cudaMalloc can synchronise the device), or a
 * plugin whose host framework owns all device memory and hands it none.  The pages have
 * no counterpart of this call; it exists only for such callers.
 * Scratch: one FL_NOALLOC_SCRATCH_BYTES array compiled into the library and
 * held by every GPU that loads it until the process exits.  A shape whose
 * fl_rmsnorm_fp8_workspace_bytes(M, N, K) exceeds that size is rejected with
 * FL_ERR_WORKSPACE.  The array is shared by every call and keeps the last call's
 * contents: calls that can overlap on the GPU (streams with no ordering between
 * them) race and must not be issued.  A call that passes every check enqueues an
 * asynchronous memset on `stream` that clears the counters the kernels wait on, then
 * the kernel; a rejected call enqueues nothing.  Nothing is allocated.  The first
 * call on a device looks up the array's device address with that device current (a
 * one-time set-up); make that first call before any stream capture.  The address is
 * kept for the life of the process, so cudaDeviceReset is not supported with this
 * call.  Device-side failures go to the device-wide status word (fl_device_status).
 * Other arguments, layouts and errors are those of fused_linear_residual_rmsnorm_fp8. */
#define FL_NOALLOC_SCRATCH_BYTES (8u << 20)
FL_API int fused_linear_residual_rmsnorm_fp8_noalloc(const void* X, const void* W, const void* b,
                                                     const void* Z, const void* gamma, float eps,
                                                     void* Yq, float* row_scale,
                                                     int M, int N, int K,
                                                     int64_t ldx, int64_t ldw, int64_t ldz, int64_t ldq,
                                                     void* stream);

/* GEMM -> residual -> RMSNorm -> GEMM, with the RMSNorm row scale deferred into
 * the second GEMM ("GEMM Epilogue 完全拆解", §模式 A: y = RMSNorm(x W0 + z, gamma) W1
 * = r (.) (((x W0 + z) (.) gamma) W1), since r is one scalar per row and commutes
 * with a matrix product; a per-column factor such as gamma does not).
 *
 * Step 1, fused_linear_residual_gamma: h1 = X W^T (+ b) + Z; writes H2 = h1 (.) gamma
 * (bf16, the unscaled input of the second GEMM), optionally H1 = h1 (bf16, the
 * residual stream after the add; NULL to skip), and rms_partials: fp32
 * [fl_rms_partials_per_row(N)][M] (tile-major), entry [j][m] = sum of h1[m, n]^2 over
 * columns n of the j-th 256-column tile.  X [M,K], W [N,K], b [N] (nullable),
 * Z [M,N] (ldz), gamma [N]; H1 and H2 share the leading dimension ldh.
 *
 * Step 2, fused_linear_rms_rowscale: Y = r (.) (H2 W1^T) (+ b1) with
 * r[m] = 1 / sqrt((sum_j rms_partials[j][m]) / n_norm + eps), the partials merged in a
 * fixed order inside the epilogue (no separate reduction launch).  H2 [M,K] with
 * K = n_norm normally, W1 [N,K], b1 [N] (nullable), Y [M,N] bf16.  Run step 2 on the
 * same stream after step 1 (or after an event) so the partials are complete.
 * M <= 32 runs both steps on the decode kernel (fl_set_linear_decode): tiles of 128 output
 * features; step 1 then enqueues a memset of its rms_partials before the kernel, which adds the
 * sums of the two 128-feature halves of every 256-column entry onto zero (the same bits in
 * either order). */
FL_API int fused_linear_residual_gamma(const void* X, const void* W, const void* b, const void* Z,
                                       const void* gamma, void* H2, void* H1, float* rms_partials,
                                       int M, int N, int K, int64_t ldx, int64_t ldw, int64_t ldz,
                                       int64_t ldh, void* stream);
FL_API int fused_linear_rms_rowscale(const void* H2, const void* W1, const void* b1,
                                     const float* rms_partials, int n_norm, float eps, void* Y,
                                     int M, int N, int K, int64_t ldh, int64_t ldw, int64_t ldy,
                                     void* stream);
/* Number of rms_partials entries per row for a normalised width of n_norm (ceil(n_norm / 256)). */
FL_API int fl_rms_partials_per_row(int n_norm);

/* LM-head cross-entropy: logits h = X W^T (+ b) over a vocabulary of V and
 * loss[m] = logsumexp_v(h[m, v]) - h[m, labels[m]], without writing the logits.
 *   "GEMM Epilogue 完全拆解", §模式 C: every 256-column tile keeps, per row, the running
 *   maximum m and s = sum exp(h - m) (a stateful epilogue) and the tile holding the
 *   label keeps that logit; the last tile of each 128-row block to finish merges the
 *   row's states in column order (m = max(m1, m2), s = s1 e^{m1-m} + s2 e^{m2-m}), so the
 *   result is deterministic and needs no waiting between CTAs.
 * X [M,K] bf16, W [V,K] bf16, b [V] bf16 (nullable), labels [M] int32 (negative: ignored
 * row, loss 0; >= V: loss NaN), loss [M] fp32 out.  logits: nullable bf16 [M,V] copy of
 * the logits (leading dimension ldl), e.g. kept for a backward pass.
 * workspace: fl_cross_entropy_workspace_bytes(M, V) bytes, 256-byte aligned and
 * zero-filled before first use; its first 256 bytes are the call's status record
 * (fl_check_device_status).  The kernel resets its counters, so it can be reused
 * by later calls on the same stream (re-zero it after FL_ERR_TIMEOUT). */
FL_API int fused_linear_cross_entropy(const void* X, const void* W, const void* b, const int32_t* labels,
                                      float* loss, void* logits, int M, int V, int K,
                                      int64_t ldx, int64_t ldw, int64_t ldl,
                                      void* workspace, size_t workspace_bytes, void* stream);
FL_API size_t fl_cross_entropy_workspace_bytes(int M, int V);

/* Linear (+ bias) with a block-scaled quantised write-back.
 *   "GEMM Epilogue 完全拆解", §仿射量化与尾声的五步: for every block of consecutive columns
 *   of a row, scale = max|y| / qmax, codes = y / scale rounded to the format (nearest
 *   even, saturating), packed compactly, and the scale array written beside them.
 *   A block whose maximum is 0 gets scale 0 and zero codes.
 *   Step 3 (optional scale-factor correction): inv_smooth, a nullable fp32 [N] vector
 *   (16-byte aligned), is the inverse smoothing coefficient of a layer fed by
 *   SmoothQuant/QuaRot-style smoothing; when given, y[m,n] = (X W^T + b)[m,n] *
 *   inv_smooth[n] is what the blocks' maxima, scales and codes describe.
 * fmt FL_QUANT_FP8_1X128: E4M3 codes, one byte per value (Yq [M,N], ldq >= N bytes);
 *     blocks of 128 columns, fp32 scales [M][lds] = max / 448.
 * fmt FL_QUANT_INT4_G32: signed 4-bit codes in [-7, 7] (two's complement), two per byte
 *     with column 2j in the low nibble of byte j (Yq [M,N/2] bytes); groups of 32,
 *     fp32 scales = max / 7.  N must be even.
 * fmt FL_QUANT_NVFP4_G16: FP4 E2M1 codes, two per byte as above; groups of 16, scales
 *     stored as E4M3 bytes [M][lds] = e4m3(max / 6), the values divided by that stored
 *     scale.  N must be even.
 * X [M,K] bf16, W [N,K] bf16, b [N] bf16 (nullable); ldq in bytes (multiple of 16),
 * lds in scale elements (>= number of blocks per row).
 * M <= 32 runs the decode kernel (fl_set_linear_decode), tiles of 128 output features
 * finished by whole tokens, so every block of a token is inside one CTA. */
enum { FL_QUANT_FP8_1X128 = 0, FL_QUANT_INT4_G32 = 1, FL_QUANT_NVFP4_G16 = 2 };
FL_API int fused_linear_quant(const void* X, const void* W, const void* b, const float* inv_smooth,
                              void* Yq, void* scales, int M, int N, int K, int64_t ldx, int64_t ldw,
                              int64_t ldq, int64_t lds, int fmt, void* stream);

/* Backward of Linear -> GELU, fused into the dgrad GEMM.
 *   "GEMM Epilogue 完全拆解", §模式 D: dH = (dZ W) * GELU'(H).  dZ [M,K] bf16 is the
 *   gradient w.r.t. the next layer's output (K = that layer's output features), W [K,N]
 *   bf16 that layer's weight as stored (N contiguous, pitch ldw >= N), H [M,N] bf16 the
 *   saved pre-activation, dH [M,N] bf16 (pitches in elements, multiples of 8).  mode
 *   FL_GELU_ERF or FL_GELU_TANH picks the derivative's form.  Accumulation in fp32,
 *   one rounding at the store. */
FL_API int fused_dgrad_gelu(const void* dZ, const void* W, const void* H, void* dH, int M, int N, int K,
                            int64_t ldz, int64_t ldw, int64_t ldh, int64_t ldo, int mode, void* stream);

/* Backward of SwiGLU through the down projection, fused into its dgrad GEMM.
 *   "GEMM Epilogue 完全拆解", §末尾布局调整 (SwiGLU 反向): dy = dO Wd, and per feature n
 *   dg = dy u SiLU'(g), du = dy SiLU(g) with SiLU'(g) = s (1 + g (1 - s)), s = sigmoid(g).
 *   The pair is packed into one 32-bit word: dGU [M, 2N] bf16 holds dg at column 2n and
 *   du at column 2n + 1.  dO [M,K] bf16, Wd [K,N] bf16 the down projection's weight as
 *   stored, G and U [M,N] bf16 the saved gate and up activations (shared pitch ldgu). */
FL_API int fused_swiglu_bwd(const void* dO, const void* Wd, const void* G, const void* U, void* dGU,
                            int M, int N, int K, int64_t ldo_in, int64_t ldw, int64_t ldgu, int64_t ldout,
                            void* stream);

/* fused_linear_gelu (bf16) on HOST buffers: copies in, GEMM + epilogue, copies out.
 *   X [M,K], W [N,K], b [N] (nullable) and Y [M,N] are contiguous bf16 arrays in host
 *   memory (page-locked for the copies to overlap; pageable memory works, serialised).
 *   The pipeline is this library's: X is cut into about 4 blocks of whole 128-row tiles
 *   and W into about 8 blocks of whole 256-column output tiles, uploaded alternately (b,
 *   X0, W0, X1, W1, ..., then the rest of W); output block (r, c) is computed as soon as
 *   X_r and W_c have landed, and returns to the host (one 2-D copy) on a second copy
 *   stream while later blocks upload and compute.
 * dev_buf: caller-owned device memory of fl_linear_gelu_host_buffer_bytes(M, N, K)
 *   bytes, 256-byte aligned (holds X, W, b and Y on the device; no allocation per call).
 * Asynchronous with respect to the host: the call enqueues everything and returns; the
 *   kernels run on `stream`, the copies on two library-owned streams ordered after the
 *   work already on `stream`, and `stream` waits for the last copy out.  The host arrays
 *   must stay valid until `stream` has completed.  N and K must be multiples of 8
 *   (FL_ERR_ALIGNMENT); FL_ERR_WORKSPACE if dev_buf is too small. */
FL_API int fused_linear_gelu_host(const void* X, const void* W, const void* b, void* Y, int M, int N, int K,
                                  int mode, void* dev_buf, size_t dev_buf_bytes, void* stream);
FL_API size_t fl_linear_gelu_host_buffer_bytes(int M, int N, int K);

/* Bytes of workspace fused_linear_residual_rmsnorm_fp8 needs for this shape
 * on the current device (0 for an empty problem). */
FL_API size_t fl_rmsnorm_fp8_workspace_bytes(int M, int N, int K);

/* Synchronises `stream`, then returns FL_OK if no kernel of this library
 * recorded a device-side failure in the device-wide status word of the current
 * device since the previous call, else the recorded code (FL_ERR_TIMEOUT), and
 * clears the record.  Calls that take a workspace record their failures in it
 * instead (fl_check_device_status).  Returns FL_ERR_CUDA if the synchronisation
 * itself fails. */
FL_API int fl_device_status(void* stream);

/* The status of the calls that used `workspace` (a workspace of
 * fused_linear_residual_rmsnorm_fp8 or fused_linear_cross_entropy).
 *   "GEMM Epilogue 完全拆解", §边界三 (布局即约定): the error contract travels with the
 *   buffer layout, so a failure is reported against the workspace the call used.
 * Synchronises `stream`, reads the status record in the workspace's first 256 bytes,
 * returns FL_OK if it is clear, else the recorded code (FL_ERR_TIMEOUT) after clearing
 * it.  Concurrent calls on other streams with other workspaces neither see nor clear
 * this record.  workspace NULL: the same as fl_device_status(stream).
 * FL_ERR_ALIGNMENT if workspace is not 256-byte aligned; FL_ERR_CUDA if the
 * synchronisation or the read fails. */
FL_API int fl_check_device_status(void* workspace, void* stream);

/* Upper bound, in nanoseconds, on every device-side wait of later launches
 * (default 2e9).  A wait that runs out sets the status word, makes the kernel
 * drain its in-flight copies, free its tensor memory and return.  0 restores
 * the default.  Process-wide; intended for tests and diagnostics. */
FL_API void fl_set_wait_timeout_ns(uint64_t ns);

/* Caps the number of CTAs of the persistent kernels and of the decode kernels
 * (0 = one per SM; the decode kernels of fused_linear_gelu, fused_swiglu and the QKV
 * calls take it as the number of SMs, and their two-per-SM shapes launch up to twice
 * as many CTAs).  Used by tests to make each CTA walk many tiles, or to run the
 * flat split-K decode kernel where the cluster one would not fit under the cap; the
 * RMSNorm workspace size depends on it, so size the workspace under the same cap.
 * Process-wide. */
FL_API void fl_set_max_ctas(int n);

/* Two-CTA tensor-core mode of the prefill kernels: with 1 (the default) a pair
 * of CTAs on neighbouring SMs shares each 256-row tile (tcgen05 cta_group::2,
 * each CTA loading half of the W tile) whenever M spans at least two 128-row
 * blocks; with 0 every CTA computes its own 128-row tile.  Results are the
 * same either way.  Process-wide; intended for tests and diagnostics. */
FL_API void fl_set_cta_pairing(int enable);

/* Cooperative launch of the kernels whose CTAs wait on one another (the RMSNorm prefill
 * kernel's row exchange): with 1 (the default) the launch carries the cooperative attribute,
 * so the driver refuses it rather than start a grid that cannot be resident at once; with 0
 * the same grid (sized to what is resident at once) launches without it.  Only for tools
 * that refuse cooperative launches of clusters, such as a kernel profiler serialising the
 * device.  Process-wide; intended for diagnostics. */
FL_API void fl_set_cooperative_launch(int enable);

/* Tensor-map descriptor cache: every call encodes the TMA descriptors of its operands; with
 * 1 (the default) an encoded descriptor is kept, keyed by (address, extents, pitch, box,
 * element type, swizzle), and reused when a later call passes the same key (a descriptor
 * holds nothing else, so reuse is exact; a new pointer or shape is a new key).  128 entries,
 * round-robin replacement, guarded by a mutex.  0 disables and empties it.
 * fl_descriptor_cache_stats returns the hits and misses counted since the process started
 * (either pointer may be NULL).  Process-wide. */
FL_API void fl_set_descriptor_cache(int enable);
FL_API void fl_descriptor_cache_stats(unsigned long long* hits, unsigned long long* misses);

/* Decode-shaped calls: with 1 (the default) fused_linear_gelu (bf16), fused_swiglu,
 * fused_qkv_rope, fused_qkv_rope_fp8kv, fused_linear_quant and both steps of the deferred-scale
 * chain with M <= 32 rows run a swap-AB kernel that streams W once (tiles of W rows
 * on the tensor cores' M side, the tokens on N, split-K across a thread-block cluster; tiles of
 * 128 output features, SwiGLU 64; more tiles than fit at once, at two CTAs per SM, in several
 * launches); with 0 they run on the prefill GEMM kernel.  Results agree within rounding (the
 * split-K sums in a different order).
 * Process-wide; intended for tests and diagnostics. */
FL_API void fl_set_linear_decode(int enable);

/* The launches a decode-shaped call would make on the current device, without making them.
 * kind: FL_DECODE_GELU (fused_linear_gelu, N output features), FL_DECODE_SWIGLU (fused_swiglu,
 * N = d_ff), FL_DECODE_QKV (fused_qkv_rope, N = 3 * n_heads * head_dim), FL_DECODE_QKV_FP8KV
 * (fused_qkv_rope_fp8kv, N = (n_heads + 2 * n_kv_heads) * head_dim), FL_DECODE_QUANT
 * (fused_linear_quant, N output features), FL_DECODE_RESID_GAMMA (fused_linear_residual_gamma) or
 * FL_DECODE_ROWSCALE (fused_linear_rms_rowscale), N output features.  On FL_OK: *cluster = CTAs
 * per W-row tile (0 when the call runs on the GEMM kernel instead: M outside 1..32, the decode
 * path off, or no shape fits), *ctas_per_sm = 1 or 2 (the kernel variant with 10 or 5 stages),
 * *launches = consecutive launches of equal tile shares (more tiles than fit at once).
 * Takes fl_set_max_ctas and fl_set_linear_decode into account.  FL_ERR_INVALID_ARG for a null
 * output pointer, a negative size or an unknown kind. */
enum { FL_DECODE_GELU = 0, FL_DECODE_SWIGLU = 1, FL_DECODE_QKV = 2, FL_DECODE_QKV_FP8KV = 3, FL_DECODE_QUANT = 4,
       FL_DECODE_RESID_GAMMA = 5, FL_DECODE_ROWSCALE = 6 };
FL_API int fl_linear_decode_shape(int kind, int M, int N, int K, int* cluster, int* ctas_per_sm, int* launches);

/* Static text for a status code. */
FL_API const char* fl_status_string(int status);

/* Library ABI version (major * 100 + minor). */
FL_API int fl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FUSED_LINEAR_H */
