/* fp64 CPU oracle for the fused Linear + epilogue path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only code that may load this library.  It shares
 * no source, header, table or helper with the CUDA library and never calls it.
 *
 * Each function is the plain definition of what the fused kernels compute,
 * written out in fp64 with ordinary loops and libm, in the order the pages
 * state it.  Inputs are the exact fp64 widening of the bf16 / fp32 operands.
 * Page citations name the page title and its section:
 *   [T] "Triton 算子融合: Linear 与 Attention" (aiqz.cc, triton-operator-fusion-linear-attention)
 *   [E] "GEMM Epilogue 完全拆解: 推理内核的最后一公里" (pinghaoyang.com.cn, gemm-epilogue-fusion)
 *   [L] "什么是算子融合？LayerNorm与GeLU融合如何为深度学习推理提速" (ipipp.com)
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* ---- Linear -------------------------------------------------------------
 * [T] §Linear算子剖析: Y[m,n] = sum_{k=0}^{K-1} X[m,k] * W[n,k] + b[n].
 * W is stored [N, K] (one row per output feature).  The sum runs in k order.
 */
static double linear_at(const double* x_row, const double* W, const double* b, long K, long n) {
    const double* w = W + (size_t)n * (size_t)K;
    double s = 0.0;
    for (long k = 0; k < K; ++k) s += x_row[k] * w[k];
    if (b) s += b[n];
    return s;
}

/* out[i, j] = Linear(X[i, :])[cols[j]] for each of the nrows given rows of X. */
void orc_linear(const double* X, long nrows, const double* W, const double* b, long K,
                const long* cols, long ncols, double* out) {
#pragma omp parallel for collapse(2) schedule(static)
    for (long i = 0; i < nrows; ++i)
        for (long j = 0; j < ncols; ++j)
            out[i * ncols + j] = linear_at(X + (size_t)i * (size_t)K, W, b, K, cols[j]);
}

/* ---- GELU ----------------------------------------------------------------
 * erf form, [T] §GELU激活融合 (the kernel line 0.5*x*(1+erf(x/sqrt 2))), which
 * is x * Phi(x) with Phi the standard normal CDF.
 */
double orc_gelu_erf(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

/* tanh form, [T] §GELU激活融合 (formula) and [L] (constant sqrt(2/pi)):
 * 0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) )).
 */
double orc_gelu_tanh(double v) {
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
}

void orc_gelu(const double* v, long n, int mode, double* y) {
    for (long i = 0; i < n; ++i) y[i] = mode == 0 ? orc_gelu_erf(v[i]) : orc_gelu_tanh(v[i]);
}

/* Linear followed by GELU (mode 0 = erf, 1 = tanh), [T] §GELU激活融合. */
void orc_linear_gelu(const double* X, long nrows, const double* W, const double* b, long K,
                     const long* cols, long ncols, int mode, double* out) {
    orc_linear(X, nrows, W, b, K, cols, ncols, out);
    orc_gelu(out, nrows * ncols, mode, out);
}

/* ---- RoPE ----------------------------------------------------------------
 * [E] §模式 B and §累加器布局 (逐对运算): each adjacent pair of features
 * (2i, 2i+1) inside a head is rotated in its plane by the angle
 * pos * theta^(-2i / head_dim); two values in, two values out.
 */
double orc_rope_angle(double pos, long pair, long head_dim, double theta) {
    return pos * pow(theta, -2.0 * (double)pair / (double)head_dim);
}

void orc_rope_rotate(double x0, double x1, double angle, double* y0, double* y1) {
    double c = cos(angle), s = sin(angle);
    *y0 = x0 * c - x1 * s;
    *y1 = x0 * s + x1 * c;
}

/* ---- Fused QKV projection + RoPE ----------------------------------------
 * [T] §QKV投影融合: [Q|K|V] = X Wqkv^T + bqkv with Q = columns [0, d),
 * K = [d, 2d), V = [2d, 3d), here d = n_heads * head_dim.
 * [E] §用形状与步长把约定钉死: rotation happens inside the epilogue, so the
 * K section is written already rotated; V is not rotated.
 * out[i, j] is column cols[j] of [Q|K|V] for row i, whose position is pos[i].
 */
void orc_qkv_rope(const double* X, long nrows, const double* Wqkv, const double* bqkv, long K,
                  long n_heads, long head_dim, double theta, const double* pos,
                  const long* cols, long ncols, double* out) {
    const long d_model = n_heads * head_dim;
#pragma omp parallel for collapse(2) schedule(static)
    for (long i = 0; i < nrows; ++i) {
        for (long j = 0; j < ncols; ++j) {
            const double* x = X + (size_t)i * (size_t)K;
            long c = cols[j];
            long section = c / d_model;
            long d = (c % d_model) % head_dim;
            if (section == 2) {
                out[i * ncols + j] = linear_at(x, Wqkv, bqkv, K, c);
                continue;
            }
            long c0 = c - (d & 1);
            double x0 = linear_at(x, Wqkv, bqkv, K, c0);
            double x1 = linear_at(x, Wqkv, bqkv, K, c0 + 1);
            double y0, y1;
            orc_rope_rotate(x0, x1, orc_rope_angle(pos[i], d / 2, head_dim, theta), &y0, &y1);
            out[i * ncols + j] = (d & 1) ? y1 : y0;
        }
    }
}

/* ---- SwiGLU --------------------------------------------------------------
 * [E] §模式 B / §末尾布局调整: gate g and value u of the same output feature
 * give one value, y = SiLU(g) * u with SiLU(g) = g / (1 + e^{-g}); the output
 * has half the width of the [gate | up] product.
 */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

void orc_swiglu(const double* X, long nrows, const double* Wg, const double* Wu,
                const double* bg, const double* bu, long K, const long* cols, long ncols,
                double* out) {
#pragma omp parallel for collapse(2) schedule(static)
    for (long i = 0; i < nrows; ++i)
        for (long j = 0; j < ncols; ++j) {
            const double* x = X + (size_t)i * (size_t)K;
            double g = linear_at(x, Wg, bg, K, cols[j]);
            double u = linear_at(x, Wu, bu, K, cols[j]);
            out[i * ncols + j] = orc_silu(g) * u;
        }
}

/* ---- FP8 E4M3 (OCP 8-bit floating point, E4M3FN variant) -----------------
 * sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities; the
 * only NaN magnitude is S.1111.111; largest finite 448; subnormals m * 2^-9.
 */
double orc_e4m3_decode(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* [E] §仿射量化与尾声的五步, step 2: round to the nearest representable value
 * (ties to the even mantissa) and clamp to [-448, 448].  Written as a search
 * over the 127 non-negative finite codes, nearest first, even code on a tie. */
int orc_e4m3_encode(double y) {
    if (isnan(y)) return 0x7F;
    int s = signbit(y) ? 1 : 0;
    double a = fabs(y);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_decode(c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (s << 7) | best;
}

void orc_e4m3_encode_array(const double* y, long n, uint8_t* q) {
    for (long i = 0; i < n; ++i) q[i] = (uint8_t)orc_e4m3_encode(y[i]);
}

void orc_e4m3_decode_array(const uint8_t* q, long n, double* y) {
    for (long i = 0; i < n; ++i) y[i] = orc_e4m3_decode(q[i]);
}

/* ---- Down projection + residual + RMSNorm + FP8 write-back --------------
 * [E] §模式 A: h = X W^T (+ b) + z; r = 1 / sqrt(mean_n h^2 + eps) is one
 * scalar per row; y = r * h (.) gamma.
 * [E] §仿射量化与尾声的五步, steps 1, 2 and 5 with one block per row:
 * s = max_n |y| / 448; q = e4m3(y / s); s is written beside q.  A row whose
 * maximum is 0 gets s = 0 and all-zero codes.
 * Outputs: q [nrows, N] codes, scale [nrows], y [nrows, N] (pre-quantisation).
 */
void orc_rmsnorm_fp8(const double* X, long nrows, const double* W, const double* b,
                     const double* Z, const double* gamma, long N, long K, double eps,
                     uint8_t* q, double* scale, double* y) {
    for (long i = 0; i < nrows; ++i) {
        const double* x = X + (size_t)i * (size_t)K;
        double* yi = y + (size_t)i * (size_t)N;
#pragma omp parallel for schedule(static)
        for (long n = 0; n < N; ++n) yi[n] = linear_at(x, W, b, K, n) + Z[(size_t)i * N + n];
        double ss = 0.0;
        for (long n = 0; n < N; ++n) ss += yi[n] * yi[n];
        double r = 1.0 / sqrt(ss / (double)N + eps);
        double amax = 0.0;
        for (long n = 0; n < N; ++n) {
            yi[n] = yi[n] * gamma[n] * r;
            if (fabs(yi[n]) > amax) amax = fabs(yi[n]);
        }
        scale[i] = amax / 448.0;
        for (long n = 0; n < N; ++n)
            q[(size_t)i * N + n] = amax > 0.0 ? (uint8_t)orc_e4m3_encode(yi[n] / scale[i]) : 0;
    }
}

/* ---- GEMM -> residual -> RMSNorm -> GEMM --------------------------------
 * [E] §模式 A: y = RMSNorm(x W0^T (+ b0) + z, gamma) W1^T (+ b1), i.e.
 * h1 = x W0^T + b0 + z,  r = 1 / sqrt(mean_n h1^2 + eps),  v = r * h1 (.) gamma,
 * y[j] = sum_n v[n] W1[j, n] + b1[j].  Written in that plain order (the
 * reparameterised order of the kernels is what the tests compare against it).
 * Also returns h1 (the residual stream after the add).
 * X [nrows, K], W0 [N, K], Z [nrows, N], gamma [N], W1 [N2, N]; out y [nrows, N2], h1 [nrows, N].
 */
void orc_residual_rmsnorm_linear(const double* X, long nrows, const double* W0, const double* b0,
                                 const double* Z, const double* gamma, long N, long K, double eps,
                                 const double* W1, const double* b1, long N2, double* y, double* h1) {
    for (long i = 0; i < nrows; ++i) {
        const double* x = X + (size_t)i * (size_t)K;
        double* hi = h1 + (size_t)i * (size_t)N;
#pragma omp parallel for schedule(static)
        for (long n = 0; n < N; ++n) hi[n] = linear_at(x, W0, b0, K, n) + Z[(size_t)i * N + n];
        double ss = 0.0;
        for (long n = 0; n < N; ++n) ss += hi[n] * hi[n];
        const double r = 1.0 / sqrt(ss / (double)N + eps);
        double* v = (double*)malloc((size_t)N * sizeof(double));
        for (long n = 0; n < N; ++n) v[n] = r * hi[n] * gamma[n];
#pragma omp parallel for schedule(static)
        for (long j = 0; j < N2; ++j) y[(size_t)i * N2 + j] = linear_at(v, W1, b1, N, j);
        free(v);
    }
}

/* ---- LM-head cross-entropy ----------------------------------------------
 * [E] §模式 C: logits h_i = x_i W^T (+ b) over the vocabulary, and
 * loss_i = -h_{i, y_i} + log sum_k exp(h_{i, k}); the log-sum-exp is evaluated in
 * the usual shifted form m + log sum_k exp(h_k - m) with m = max_k h_k.
 * A negative label marks an ignored row (loss 0).  X [nrows, K], W [V, K].
 */
void orc_linear_cross_entropy(const double* X, long nrows, const double* W, const double* b, long V, long K,
                              const long* labels, double* loss) {
    for (long i = 0; i < nrows; ++i) {
        const double* x = X + (size_t)i * (size_t)K;
        double* h = (double*)malloc((size_t)V * sizeof(double));
#pragma omp parallel for schedule(static)
        for (long v = 0; v < V; ++v) h[v] = linear_at(x, W, b, K, v);
        if (labels[i] < 0) {
            loss[i] = 0.0;
        } else if (labels[i] >= V) {
            loss[i] = NAN;
        } else {
            double m = -INFINITY;
            for (long v = 0; v < V; ++v) m = h[v] > m ? h[v] : m;
            double s = 0.0;
            for (long v = 0; v < V; ++v) s += exp(h[v] - m);
            loss[i] = m + log(s) - h[labels[i]];
        }
        free(h);
    }
}

/* ---- Block-scaled quantised write-back ------------------------------------
 * [E] §仿射量化与尾声的五步: per block, (1) s = max|x| / qmax, (2) q = round(x / s)
 * clamped to [-qmax, qmax], (4) compact layout, (5) the scale written beside the codes.
 * A block whose maximum is 0 gets s = 0 and zero codes.
 *
 * FP4 E2M1 (OCP microscaling formats): sign, 2 exponent bits (bias 1), 1 mantissa
 * bit; exponent 0 is subnormal (m * 0.5); largest finite 6; no inf / NaN.
 */
double orc_e2m1_decode(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Nearest of the 8 non-negative codes (even code on a tie), saturating at 6. */
int orc_e2m1_encode(double y) {
    int s = signbit(y) ? 1 : 0;
    double a = fabs(y);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 7; ++c) {
        double d = fabs(orc_e2m1_decode(c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (s << 3) | best;
}

/* Linear followed by block-scaled quantisation of every row.
 * Step 3 of [E] §仿射量化与尾声的五步 (optional scale-factor correction): when the
 * activation leaves a SmoothQuant/QuaRot-style smoothed layer, the epilogue multiplies it
 * by the inverse smoothing coefficient before quantising, so the codes hold what the next
 * kernel expects.  Here that is a per-output-column factor: y[n] <- y[n] * inv_smooth[n]
 * (NULL: no correction), applied before the block maximum of step 1, since the codes and
 * the scale must describe the corrected values.
 * fmt 0: FP8 E4M3, blocks of 128 columns, fp32 scale = amax / 448, codes 1 byte each.
 * fmt 1: INT4 symmetric, groups of 32, fp32 scale = amax / 7, code = round-half-even(y / s)
 *        clamped to [-7, 7], two's-complement nibble; column 2j in the low nibble of byte j.
 * fmt 2: NVFP4, groups of 16, scale = E4M3 code of amax / 6 (the stored scale is what the
 *        codes are divided by), values E2M1, column 2j in the low nibble of byte j.
 * Outputs: q [nrows, qbytes_per_row] (qbytes = N for fmt 0, N/2 otherwise),
 *          scale [nrows, nblocks] as fp64 (fmt 0, 1) or as E4M3 codes widened to fp64 (fmt 2),
 *          y [nrows, N] the unquantised (corrected) Linear output. */
void orc_linear_quant(const double* X, long nrows, const double* W, const double* b, long N, long K, int fmt,
                      const double* inv_smooth, uint8_t* q, double* scale, double* y) {
    const long bs = fmt == 0 ? 128 : (fmt == 1 ? 32 : 16);
    const long nblocks = (N + bs - 1) / bs;
    const long qbytes = fmt == 0 ? N : (N + 1) / 2;
    for (long i = 0; i < nrows; ++i) {
        const double* x = X + (size_t)i * (size_t)K;
        double* yi = y + (size_t)i * (size_t)N;
#pragma omp parallel for schedule(static)
        for (long n = 0; n < N; ++n) yi[n] = linear_at(x, W, b, K, n);
        if (inv_smooth)
            for (long n = 0; n < N; ++n) yi[n] *= inv_smooth[n];
        uint8_t* qi = q + (size_t)i * (size_t)qbytes;
        for (long n = 0; n < qbytes; ++n) qi[n] = 0;
        for (long blk = 0; blk < nblocks; ++blk) {
            const long c0 = blk * bs, c1 = c0 + bs < N ? c0 + bs : N;
            double amax = 0.0;
            for (long n = c0; n < c1; ++n) amax = fabs(yi[n]) > amax ? fabs(yi[n]) : amax;
            double s;
            if (fmt == 0) s = amax / 448.0;
            else if (fmt == 1) s = amax / 7.0;
            else s = orc_e4m3_decode(orc_e4m3_encode(amax / 6.0));
            scale[i * nblocks + blk] = fmt == 2 ? (double)orc_e4m3_encode(amax / 6.0) : s;
            for (long n = c0; n < c1; ++n) {
                const double v = s > 0.0 ? yi[n] / s : 0.0;
                if (fmt == 0) {
                    qi[n] = s > 0.0 ? (uint8_t)orc_e4m3_encode(v) : 0;
                } else {
                    int nib;
                    if (fmt == 1) {
                        double r = nearbyint(v);  /* default rounding mode: to nearest, ties to even */
                        if (r > 7.0) r = 7.0;
                        if (r < -7.0) r = -7.0;
                        nib = ((int)r) & 15;
                    } else {
                        nib = s > 0.0 ? orc_e2m1_encode(v) : 0;
                    }
                    qi[n / 2] |= (uint8_t)(nib << (4 * (n & 1)));
                }
            }
        }
    }
}

/* ---- QKV projection + RoPE with the K/V cache written in FP8 -------------
 * [E] §一个瓦片的字节账 (the decode K/V write-back quantised to FP8 in the epilogue,
 * halving its bytes) with the scale of [E] §仿射量化与尾声的五步 taken over one
 * head's head_dim values of one token (a 1 x head_dim block; head_dim 128 gives
 * the 1 x 128 blocks of fine-grained FP8 scaling).
 * Widths: Q = n_heads * head_dim, K = V = n_kv_heads * head_dim (grouped-query
 * attention when n_kv_heads < n_heads); the rows of Wqkv are [Q | K | V].
 * Q and K are rotated as in orc_qkv_rope ([T] §QKV投影融合, adjacent pairs);
 * V is not.  Q stays unquantised (fp64 out).  For K and V, per (row, kv head):
 * s = max|y| / 448 over the head, codes e4m3(y / s); a head whose maximum is 0
 * gets s = 0 and zero codes.
 * Outputs: q [nrows, n_heads*head_dim] fp64; kq, vq [nrows, n_kv_heads*head_dim]
 * E4M3 codes; ks, vs [nrows, n_kv_heads] scales; kv [nrows, 2*n_kv_heads*head_dim]
 * the unquantised rotated K then V (for error bounds in the tests). */
void orc_qkv_rope_kv_fp8(const double* X, long nrows, const double* Wqkv, const double* bqkv, long K,
                         long n_heads, long n_kv_heads, long head_dim, double theta, const double* pos,
                         double* q, uint8_t* kq, double* ks, uint8_t* vq, double* vs, double* kv) {
    const long qw = n_heads * head_dim, kvw = n_kv_heads * head_dim;
    const long width = qw + 2 * kvw;
    double* row = (double*)malloc((size_t)width * sizeof(double));
    for (long i = 0; i < nrows; ++i) {
        const double* x = X + (size_t)i * (size_t)K;
#pragma omp parallel for schedule(static)
        for (long c = 0; c < width; ++c) row[c] = linear_at(x, Wqkv, bqkv, K, c);
        /* rotate every adjacent pair of the Q and K sections */
        for (long c = 0; c < qw + kvw; c += 2) {
            const long d = (c < qw ? c : c - qw) % head_dim;
            double y0, y1;
            orc_rope_rotate(row[c], row[c + 1], orc_rope_angle(pos[i], d / 2, head_dim, theta), &y0, &y1);
            row[c] = y0;
            row[c + 1] = y1;
        }
        for (long c = 0; c < qw; ++c) q[(size_t)i * (size_t)qw + (size_t)c] = row[c];
        for (long c = 0; c < 2 * kvw; ++c) kv[(size_t)i * (size_t)(2 * kvw) + (size_t)c] = row[qw + c];
        for (long sec = 0; sec < 2; ++sec) {
            const double* y = row + qw + sec * kvw;
            uint8_t* codes = (sec == 0 ? kq : vq) + (size_t)i * (size_t)kvw;
            double* scale = (sec == 0 ? ks : vs) + (size_t)i * (size_t)n_kv_heads;
            for (long h = 0; h < n_kv_heads; ++h) {
                double amax = 0.0;
                for (long d = 0; d < head_dim; ++d) {
                    const double a = fabs(y[h * head_dim + d]);
                    amax = a > amax ? a : amax;
                }
                const double sc = amax / 448.0;
                scale[h] = sc;
                for (long d = 0; d < head_dim; ++d)
                    codes[h * head_dim + d] = sc > 0.0 ? (uint8_t)orc_e4m3_encode(y[h * head_dim + d] / sc) : 0;
            }
        }
    }
    free(row);
}

/* ---- Backward epilogues ---------------------------------------------------
 * [E] §模式 D: for blocks h = x W, x' = f(h) with f acting per element, the
 * backward pass has the same shape: the gradient w.r.t. the block input is a
 * GEMM with the weight, and multiplying by f'(h) is an element-wise step that
 * belongs in the epilogue of the GEMM producing that gradient.
 * With W stored [n_out, n_in] (one row per output feature, as in orc_linear),
 * the gradient w.r.t. the input x is dX[m, n] = sum_k dZ[m, k] W[k, n], k over
 * the n_out outputs: the contraction runs over W's rows. */

/* d/dx of the erf form: Phi(x) + x phi(x), phi(x) = exp(-x^2/2) / sqrt(2 pi). */
double orc_gelu_erf_grad(double x) {
    return 0.5 * (1.0 + erf(x / sqrt(2.0))) + x * exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
}

/* d/dx of the tanh form with u = c (x + a x^3), c = sqrt(2/pi), a = 0.044715:
 * 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) c (1 + 3 a x^2). */
double orc_gelu_tanh_grad(double x) {
    const double c = sqrt(2.0 / M_PI), a = 0.044715;
    const double t = tanh(c * (x + a * x * x * x));
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * c * (1.0 + 3.0 * a * x * x);
}

/* dgrad with W as stored: acc[i, n] = sum_k dZ[i, k] W[k, n] (k in order). */
static double dgrad_at(const double* dz_row, const double* W, long Kp, long N, long n) {
    double s = 0.0;
    for (long k = 0; k < Kp; ++k) s += dz_row[k] * W[(size_t)k * (size_t)N + (size_t)n];
    return s;
}

/* GELU backward fused into the dgrad GEMM: dH[i, n] = (dZ W)[i, n] * GELU'(H[i, n])
 * (mode 0 = erf form, 1 = tanh form).  dZ [nrows, Kp], W [Kp, N], H [nrows, N] the
 * saved pre-activation; out [nrows, ncols] at the columns cols. */
void orc_dgrad_gelu(const double* dZ, long nrows, const double* W, long Kp, long N, const double* H, int mode,
                    const long* cols, long ncols, double* out) {
#pragma omp parallel for collapse(2) schedule(static)
    for (long i = 0; i < nrows; ++i)
        for (long j = 0; j < ncols; ++j) {
            const long n = cols[j];
            const double h = H[(size_t)i * (size_t)N + (size_t)n];
            const double d = mode == 0 ? orc_gelu_erf_grad(h) : orc_gelu_tanh_grad(h);
            out[i * ncols + j] = dgrad_at(dZ + (size_t)i * (size_t)Kp, W, Kp, N, n) * d;
        }
}

/* SwiGLU backward, [E] §末尾布局调整 (SwiGLU 反向): y = SiLU(g) u, so with the upstream
 * gradient dy = (dO W_down)[i, n] of y,
 *   dg = dy * u * SiLU'(g),  SiLU'(g) = s (1 + g (1 - s)),  s = 1 / (1 + e^{-g}),
 *   du = dy * SiLU(g).
 * One input value gives two outputs: the result is twice as wide, the pair of feature n
 * at columns 2n (dg) and 2n + 1 (du).  dO [nrows, Kp], Wd [Kp, N], G and U [nrows, N]
 * the saved gate and up activations; out [nrows, 2 ncols] for the features cols. */
void orc_swiglu_bwd(const double* dO, long nrows, const double* Wd, long Kp, long N, const double* G,
                    const double* U, const long* cols, long ncols, double* out) {
#pragma omp parallel for collapse(2) schedule(static)
    for (long i = 0; i < nrows; ++i)
        for (long j = 0; j < ncols; ++j) {
            const long n = cols[j];
            const double g = G[(size_t)i * (size_t)N + (size_t)n];
            const double u = U[(size_t)i * (size_t)N + (size_t)n];
            const double dy = dgrad_at(dO + (size_t)i * (size_t)Kp, Wd, Kp, N, n);
            const double s = 1.0 / (1.0 + exp(-g));
            out[i * 2 * ncols + 2 * j] = dy * u * s * (1.0 + g * (1.0 - s));
            out[i * 2 * ncols + 2 * j + 1] = dy * g * s;
        }
}

/* Number of OpenMP threads the parallel loops above use. */
int orc_num_threads(void) {
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
