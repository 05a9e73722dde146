"""Pins for the fp64 oracle: each check ties it to something other than itself.

Kinds of pin used here: hand sums and brute force on tiny inputs, closed
forms and identities of the mathematics, library routines computing the same
quantity by another route (scipy, torch fp64 CPU ops, torch's float8 type),
and constants printed on the pages (tests/golden/).  Each is chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign, a swapped index or
operand, a wrong exponent) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            vals[parts[0]] = [float(p) for p in parts[1:]]
    return vals


# --------------------------------------------------------------------- Linear
def test_linear_hand_sum():
    # Y = X W^T + b, hand-summed: rows of X times rows of W.
    X = np.array([[1, 2, 3], [4, 5, 6]], float)
    W = np.array([[1, 0, -1], [2, 1, 0]], float)
    b = np.array([10, 20], float)
    Y = oracle.linear(X, W, b)
    assert Y.tolist() == [[8.0, 24.0], [8.0, 33.0]]


def test_linear_brute_force_nonsquare():
    rng = np.random.default_rng(1)
    X = rng.integers(-4, 5, size=(4, 8)).astype(float)
    W = rng.integers(-4, 5, size=(5, 8)).astype(float)   # N=5 != M=4 != K=8
    b = rng.integers(-4, 5, size=5).astype(float)
    ref = [[sum(X[m, k] * W[n, k] for k in range(8)) + b[n] for n in range(5)] for m in range(4)]
    assert oracle.linear(X, W, b).tolist() == ref
    # column subset selection keeps the requested order
    assert oracle.linear(X, W, b, cols=[3, 0]).tolist() == [[r[3], r[0]] for r in ref]


def test_linear_special_cases():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((3, 6))
    assert np.array_equal(oracle.linear(X, np.eye(6)), X)              # identity W returns X
    x1, w1 = rng.standard_normal((5, 1)), rng.standard_normal((7, 1))
    assert np.allclose(oracle.linear(x1, w1), np.outer(x1[:, 0], w1[:, 0]), rtol=0, atol=0)  # K=1
    assert np.all(oracle.linear(np.ones((2, 9)), np.ones((3, 9))) == 9.0)  # all-ones gives K
    Xb, Wb = rng.standard_normal((16, 40)), rng.standard_normal((24, 40))
    assert np.allclose(oracle.linear(Xb, Wb), Xb @ Wb.T, rtol=1e-13, atol=1e-13)  # library matmul


# ----------------------------------------------------------------------- GELU
def test_gelu_closed_forms():
    for mode in (oracle.GELU_ERF, oracle.GELU_TANH):
        g = oracle.gelu(np.array([0.0, 10.0, -10.0, 50.0]), mode)
        assert g[0] == 0.0
        assert abs(g[1] - 10.0) < 1e-15
        assert abs(g[2]) < 1e-20
        assert g[3] == 50.0
    # erf form equals x * Phi(x); Phi from scipy's normal CDF (independent route)
    from scipy.special import ndtr
    x = np.linspace(-8, 8, 2001)
    assert np.allclose(oracle.gelu(x, oracle.GELU_ERF), x * ndtr(x), rtol=1e-14, atol=1e-14)
    assert oracle.gelu_erf(1.0) == pytest.approx(0.8413447460685429, rel=1e-15, abs=0)


def test_gelu_matches_torch_fp64():
    x = torch.linspace(-12, 12, 4801, dtype=torch.float64)
    e = F.gelu(x).numpy()
    t = F.gelu(x, approximate="tanh").numpy()
    assert np.allclose(oracle.gelu(x.numpy(), oracle.GELU_ERF), e, rtol=1e-14, atol=1e-15)
    assert np.allclose(oracle.gelu(x.numpy(), oracle.GELU_TANH), t, rtol=1e-14, atol=1e-15)


def test_gelu_printed_constants():
    g = _golden("gelu_constants.txt")
    x = np.linspace(-6, 6, 1201)
    from scipy.special import erf
    printed_erf = 0.5 * x * (1.0 + erf(x * g["erf_arg_scale"][0]))
    assert np.max(np.abs(oracle.gelu(x, oracle.GELU_ERF) - printed_erf)) < 1e-8
    c, a = g["tanh_arg_scale"][0], g["tanh_cubic"][0]
    printed_tanh = 0.5 * x * (1.0 + np.tanh(c * (x + a * x ** 3)))
    assert np.max(np.abs(oracle.gelu(x, oracle.GELU_TANH) - printed_tanh)) < 1e-9


def test_gelu_erf_tanh_gap():
    g = _golden("gelu_constants.txt")
    x = np.linspace(-10, 10, 200001)
    gap = np.abs(oracle.gelu(x, oracle.GELU_ERF) - oracle.gelu(x, oracle.GELU_TANH))
    # "about 1e-3": the largest gap lies within one decade below the printed order
    order = g["erf_tanh_gap_order"][0]
    assert order / 10 < gap.max() < order
    assert gap.max() == pytest.approx(4.73e-4, rel=0.01)
    assert abs(x[np.argmax(gap)] + 2.70) < 0.05


def test_gelu_tanh_bracket():
    # 1 + tanh(z) lies in (0, 2): gelu_tanh(x) / x lies in (0, 1) for x != 0
    x = np.concatenate([np.linspace(-20, -1e-3, 500), np.linspace(1e-3, 20, 500)])
    r = oracle.gelu(x, oracle.GELU_TANH) / x
    assert np.all(r >= 0) and np.all(r <= 1)


# ----------------------------------------------------------------------- RoPE
def test_rope_angle_and_sign():
    assert oracle.rope_angle(0, 5, 128, 1e4) == 0.0
    assert oracle.rope_angle(1, 0, 128, 1e4) == 1.0                  # pair 0: 1 rad per position
    assert oracle.rope_angle(100, 32, 128, 1e4) == pytest.approx(1.0, rel=1e-15)  # 1e4^(-64/128)=0.01
    assert oracle.rope_angle(1, 63, 128, 1e4) == pytest.approx(1e4 ** (-126 / 128), rel=1e-15)
    y0, y1 = oracle.rope_rotate(1.0, 0.0, 1.0)
    assert (y0, y1) == pytest.approx((math.cos(1), math.sin(1)), abs=1e-16)
    y0, y1 = oracle.rope_rotate(0.0, 1.0, 1.0)
    assert (y0, y1) == pytest.approx((-math.sin(1), math.cos(1)), abs=1e-16)


def test_rope_invariants():
    rng = np.random.default_rng(3)
    for _ in range(200):
        x0, x1, a, b = rng.standard_normal(4) * [1, 1, 50, 50]
        y0, y1 = oracle.rope_rotate(x0, x1, a)
        assert math.hypot(y0, y1) == pytest.approx(math.hypot(x0, x1), abs=1e-12)   # norm kept
        z0, z1 = oracle.rope_rotate(y0, y1, b)
        w0, w1 = oracle.rope_rotate(x0, x1, a + b)                                 # R(a)R(b)=R(a+b)
        assert (z0, z1) == pytest.approx((w0, w1), abs=1e-11)


def _rope_torch_complex(v, pos, head_dim, theta):
    """RoPE as complex multiplication (independent formulation): [M, H*D] fp64."""
    M = v.shape[0]
    t = torch.from_numpy(v).reshape(M, -1, head_dim // 2, 2)
    z = torch.view_as_complex(t.contiguous())
    i = torch.arange(head_dim // 2, dtype=torch.float64)
    freq = theta ** (-2.0 * i / head_dim)
    ang = torch.from_numpy(np.asarray(pos, float))[:, None] * freq[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return torch.view_as_real(z * rot).reshape(M, -1).numpy()


def test_qkv_rope_composite_against_complex_rotation():
    rng = np.random.default_rng(4)
    M, K, H, D = 5, 24, 2, 16
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((3 * H * D, K)) / math.sqrt(K)
    b = rng.standard_normal(3 * H * D) * 0.02
    pos = np.array([0, 1, 7, 2047, 300])
    out = oracle.qkv_rope(X, W, b, H, D, 10000.0, pos)
    plain = X @ W.T + b
    d = H * D
    assert np.allclose(out[:, 2 * d:], plain[:, 2 * d:], rtol=1e-13, atol=1e-13)       # V untouched
    assert np.allclose(out[0], plain[0], rtol=1e-13, atol=1e-13)                       # pos 0
    assert np.allclose(out[:, :d], _rope_torch_complex(plain[:, :d], pos, D, 1e4), atol=1e-12)
    assert np.allclose(out[:, d:2 * d], _rope_torch_complex(plain[:, d:2 * d], pos, D, 1e4), atol=1e-12)
    # relative position: <RoPE(q, m), RoPE(k, n)> depends only on m - n
    q, k = plain[1, :D], plain[1, d:d + D]
    def dot_at(m, n):
        a = _rope_torch_complex(q[None], [m], D, 1e4)[0]
        c = _rope_torch_complex(k[None], [n], D, 1e4)[0]
        return float(a @ c)
    assert dot_at(10, 3) == pytest.approx(dot_at(107, 100), abs=1e-10)


# --------------------------------------------------------------------- SwiGLU
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(50.0) == pytest.approx(50.0, abs=1e-18)
    assert abs(oracle.silu(-50.0)) < 1e-18
    for x in np.linspace(-9, 9, 37):
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, abs=1e-14)   # x*s(x) - (-x)s(-x) = x


def test_swiglu_matches_torch_fp64():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((6, 32))
    Wg, Wu = rng.standard_normal((10, 32)) / 6, rng.standard_normal((10, 32)) / 6
    bg, bu = rng.standard_normal(10) * 0.02, rng.standard_normal(10) * 0.02
    Xt = torch.from_numpy(X)
    ref = (F.silu(Xt @ torch.from_numpy(Wg).T + torch.from_numpy(bg))
           * (Xt @ torch.from_numpy(Wu).T + torch.from_numpy(bu))).numpy()
    assert np.allclose(oracle.swiglu(X, Wg, Wu, bg, bu), ref, rtol=1e-13, atol=1e-14)
    # u == 1 reduces SwiGLU to SiLU of the gate projection
    ones = oracle.swiglu(X, Wg, np.zeros_like(Wu), bg, np.ones(10))
    assert np.allclose(ones, F.silu(Xt @ torch.from_numpy(Wg).T + torch.from_numpy(bg)).numpy(),
                       rtol=1e-14, atol=1e-15)
    # gate and up are not interchangeable
    assert not np.allclose(oracle.swiglu(X, Wu, Wg, bu, bg), oracle.swiglu(X, Wg, Wu, bg, bu))


# ------------------------------------------------------------------------ FP8
def test_e4m3_decode_table():
    d = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert d[0x00] == 0.0 and d[0x01] == 2.0 ** -9 and d[0x07] == 7 * 2.0 ** -9
    assert d[0x08] == 2.0 ** -6 and d[0x38] == 1.0 and d[0x7E] == 448.0
    assert math.isnan(d[0x7F]) and math.isnan(d[0xFF])
    assert d[0xFE] == -448.0 and d[0x80] == 0.0 and math.copysign(1, d[0x80]) < 0
    # library decode of the same bytes (torch's float8_e4m3fn type)
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fin = ~np.isnan(t)
    assert np.array_equal(np.isnan(d), ~fin) and np.array_equal(d[fin], t[fin])


def test_e4m3_encode_round_trip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
    enc = lambda v: int(oracle.e4m3_encode(np.array([v]))[0])
    assert enc(1.0625) == 0x38          # midpoint 1 | 1.125 -> even mantissa (1.0)
    assert enc(1.1875) == 0x3A          # midpoint 1.125 | 1.25 -> even mantissa (1.25)
    assert enc(2.0 ** -10) == 0x00      # midpoint 0 | 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02  # midpoint 2^-9 | 2^-8 -> code 2
    assert enc(449.0) == 0x7E and enc(1e6) == 0x7E and enc(-500.0) == 0xFE
    assert enc(-1e-6) == 0x80


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(6)
    v = np.concatenate([rng.standard_normal(20000) * 40, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(5000) * 1e-2]).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v.astype(np.float64)), lib)


# -------------------------------------------------------------------- RMSNorm
def _rms_case(seed, r=4, N=96, K=40, with_b=True):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((r, K))
    W = rng.standard_normal((N, K)) / math.sqrt(K)
    b = rng.standard_normal(N) * 0.02 if with_b else None
    Z = rng.standard_normal((r, N))
    g = 1.0 + 0.1 * rng.standard_normal(N)
    return X, W, b, Z, g


def test_rmsnorm_matches_torch_fp64():
    X, W, b, Z, g = _rms_case(7)
    q, s, y = oracle.rmsnorm_fp8(X, W, b, Z, g, 1e-6)
    h = torch.from_numpy(X @ W.T + b + Z)
    ref = F.rms_norm(h, (W.shape[0],), weight=torch.from_numpy(g), eps=1e-6).numpy()
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-14)
    assert np.allclose(s, np.abs(ref).max(axis=1) / 448.0, rtol=1e-14)
    lib = torch.from_numpy((ref / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
    lib = lib.view(torch.uint8).numpy()
    assert np.mean(lib == q) > 0.999


def test_rmsnorm_unit_rms_and_invariance():
    X, W, b, Z, _ = _rms_case(8, r=3, N=128)
    ones = np.ones(128)
    _, _, y = oracle.rmsnorm_fp8(X, W, b, Z, ones, 1e-6)
    rms = np.sqrt(np.mean(y ** 2, axis=1))
    assert np.all(np.abs(rms - 1.0) < 1e-6)
    # with X = 0 the row is the residual alone; scaling it leaves the output unchanged
    zX = np.zeros_like(X)
    _, _, y1 = oracle.rmsnorm_fp8(zX, W, None, Z, ones, 1e-12)
    _, _, y2 = oracle.rmsnorm_fp8(zX, W, None, 7.5 * Z, ones, 1e-12)
    assert np.allclose(y1, y2, rtol=1e-10, atol=1e-12)
    # constant row c: every output equals sign(c) / sqrt(1 + eps / c^2)
    c = -0.3
    _, _, yc = oracle.rmsnorm_fp8(zX[:1], W, None, np.full((1, 128), c), ones, 1e-6)
    assert np.allclose(yc, -1.0 / math.sqrt(1 + 1e-6 / c ** 2), rtol=1e-14)


def test_rmsnorm_fp8_codes_and_scale():
    X, W, b, Z, g = _rms_case(9, r=5, N=200)
    q, s, y = oracle.rmsnorm_fp8(X, W, b, Z, g, 1e-6)
    for i in range(5):
        j = int(np.argmax(np.abs(y[i])))
        assert q[i, j] == (0xFE if y[i, j] < 0 else 0x7E)          # row maximum maps to +-448
    deq = oracle.e4m3_decode(q) * s[:, None]
    assert np.all(np.abs(deq - y) <= np.maximum(np.abs(y) * 2.0 ** -4, s[:, None] * 2.0 ** -9) + 1e-15)
    # a zero row gives scale 0 and zero codes
    q0, s0, _ = oracle.rmsnorm_fp8(np.zeros((1, 40)), W, None, np.zeros((1, 200)), g, 1e-6)
    assert s0[0] == 0.0 and not q0.any()


# ------------------------------------------------ GEMM -> residual -> RMSNorm -> GEMM
def test_residual_rmsnorm_linear_matches_torch_fp64():
    rng = np.random.default_rng(10)
    r, K, N, N2 = 4, 48, 64, 40
    X = rng.standard_normal((r, K))
    W0, W1 = rng.standard_normal((N, K)) / math.sqrt(K), rng.standard_normal((N2, N)) / math.sqrt(N)
    b0, b1 = rng.standard_normal(N) * 0.02, rng.standard_normal(N2) * 0.02
    Z, g = rng.standard_normal((r, N)), 1.0 + 0.1 * rng.standard_normal(N)
    y, h1 = oracle.residual_rmsnorm_linear(X, W0, b0, Z, g, 1e-6, W1, b1)
    t = lambda a: torch.from_numpy(a)
    h = F.linear(t(X), t(W0), t(b0)) + t(Z)
    ref = F.linear(F.rms_norm(h, (N,), weight=t(g), eps=1e-6), t(W1), t(b1)).numpy()
    assert np.allclose(h1, h.numpy(), rtol=1e-13, atol=1e-13)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)
    # the row scale is one scalar per row: it commutes with the second GEMM (the deferral the kernels use)
    rr = 1.0 / np.sqrt(np.mean(h1 ** 2, axis=1) + 1e-6)
    deferred = rr[:, None] * ((h1 * g) @ W1.T) + b1
    assert np.allclose(y, deferred, rtol=1e-12, atol=1e-13)
    # a per-column factor does not commute: moving gamma after W1 changes the result
    assert not np.allclose(y, rr[:, None] * (h1 @ W1.T) * g[:N2] + b1, rtol=1e-3, atol=1e-3)


# ------------------------------------------------------------- LM-head cross-entropy
def test_cross_entropy_matches_torch_and_closed_forms():
    rng = np.random.default_rng(11)
    r, K, V = 6, 32, 300
    X = rng.standard_normal((r, K))
    W = rng.standard_normal((V, K)) / math.sqrt(K)
    b = rng.standard_normal(V) * 0.1
    y = rng.integers(0, V, size=r)
    loss = oracle.linear_cross_entropy(X, W, b, y)
    logits = F.linear(torch.from_numpy(X), torch.from_numpy(W), torch.from_numpy(b))
    ref = F.cross_entropy(logits, torch.from_numpy(y), reduction="none").numpy()
    assert np.allclose(loss, ref, rtol=1e-13, atol=1e-13)
    # uniform logits: loss = log V exactly; a dominant label logit: loss -> 0
    assert np.allclose(oracle.linear_cross_entropy(X, np.zeros((V, K)), None, y), math.log(V), rtol=0, atol=1e-13)
    bb = np.zeros(V)
    bb[7] = 60.0
    assert oracle.linear_cross_entropy(X[:1], np.zeros((V, K)), bb, [7])[0] < 1e-20
    # large logits do not overflow (shifted form), ignored and out-of-range labels
    big = oracle.linear_cross_entropy(X[:1], W * 1e3, None, [3])[0]
    assert np.isfinite(big) and big >= 0
    assert oracle.linear_cross_entropy(X[:2], W, b, [-100, V])[0] == 0.0
    assert math.isnan(oracle.linear_cross_entropy(X[:2], W, b, [-100, V])[1])


def test_online_lse_merge_matches_library():
    # the per-tile (m, s) merge the kernel uses reproduces torch.logsumexp over the whole row
    rng = np.random.default_rng(12)
    h = rng.standard_normal(1000) * 5
    m, s = -np.inf, 0.0
    for tile in np.array_split(h, 7):
        mt, st = tile.max(), np.exp(tile - tile.max()).sum()
        mn = max(m, mt)
        s = s * math.exp(m - mn) + st * math.exp(mt - mn)
        m = mn
    assert m + math.log(s) == pytest.approx(torch.logsumexp(torch.from_numpy(h), 0).item(), rel=1e-14)


# ------------------------------------------------------- block-scaled quantised write-back
def test_e2m1_table_and_rounding():
    # OCP FP4 E2M1 magnitudes, listed from the format definition
    assert [oracle.e2m1_decode(c) for c in range(8)] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [oracle.e2m1_decode(c | 8) for c in range(1, 8)] == [-0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert [oracle.e2m1_encode(oracle.e2m1_decode(c)) for c in range(16) if c != 8] == [c for c in range(16) if c != 8]
    assert oracle.e2m1_encode(2.5) == 4 and oracle.e2m1_encode(3.5) == 6   # ties to the even code (2.0, 4.0)
    assert oracle.e2m1_encode(0.25) == 0 and oracle.e2m1_encode(5.0) == 6  # 0 | 0.5 -> 0; 4 | 6 -> 6 (even)
    assert oracle.e2m1_encode(100.0) == 7 and oracle.e2m1_encode(-7.0) == 15


def _unpack_nibbles(q, n):
    lo, hi = q & 15, q >> 4
    out = np.empty((q.shape[0], 2 * q.shape[1]), dtype=np.int64)
    out[:, 0::2], out[:, 1::2] = lo, hi
    return out[:, :n]


def test_quant_formats_round_trip_and_layout():
    rng = np.random.default_rng(13)
    r, K, N = 3, 24, 256
    X = rng.standard_normal((r, K))
    W = rng.standard_normal((N, K)) / math.sqrt(K)
    y = X @ W.T
    # FP8 1x128: scale = blockwise amax / 448 and the block maximum encodes to +-448
    q, s, yy = oracle.linear_quant(X, W, None, oracle.QUANT_FP8_1X128)
    assert np.allclose(yy, y, rtol=1e-13, atol=1e-13)
    for blk in range(2):
        seg = y[:, blk * 128:(blk + 1) * 128]
        assert np.allclose(s[:, blk], np.abs(seg).max(axis=1) / 448, rtol=1e-14)
        dq = oracle.e4m3_decode(q[:, blk * 128:(blk + 1) * 128]) * s[:, blk:blk + 1]
        assert np.all(np.abs(dq - seg) <= np.abs(seg) * 2.0 ** -4 + s[:, blk:blk + 1] * 2.0 ** -9)
    # INT4 g32: nibble two's complement, low nibble first, values = numpy rint (half to even) clamp 7
    q, s, _ = oracle.linear_quant(X, W, None, oracle.QUANT_INT4_G32)
    nib = _unpack_nibbles(q, N)
    vals = np.where(nib >= 8, nib - 16, nib)
    sref = np.abs(y.reshape(r, -1, 32)).max(axis=2) / 7
    assert np.allclose(s, sref, rtol=1e-14)
    expect = np.clip(np.rint(y / np.repeat(sref, 32, axis=1)), -7, 7)
    assert np.array_equal(vals, expect)
    # NVFP4 g16: the stored E4M3 scale divides the values; decoded values stay within half an ulp
    q, s, _ = oracle.linear_quant(X, W, None, oracle.QUANT_NVFP4_G16)
    sc = oracle.e4m3_decode(s.astype(np.uint8))
    assert np.array_equal(s.astype(np.uint8), oracle.e4m3_encode(np.abs(y.reshape(r, -1, 16)).max(axis=2) / 6))
    dec = np.vectorize(oracle.e2m1_decode)(_unpack_nibbles(q, N)) * np.repeat(sc, 16, axis=1)
    rel = np.abs(dec - y) / np.repeat(sc, 16, axis=1)
    assert rel.max() <= 1.0 + 1e-12  # at most one E2M1 step (1.0 at the top of the range, 2 -> 3 -> 4 -> 6)
    # a zero block gives scale 0 and zero codes
    q0, s0, _ = oracle.linear_quant(np.zeros((1, K)), W, None, oracle.QUANT_INT4_G32)
    assert not q0.any() and not s0.any()


def test_quant_smoothing_factor_of_ones_changes_nothing():
    """Step 3 of the five-step quantised write-back with every factor 1 is the plain
    block-scaled output, in all three formats."""
    rng = np.random.default_rng(21)
    X = rng.standard_normal((2, 40))
    W = rng.standard_normal((96, 40)) / math.sqrt(40)
    for fmt in (oracle.QUANT_FP8_1X128, oracle.QUANT_INT4_G32, oracle.QUANT_NVFP4_G16):
        q0, s0, y0 = oracle.linear_quant(X, W, None, fmt)
        q1, s1, y1 = oracle.linear_quant(X, W, None, fmt, inv_smooth=np.ones(96))
        assert np.array_equal(q0, q1) and np.array_equal(s0, s1) and np.array_equal(y0, y1)


def test_quant_smoothing_undoes_a_per_column_weight_scale():
    """Scaling output column n of the Linear (row n of W and b[n]) by c_n and correcting
    with the inverse factor 1/c_n gives back the unscaled codes and scales exactly (c_n
    powers of two, so every product is exact).  A factor that divided instead of
    multiplying, or that was indexed by anything but the output column, fails this."""
    rng = np.random.default_rng(22)
    N, K = 160, 48
    X = rng.standard_normal((3, K))
    W = rng.standard_normal((N, K)) / math.sqrt(K)
    b = rng.standard_normal(N) * 0.1
    c = 2.0 ** rng.integers(-3, 4, size=N)
    for fmt in (oracle.QUANT_FP8_1X128, oracle.QUANT_INT4_G32, oracle.QUANT_NVFP4_G16):
        q0, s0, y0 = oracle.linear_quant(X, W, b, fmt)
        q1, s1, y1 = oracle.linear_quant(X, W * c[:, None], b * c, fmt, inv_smooth=1.0 / c)
        assert np.array_equal(q0, q1) and np.array_equal(s0, s1)
        assert np.array_equal(y0, y1)
    # a correction that is not undone moves the codes
    q2, _, _ = oracle.linear_quant(X, W * c[:, None], b * c, oracle.QUANT_FP8_1X128)
    assert not np.array_equal(oracle.linear_quant(X, W, b, oracle.QUANT_FP8_1X128)[0], q2)


def test_quant_smoothing_hand_computed_nvfp4_block():
    """One 1 x 16 NVFP4 group worked by hand.  X = [1], W[n] = n + 1, so the Linear output
    is 1, 2, ..., 16; the inverse smoothing factor is 1/2 on even columns and 1 on odd ones,
    so the corrected values are 0.5, 2, 1.5, 4, 2.5, 6, 3.5, 8, 4.5, 10, 5.5, 12, 6.5, 14,
    7.5, 16.  Their maximum 16 gives 16 / 6 = 2.667, whose nearest E4M3 value is 2.75 =
    1.375 * 2^1 (exponent field 8, mantissa 3: code 0x43).  Divided by 2.75 the values are
    0.18, 0.73, 0.55, 1.45, 0.91, 2.18, 1.27, 2.91, 1.64, 3.64, 2.0, 4.36, 2.36, 5.09, 2.73,
    5.82, and the nearest E2M1 values 0, 0.5, 0.5, 1.5, 1, 2, 1.5, 3, 1.5, 4, 2, 4, 2, 6, 3, 6
    are codes 0 1 1 3 2 4 3 5 3 6 4 6 4 7 5 7, packed low nibble first."""
    X = np.ones((1, 1))
    W = np.arange(1.0, 17.0)[:, None]
    inv = np.where(np.arange(16) % 2 == 0, 0.5, 1.0)
    q, s, y = oracle.linear_quant(X, W, None, oracle.QUANT_NVFP4_G16, inv_smooth=inv)
    assert np.array_equal(y[0], [0.5, 2, 1.5, 4, 2.5, 6, 3.5, 8, 4.5, 10, 5.5, 12, 6.5, 14, 7.5, 16])
    assert int(s[0, 0]) == 0x43
    assert list(q[0]) == [0x10, 0x31, 0x42, 0x53, 0x63, 0x64, 0x74, 0x75]
    # without the correction column 0 is 1 / 2.75 = 0.36, which rounds to 0.5 (code 1)
    q_plain, s_plain, _ = oracle.linear_quant(X, W, None, oracle.QUANT_NVFP4_G16)
    assert int(s_plain[0, 0]) == 0x43 and q_plain[0, 0] & 15 == 1


def test_quant_smoothing_block_maximum_maps_to_the_top_code():
    """FP8 1x128 with a correction: the block maximum is taken after the correction, so the
    corrected maximum codes to +-448 (0x7E / 0xFE) and the scale is that maximum / 448."""
    rng = np.random.default_rng(23)
    X = rng.standard_normal((4, 32))
    W = rng.standard_normal((256, 32)) / math.sqrt(32)
    inv = rng.uniform(0.25, 4.0, size=256)
    q, s, y = oracle.linear_quant(X, W, None, oracle.QUANT_FP8_1X128, inv_smooth=inv)
    ref = (X @ W.T) * inv
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)
    for blk in range(2):
        seg = ref[:, blk * 128:(blk + 1) * 128]
        assert np.allclose(s[:, blk], np.abs(seg).max(axis=1) / 448, rtol=1e-13)
        top = np.argmax(np.abs(seg), axis=1)
        codes = q[np.arange(4), blk * 128 + top]
        assert set(codes.tolist()) <= {0x7E, 0xFE}


def test_qkv_rope_kv_fp8_against_complex_rotation_and_e4m3_bounds():
    """GQA widths (4 query heads, 2 kv heads): Q and K against RoPE as complex
    multiplication of a numpy projection, V against the projection alone; each
    (row, kv head) block's maximum encodes to +-448 and its dequantised values
    lie within half an E4M3 step; an all-zero head gets scale 0 and zero codes."""
    rng = np.random.default_rng(11)
    M, K, H, Hkv, D = 6, 40, 4, 2, 16
    X = rng.standard_normal((M, K))
    X[3] = 0.0
    W = rng.standard_normal(((H + 2 * Hkv) * D, K)) / math.sqrt(K)
    b = rng.standard_normal((H + 2 * Hkv) * D) * 0.02
    b[H * D + Hkv * D:H * D + Hkv * D + D] = 0.0  # V head 0 of the zero row stays exactly 0
    pos = np.array([0, 1, 7, 2047, 300, 5])
    o = oracle.qkv_rope_kv_fp8(X, W, b, H, Hkv, D, 10000.0, pos)
    P = X @ W.T + b
    qw, kvw = H * D, Hkv * D
    np.testing.assert_allclose(o["q"], _rope_torch_complex(P[:, :qw], pos, D, 1e4), rtol=0, atol=1e-12)
    k_ref = _rope_torch_complex(P[:, qw:qw + kvw], pos, D, 1e4)
    v_ref = P[:, qw + kvw:]
    np.testing.assert_allclose(o["kv"], np.concatenate([k_ref, v_ref], axis=1), rtol=0, atol=1e-12)
    for codes, scale, ref in ((o["kq"], o["ks"], k_ref), (o["vq"], o["vs"], v_ref)):
        blocks = ref.reshape(M, Hkv, D)
        amax = np.abs(blocks).max(axis=2)
        np.testing.assert_allclose(scale, amax / 448.0, rtol=1e-15, atol=0)
        deq = oracle.e4m3_decode(codes).reshape(M, Hkv, D) * scale[:, :, None]
        bound = 2.0 ** -4 * np.abs(blocks) + 2.0 ** -10 * scale[:, :, None]
        assert np.all(np.abs(deq - blocks) <= bound * (1 + 1e-12))
        c = codes.reshape(M, Hkv, D)
        for i in range(M):
            for h in range(Hkv):
                if amax[i, h] > 0:
                    j = int(np.argmax(np.abs(blocks[i, h])))
                    assert c[i, h, j] == (0x7E if blocks[i, h, j] > 0 else 0xFE)
    assert o["vs"][3, 0] == 0.0 and not o["vq"][3, :D].any()
    # the pages' K/V byte ledger for one token of an 8-kv-head, head_dim-128 model:
    # 4096 bytes per layer in bf16, 2048 in FP8; 64 KiB over 32 layers
    kv_bytes_fp8 = 2 * 8 * 128 * np.dtype(np.uint8).itemsize
    assert (kv_bytes_fp8, 2 * kv_bytes_fp8, 32 * kv_bytes_fp8) == (2048, 4096, 64 * 1024)


@pytest.mark.parametrize("mode", [oracle.GELU_ERF, oracle.GELU_TANH])
def test_gelu_grad_against_differences_and_autograd(mode):
    """GELU' against central differences of the (pinned) forward GELU, against torch's
    fp64 autograd of F.gelu, and at closed-form points."""
    xs = np.concatenate([np.linspace(-8, 8, 161), [-30.0, -0.3, 1e-3, 30.0]])
    step = 1e-5
    fwd = oracle.gelu_erf if mode == oracle.GELU_ERF else oracle.gelu_tanh
    for x in xs:
        fd = (fwd(x + step) - fwd(x - step)) / (2 * step)
        assert oracle.gelu_grad(x, mode) == pytest.approx(fd, abs=1e-8)
    t = torch.tensor(xs, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(t, approximate="none" if mode == oracle.GELU_ERF else "tanh").sum().backward()
    got = np.array([oracle.gelu_grad(x, mode) for x in xs])
    # atol: where tanh(u) rounds next to -1 (absolute step 1.1e-16) the derivative's second
    # term multiplies that rounding by x c (1 + 3 a x^2) ~ 50 near x = -7
    np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-13, atol=1e-14)
    assert oracle.gelu_grad(0.0, mode) == 0.5                      # Phi(0) = 1/2, 0 * phi(0) = 0
    assert oracle.gelu_grad(30.0, mode) == pytest.approx(1.0, abs=1e-15)
    assert abs(oracle.gelu_grad(-30.0, mode)) < 1e-15


def test_dgrad_gelu_against_numpy_and_autograd():
    """(dZ W) * GELU'(H) with W stored [n_out, n_in]: against numpy's matmul times torch's
    autograd derivative, and a transposed-operand mistake fails (W not square)."""
    rng = np.random.default_rng(21)
    M, Kp, N = 7, 12, 9
    dZ, W, H = rng.standard_normal((M, Kp)), rng.standard_normal((Kp, N)), rng.standard_normal((M, N)) * 2
    for mode, approx in ((oracle.GELU_ERF, "none"), (oracle.GELU_TANH, "tanh")):
        h = torch.tensor(H, requires_grad=True)
        torch.nn.functional.gelu(h, approximate=approx).backward(torch.tensor(dZ @ W))
        np.testing.assert_allclose(oracle.dgrad_gelu(dZ, W, H, mode), h.grad.numpy(), rtol=1e-12, atol=1e-13)
        cols = np.array([8, 0, 3])
        np.testing.assert_allclose(oracle.dgrad_gelu(dZ, W, H, mode, cols), h.grad.numpy()[:, cols], rtol=1e-12,
                                   atol=1e-13)


def test_swiglu_bwd_against_autograd_and_layout():
    """SwiGLU backward pairs against torch fp64 autograd of silu(g) * u with dy = dO Wd;
    the pair of feature n sits at columns 2n (gate) and 2n + 1 (up); g = 0 gives
    dg = dy u / 2 and du = 0."""
    rng = np.random.default_rng(22)
    M, Kp, N = 6, 10, 8
    dO, Wd = rng.standard_normal((M, Kp)), rng.standard_normal((Kp, N))
    G, U = rng.standard_normal((M, N)) * 3, rng.standard_normal((M, N))
    G[2, 5] = 0.0
    g = torch.tensor(G, requires_grad=True)
    u = torch.tensor(U, requires_grad=True)
    dy = dO @ Wd
    (torch.nn.functional.silu(g) * u).backward(torch.tensor(dy))
    out = oracle.swiglu_bwd(dO, Wd, G, U)
    assert out.shape == (M, 2 * N)
    np.testing.assert_allclose(out[:, 0::2], g.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out[:, 1::2], u.grad.numpy(), rtol=1e-12, atol=1e-13)
    assert out[2, 10] == pytest.approx(dy[2, 5] * U[2, 5] / 2, rel=1e-14) and out[2, 11] == 0.0
    sub = oracle.swiglu_bwd(dO, Wd, G, U, cols=np.array([7, 1]))
    np.testing.assert_allclose(sub, out[:, [14, 15, 2, 3]], rtol=0, atol=0)
