"""fp64 CPU oracle for the fused Linear + epilogue path (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The CUDA library never imports it,
and the two share no code.  The arithmetic lives in ``oracle.c`` (plain C,
fp64, OpenMP over independent outputs); this module only compiles it and
marshals numpy arrays.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, library routines (libm / torch fp64 CPU ops / scipy),
brute force on tiny inputs, or values printed on the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib_handle = None

GELU_ERF, GELU_TANH = 0, 1


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` to ``liboracle.so`` (gcc -O2, OpenMP, no fast-math)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    lib = ctypes.CDLL(build())
    P, L, D, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_double, ctypes.c_int
    sig = {
        "orc_linear": [P, L, P, P, L, P, L, P],
        "orc_linear_gelu": [P, L, P, P, L, P, L, I, P],
        "orc_gelu": [P, L, I, P],
        "orc_qkv_rope": [P, L, P, P, L, L, L, D, P, P, L, P],
        "orc_swiglu": [P, L, P, P, P, P, L, P, L, P],
        "orc_rmsnorm_fp8": [P, L, P, P, P, P, L, L, D, P, P, P],
        "orc_e4m3_encode_array": [P, L, P],
        "orc_e4m3_decode_array": [P, L, P],
        "orc_rope_rotate": [D, D, D, P, P],
        "orc_residual_rmsnorm_linear": [P, L, P, P, P, P, L, L, D, P, P, L, P, P],
        "orc_linear_cross_entropy": [P, L, P, P, L, L, P, P],
        "orc_linear_quant": [P, L, P, P, L, L, I, P, P, P, P],
        "orc_qkv_rope_kv_fp8": [P, L, P, P, L, L, L, L, D, P, P, P, P, P, P, P],
        "orc_dgrad_gelu": [P, L, P, L, L, P, I, P, L, P],
        "orc_swiglu_bwd": [P, L, P, L, L, P, P, P, L, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = None
    for name in ("orc_gelu_erf", "orc_gelu_tanh", "orc_silu", "orc_gelu_erf_grad", "orc_gelu_tanh_grad"):
        getattr(lib, name).argtypes = [D]
        getattr(lib, name).restype = D
    lib.orc_rope_angle.argtypes = [D, L, L, D]
    lib.orc_rope_angle.restype = D
    lib.orc_e4m3_encode.argtypes = [D]
    lib.orc_e4m3_encode.restype = I
    lib.orc_e4m3_decode.argtypes = [I]
    lib.orc_e4m3_decode.restype = D
    lib.orc_e2m1_decode.argtypes = [I]
    lib.orc_e2m1_decode.restype = D
    lib.orc_e2m1_encode.argtypes = [D]
    lib.orc_e2m1_encode.restype = I
    lib.orc_num_threads.argtypes = []
    lib.orc_num_threads.restype = I
    _lib_handle = lib
    return lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _cols(cols, n):
    if cols is None:
        cols = np.arange(n)
    return np.ascontiguousarray(cols, dtype=np.int64)


def num_threads() -> int:
    return _lib().orc_num_threads()


def linear(X, W, b=None, cols=None) -> np.ndarray:
    """Y = X W^T + b for the rows of X given, at the requested output columns."""
    X, W, b = _f64(X), _f64(W), _f64(b)
    K = X.shape[1]
    c = _cols(cols, W.shape[0])
    out = np.empty((X.shape[0], len(c)), dtype=np.float64)
    _lib().orc_linear(_ptr(X), X.shape[0], _ptr(W), _ptr(b), K, _ptr(c), len(c), _ptr(out))
    return out


def linear_gelu(X, W, b=None, mode=GELU_TANH, cols=None) -> np.ndarray:
    X, W, b = _f64(X), _f64(W), _f64(b)
    c = _cols(cols, W.shape[0])
    out = np.empty((X.shape[0], len(c)), dtype=np.float64)
    _lib().orc_linear_gelu(_ptr(X), X.shape[0], _ptr(W), _ptr(b), X.shape[1], _ptr(c), len(c),
                           int(mode), _ptr(out))
    return out


def gelu(v, mode) -> np.ndarray:
    v = _f64(v)
    out = np.empty_like(v)
    _lib().orc_gelu(_ptr(v), v.size, int(mode), _ptr(out))
    return out


def gelu_erf(x: float) -> float:
    return _lib().orc_gelu_erf(float(x))


def gelu_tanh(x: float) -> float:
    return _lib().orc_gelu_tanh(float(x))


def silu(x: float) -> float:
    return _lib().orc_silu(float(x))


def rope_angle(pos: float, pair: int, head_dim: int, theta: float) -> float:
    return _lib().orc_rope_angle(float(pos), int(pair), int(head_dim), float(theta))


def rope_rotate(x0: float, x1: float, angle: float):
    y0, y1 = ctypes.c_double(), ctypes.c_double()
    _lib().orc_rope_rotate(float(x0), float(x1), float(angle), ctypes.byref(y0), ctypes.byref(y1))
    return y0.value, y1.value


def qkv_rope(X, Wqkv, bqkv, n_heads, head_dim, theta, pos, cols=None) -> np.ndarray:
    """Columns of [Q|K|V] after RoPE on Q and K; ``pos`` holds each row's position."""
    X, Wqkv, bqkv = _f64(X), _f64(Wqkv), _f64(bqkv)
    pos = _f64(np.asarray(pos))
    c = _cols(cols, Wqkv.shape[0])
    out = np.empty((X.shape[0], len(c)), dtype=np.float64)
    _lib().orc_qkv_rope(_ptr(X), X.shape[0], _ptr(Wqkv), _ptr(bqkv), X.shape[1], int(n_heads),
                        int(head_dim), float(theta), _ptr(pos), _ptr(c), len(c), _ptr(out))
    return out


def swiglu(X, Wg, Wu, bg=None, bu=None, cols=None) -> np.ndarray:
    X, Wg, Wu, bg, bu = _f64(X), _f64(Wg), _f64(Wu), _f64(bg), _f64(bu)
    c = _cols(cols, Wg.shape[0])
    out = np.empty((X.shape[0], len(c)), dtype=np.float64)
    _lib().orc_swiglu(_ptr(X), X.shape[0], _ptr(Wg), _ptr(Wu), _ptr(bg), _ptr(bu), X.shape[1],
                      _ptr(c), len(c), _ptr(out))
    return out


def rmsnorm_fp8(X, W, b, Z, gamma, eps):
    """Returns (codes uint8 [r, N], scale fp64 [r], y fp64 [r, N]) for the rows given."""
    X, W, b, Z, gamma = _f64(X), _f64(W), _f64(b), _f64(Z), _f64(gamma)
    r, K = X.shape
    N = W.shape[0]
    q = np.empty((r, N), dtype=np.uint8)
    scale = np.empty(r, dtype=np.float64)
    y = np.empty((r, N), dtype=np.float64)
    _lib().orc_rmsnorm_fp8(_ptr(X), r, _ptr(W), _ptr(b), _ptr(Z), _ptr(gamma), N, K, float(eps),
                           _ptr(q), _ptr(scale), _ptr(y))
    return q, scale, y


def e4m3_encode(y) -> np.ndarray:
    y = _f64(y)
    q = np.empty(y.shape, dtype=np.uint8)
    _lib().orc_e4m3_encode_array(_ptr(y), y.size, _ptr(q))
    return q


def e4m3_decode(q) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    y = np.empty(q.shape, dtype=np.float64)
    _lib().orc_e4m3_decode_array(_ptr(q), q.size, _ptr(y))
    return y


def residual_rmsnorm_linear(X, W0, b0, Z, gamma, eps, W1, b1=None):
    """(y, h1): y = RMSNorm(X W0^T + b0 + Z, gamma) W1^T + b1 for the rows given; h1 = X W0^T + b0 + Z."""
    X, W0, b0, Z, gamma, W1, b1 = _f64(X), _f64(W0), _f64(b0), _f64(Z), _f64(gamma), _f64(W1), _f64(b1)
    r, K = X.shape
    N, N2 = W0.shape[0], W1.shape[0]
    y = np.empty((r, N2), dtype=np.float64)
    h1 = np.empty((r, N), dtype=np.float64)
    _lib().orc_residual_rmsnorm_linear(_ptr(X), r, _ptr(W0), _ptr(b0), _ptr(Z), _ptr(gamma), N, K, float(eps),
                                       _ptr(W1), _ptr(b1), N2, _ptr(y), _ptr(h1))
    return y, h1


def linear_cross_entropy(X, W, b, labels) -> np.ndarray:
    """Per-row loss -h[y] + logsumexp(h) with h = X W^T + b; label < 0 gives 0, label >= V gives NaN."""
    X, W, b = _f64(X), _f64(W), _f64(b)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    out = np.empty(X.shape[0], dtype=np.float64)
    _lib().orc_linear_cross_entropy(_ptr(X), X.shape[0], _ptr(W), _ptr(b), W.shape[0], X.shape[1], _ptr(lab),
                                    _ptr(out))
    return out


QUANT_FP8_1X128, QUANT_INT4_G32, QUANT_NVFP4_G16 = 0, 1, 2
QUANT_BLOCK = {QUANT_FP8_1X128: 128, QUANT_INT4_G32: 32, QUANT_NVFP4_G16: 16}


def e2m1_decode(code: int) -> float:
    return _lib().orc_e2m1_decode(int(code))


def e2m1_encode(y: float) -> int:
    return _lib().orc_e2m1_encode(float(y))


def linear_quant(X, W, b, fmt, inv_smooth=None):
    """(codes uint8 [r, qbytes], scales [r, nblocks], y fp64 [r, N]) of the block-scaled Linear output.

    inv_smooth: optional per-column factor [N] applied to the Linear output before the
    block maxima (step 3 of the five-step quantised write-back); y is the corrected output."""
    X, W, b, inv_smooth = _f64(X), _f64(W), _f64(b), _f64(inv_smooth)
    r, K = X.shape
    N = W.shape[0]
    bs = QUANT_BLOCK[fmt]
    nb = -(-N // bs)
    qbytes = N if fmt == QUANT_FP8_1X128 else -(-N // 2)
    q = np.empty((r, qbytes), dtype=np.uint8)
    sc = np.empty((r, nb), dtype=np.float64)
    y = np.empty((r, N), dtype=np.float64)
    if inv_smooth is not None and inv_smooth.shape != (N,):
        raise ValueError("inv_smooth must have N entries")
    _lib().orc_linear_quant(_ptr(X), r, _ptr(W), _ptr(b), N, K, int(fmt), _ptr(inv_smooth), _ptr(q), _ptr(sc),
                            _ptr(y))
    return q, sc, y


def qkv_rope_kv_fp8(X, Wqkv, bqkv, n_heads, n_kv_heads, head_dim, theta, pos):
    """QKV + RoPE with K and V quantised to E4M3 per (row, kv head).

    Returns dict with q (fp64 [r, H*D]), kq / vq (uint8 [r, Hkv*D]), ks / vs (fp64 [r, Hkv])
    and kv (fp64 [r, 2*Hkv*D], the unquantised rotated K then V).
    """
    X, Wqkv, bqkv = _f64(X), _f64(Wqkv), _f64(bqkv)
    pos = _f64(np.asarray(pos))
    r, K = X.shape
    qw, kvw = n_heads * head_dim, n_kv_heads * head_dim
    assert Wqkv.shape[0] == qw + 2 * kvw
    out = {"q": np.empty((r, qw)), "kq": np.empty((r, kvw), dtype=np.uint8), "ks": np.empty((r, n_kv_heads)),
           "vq": np.empty((r, kvw), dtype=np.uint8), "vs": np.empty((r, n_kv_heads)), "kv": np.empty((r, 2 * kvw))}
    _lib().orc_qkv_rope_kv_fp8(_ptr(X), r, _ptr(Wqkv), _ptr(bqkv), K, int(n_heads), int(n_kv_heads), int(head_dim),
                               float(theta), _ptr(pos), _ptr(out["q"]), _ptr(out["kq"]), _ptr(out["ks"]),
                               _ptr(out["vq"]), _ptr(out["vs"]), _ptr(out["kv"]))
    return out


def gelu_grad(x: float, mode) -> float:
    """GELU'(x), mode GELU_ERF or GELU_TANH."""
    f = _lib().orc_gelu_erf_grad if mode == GELU_ERF else _lib().orc_gelu_tanh_grad
    return f(float(x))


def dgrad_gelu(dZ, W, H, mode, cols=None) -> np.ndarray:
    """(dZ W)[i, n] * GELU'(H[i, n]) with W stored [Kp, N] (the contraction runs over its rows)."""
    dZ, W, H = _f64(dZ), _f64(W), _f64(H)
    Kp, N = W.shape
    c = _cols(cols, N)
    out = np.empty((dZ.shape[0], len(c)), dtype=np.float64)
    _lib().orc_dgrad_gelu(_ptr(dZ), dZ.shape[0], _ptr(W), Kp, N, _ptr(H), int(mode), _ptr(c), len(c), _ptr(out))
    return out


def swiglu_bwd(dO, Wd, G, U, cols=None) -> np.ndarray:
    """Interleaved (dg, du) pairs [r, 2 len(cols)] of SwiGLU's backward with dy = dO Wd, Wd stored [Kp, N]."""
    dO, Wd, G, U = _f64(dO), _f64(Wd), _f64(G), _f64(U)
    Kp, N = Wd.shape
    c = _cols(cols, N)
    out = np.empty((dO.shape[0], 2 * len(c)), dtype=np.float64)
    _lib().orc_swiglu_bwd(_ptr(dO), dO.shape[0], _ptr(Wd), Kp, N, _ptr(G), _ptr(U), _ptr(c), len(c), _ptr(out))
    return out
