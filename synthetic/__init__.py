"""Seeded synthetic operands for the fused-Linear workloads.

This module is shared by the fp64 oracle (``oracle/``) and the CUDA path
(``gemm_epilogue_tcgen05_gb300``).  It holds no arithmetic of the method
itself: it only draws numbers.  Every value is a pure function of
``(seed, stream, element index)``, so a block of rows can be regenerated on
its own and both sides always see the same bits.

Recipe (one element):

1. splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
   generators", OOPSLA 2014) gives 64 random bits per counter value.  The
   stream key is ``mix64(seed * 256 + stream)``; counter ``c`` yields
   ``mix64(key + (c + 1) * 0x9E3779B97F4A7C15)``.
2. Element pair ``(2j, 2j+1)`` uses counters ``2j`` and ``2j+1`` as two
   uniforms ``u1 = (hi53(a) + 1) / 2^53`` in (0, 1] and
   ``u2 = hi53(b) / 2^53`` in [0, 1).
3. Box-Muller (1958): ``rho = sqrt(-2 ln u1)``; element ``2j`` is
   ``rho * cos(2 pi u2)`` and element ``2j+1`` is ``rho * sin(2 pi u2)``.
4. ``value = mean + std * normal`` in fp64, rounded to fp32 (round to
   nearest even), then, for bf16 operands, the fp32 bits are rounded to
   bf16 (round to nearest even).

Streams within a workload: X = 0, W = 1, b = 2, Z = 3, gamma = 4,
W_up = 5, b_up = 6, W2 (second GEMM of a chain) = 7, labels = 8,
inverse smoothing factors = 9.
Labels are uniform integers: (top 53 bits of counter i) mod V.
Inverse smoothing factors are log-normal with median 1: exp(0.5 z) for a
standard normal z of stream 9 (fp64), rounded to fp32.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21  # elements per vectorised chunk (bounds host memory)

STREAM_X, STREAM_W, STREAM_B, STREAM_Z, STREAM_GAMMA, STREAM_WUP, STREAM_BUP, STREAM_W2, STREAM_LABEL, \
    STREAM_SMOOTH = range(10)


def _mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrap-around arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed * 256 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix64(base)[0]


def _normal_chunk(key: np.uint64, lo: int, n: int, out: np.ndarray) -> None:
    two_pi = 2.0 * math.pi
    inv53 = 1.0 / float(1 << 53)
    j0 = lo >> 1
    j1 = (lo + n - 1) >> 1
    j = np.arange(j0, j1 + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        a = _mix64(key + (np.uint64(2) * j + np.uint64(1)) * GOLDEN_GAMMA)
        b = _mix64(key + (np.uint64(2) * j + np.uint64(2)) * GOLDEN_GAMMA)
    u1 = ((a >> np.uint64(11)).astype(np.float64) + 1.0) * inv53
    u2 = (b >> np.uint64(11)).astype(np.float64) * inv53
    rho = np.sqrt(-2.0 * np.log(u1))
    ang = two_pi * u2
    pair = np.empty(2 * len(j), dtype=np.float64)
    pair[0::2] = rho * np.cos(ang)
    pair[1::2] = rho * np.sin(ang)
    off = lo - 2 * j0
    out[:] = pair[off:off + n]


def normal_f64_numpy(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Standard normals for element indices ``[start, start + count)``.

    Plain numpy statement of the recipe; :func:`normal_f64` is the fast C
    implementation of the same recipe and is checked against this one.
    """
    out = np.empty(count, dtype=np.float64)
    key = stream_key(seed, stream)
    jobs = [(p, min(_CHUNK, count - p)) for p in range(0, count, _CHUNK)]
    if len(jobs) <= 1:
        for p, n in jobs:
            _normal_chunk(key, start + p, n, out[p:p + n])
        return out
    # numpy releases the GIL inside these array kernels, so chunks run in parallel.
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
        list(ex.map(lambda job: _normal_chunk(key, start + job[0], job[1],
                                              out[job[0]:job[0] + job[1]]), jobs))
    return out


_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib_handle = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` beside it (plain gcc + OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        lib.synth_stream_key.restype = ctypes.c_uint64
        lib.synth_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.synth_normal_f64.argtypes = [ctypes.c_uint64, i64, i64, p]
        lib.synth_draw_f32.argtypes = [ctypes.c_uint64, i64, i64, ctypes.c_double, ctypes.c_double, p]
        lib.synth_draw_bf16.argtypes = [ctypes.c_uint64, i64, i64, ctypes.c_double, ctypes.c_double, p]
        _lib_handle = lib
    return _lib_handle


def normal_f64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Standard normals for element indices ``[start, start + count)`` (C implementation)."""
    out = np.empty(count, dtype=np.float64)
    lib = _lib()
    lib.synth_normal_f64(lib.synth_stream_key(seed, stream), start, count, out.ctypes.data)
    return out


def draw_labels(seed: int, stream: int, count: int, vocab: int) -> np.ndarray:
    """Uniform int32 labels in [0, vocab): (mix64(key + (i + 1) * golden) >> 11) mod vocab."""
    key = stream_key(seed, stream)
    i = np.arange(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix64(key + (i + np.uint64(1)) * GOLDEN_GAMMA)
    return ((z >> np.uint64(11)) % np.uint64(vocab)).astype(np.int32)


def draw_inv_smooth(seed: int, count: int) -> np.ndarray:
    """Per-column inverse smoothing factors, fp32: exp(0.5 z), z standard normal (stream 9)."""
    z = normal_f64(seed, STREAM_SMOOTH, 0, count)
    return np.exp(0.5 * z).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even); returns uint16 bit patterns."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((bits + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def draw(seed: int, stream: int, shape, mean: float, std: float, dtype: str,
         row_start: int = 0, row_count: int | None = None) -> np.ndarray:
    """Draw a tensor (or a block of its rows) of the given logical shape.

    ``dtype`` is ``"bf16"`` (returns uint16 bit patterns) or ``"f32"``
    (returns float32).  Rows ``[row_start, row_start + row_count)`` of the
    full tensor are produced; the values do not depend on how many rows are
    requested.
    """
    shape = tuple(int(s) for s in shape)
    cols = 1
    for s in shape[1:]:
        cols *= s
    rows = shape[0]
    if row_count is None:
        row_count = rows - row_start
    out_shape = (row_count,) + shape[1:]
    n = row_count * cols
    lib = _lib()
    key = lib.synth_stream_key(seed, stream)
    if dtype == "f32":
        out = np.empty(n, dtype=np.float32)
        lib.synth_draw_f32(key, row_start * cols, n, float(mean), float(std), out.ctypes.data)
        return out.reshape(out_shape)
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        lib.synth_draw_bf16(key, row_start * cols, n, float(mean), float(std), out.ctypes.data)
        return out.reshape(out_shape)
    raise ValueError(f"unknown dtype {dtype}")


def draw_numpy(seed: int, stream: int, shape, mean: float, std: float, dtype: str,
               row_start: int = 0, row_count: int | None = None) -> np.ndarray:
    """:func:`draw` written in numpy only (slow; used to check the C implementation)."""
    shape = tuple(int(s) for s in shape)
    cols = 1
    for s in shape[1:]:
        cols *= s
    if row_count is None:
        row_count = shape[0] - row_start
    z = normal_f64_numpy(seed, stream, row_start * cols, row_count * cols)
    v = (mean + std * z).astype(np.float32)
    out_shape = (row_count,) + shape[1:]
    if dtype == "f32":
        return v.reshape(out_shape)
    return f32_to_bf16_bits(v).reshape(out_shape)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype and the distribution of each operand."""
    name: str
    kind: str            # "gelu_erf" | "gelu_tanh" | "qkv_rope" | "swiglu" | "rmsnorm_fp8" | "rms_chain" | "cross_entropy" | "quant" | "qkv_fp8kv" | "gelu_bwd" | "swiglu_bwd"
    M: int
    N: int               # output features (QKV: 3*H*D; SwiGLU: d_ff)
    K: int
    dtype: str = "bf16"  # "bf16" or "f32"
    has_bias: bool = True
    n_heads: int = 0
    head_dim: int = 0
    seq_len: int = 0
    theta: float = 10000.0
    eps: float = 1e-6
    seed: int = 0
    N2: int = 0          # rms_chain: output features of the second GEMM (its K is N)
    quant: str = ""      # quant: "fp8_1x128" | "int4_g32" | "nvfp4_g16"
    n_kv_heads: int = 0  # qkv_fp8kv: key/value heads (grouped-query attention)
    smooth: bool = False  # quant: per-column inverse smoothing factors (fp32 [N], "inv_smooth")
    extra: dict = field(default_factory=dict, compare=False, hash=False)


# The workloads named for this path: (configuration, shapes and distributions).
WORKLOADS = {
    "tiny_gelu_erf_f32": Workload("tiny_gelu_erf_f32", "gelu_erf", 64, 256, 128, dtype="f32"),
    "gelu_tanh_8192x16384x4096": Workload("gelu_tanh_8192x16384x4096", "gelu_tanh", 8192, 16384, 4096),
    "qkv_rope_8192x12288x4096": Workload("qkv_rope_8192x12288x4096", "qkv_rope", 8192, 12288, 4096,
                                         has_bias=False, n_heads=32, head_dim=128, seq_len=2048),
    # grouped-query QKV (32 query heads, 8 kv heads of 128) writing the K/V cache entry in FP8
    "qkv_fp8kv_8192x6144x4096": Workload("qkv_fp8kv_8192x6144x4096", "qkv_fp8kv", 8192, 6144, 4096,
                                         has_bias=False, n_heads=32, n_kv_heads=8, head_dim=128, seq_len=2048),
    "swiglu_8192x14336x4096": Workload("swiglu_8192x14336x4096", "swiglu", 8192, 14336, 4096,
                                       has_bias=False),
    "rmsnorm_fp8_prefill_8192x4096x14336": Workload("rmsnorm_fp8_prefill_8192x4096x14336", "rmsnorm_fp8",
                                                    8192, 4096, 14336, has_bias=False),
    "rmsnorm_fp8_decode_32x4096x14336": Workload("rmsnorm_fp8_decode_32x4096x14336", "rmsnorm_fp8",
                                                 32, 4096, 14336, has_bias=False),
    # attention output projection -> residual -> RMSNorm -> gate (or up) projection, d 4096, d_ff 14336
    "rms_chain_8192x4096x4096_to_14336": Workload("rms_chain_8192x4096x4096_to_14336", "rms_chain",
                                                  8192, 4096, 4096, has_bias=False, N2=14336),
    # LM head over a 32K vocabulary with the cross-entropy in the epilogue
    "lm_head_ce_8192x32768x4096": Workload("lm_head_ce_8192x32768x4096", "cross_entropy", 8192, 32768, 4096,
                                           has_bias=False),
    # backward of the MLP blocks: dgrad of the down projection (K = d_model) with the
    # activation derivative in the epilogue; N = d_ff features of the saved activations
    "gelu_bwd_8192x16384x4096": Workload("gelu_bwd_8192x16384x4096", "gelu_bwd", 8192, 16384, 4096,
                                         has_bias=False),
    "swiglu_bwd_8192x14336x4096": Workload("swiglu_bwd_8192x14336x4096", "swiglu_bwd", 8192, 14336, 4096,
                                           has_bias=False),
    # up-projection whose output is written block-scaled for a low-precision consumer
    "quant_fp8_1x128_8192x16384x4096": Workload("quant_fp8_1x128_8192x16384x4096", "quant", 8192, 16384, 4096,
                                                quant="fp8_1x128"),
    "quant_int4_g32_8192x16384x4096": Workload("quant_int4_g32_8192x16384x4096", "quant", 8192, 16384, 4096,
                                               quant="int4_g32"),
    "quant_nvfp4_g16_8192x16384x4096": Workload("quant_nvfp4_g16_8192x16384x4096", "quant", 8192, 16384, 4096,
                                                quant="nvfp4_g16"),
    # the same with the output of a smoothed layer: inverse smoothing factor per column first
    "quant_fp8_1x128_smooth_8192x16384x4096": Workload("quant_fp8_1x128_smooth_8192x16384x4096", "quant", 8192,
                                                       16384, 4096, quant="fp8_1x128", smooth=True),
    # decode shapes (32 tokens) of the up projection with GELU and of the fused QKV projection
    "gelu_decode_32x16384x4096": Workload("gelu_decode_32x16384x4096", "gelu_tanh", 32, 16384, 4096),
    "qkv_decode_32x12288x4096": Workload("qkv_decode_32x12288x4096", "qkv_rope", 32, 12288, 4096,
                                         has_bias=False, n_heads=32, head_dim=128, seq_len=2048),
    "qkv_fp8kv_decode_32x6144x4096": Workload("qkv_fp8kv_decode_32x6144x4096", "qkv_fp8kv", 32, 6144, 4096,
                                              has_bias=False, n_heads=32, n_kv_heads=8, head_dim=128,
                                              seq_len=2048),
    "swiglu_decode_32x14336x4096": Workload("swiglu_decode_32x14336x4096", "swiglu", 32, 14336, 4096,
                                            has_bias=False),
    # decode shape of the block-scaled up projection (FP8 activations for a low-precision consumer)
    "quant_fp8_1x128_decode_32x16384x4096": Workload("quant_fp8_1x128_decode_32x16384x4096", "quant", 32, 16384,
                                                     4096, quant="fp8_1x128"),
}


def operand_specs(w: Workload):
    """(name, stream, shape, mean, std, dtype) for every operand of a workload."""
    dt = w.dtype
    w_std = 1.0 / math.sqrt(w.K)
    if w.kind == "gelu_bwd":  # upstream gradient, next layer's weight [K, N] as stored, saved H
        return [("dZ", STREAM_X, (w.M, w.K), 0.0, 1.0, dt), ("W", STREAM_W, (w.K, w.N), 0.0, w_std, dt),
                ("H", STREAM_Z, (w.M, w.N), 0.0, 1.0, dt)]
    if w.kind == "swiglu_bwd":  # upstream gradient, down projection [K, N] as stored, saved gate and up
        return [("dO", STREAM_X, (w.M, w.K), 0.0, 1.0, dt), ("Wd", STREAM_W, (w.K, w.N), 0.0, w_std, dt),
                ("G", STREAM_Z, (w.M, w.N), 0.0, 1.0, dt), ("U", STREAM_GAMMA, (w.M, w.N), 0.0, 1.0, dt)]
    specs = [("X", STREAM_X, (w.M, w.K), 0.0, 1.0, dt)]
    if w.kind == "swiglu":
        specs += [("Wgate", STREAM_W, (w.N, w.K), 0.0, w_std, dt),
                  ("Wup", STREAM_WUP, (w.N, w.K), 0.0, w_std, dt)]
        if w.has_bias:
            specs += [("bgate", STREAM_B, (w.N,), 0.0, 0.02, dt),
                      ("bup", STREAM_BUP, (w.N,), 0.0, 0.02, dt)]
        return specs
    specs.append(("W", STREAM_W, (w.N, w.K), 0.0, w_std, dt))
    if w.has_bias:
        specs.append(("b", STREAM_B, (w.N,), 0.0, 0.02, dt))
    if w.kind in ("rmsnorm_fp8", "rms_chain"):
        specs += [("Z", STREAM_Z, (w.M, w.N), 0.0, 1.0, dt),
                  ("gamma", STREAM_GAMMA, (w.N,), 1.0, 0.1, dt)]
    if w.kind == "rms_chain":
        specs.append(("W2", STREAM_W2, (w.N2, w.N), 0.0, 1.0 / math.sqrt(w.N), dt))
    return specs


def make_labels(w: Workload) -> np.ndarray:
    return draw_labels(w.seed, STREAM_LABEL, w.M, w.N)


ROW_OPERANDS = ("X", "Z", "dZ", "H", "dO", "G", "U")  # operands with one row per token


def make_operands(w: Workload, rows: tuple[int, int] | None = None) -> dict:
    """All operands of ``w`` as host arrays (bf16 as uint16 bits, f32 as float32).

    With ``rows=(start, count)`` only that block of the row-indexed operands
    (those in ROW_OPERANDS) is produced; weights and vectors are always produced whole.
    """
    out = {}
    for name, stream, shape, mean, std, dt in operand_specs(w):
        if rows is not None and name in ROW_OPERANDS:
            out[name] = draw(w.seed, stream, shape, mean, std, dt, rows[0], rows[1])
        else:
            out[name] = draw(w.seed, stream, shape, mean, std, dt)
    if w.smooth:
        out["inv_smooth"] = draw_inv_smooth(w.seed, w.N)
    return out


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 copy of an operand produced by :func:`draw` (fp32 arrays are widened as they
    are, whatever the workload's dtype: the inverse smoothing factors are always fp32)."""
    if dtype == "bf16" and a.dtype != np.float32:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields replaced (used for smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)
