"""GB300 (sm_103a) fused Linear + epilogue library: Python binding.

This module only marshals arguments: it turns torch CUDA tensors into device
pointers, leading dimensions and a stream handle, and calls the C ABI of
``libfusedlinear.so`` (declared in ``include/fused_linear.h``), whose CUDA
kernels do every step of the computation.  There is no other code path: if
the library is not built or cannot be loaded, every call raises.

Functions carry the C names: :func:`fused_linear_gelu` (and its host-buffer
form :func:`fused_linear_gelu_host`), :func:`fused_qkv_rope`,
:func:`fused_qkv_rope_fp8kv`, :func:`fused_swiglu`,
:func:`fused_linear_residual_rmsnorm_fp8` (and
:func:`fused_linear_residual_rmsnorm_fp8_noalloc`, which takes no workspace),
the deferred-scale chain :func:`fused_linear_residual_gamma` and
:func:`fused_linear_rms_rowscale`, :func:`fused_linear_cross_entropy`,
:func:`fused_linear_quant`, and the backward epilogues
:func:`fused_dgrad_gelu` and :func:`fused_swiglu_bwd`.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "libfusedlinear.so")
HEADER = os.path.join(ROOT, "include", "fused_linear.h")

FL_OK, FL_ERR_INVALID_ARG, FL_ERR_UNSUPPORTED, FL_ERR_ALIGNMENT, FL_ERR_WORKSPACE, FL_ERR_CUDA, \
    FL_ERR_TIMEOUT, FL_ERR_ARCH = range(8)
FL_F32, FL_BF16 = 0, 1
FL_GELU_ERF, FL_GELU_TANH = 0, 1

_lib = None


class FusedLinearError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Loads the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run gemm_epilogue_tcgen05_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.fused_linear_gelu.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, I, I, P]
    lib.fused_qkv_rope.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, I64, I64, I64, P]
    lib.fused_swiglu.argtypes = [P, P, P, P, P, P, I, I, I, I64, I64, I64, P]
    lib.fused_linear_residual_rmsnorm_fp8.argtypes = [P, P, P, P, P, F, P, P, P, I, I, I, I64, I64, I64, I64,
                                                      P, SZ, P]
    for f in (lib.fused_linear_gelu, lib.fused_qkv_rope, lib.fused_swiglu,
              lib.fused_linear_residual_rmsnorm_fp8):
        f.restype = I
    lib.fused_linear_residual_gamma.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I64, I64, I64, I64, P]
    lib.fused_linear_rms_rowscale.argtypes = [P, P, P, P, I, F, P, I, I, I, I64, I64, I64, P]
    lib.fused_linear_residual_gamma.restype = I
    lib.fused_linear_rms_rowscale.restype = I
    lib.fused_linear_cross_entropy.argtypes = [P, P, P, P, P, P, I, I, I, I64, I64, I64, P, SZ, P]
    lib.fused_linear_cross_entropy.restype = I
    lib.fused_qkv_rope_fp8kv.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I64, I64, I64, I64, I64, P]
    lib.fused_qkv_rope_fp8kv.restype = I
    lib.fused_dgrad_gelu.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, I64, I, P]
    lib.fused_dgrad_gelu.restype = I
    lib.fused_swiglu_bwd.argtypes = [P, P, P, P, P, I, I, I, I64, I64, I64, I64, P]
    lib.fused_swiglu_bwd.restype = I
    lib.fused_linear_gelu_host.argtypes = [P, P, P, P, I, I, I, I, P, SZ, P]
    lib.fused_linear_gelu_host.restype = I
    lib.fl_linear_gelu_host_buffer_bytes.argtypes = [I, I, I]
    lib.fl_linear_gelu_host_buffer_bytes.restype = SZ
    lib.fused_linear_quant.argtypes = [P, P, P, P, P, P, I, I, I, I64, I64, I64, I64, I, P]
    lib.fused_linear_quant.restype = I
    lib.fl_cross_entropy_workspace_bytes.argtypes = [I, I]
    lib.fl_cross_entropy_workspace_bytes.restype = SZ
    lib.fl_rms_partials_per_row.argtypes = [I]
    lib.fl_rms_partials_per_row.restype = I
    lib.fused_linear_residual_rmsnorm_fp8_noalloc.argtypes = [P, P, P, P, P, F, P, P, I, I, I, I64, I64, I64,
                                                              I64, P]
    lib.fused_linear_residual_rmsnorm_fp8_noalloc.restype = I
    lib.fl_rmsnorm_fp8_workspace_bytes.argtypes = [I, I, I]
    lib.fl_rmsnorm_fp8_workspace_bytes.restype = SZ
    lib.fl_device_status.argtypes = [P]
    lib.fl_device_status.restype = I
    lib.fl_check_device_status.argtypes = [P, P]
    lib.fl_check_device_status.restype = I
    lib.fl_set_cooperative_launch.argtypes = [I]
    lib.fl_set_cooperative_launch.restype = None
    lib.fl_set_descriptor_cache.argtypes = [I]
    lib.fl_set_descriptor_cache.restype = None
    lib.fl_descriptor_cache_stats.argtypes = [P, P]
    lib.fl_descriptor_cache_stats.restype = None
    lib.fl_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.fl_set_wait_timeout_ns.restype = None
    lib.fl_set_max_ctas.argtypes = [I]
    lib.fl_set_max_ctas.restype = None
    lib.fl_set_cta_pairing.argtypes = [I]
    lib.fl_set_cta_pairing.restype = None
    lib.fl_set_linear_decode.argtypes = [I]
    lib.fl_set_linear_decode.restype = None
    lib.fl_linear_decode_shape.argtypes = [I, I, I, I, P, P, P]
    lib.fl_linear_decode_shape.restype = I
    lib.fl_status_string.argtypes = [I]
    lib.fl_status_string.restype = ctypes.c_char_p
    lib.fl_version.argtypes = []
    lib.fl_version.restype = I
    _lib = lib
    return lib


def header_symbols() -> list[str]:
    """Names of every entry point declared (FL_API) in include/fused_linear.h."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^FL_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)


def status_string(status: int) -> str:
    return load().fl_status_string(int(status)).decode()


def version() -> int:
    return load().fl_version()


def _check(fn: str, status: int):
    if status != FL_OK:
        raise FusedLinearError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _mat(t, name, dtype):
    if t.dim() != 2 or t.dtype != dtype or not t.is_cuda or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name}: expected a 2-D {dtype} CUDA tensor with unit column stride")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _vec(t, name, dtype, n):
    if t is None:
        return None
    if t.dtype != dtype or not t.is_cuda or t.numel() != n or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous {dtype} CUDA vector of length {n}")
    return t


def _out(rows: int, cols: int, dtype, device):
    """An output [rows, cols] whose row pitch is rounded up to 16 bytes (the TMA store rule)."""
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((rows, -(-cols // per) * per), dtype=dtype, device=device)[:, :cols]


def _ld(t, width, fallback):
    # Leading dimension of a [rows, width] row-major matrix.  A one-row matrix
    # never reads past its first row, so any pitch >= width works; take one
    # that satisfies the 16-byte pitch rule.
    if t.shape[0] > 1:
        return t.stride(0)
    return max(-(-fallback // 16) * 16, 16)


def fused_linear_gelu(X, W, b=None, Y=None, mode: str = "tanh", stream=None):
    """Y = GELU(X W^T + b); bf16 (tcgen05) or fp32 operands."""
    dtype = X.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("X must be bf16 or fp32")
    M, K = X.shape
    N = W.shape[0]
    _mat(X, "X", dtype)
    _mat(W, "W", dtype)
    _vec(b, "b", dtype, N)
    if Y is None:
        Y = _out(M, N, dtype, X.device)
    _mat(Y, "Y", dtype)
    m = {"erf": FL_GELU_ERF, "tanh": FL_GELU_TANH}[mode]
    st = load().fused_linear_gelu(_ptr(X), _ptr(W), _ptr(b), _ptr(Y), M, N, K, _ld(X, K, K), _ld(W, K, K),
                                  _ld(Y, N, N), FL_BF16 if dtype == torch.bfloat16 else FL_F32, m,
                                  _stream(stream))
    _check("fused_linear_gelu", st)
    return Y


def linear_gelu_host_buffer(M: int, N: int, K: int, device=None) -> torch.Tensor:
    """Device buffer for fused_linear_gelu_host (256-byte aligned, as torch allocates)."""
    n = int(load().fl_linear_gelu_host_buffer_bytes(M, N, K))
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def fused_linear_gelu_host(X, W, b=None, Y=None, mode: str = "tanh", dev_buf=None, stream=None):
    """fused_linear_gelu on host (CPU, ideally pinned) bf16 tensors, copies overlapped with the GEMM.

    Returns Y (host); it is complete once `stream` (default: the current stream) has finished.
    """
    M, K = X.shape
    N = W.shape[0]
    for t, nm in ((X, "X"), (W, "W"), (b, "b"), (Y, "Y")):
        if t is not None and (t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous()):
            raise ValueError(f"{nm}: expected a contiguous bf16 host tensor")
    if b is not None and b.numel() != N:
        raise ValueError("b must have N elements")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [M, N]")
    if dev_buf is None:
        dev_buf = linear_gelu_host_buffer(M, N, K)
    if mode not in ("tanh", "erf"):
        raise ValueError("mode must be 'tanh' or 'erf'")
    st = load().fused_linear_gelu_host(_ptr(X), _ptr(W), _ptr(b), _ptr(Y), M, N, K,
                                       FL_GELU_TANH if mode == "tanh" else FL_GELU_ERF, _ptr(dev_buf),
                                       dev_buf.numel(), _stream(stream))
    _check("fused_linear_gelu_host", st)
    return Y


def fused_qkv_rope(X, Wqkv, bqkv=None, n_heads: int = 32, head_dim: int = 128, seq_len: int = 2048,
                   theta: float = 10000.0, positions=None, out=None, stream=None):
    """Returns (Q, K, V), Q and K already rotated (RoPE on adjacent pairs)."""
    M, K = X.shape
    d = n_heads * head_dim
    _mat(X, "X", torch.bfloat16)
    _mat(Wqkv, "Wqkv", torch.bfloat16)
    _vec(bqkv, "bqkv", torch.bfloat16, 3 * d)
    if positions is not None and (positions.dtype != torch.int32 or positions.numel() != M
                                  or not positions.is_cuda or not positions.is_contiguous()):
        raise ValueError("positions must be a contiguous int32 CUDA vector of length M")
    if out is None:
        out = tuple(torch.empty((M, d), dtype=torch.bfloat16, device=X.device) for _ in range(3))
    Q, Ko, V = out
    lds = {_ld(t, d, d) for t in out}
    for t, nm in zip(out, "QKV"):
        _mat(t, nm, torch.bfloat16)
    if len(lds) != 1:
        raise ValueError("Q, K and V must share one leading dimension")
    st = load().fused_qkv_rope(_ptr(X), _ptr(Wqkv), _ptr(bqkv), _ptr(Q), _ptr(Ko), _ptr(V), _ptr(positions),
                               M, K, n_heads, head_dim, seq_len, float(theta), _ld(X, K, K), _ld(Wqkv, K, K),
                               lds.pop(), _stream(stream))
    _check("fused_qkv_rope", st)
    return Q, Ko, V


def fused_qkv_rope_fp8kv(X, Wqkv, bqkv=None, n_heads: int = 32, n_kv_heads: int = 8, head_dim: int = 128,
                         seq_len: int = 2048, theta: float = 10000.0, positions=None, out=None, stream=None):
    """QKV + RoPE with the K/V cache entry in FP8; returns (Q, Kq, Vq, k_scale, v_scale).

    Q bf16 [M, n_heads*head_dim] (rotated); Kq (rotated) and Vq E4M3 bytes
    [M, n_kv_heads*head_dim]; k_scale, v_scale fp32 [M, n_kv_heads].
    """
    M, K = X.shape
    dq, dkv = n_heads * head_dim, n_kv_heads * head_dim
    _mat(X, "X", torch.bfloat16)
    _mat(Wqkv, "Wqkv", torch.bfloat16)
    _vec(bqkv, "bqkv", torch.bfloat16, dq + 2 * dkv)
    if positions is not None and (positions.dtype != torch.int32 or positions.numel() != M
                                  or not positions.is_cuda or not positions.is_contiguous()):
        raise ValueError("positions must be a contiguous int32 CUDA vector of length M")
    if out is None:
        out = (torch.empty((M, dq), dtype=torch.bfloat16, device=X.device),
               torch.empty((M, dkv), dtype=torch.uint8, device=X.device),
               torch.empty((M, dkv), dtype=torch.uint8, device=X.device),
               torch.empty((M, n_kv_heads), dtype=torch.float32, device=X.device),
               torch.empty((M, n_kv_heads), dtype=torch.float32, device=X.device))
    Q, Kq, Vq, ks, vs = out
    _mat(Q, "Q", torch.bfloat16)
    for t, nm in ((Kq, "Kq"), (Vq, "Vq")):
        _mat(t, nm, torch.uint8)
    for t, nm in ((ks, "k_scale"), (vs, "v_scale")):
        _mat(t, nm, torch.float32)
    ldkv = {_ld(Kq, dkv, dkv), _ld(Vq, dkv, dkv)}
    lds = {_ld(ks, n_kv_heads, n_kv_heads), _ld(vs, n_kv_heads, n_kv_heads)}
    if len(ldkv) != 1 or len(lds) != 1:
        raise ValueError("Kq and Vq (and their scales) must share one leading dimension")
    st = load().fused_qkv_rope_fp8kv(_ptr(X), _ptr(Wqkv), _ptr(bqkv), _ptr(Q), _ptr(Kq), _ptr(Vq), _ptr(ks),
                                     _ptr(vs), _ptr(positions), M, K, n_heads, n_kv_heads, head_dim, seq_len,
                                     float(theta), _ld(X, K, K), _ld(Wqkv, K, K), _ld(Q, dq, dq), ldkv.pop(),
                                     lds.pop(), _stream(stream))
    _check("fused_qkv_rope_fp8kv", st)
    return Q, Kq, Vq, ks, vs


def fused_swiglu(X, Wgate, Wup, bgate=None, bup=None, Y=None, stream=None):
    """Y = SiLU(X Wgate^T + bgate) * (X Wup^T + bup)."""
    M, K = X.shape
    N = Wgate.shape[0]
    _mat(X, "X", torch.bfloat16)
    ldg = _mat(Wgate, "Wgate", torch.bfloat16)
    ldu = _mat(Wup, "Wup", torch.bfloat16)
    if Wup.shape != Wgate.shape or (N > 1 and ldg != ldu):
        raise ValueError("Wgate and Wup must have the same shape and leading dimension")
    _vec(bgate, "bgate", torch.bfloat16, N)
    _vec(bup, "bup", torch.bfloat16, N)
    if Y is None:
        Y = _out(M, N, torch.bfloat16, X.device)
    _mat(Y, "Y", torch.bfloat16)
    st = load().fused_swiglu(_ptr(X), _ptr(Wgate), _ptr(Wup), _ptr(bgate), _ptr(bup), _ptr(Y), M, N, K,
                             _ld(X, K, K), _ld(Wgate, K, K), _ld(Y, N, N), _stream(stream))
    _check("fused_swiglu", st)
    return Y


def rmsnorm_fp8_workspace_bytes(M: int, N: int, K: int) -> int:
    return load().fl_rmsnorm_fp8_workspace_bytes(M, N, K)


def rmsnorm_fp8_workspace(M: int, N: int, K: int, device=None) -> torch.Tensor:
    """A zero-filled workspace of the size the library asks for (torch allocation)."""
    n = max(rmsnorm_fp8_workspace_bytes(M, N, K), 1)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def fused_linear_residual_rmsnorm_fp8(X, W, b, Z, gamma, eps: float = 1e-6, Yq=None, row_scale=None,
                                      workspace=None, h_out=None, stream=None):
    """Returns (Yq, row_scale): E4M3 codes as uint8 [M, N] and fp32 scales [M].

    h_out: None (default), True (allocate one) or a bf16 [M, N] tensor with Z's row pitch;
    when given, h = X W^T + b + Z is written there too and (Yq, row_scale, h_out) is returned."""
    M, K = X.shape
    N = W.shape[0]
    _mat(X, "X", torch.bfloat16)
    _mat(W, "W", torch.bfloat16)
    _mat(Z, "Z", torch.bfloat16)
    _vec(b, "b", torch.bfloat16, N)
    _vec(gamma, "gamma", torch.bfloat16, N)
    if Yq is None:  # row pitch rounded up to 16 bytes, as the TMA store needs
        Yq = _out(M, N, torch.uint8, X.device)
    if Yq.dtype != torch.uint8:
        Yq = Yq.view(torch.uint8)
    _mat(Yq, "Yq", torch.uint8)
    if row_scale is None:
        row_scale = torch.empty(M, dtype=torch.float32, device=X.device)
    _vec(row_scale, "row_scale", torch.float32, M)
    want_h = h_out is not None
    if h_out is True:
        h_out = torch.empty_strided((M, N), (_ld(Z, N, N), 1), dtype=torch.bfloat16, device=X.device)
    if want_h:
        _mat(h_out, "h_out", torch.bfloat16)
        if tuple(h_out.shape) != (M, N) or (M > 1 and h_out.stride(0) != Z.stride(0)):
            raise ValueError("h_out must be [M, N] with Z's row pitch")
    if workspace is None:
        workspace = rmsnorm_fp8_workspace(M, N, K, X.device)
    st = load().fused_linear_residual_rmsnorm_fp8(
        _ptr(X), _ptr(W), _ptr(b), _ptr(Z), _ptr(gamma), float(eps), _ptr(Yq), _ptr(row_scale),
        _ptr(h_out) if want_h else None, M, N, K, _ld(X, K, K), _ld(W, K, K), _ld(Z, N, N), _ld(Yq, N, N),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check("fused_linear_residual_rmsnorm_fp8", st)
    return (Yq, row_scale, h_out) if want_h else (Yq, row_scale)


def fused_linear_residual_rmsnorm_fp8_noalloc(X, W, b, Z, gamma, Yq, row_scale, eps: float = 1e-6,
                                              stream=None):
    """The same codes and scales as :func:`fused_linear_residual_rmsnorm_fp8`, through the entry point
    that needs no workspace (it uses a scratch array built into the library; calls that may overlap
    on the GPU must not be issued).  Yq (uint8 [M, N]) and row_scale (fp32 [M]) are the caller's:
    the call allocates nothing.  Returns (Yq, row_scale)."""
    M, K = X.shape
    N = W.shape[0]
    _mat(X, "X", torch.bfloat16)
    _mat(W, "W", torch.bfloat16)
    _mat(Z, "Z", torch.bfloat16)
    _vec(b, "b", torch.bfloat16, N)
    _vec(gamma, "gamma", torch.bfloat16, N)
    _mat(Yq, "Yq", torch.uint8)
    _vec(row_scale, "row_scale", torch.float32, M)
    st = load().fused_linear_residual_rmsnorm_fp8_noalloc(
        _ptr(X), _ptr(W), _ptr(b), _ptr(Z), _ptr(gamma), float(eps), _ptr(Yq), _ptr(row_scale), M, N, K,
        _ld(X, K, K), _ld(W, K, K), _ld(Z, N, N), _ld(Yq, N, N), _stream(stream))
    _check("fused_linear_residual_rmsnorm_fp8_noalloc", st)
    return Yq, row_scale


def rms_partials_per_row(n_norm: int) -> int:
    return load().fl_rms_partials_per_row(int(n_norm))


def fused_linear_residual_gamma(X, W, b, Z, gamma, store_h1: bool = True, H2=None, H1=None, rms_partials=None,
                                stream=None):
    """Step 1 of GEMM -> residual -> RMSNorm -> GEMM: returns (H2 = h1 * gamma, H1 = h1 or None, partials)."""
    M, K = X.shape
    N = W.shape[0]
    _mat(X, "X", torch.bfloat16)
    _mat(W, "W", torch.bfloat16)
    _mat(Z, "Z", torch.bfloat16)
    _vec(b, "b", torch.bfloat16, N)
    _vec(gamma, "gamma", torch.bfloat16, N)
    if H2 is None:
        H2 = _out(M, N, torch.bfloat16, X.device)
    if H1 is None and store_h1:
        H1 = _out(M, N, torch.bfloat16, X.device)
    _mat(H2, "H2", torch.bfloat16)
    if H1 is not None and (_mat(H1, "H1", torch.bfloat16) != _mat(H2, "H2", torch.bfloat16) and M > 1):
        raise ValueError("H1 and H2 must share one leading dimension")
    npart = rms_partials_per_row(N)
    if rms_partials is None:
        rms_partials = torch.empty((npart, M), dtype=torch.float32, device=X.device)
    if rms_partials.dtype != torch.float32 or rms_partials.numel() < npart * M or not rms_partials.is_contiguous():
        raise ValueError("rms_partials must be a contiguous fp32 tensor of [ceil(N/256), M] entries")
    st = load().fused_linear_residual_gamma(_ptr(X), _ptr(W), _ptr(b), _ptr(Z), _ptr(gamma), _ptr(H2), _ptr(H1),
                                            _ptr(rms_partials), M, N, K, _ld(X, K, K), _ld(W, K, K), _ld(Z, N, N),
                                            _ld(H2, N, N), _stream(stream))
    _check("fused_linear_residual_gamma", st)
    return H2, H1, rms_partials


def fused_linear_rms_rowscale(H2, W1, b1, rms_partials, n_norm: int, eps: float = 1e-6, Y=None, stream=None):
    """Step 2: Y = r * (H2 W1^T) + b1, r = 1/sqrt(sum of the row's partials / n_norm + eps)."""
    M, K = H2.shape
    N = W1.shape[0]
    _mat(H2, "H2", torch.bfloat16)
    _mat(W1, "W1", torch.bfloat16)
    _vec(b1, "b1", torch.bfloat16, N)
    if Y is None:
        Y = _out(M, N, torch.bfloat16, H2.device)
    _mat(Y, "Y", torch.bfloat16)
    st = load().fused_linear_rms_rowscale(_ptr(H2), _ptr(W1), _ptr(b1), _ptr(rms_partials), int(n_norm), float(eps),
                                          _ptr(Y), M, N, K, _ld(H2, K, K), _ld(W1, K, K), _ld(Y, N, N),
                                          _stream(stream))
    _check("fused_linear_rms_rowscale", st)
    return Y


def cross_entropy_workspace(M: int, V: int, device=None) -> torch.Tensor:
    n = max(load().fl_cross_entropy_workspace_bytes(int(M), int(V)), 1)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def fused_linear_cross_entropy(X, W, b, labels, loss=None, logits=None, store_logits: bool = False,
                               workspace=None, stream=None):
    """Per-row loss logsumexp(X W^T + b) - (X W^T + b)[label]; returns (loss, logits or None)."""
    M, K = X.shape
    V = W.shape[0]
    _mat(X, "X", torch.bfloat16)
    _mat(W, "W", torch.bfloat16)
    _vec(b, "b", torch.bfloat16, V)
    if labels.dtype != torch.int32 or labels.numel() != M or not labels.is_cuda or not labels.is_contiguous():
        raise ValueError("labels must be a contiguous int32 CUDA vector of length M")
    if loss is None:
        loss = torch.empty(M, dtype=torch.float32, device=X.device)
    _vec(loss, "loss", torch.float32, M)
    if logits is None and store_logits:
        logits = _out(M, V, torch.bfloat16, X.device)
    ldl = 0
    if logits is not None:
        _mat(logits, "logits", torch.bfloat16)
        ldl = _ld(logits, V, V)
    if workspace is None:
        workspace = cross_entropy_workspace(M, V, X.device)
    st = load().fused_linear_cross_entropy(_ptr(X), _ptr(W), _ptr(b), _ptr(labels), _ptr(loss), _ptr(logits), M, V, K,
                                           _ld(X, K, K), _ld(W, K, K), ldl, _ptr(workspace), workspace.numel(),
                                           _stream(stream))
    _check("fused_linear_cross_entropy", st)
    return loss, logits


QUANT_FP8_1X128, QUANT_INT4_G32, QUANT_NVFP4_G16 = 0, 1, 2
QUANT_BLOCK = {QUANT_FP8_1X128: 128, QUANT_INT4_G32: 32, QUANT_NVFP4_G16: 16}


def fused_linear_quant(X, W, b=None, fmt: int = QUANT_FP8_1X128, Yq=None, scales=None, inv_smooth=None,
                       stream=None):
    """Block-scaled quantised Linear output; returns (codes uint8, scales).

    inv_smooth: optional fp32 [N] inverse smoothing factor, multiplied into each output
    column before the block maxima (the optional correction step of the quantised write-back).
    FP8 1x128: codes [M, N] E4M3, scales fp32 [M, ceil(N/128)].
    INT4 g32:  codes [M, N/2] (column 2j in the low nibble of byte j), scales fp32 [M, ceil(N/32)].
    NVFP4 g16: codes [M, N/2] E2M1 pairs, scales E4M3 bytes (uint8) [M, ceil(N/16)].
    """
    if fmt not in QUANT_BLOCK:
        raise ValueError(f"unknown quantisation format {fmt}")
    M, K = X.shape
    N = W.shape[0]
    _mat(X, "X", torch.bfloat16)
    _mat(W, "W", torch.bfloat16)
    _vec(b, "b", torch.bfloat16, N)
    _vec(inv_smooth, "inv_smooth", torch.float32, N)
    qbytes = N if fmt == QUANT_FP8_1X128 else N // 2
    nblocks = -(-N // QUANT_BLOCK[fmt])
    sdt = torch.uint8 if fmt == QUANT_NVFP4_G16 else torch.float32
    if Yq is None:  # row pitch rounded up to 16 bytes, as the TMA store needs
        Yq = _out(M, qbytes, torch.uint8, X.device)
    if scales is None:
        scales = torch.empty((M, nblocks), dtype=sdt, device=X.device)
    _mat(Yq, "Yq", torch.uint8)
    _mat(scales, "scales", sdt)
    st = load().fused_linear_quant(_ptr(X), _ptr(W), _ptr(b), _ptr(inv_smooth), _ptr(Yq), _ptr(scales), M, N, K,
                                   _ld(X, K, K),
                                   _ld(W, K, K), _ld(Yq, qbytes, qbytes), _ld(scales, nblocks, nblocks), int(fmt),
                                   _stream(stream))
    _check("fused_linear_quant", st)
    return Yq, scales


def fused_dgrad_gelu(dZ, W, H, mode: str = "tanh", dH=None, stream=None):
    """dH = (dZ W) * GELU'(H): the next layer's weight W [K, N] as stored, H the saved pre-activation."""
    M, K = dZ.shape
    if W.shape[0] != K:
        raise ValueError("W must be [K, N] with K = dZ.shape[1]")
    N = W.shape[1]
    _mat(dZ, "dZ", torch.bfloat16)
    _mat(W, "W", torch.bfloat16)
    _mat(H, "H", torch.bfloat16)
    if tuple(H.shape) != (M, N):
        raise ValueError("H must be [M, N]")
    if dH is None:
        dH = _out(M, N, torch.bfloat16, dZ.device)
    _mat(dH, "dH", torch.bfloat16)
    if mode not in ("tanh", "erf"):
        raise ValueError("mode must be 'tanh' or 'erf'")
    st = load().fused_dgrad_gelu(_ptr(dZ), _ptr(W), _ptr(H), _ptr(dH), M, N, K, _ld(dZ, K, K), _ld(W, N, N),
                                 _ld(H, N, N), _ld(dH, N, N), FL_GELU_TANH if mode == "tanh" else FL_GELU_ERF,
                                 _stream(stream))
    _check("fused_dgrad_gelu", st)
    return dH


def fused_swiglu_bwd(dO, Wd, G, U, dGU=None, stream=None):
    """SwiGLU backward through the down projection Wd [K, N] (as stored): returns dGU [M, 2N]
    with dg at column 2n and du at column 2n + 1."""
    M, K = dO.shape
    if Wd.shape[0] != K:
        raise ValueError("Wd must be [K, N] with K = dO.shape[1]")
    N = Wd.shape[1]
    _mat(dO, "dO", torch.bfloat16)
    _mat(Wd, "Wd", torch.bfloat16)
    _mat(G, "G", torch.bfloat16)
    _mat(U, "U", torch.bfloat16)
    if tuple(G.shape) != (M, N) or tuple(U.shape) != (M, N) or _ld(G, N, N) != _ld(U, N, N):
        raise ValueError("G and U must be [M, N] with one shared pitch")
    if dGU is None:
        dGU = _out(M, 2 * N, torch.bfloat16, dO.device)
    _mat(dGU, "dGU", torch.bfloat16)
    st = load().fused_swiglu_bwd(_ptr(dO), _ptr(Wd), _ptr(G), _ptr(U), _ptr(dGU), M, N, K, _ld(dO, K, K),
                                 _ld(Wd, N, N), _ld(G, N, N), _ld(dGU, 2 * N, 2 * N), _stream(stream))
    _check("fused_swiglu_bwd", st)
    return dGU


def device_status(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device-wide failure code."""
    return load().fl_device_status(_stream(stream))


def check_device_status(workspace=None, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the failure code recorded in `workspace`
    (a workspace of the RMSNorm + FP8 or cross-entropy calls); None: the device-wide word."""
    return load().fl_check_device_status(_ptr(workspace), _stream(stream))


def set_cooperative_launch(enable: bool) -> None:
    """Cooperative attribute on the RMSNorm prefill launch (default on); off only for profilers
    that refuse cooperative launches of clusters."""
    load().fl_set_cooperative_launch(1 if enable else 0)


def set_descriptor_cache(enable: bool) -> None:
    """Tensor-map descriptor cache on (default) or off (and emptied)."""
    load().fl_set_descriptor_cache(1 if enable else 0)


def descriptor_cache_stats() -> tuple[int, int]:
    """(hits, misses) of the tensor-map descriptor cache since the process started."""
    h, m = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    load().fl_descriptor_cache_stats(ctypes.byref(h), ctypes.byref(m))
    return h.value, m.value


def set_wait_timeout_ns(ns: int) -> None:
    load().fl_set_wait_timeout_ns(int(ns))


def set_max_ctas(n: int) -> None:
    load().fl_set_max_ctas(int(n))


def set_cta_pairing(enable: bool) -> None:
    """Two-CTA (cta_group::2) prefill tiles on (default) or off; results are the same."""
    load().fl_set_cta_pairing(1 if enable else 0)


DECODE_GELU, DECODE_SWIGLU, DECODE_QKV, DECODE_QKV_FP8KV, DECODE_QUANT = 0, 1, 2, 3, 4
DECODE_RESID_GAMMA, DECODE_ROWSCALE = 5, 6


def linear_decode_shape(kind: int, M: int, N: int, K: int) -> tuple[int, int, int]:
    """(CTAs per W-row tile, CTAs per SM, launches) that a decode-shaped call would use on the current
    device; (0, 0, 0) when it would run on the GEMM kernel.  N: the rows of W (SwiGLU: d_ff; QKV:
    3 * d_model; QKV + FP8 K/V: (n_heads + 2 * n_kv_heads) * head_dim; block-scaled and the chain: N)."""
    out = [ctypes.c_int(0) for _ in range(3)]
    _check("fl_linear_decode_shape", load().fl_linear_decode_shape(kind, M, N, K, *(ctypes.byref(o) for o in out)))
    return tuple(o.value for o in out)


def set_linear_decode(enable: bool) -> None:
    """Decode kernels for M <= 32 calls of fused_linear_gelu (bf16), fused_swiglu, fused_qkv_rope,
    fused_qkv_rope_fp8kv, fused_linear_quant and both chain steps on (default) or off (the prefill
    GEMM kernel then takes them)."""
    load().fl_set_linear_decode(1 if enable else 0)
