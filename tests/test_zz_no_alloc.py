"""The no-allocation RMSNorm + FP8 entry point, called through the C ABI.

Some callers cannot allocate device memory while they run: a serving loop
that must not stall in the allocator (cudaMalloc can synchronise the whole
device), or a plugin whose host framework owns all GPU memory and hands it
none.  They cannot pass a workspace, so
fused_linear_residual_rmsnorm_fp8_noalloc uses a scratch array built into the
library instead.  These tests check, on two calls in a row (the second call
reuses the scratch the first one left behind), for a decode and a prefill
shape, that it produces the codes and scales of the workspace entry point and
of the fp64 oracle, and that shapes it cannot serve are rejected.  The file
is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gemm_epilogue_tcgen05_gb300 as fl
import oracle
import synthetic as syn
from parity_utils import assert_fp8_close, dev_bf16, f64

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    f = fl.load().fused_linear_residual_rmsnorm_fp8_noalloc
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, I, I, I, I64, I64, I64, I64, P]
    f.restype = I
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("M,N,K,bias", [(32, 4096, 2048, False), (300, 1024, 520, True)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(M, N, K, bias):
    Xh = syn.draw(0, syn.STREAM_X, (M, K), 0.0, 1.0, "bf16")
    Wh = syn.draw(0, syn.STREAM_W, (N, K), 0.0, K ** -0.5, "bf16")
    bh = syn.draw(0, syn.STREAM_B, (N,), 0.0, 0.02, "bf16") if bias else None
    Zh = syn.draw(0, syn.STREAM_Z, (M, N), 0.0, 1.0, "bf16")
    gh = syn.draw(0, syn.STREAM_GAMMA, (N,), 1.0, 0.1, "bf16")
    X, W, Z, g = dev_bf16(Xh), dev_bf16(Wh), dev_bf16(Zh), dev_bf16(gh)
    b = dev_bf16(bh) if bias else None
    q_ws, s_ws = fl.fused_linear_residual_rmsnorm_fp8(X, W, b, Z, g, 1e-6)
    q_ws, s_ws = q_ws.cpu().numpy(), s_ws.cpu().numpy().astype(np.float64)
    q_or, s_or, _ = oracle.rmsnorm_fp8(f64(Xh), f64(Wh), None if bh is None else f64(bh), f64(Zh), f64(gh), 1e-6)
    fn = _noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        Yq = torch.zeros((M, N), dtype=torch.uint8, device="cuda")
        sc = torch.zeros(M, dtype=torch.float32, device="cuda")
        st = fn(_ptr(X), _ptr(W), _ptr(b), _ptr(Z), _ptr(g), 1e-6, _ptr(Yq), _ptr(sc), M, N, K,
                X.stride(0), W.stride(0), Z.stride(0), Yq.stride(0), stream)
        assert st == fl.FL_OK, fl.status_string(st)
        assert fl.device_status() == fl.FL_OK
        q, s = Yq.cpu().numpy(), sc.cpu().numpy().astype(np.float64)
        assert_fp8_close(q, s, q_ws, s_ws, f"noalloc {M}x{N}x{K} call {call} vs workspace entry point")
        assert_fp8_close(q, s, q_or, s_or, f"noalloc {M}x{N}x{K} call {call} vs oracle")
    # the Python binding of the same entry point: the same call, bit for bit
    Yb = torch.zeros((M, N), dtype=torch.uint8, device="cuda")
    sb = torch.zeros(M, dtype=torch.float32, device="cuda")
    fl.fused_linear_residual_rmsnorm_fp8_noalloc(X, W, b, Z, g, Yb, sb, 1e-6)
    assert torch.equal(Yb, Yq) and torch.equal(sb, sc)


def test_noalloc_rejects_shapes_it_cannot_serve():
    fn = _noalloc_fn()
    a = ctypes.c_void_p(torch.empty(16, dtype=torch.uint8, device="cuda").data_ptr())
    # prefill partials alone need 32 MiB: beyond the 8 MiB scratch
    M, N, K = 8192, 131072, 64
    assert fl.rmsnorm_fp8_workspace_bytes(M, N, K) > (8 << 20)
    assert fn(a, a, None, a, a, 1e-6, a, a, M, N, K, K, K, N, N, None) == fl.FL_ERR_WORKSPACE
    # a row wider than 256 columns per SM fits the scratch but not the prefill kernel's grid
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 64, 256 * (sms + 1), 64
    assert fl.rmsnorm_fp8_workspace_bytes(M, N, K) <= (8 << 20)
    assert fn(a, a, None, a, a, 1e-6, a, a, M, N, K, K, K, N, N, None) == fl.FL_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert fl.device_status() == fl.FL_OK
