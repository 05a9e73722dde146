"""The no-allocation RMSNorm + FP8 entry point, called through the C ABI.

Some callers cannot allocate device memory while they run (a decode step
being recorded into a CUDA graph, a serving loop that must not stall in the
allocator, a plugin whose host framework owns all GPU memory), so they cannot
pass a workspace.  fused_linear_residual_rmsnorm_fp8_noalloc uses a scratch
array built into the library instead.  This test checks that it produces what
the workspace entry point produces, on two calls in a row (the second call
reuses the scratch the first one left behind), for a decode and a prefill
shape.  It lives in its own file named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gemm_epilogue_tcgen05_gb300 as fl
import synthetic as syn
from parity_utils import assert_fp8_close, dev_bf16

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
def test_noalloc_matches_workspace_entry_point_twice(M, N, K, bias):
    X = dev_bf16(syn.draw(0, syn.STREAM_X, (M, K), 0.0, 1.0, "bf16"))
    W = dev_bf16(syn.draw(0, syn.STREAM_W, (N, K), 0.0, K ** -0.5, "bf16"))
    b = dev_bf16(syn.draw(0, syn.STREAM_B, (N,), 0.0, 0.02, "bf16")) if bias else None
    Z = dev_bf16(syn.draw(0, syn.STREAM_Z, (M, N), 0.0, 1.0, "bf16"))
    g = dev_bf16(syn.draw(0, syn.STREAM_GAMMA, (N,), 1.0, 0.1, "bf16"))
    q_ref, s_ref = fl.fused_linear_residual_rmsnorm_fp8(X, W, b, Z, g, 1e-6)
    q_ref, s_ref = q_ref.cpu().numpy(), s_ref.cpu().numpy().astype(np.float64)
    fn = _noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        Yq = torch.zeros((M, N), dtype=torch.uint8, device="cuda")
        sc = torch.zeros(M, dtype=torch.float32, device="cuda")
        st = fn(_ptr(X), _ptr(W), _ptr(b), _ptr(Z), _ptr(g), 1e-6, _ptr(Yq), _ptr(sc), M, N, K,
                X.stride(0), W.stride(0), Z.stride(0), Yq.stride(0), stream)
        assert st == fl.FL_OK, fl.status_string(st)
        assert fl.device_status() == fl.FL_OK
        assert_fp8_close(Yq.cpu().numpy(), sc.cpu().numpy().astype(np.float64), q_ref, s_ref,
                         f"noalloc {M}x{N}x{K}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fn = _noalloc_fn()
    M, N, K = 8192, 131072, 64  # prefill partials alone need 32 MiB
    assert fl.rmsnorm_fp8_workspace_bytes(M, N, K) > (8 << 20)
    a = ctypes.c_void_p(torch.empty(16, dtype=torch.uint8, device="cuda").data_ptr())
    st = fn(a, a, None, a, a, 1e-6, a, a, M, N, K, K, K, N, N, None)
    assert st == fl.FL_ERR_WORKSPACE
