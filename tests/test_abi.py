"""The C-ABI library on the host (no GPU needed): it builds, loads, exports
every entry point the header declares, and rejects bad arguments before it
touches the device."""
import ctypes

import pytest

import gemm_epilogue_tcgen05_gb300 as fl
from gemm_epilogue_tcgen05_gb300 import build as cuda_build


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return fl.load()


def test_exports_every_declared_symbol(lib):
    names = fl.header_symbols()
    assert {"fused_linear_gelu", "fused_qkv_rope", "fused_swiglu",
            "fused_linear_residual_rmsnorm_fp8"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/fused_linear.h but not exported"


def test_every_compute_entry_point_has_a_binding_of_the_same_name(lib):
    """Each computing call the header declares (the fl_* names are queries and switches) has a
    function of the same name in the Python binding."""
    compute = [n for n in fl.header_symbols() if not n.startswith("fl_")]
    assert len(compute) >= 12
    missing = [n for n in compute if not callable(getattr(fl, n, None))]
    assert not missing, f"no binding for {missing}"


def test_status_strings_and_version(lib):
    assert fl.version() == 200
    assert fl.status_string(fl.FL_OK) == "ok"
    assert "timed out" in fl.status_string(fl.FL_ERR_TIMEOUT)
    assert fl.status_string(99) == "unknown status"


P = ctypes.c_void_p


def test_gelu_rejects_bad_arguments_on_host(lib):
    a = P(0x10000)
    # negative sizes, bad dtype / mode, missing pointers, short leading dimension
    assert lib.fused_linear_gelu(a, a, None, a, -1, 8, 8, 8, 8, 8, 1, 1, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_gelu(a, a, None, a, 8, 8, 8, 8, 8, 8, 7, 1, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_gelu(a, a, None, a, 8, 8, 8, 8, 8, 8, 1, 5, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_gelu(None, a, None, a, 8, 8, 8, 8, 8, 8, 1, 1, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_gelu(a, a, None, a, 8, 8, 16, 8, 16, 8, 1, 1, None) == fl.FL_ERR_INVALID_ARG
    # misaligned base pointer, row pitch not a multiple of 16 bytes
    assert lib.fused_linear_gelu(P(0x10002), a, None, a, 8, 8, 8, 8, 8, 8, 1, 1, None) == fl.FL_ERR_ALIGNMENT
    assert lib.fused_linear_gelu(a, a, None, a, 8, 8, 12, 12, 12, 8, 1, 1, None) == fl.FL_ERR_ALIGNMENT
    # empty problems succeed without touching the device
    assert lib.fused_linear_gelu(None, None, None, None, 0, 8, 8, 8, 8, 8, 1, 1, None) == fl.FL_OK
    assert lib.fused_linear_gelu(None, None, None, None, 8, 0, 8, 8, 8, 8, 1, 1, None) == fl.FL_OK


def test_other_entry_points_reject_bad_arguments_on_host(lib):
    a = P(0x10000)
    # QKV: head_dim other than 128, or a model width that is not a multiple of 256
    assert lib.fused_qkv_rope(a, a, None, a, a, a, None, 8, 64, 1, 64, 16, 1e4, 64, 64, 64,
                              None) == fl.FL_ERR_UNSUPPORTED
    assert lib.fused_qkv_rope(a, a, None, a, a, a, None, 8, 64, 3, 128, 16, 1e4, 64, 64, 384,
                              None) == fl.FL_ERR_UNSUPPORTED
    assert lib.fused_qkv_rope(a, a, None, a, a, a, None, 8, 64, 2, 128, 0, 1e4, 64, 64, 256,
                              None) == fl.FL_ERR_INVALID_ARG  # no positions and no sequence length
    assert lib.fused_qkv_rope(a, a, None, a, a, a, None, 8, 64, 2, 128, 16, -1.0, 64, 64, 256,
                              None) == fl.FL_ERR_INVALID_ARG
    # SwiGLU: misaligned up-projection weights
    assert lib.fused_swiglu(a, a, P(0x10008), None, None, a, 8, 8, 8, 8, 8, 8, None) == fl.FL_ERR_ALIGNMENT
    # RMSNorm: missing gamma, negative eps, FP8 pitch not a multiple of 16
    f = ctypes.c_float
    assert lib.fused_linear_residual_rmsnorm_fp8(a, a, None, a, None, f(1e-6), a, a, None, 8, 16, 8, 8, 8, 16, 16,
                                                 a, 1 << 20, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_residual_rmsnorm_fp8(a, a, None, a, a, f(-1.0), a, a, None, 8, 16, 8, 8, 8, 16, 16,
                                                 a, 1 << 20, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_residual_rmsnorm_fp8(a, a, None, a, a, f(1e-6), a, a, None, 8, 24, 8, 8, 8, 24, 24,
                                                 a, 1 << 20, None) == fl.FL_ERR_ALIGNMENT
    # h_out: may not overlap the residual Z (same pitch), must be 16-byte aligned
    z = 0x100000
    for h in (z, z + 16 * 2 * 7, z - 16):  # same base, inside the last row, one row-end before the start
        assert lib.fused_linear_residual_rmsnorm_fp8(a, a, None, P(z), a, f(1e-6), a, a, P(h), 8, 16, 8, 8, 8, 16,
                                                     16, a, 1 << 20, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_residual_rmsnorm_fp8(a, a, None, P(z), a, f(1e-6), a, a, P(z + 4096 + 8), 8, 16, 8, 8,
                                                 8, 16, 16, a, 1 << 20, None) == fl.FL_ERR_ALIGNMENT


def test_quant_rejects_bad_arguments_on_host(lib):
    a = P(0x10000)
    # unknown format, odd N for a 4-bit format, short scale pitch, code pitch not a multiple of 16
    assert lib.fused_linear_quant(a, a, None, None, a, a, 8, 32, 16, 16, 16, 32, 4, 3, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_quant(a, a, None, None, a, a, 8, 33, 16, 16, 16, 32, 4, 1, None) == fl.FL_ERR_UNSUPPORTED
    assert lib.fused_linear_quant(a, a, None, None, a, a, 8, 256, 16, 16, 16, 128, 7, 1, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_quant(a, a, None, None, a, a, 8, 264, 16, 16, 16, 264, 3, 0, None) == fl.FL_ERR_ALIGNMENT
    assert lib.fused_linear_quant(a, a, None, None, a, None, 8, 32, 16, 16, 16, 32, 1, 0, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_quant(None, None, None, None, None, None, 0, 32, 16, 16, 16, 32, 1, 0, None) == fl.FL_OK
    # the inverse smoothing vector must be 16-byte aligned like every other operand
    assert lib.fused_linear_quant(a, a, None, P(0x10004), a, a, 8, 32, 16, 16, 16, 32, 1, 0,
                                  None) == fl.FL_ERR_ALIGNMENT


def test_qkv_fp8kv_rejects_bad_arguments_on_host(lib):
    a = P(0x10000)
    f = ctypes.c_float
    # odd kv head count, head_dim other than 128, short scale pitch, KV pitch not a multiple of 16
    assert lib.fused_qkv_rope_fp8kv(a, a, None, a, a, a, a, a, None, 8, 64, 2, 1, 128, 16, f(1e4), 64, 64, 256, 128,
                                    1, None) == fl.FL_ERR_UNSUPPORTED
    assert lib.fused_qkv_rope_fp8kv(a, a, None, a, a, a, a, a, None, 8, 64, 4, 4, 64, 16, f(1e4), 64, 64, 256, 256,
                                    4, None) == fl.FL_ERR_UNSUPPORTED
    assert lib.fused_qkv_rope_fp8kv(a, a, None, a, a, a, a, a, None, 8, 64, 2, 2, 128, 16, f(1e4), 64, 64, 256, 256,
                                    1, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_qkv_rope_fp8kv(a, a, None, a, a, a, a, a, None, 8, 64, 2, 2, 128, 16, f(1e4), 64, 64, 256, 264,
                                    2, None) == fl.FL_ERR_ALIGNMENT
    assert lib.fused_qkv_rope_fp8kv(a, a, None, a, a, a, None, a, None, 8, 64, 2, 2, 128, 16, f(1e4), 64, 64, 256,
                                    256, 2, None) == fl.FL_ERR_INVALID_ARG


def test_backward_entry_points_reject_bad_arguments_on_host(lib):
    a = P(0x10000)
    # bad GELU form, W pitch below N, H pitch not a multiple of 8 elements, missing U
    assert lib.fused_dgrad_gelu(a, a, a, a, 8, 16, 8, 8, 16, 16, 16, 7, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_dgrad_gelu(a, a, a, a, 8, 16, 8, 8, 8, 16, 16, 1, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_dgrad_gelu(a, a, a, a, 8, 16, 8, 8, 16, 20, 16, 1, None) == fl.FL_ERR_ALIGNMENT
    assert lib.fused_swiglu_bwd(a, a, a, None, a, 8, 16, 8, 8, 16, 16, 32, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_swiglu_bwd(a, a, a, a, a, 8, 16, 8, 8, 16, 16, 24, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_swiglu_bwd(None, None, None, None, None, 0, 16, 8, 8, 16, 16, 32, None) == fl.FL_OK


def test_host_pipeline_rejects_bad_arguments_on_host(lib):
    a = P(0x10000)
    need = lib.fl_linear_gelu_host_buffer_bytes(64, 256, 64)
    assert need >= 2 * (64 * 64 + 256 * 64 + 256 + 64 * 256)
    # bad mode, missing device buffer, N not a multiple of 8, buffer too small, misaligned buffer
    assert lib.fused_linear_gelu_host(a, a, None, a, 64, 256, 64, 3, a, need, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_gelu_host(a, a, None, a, 64, 256, 64, 1, None, need, None) == fl.FL_ERR_INVALID_ARG
    assert lib.fused_linear_gelu_host(a, a, None, a, 64, 252, 64, 1, a, need, None) == fl.FL_ERR_ALIGNMENT
    assert lib.fused_linear_gelu_host(a, a, None, a, 64, 256, 64, 1, a, need - 1, None) == fl.FL_ERR_WORKSPACE
    assert lib.fused_linear_gelu_host(a, a, None, a, 64, 256, 64, 1, P(0x10010), need, None) == fl.FL_ERR_ALIGNMENT
    assert lib.fused_linear_gelu_host(None, None, None, None, 0, 256, 64, 1, None, 0, None) == fl.FL_OK


def test_decode_shape_query_on_host(lib):
    out = [ctypes.c_int(7) for _ in range(3)]
    refs = [ctypes.byref(o) for o in out]
    # unknown kind, negative size, null output: rejected before the device is touched
    assert lib.fl_linear_decode_shape(7, 8, 4096, 4096, *refs) == fl.FL_ERR_INVALID_ARG
    assert lib.fl_linear_decode_shape(-1, 8, 4096, 4096, *refs) == fl.FL_ERR_INVALID_ARG
    assert lib.fl_linear_decode_shape(fl.DECODE_GELU, -1, 4096, 4096, *refs) == fl.FL_ERR_INVALID_ARG
    assert lib.fl_linear_decode_shape(fl.DECODE_GELU, 8, 4096, 4096, None, refs[1], refs[2]) == fl.FL_ERR_INVALID_ARG
    # not a decode call (M outside 1..32, or nothing to do): FL_OK and all zeros, no device needed
    for M, N, K in ((33, 4096, 4096), (0, 4096, 4096), (8, 0, 4096), (8, 4096, 0)):
        for o in out:
            o.value = 7
        assert lib.fl_linear_decode_shape(fl.DECODE_SWIGLU, M, N, K, *refs) == fl.FL_OK
        assert [o.value for o in out] == [0, 0, 0]
    assert fl.linear_decode_shape(fl.DECODE_QKV, 64, 12288, 4096) == (0, 0, 0)
    assert fl.linear_decode_shape(fl.DECODE_QUANT, 64, 16384, 4096) == (0, 0, 0)
    assert fl.linear_decode_shape(fl.DECODE_RESID_GAMMA, 64, 4096, 4096) == (0, 0, 0)
    assert fl.linear_decode_shape(fl.DECODE_ROWSCALE, 64, 14336, 4096) == (0, 0, 0)


def test_workspace_status_check_and_diagnostic_switches_on_host(lib):
    # a workspace that is not 256-byte aligned cannot hold a status record
    assert lib.fl_check_device_status(P(0x10010), None) == fl.FL_ERR_ALIGNMENT
    # the diagnostic switches take any int and need no device
    for f in (lib.fl_set_cooperative_launch, lib.fl_set_descriptor_cache):
        f(0)
        f(1)
    h, m = ctypes.c_ulonglong(7), ctypes.c_ulonglong(7)
    lib.fl_descriptor_cache_stats(ctypes.byref(h), ctypes.byref(m))
    assert h.value >= 0 and m.value >= 0
    lib.fl_descriptor_cache_stats(None, None)


def test_noalloc_rejects_bad_arguments_before_any_device_work(lib):
    f = lib.fused_linear_residual_rmsnorm_fp8_noalloc
    I64 = ctypes.c_int64
    f.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, I64, I64, I64, I64,
                  P]
    a = P(0x10000)
    assert f(a, a, None, a, a, 1e-6, a, a, -1, 16, 8, 8, 8, 16, 16, None) == fl.FL_ERR_INVALID_ARG
    assert f(a, a, None, a, a, -1.0, a, a, 8, 16, 8, 8, 8, 16, 16, None) == fl.FL_ERR_INVALID_ARG
    assert f(None, None, None, None, None, 1e-6, None, None, 0, 16, 8, 8, 8, 16, 16, None) == fl.FL_OK
