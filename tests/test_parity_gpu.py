"""GPU parity: every entry point, through the C ABI, against the fp64 oracle.

Small cases span several tiles with ragged edges in M, N and K and are
compared element by element.  The full-size workloads run in the same launch
configuration the benchmark times and are compared on sampled rows (every
column of each sampled row, so every N-tile is covered).
"""
import numpy as np
import pytest
import torch

import gemm_epilogue_tcgen05_gb300 as fl
import oracle
import synthetic as syn
from parity_utils import (assert_bf16_close, assert_f32_close, assert_fp8_close, assert_quant_close, dev_bf16,
                          dev_f32, f64, host, sample_rows)
from parity_utils import assert_loss_close as _assert_loss_close
from parity_utils import check_kv_fp8 as _check_kv_fp8
from parity_utils import qkv_ref as _qkv_ref
from parity_utils import assert_ws_reset as _assert_ws_reset
from parity_utils import rms_case as _rms_case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    fl.set_max_ctas(0)
    fl.set_wait_timeout_ns(0)
    fl.set_cta_pairing(True)
    yield
    fl.set_max_ctas(0)
    fl.set_wait_timeout_ns(0)
    fl.set_cta_pairing(True)
    assert fl.device_status() == fl.FL_OK


def _draw(shape, stream, std=1.0, mean=0.0, seed=0, dtype="bf16"):
    return syn.draw(seed, stream, shape, mean, std, dtype)


# ------------------------------------------------------------------ GELU
@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", ["tanh", "erf"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (130, 264, 72), (300, 520, 200), (256, 256, 1024)])
def test_gelu_small(mode, M, N, K, seed):
    X = _draw((M, K), syn.STREAM_X, seed=seed)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=seed)
    b = _draw((N,), syn.STREAM_B, 0.02, seed=seed)
    Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), dev_bf16(b), mode=mode)
    m = oracle.GELU_TANH if mode == "tanh" else oracle.GELU_ERF
    assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), f64(b), m), f"gelu {mode} {M}x{N}x{K} seed {seed}")


def test_gelu_no_bias_and_k_zero():
    M, N, K = 70, 296, 96  # 296 bf16 = 592 bytes: a 16-byte row pitch
    X, W = _draw((M, K), syn.STREAM_X), _draw((N, K), syn.STREAM_W, K ** -0.5)
    Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), None, mode="tanh")
    assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), None, oracle.GELU_TANH), "no bias")
    b = _draw((N,), syn.STREAM_B, 0.5)
    Xe = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    We = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    Y0 = fl.fused_linear_gelu(Xe, We, dev_bf16(b), mode="erf")
    ref = oracle.gelu(np.broadcast_to(f64(b), (M, N)).copy(), oracle.GELU_ERF)
    assert_bf16_close(host(Y0), ref, "K=0")


def test_gelu_empty_is_noop():
    Y = torch.full((0, 16), 7.0, dtype=torch.bfloat16, device="cuda")
    fl.fused_linear_gelu(torch.empty((0, 8), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda"), None, Y=Y)


def test_gelu_strided_operands_and_few_ctas():
    # leading dimensions wider than the rows, and 3 CTAs walking 5x5 tiles each
    M, N, K = 640, 1280, 256
    X = _draw((M, K + 64), syn.STREAM_X)
    W = _draw((N, K + 32), syn.STREAM_W, K ** -0.5)
    b = _draw((N,), syn.STREAM_B, 0.02)
    Xd, Wd = dev_bf16(X)[:, :K], dev_bf16(W)[:, :K]
    Yfull = torch.zeros((M, N + 40), dtype=torch.bfloat16, device="cuda")
    fl.set_max_ctas(3)
    fl.fused_linear_gelu(Xd, Wd, dev_bf16(b), Y=Yfull[:, :N], mode="tanh")
    ref = oracle.linear_gelu(f64(X[:, :K]), f64(W[:, :K]), f64(b), oracle.GELU_TANH)
    assert_bf16_close(host(Yfull[:, :N]), ref, "strided/few CTAs")
    assert torch.count_nonzero(Yfull[:, N:]) == 0, "wrote outside the output columns"


def test_gelu_tiny_fp32_workload():
    w = syn.WORKLOADS["tiny_gelu_erf_f32"]
    ops = syn.make_operands(w)
    Y = fl.fused_linear_gelu(dev_f32(ops["X"]), dev_f32(ops["W"]), dev_f32(ops["b"]), mode="erf")
    ref = oracle.linear_gelu(ops["X"].astype(np.float64), ops["W"].astype(np.float64),
                             ops["b"].astype(np.float64), oracle.GELU_ERF)
    assert_f32_close(host(Y), ref, "tiny fp32 erf")


@pytest.mark.parametrize("mode", ["erf", "tanh"])
@pytest.mark.parametrize("M,N,K,bias", [(1, 8, 8, True), (130, 264, 72, True), (300, 520, 200, False),
                                        (64, 256, 1000, True)])
def test_gelu_fp32_tf32x3(mode, M, N, K, bias):
    """fp32 operands on the tensor cores as three TF32 products: within 1e-4 of the oracle."""
    X = _draw((M, K), syn.STREAM_X, dtype="f32")
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, dtype="f32")
    b = _draw((N,), syn.STREAM_B, 0.5, dtype="f32") if bias else None
    Y = fl.fused_linear_gelu(dev_f32(X), dev_f32(W), dev_f32(b) if bias else None, mode=mode)
    m = oracle.GELU_ERF if mode == "erf" else oracle.GELU_TANH
    ref = oracle.linear_gelu(f64(X, "f32"), f64(W, "f32"), f64(b, "f32") if bias else None, m)
    assert_f32_close(host(Y), ref, f"fp32 {mode} {M}x{N}x{K}")


def test_gelu_fp32_strided_and_k_zero():
    M, N, K = 70, 296, 96
    X = _draw((M, K + 4), syn.STREAM_X, dtype="f32")
    W = _draw((N, K + 8), syn.STREAM_W, K ** -0.5, dtype="f32")
    Yfull = torch.zeros((M, N + 12), dtype=torch.float32, device="cuda")
    fl.fused_linear_gelu(dev_f32(X)[:, :K], dev_f32(W)[:, :K], None, Y=Yfull[:, :N], mode="erf")
    ref = oracle.linear_gelu(f64(X[:, :K], "f32"), f64(W[:, :K], "f32"), None, oracle.GELU_ERF)
    assert_f32_close(host(Yfull[:, :N]), ref, "fp32 strided")
    assert torch.count_nonzero(Yfull[:, N:]) == 0
    b = _draw((N,), syn.STREAM_B, 0.5, dtype="f32")
    Y0 = fl.fused_linear_gelu(torch.empty((M, 0), dtype=torch.float32, device="cuda"),
                              torch.empty((N, 0), dtype=torch.float32, device="cuda"), dev_f32(b), mode="tanh")
    assert_f32_close(host(Y0), oracle.gelu(np.broadcast_to(f64(b, "f32"), (M, N)).copy(), oracle.GELU_TANH), "fp32 K=0")


def test_gelu_full_workload_sampled():
    w = syn.WORKLOADS["gelu_tanh_8192x16384x4096"]
    ops = syn.make_operands(w)
    Y = fl.fused_linear_gelu(dev_bf16(ops["X"]), dev_bf16(ops["W"]), dev_bf16(ops["b"]), mode="tanh")
    rows = sample_rows(w.M)
    got = host(Y[torch.from_numpy(rows).cuda()])
    ref = oracle.linear_gelu(f64(ops["X"][rows]), f64(ops["W"]), f64(ops["b"]), oracle.GELU_TANH)
    assert_bf16_close(got, ref, "gelu full")


@pytest.mark.parametrize("pairing", [True, False])
def test_every_prefill_epilogue_in_both_cta_modes(pairing):
    # one CTA per 128-row tile, or a CTA pair per 256-row tile (cta_group::2); 3 row blocks
    # make the pair's second half run past M on the last tile
    fl.set_cta_pairing(pairing)
    M, N, K = 300, 512, 200
    X = _draw((M, K), syn.STREAM_X)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5)
    Wu = _draw((N, K), syn.STREAM_WUP, K ** -0.5)
    b = _draw((N,), syn.STREAM_B, 0.02)
    Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), dev_bf16(b), mode="tanh")
    assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), f64(b), oracle.GELU_TANH), "gelu")
    Ys = fl.fused_swiglu(dev_bf16(X), dev_bf16(W), dev_bf16(Wu), dev_bf16(b), None)
    assert_bf16_close(host(Ys), oracle.swiglu(f64(X), f64(W), f64(Wu), f64(b), None), "swiglu")
    H, D = 2, 128
    Wq = _draw((3 * H * D, K), syn.STREAM_W, K ** -0.5)
    q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, head_dim=D, seq_len=77)
    ref = oracle.qkv_rope(f64(X), f64(Wq), None, H, D, 1e4, np.arange(M) % 77)
    assert_bf16_close(host(torch.cat([q, k, v], 1)), ref, "qkv")
    Z = _draw((M, N), syn.STREAM_Z)
    g = _draw((N,), syn.STREAM_GAMMA, 0.1, 1.0)
    qq, ss = fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(X), dev_bf16(W), dev_bf16(b), dev_bf16(Z),
                                                  dev_bf16(g), 1e-6)
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), f64(b), f64(Z), f64(g), 1e-6)
    assert_fp8_close(qq.cpu().numpy(), ss.cpu().numpy().astype(np.float64), q_ref, s_ref, "rmsnorm")


@pytest.mark.parametrize("pairing", [True, False])
def test_gelu_many_tiles_per_cta_both_modes(pairing):
    # two CTAs (one pair) walk 3 x 6 tiles: accumulator buffers and stage phases wrap many times
    fl.set_cta_pairing(pairing)
    fl.set_max_ctas(2)
    M, N, K = 768, 1536, 320
    X = _draw((M, K), syn.STREAM_X, seed=5)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=5)
    Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), None, mode="erf")
    assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), None, oracle.GELU_ERF), "many tiles")


# ------------------------------------------------------------------ QKV + RoPE
def test_qkv_rope_small_bias_and_positions():
    M, K, H, D = 300, 192, 2, 128
    X = _draw((M, K), syn.STREAM_X)
    Wq = _draw((3 * H * D, K), syn.STREAM_W, K ** -0.5)
    bq = _draw((3 * H * D,), syn.STREAM_B, 0.02)
    q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), dev_bf16(bq), n_heads=H, head_dim=D, seq_len=100)
    ref = _qkv_ref(X, Wq, bq, H, D, np.arange(M) % 100)
    d = H * D
    assert_bf16_close(host(q), ref[:, :d], "Q")
    assert_bf16_close(host(k), ref[:, d:2 * d], "K (rotated)")
    assert_bf16_close(host(v), ref[:, 2 * d:], "V")
    pos = np.random.default_rng(1).integers(0, 8192, size=M).astype(np.int32)
    q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, head_dim=D,
                                positions=torch.from_numpy(pos).cuda())
    ref = _qkv_ref(X, Wq, None, H, D, pos)
    assert_bf16_close(host(torch.cat([q, k, v], 1)), ref, "explicit positions")


def test_qkv_rope_full_workload_sampled():
    w = syn.WORKLOADS["qkv_rope_8192x12288x4096"]
    ops = syn.make_operands(w)
    q, k, v = fl.fused_qkv_rope(dev_bf16(ops["X"]), dev_bf16(ops["W"]), None, n_heads=w.n_heads,
                                head_dim=w.head_dim, seq_len=w.seq_len, theta=w.theta)
    rows = sample_rows(w.M)
    ri = torch.from_numpy(rows).cuda()
    got = host(torch.cat([q[ri], k[ri], v[ri]], 1))
    ref = _qkv_ref(ops["X"][rows], ops["W"], None, w.n_heads, w.head_dim, rows % w.seq_len, w.theta)
    assert_bf16_close(got, ref, "qkv full")


# ------------------------------------------------------------------ decode shapes (M <= 32) of GELU, SwiGLU, QKV
@pytest.mark.parametrize("decode", [True, False])
@pytest.mark.parametrize("M,N,K", [(32, 1024, 1024), (5, 4096, 512), (17, 8000, 320), (1, 16384, 256),
                                   (32, 1000, 200), (9, 136, 64), (32, 4096, 2048), (32, 4096, 4096),
                                   (7, 6100, 4000), (3, 2048, 8192), (32, 3072, 8192), (32, 13312, 2048),
                                   (17, 11200, 4096), (5, 12800, 4096), (3, 20480, 512)])
def test_gelu_decode_shapes(decode, M, N, K):
    """Swap-AB decode kernel and, with the decode path off, the GEMM kernel on the same small M.  On
    152 SMs the decode shapes take one CTA per tile (the first six: few k blocks, or 128 tiles),
    clusters of 2, of 4, of 4 at two CTAs per SM (48 ragged tiles, ragged K), of 8 at two per SM
    (16 and 24 tiles), of 2 at two per SM, of 3 at two per SM (uneven shares of the tile, ragged N),
    of 2 at two per SM again (100 tiles: more clusters of 3 than fit at once), and one CTA per tile at
    two per SM (160 tiles, more than SMs)."""
    fl.set_linear_decode(decode)
    try:
        X = _draw((M, K), syn.STREAM_X, seed=M)
        W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=M)
        b = _draw((N,), syn.STREAM_B, 0.3, seed=M)
        for mode, bias in (("tanh", b), ("erf", None)):
            Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), None if bias is None else dev_bf16(bias), mode=mode)
            m = oracle.GELU_TANH if mode == "tanh" else oracle.GELU_ERF
            assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), None if bias is None else f64(bias), m),
                              f"gelu decode={decode} {mode} {M}x{N}x{K}")
    finally:
        fl.set_linear_decode(True)


_DECODE_SHAPES = [  # (kind, M, N = rows of W, K) -> (CTAs per tile, CTAs per SM, launches) on 152 SMs
    (fl.DECODE_GELU, 32, 1024, 1024, (1, 1, 1)), (fl.DECODE_GELU, 5, 4096, 512, (1, 1, 1)),
    (fl.DECODE_GELU, 17, 8000, 320, (1, 1, 1)), (fl.DECODE_GELU, 1, 16384, 256, (1, 1, 1)),
    (fl.DECODE_GELU, 32, 1000, 200, (1, 1, 1)), (fl.DECODE_GELU, 9, 136, 64, (1, 1, 1)),
    (fl.DECODE_GELU, 32, 4096, 2048, (2, 1, 1)), (fl.DECODE_GELU, 32, 4096, 4096, (4, 1, 1)),
    (fl.DECODE_GELU, 7, 6100, 4000, (4, 2, 1)), (fl.DECODE_GELU, 3, 2048, 8192, (8, 2, 1)),
    (fl.DECODE_GELU, 32, 3072, 8192, (8, 2, 1)), (fl.DECODE_GELU, 32, 13312, 2048, (2, 2, 1)),
    (fl.DECODE_GELU, 17, 11200, 4096, (3, 2, 1)), (fl.DECODE_GELU, 5, 12800, 4096, (2, 2, 1)),
    (fl.DECODE_GELU, 3, 20480, 512, (1, 2, 1)), (fl.DECODE_GELU, 3, 40960, 136, (1, 2, 2)),
    (fl.DECODE_GELU, 32, 16384, 4096, (1, 1, 1)),
    (fl.DECODE_SWIGLU, 32, 1024, 1024, (1, 1, 1)), (fl.DECODE_SWIGLU, 9, 5000, 768, (1, 1, 1)),
    (fl.DECODE_SWIGLU, 4, 3000, 4096, (4, 2, 1)), (fl.DECODE_SWIGLU, 6, 6000, 4096, (3, 2, 1)),
    (fl.DECODE_SWIGLU, 5, 10000, 256, (1, 2, 1)), (fl.DECODE_SWIGLU, 3, 20000, 136, (1, 2, 2)),
    (fl.DECODE_SWIGLU, 32, 14336, 4096, (1, 2, 1)),
    (fl.DECODE_QKV, 32, 1536, 1024, (1, 1, 1)), (fl.DECODE_QKV, 7, 6144, 4096, (4, 2, 1)),
    (fl.DECODE_QKV, 1, 12288, 4096, (3, 2, 1)), (fl.DECODE_QKV, 2, 1536, 8192, (8, 1, 1)),
    (fl.DECODE_QKV, 1, 24576, 256, (1, 2, 1)), (fl.DECODE_QKV, 3, 49152, 136, (1, 2, 2)),
    (fl.DECODE_QKV_FP8KV, 7, 6144, 4096, (4, 2, 1)), (fl.DECODE_QKV_FP8KV, 3, 10240, 4096, (3, 2, 1)),
    (fl.DECODE_QKV_FP8KV, 5, 3072, 2048, (2, 1, 1)), (fl.DECODE_QKV_FP8KV, 2, 1536, 8192, (8, 1, 1)),
    (fl.DECODE_QKV_FP8KV, 2, 20480, 256, (1, 2, 1)), (fl.DECODE_QKV_FP8KV, 3, 40960, 136, (1, 2, 2)),
    (fl.DECODE_QKV, 64, 12288, 4096, (0, 0, 0)),
]


def test_linear_decode_launch_shapes():
    """The launch shape of every decode case the parity tests run (and of the bench rows), as the
    library reports it: on a 152-SM GB300 the cases cover one CTA per tile, clusters of 2, 4 and 8 at
    one CTA per SM, of 1, 2, 3, 4 and 8 at two per SM, and several launches; under a cap of 8 SMs a
    40-tile call takes three launches."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected shapes are those of a 152-SM GB300")
    for kind, M, N, K, want in _DECODE_SHAPES:
        assert fl.linear_decode_shape(kind, M, N, K) == want, (kind, M, N, K)
    fl.set_max_ctas(8)
    assert fl.linear_decode_shape(fl.DECODE_GELU, 3, 5000, 136) == (1, 2, 3)
    fl.set_max_ctas(0)
    fl.set_linear_decode(False)
    try:
        assert fl.linear_decode_shape(fl.DECODE_GELU, 32, 4096, 4096) == (0, 0, 0)
    finally:
        fl.set_linear_decode(True)


@pytest.mark.parametrize("decode", [True, False])
@pytest.mark.parametrize("M,N,K", [(32, 1024, 1024), (9, 5000, 768), (3, 2000, 136), (32, 200, 64),
                                   (4, 3000, 4096), (6, 6000, 4096), (5, 10000, 256)])
# 47 tiles: clusters of 4, 94: of 3, both at two CTAs per SM; 157 tiles: one CTA per tile, two per SM
def test_swiglu_decode_shapes(decode, M, N, K):
    fl.set_linear_decode(decode)
    try:
        X = _draw((M, K), syn.STREAM_X, seed=M)
        Wg, Wu = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=M), _draw((N, K), syn.STREAM_WUP, K ** -0.5, seed=M)
        bg, bu = _draw((N,), syn.STREAM_B, 0.1, seed=M), _draw((N,), syn.STREAM_BUP, 0.1, seed=M)
        Y = fl.fused_swiglu(dev_bf16(X), dev_bf16(Wg), dev_bf16(Wu), dev_bf16(bg), dev_bf16(bu))
        assert_bf16_close(host(Y), oracle.swiglu(f64(X), f64(Wg), f64(Wu), f64(bg), f64(bu)),
                          f"swiglu decode={decode} {M}x{N}x{K}")
        Y = fl.fused_swiglu(dev_bf16(X), dev_bf16(Wg), dev_bf16(Wu), None, None)
        assert_bf16_close(host(Y), oracle.swiglu(f64(X), f64(Wg), f64(Wu), None, None),
                          f"swiglu decode={decode} no bias {M}x{N}x{K}")
    finally:
        fl.set_linear_decode(True)


@pytest.mark.parametrize("decode", [True, False])
@pytest.mark.parametrize("M,H,K", [(32, 4, 1024), (7, 16, 4096), (1, 32, 4096), (20, 2, 200), (2, 4, 8192),
                                   (1, 64, 256)])
def test_qkv_rope_decode_shapes(decode, M, H, K):
    """Head tiles on one CTA each, on clusters of 4 and of 3 at two CTAs per SM (48 and 96 tiles), on
    clusters of 8 (12 tiles of K = 8192) and on one CTA each at two per SM (192 tiles); the GEMM
    kernel with the decode path off."""
    fl.set_linear_decode(decode)
    try:
        D = 128
        X = _draw((M, K), syn.STREAM_X, seed=M)
        Wq = _draw((3 * H * D, K), syn.STREAM_W, K ** -0.5, seed=M)
        bq = _draw((3 * H * D,), syn.STREAM_B, 0.02, seed=M)
        d = H * D
        q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), dev_bf16(bq), n_heads=H, head_dim=D, seq_len=5)
        ref = _qkv_ref(X, Wq, bq, H, D, np.arange(M) % 5)
        assert_bf16_close(host(torch.cat([q, k, v], 1)), ref, f"qkv decode={decode} M={M} H={H} K={K}")
        # decode positions deep into a long context (the angle reduction matters there)
        pos = np.random.default_rng(M).integers(0, 1 << 20, size=M).astype(np.int32)
        q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, head_dim=D,
                                    positions=torch.from_numpy(pos).cuda())
        ref = _qkv_ref(X, Wq, None, H, D, pos)
        assert_bf16_close(host(torch.cat([q, k, v], 1)), ref, f"qkv decode={decode} positions M={M} H={H}")
    finally:
        fl.set_linear_decode(True)


# ------------------------------------------------------------------ SwiGLU
def test_swiglu_small_ragged_with_bias():
    M, N, K = 300, 200, 136
    X = _draw((M, K), syn.STREAM_X)
    Wg, Wu = _draw((N, K), syn.STREAM_W, K ** -0.5), _draw((N, K), syn.STREAM_WUP, K ** -0.5)
    bg, bu = _draw((N,), syn.STREAM_B, 0.1), _draw((N,), syn.STREAM_BUP, 0.1)
    Y = fl.fused_swiglu(dev_bf16(X), dev_bf16(Wg), dev_bf16(Wu), dev_bf16(bg), dev_bf16(bu))
    assert_bf16_close(host(Y), oracle.swiglu(f64(X), f64(Wg), f64(Wu), f64(bg), f64(bu)), "swiglu small")


def test_swiglu_full_workload_sampled():
    w = syn.WORKLOADS["swiglu_8192x14336x4096"]
    ops = syn.make_operands(w)
    Y = fl.fused_swiglu(dev_bf16(ops["X"]), dev_bf16(ops["Wgate"]), dev_bf16(ops["Wup"]))
    rows = sample_rows(w.M)
    got = host(Y[torch.from_numpy(rows).cuda()])
    ref = oracle.swiglu(f64(ops["X"][rows]), f64(ops["Wgate"]), f64(ops["Wup"]))
    assert_bf16_close(got, ref, "swiglu full")


# ------------------------------------------------------------------ residual + RMSNorm + FP8
def _rms_run(X, W, b, Z, g, ldq=None, workspace=None):
    M, N = Z.shape
    Yq = None
    if ldq is not None:
        Yq = torch.zeros((M, ldq), dtype=torch.uint8, device="cuda")[:, :N]
    q, s = fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(X), dev_bf16(W), None if b is None else dev_bf16(b),
                                                dev_bf16(Z), dev_bf16(g), 1e-6, Yq=Yq, workspace=workspace)
    return q.cpu().numpy(), s.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K,bias,ldq", [(300, 1024, 520, True, None), (200, 1000, 256, False, 1008),
                                             (129, 256, 64, True, None), (64, 4096, 192, False, None)])
def test_rmsnorm_fp8_prefill_small(M, N, K, bias, ldq):
    X, W, b, Z, g = _rms_case(M, N, K, bias)
    q, s = _rms_run(X, W, b, Z, g, ldq=ldq)
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None if b is None else f64(b), f64(Z), f64(g), 1e-6)
    assert_fp8_close(q, s, q_ref, s_ref, f"prefill {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,bias", [(32, 4096, 1024, False), (1, 512, 200, True), (17, 1000, 320, True),
                                        (32, 256, 64, False),
                                        # cluster decode kernel with clusters of 8, 2 and 1 CTAs (4: the first case)
                                        (32, 2048, 512, True), (8, 7680, 256, True), (5, 15360, 128, False)])
def test_rmsnorm_fp8_decode_small(M, N, K, bias):
    X, W, b, Z, g = _rms_case(M, N, K, bias)
    ldq = -(-N // 16) * 16
    q, s = _rms_run(X, W, b, Z, g, ldq=ldq if ldq != N else None)
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None if b is None else f64(b), f64(Z), f64(g), 1e-6)
    assert_fp8_close(q, s, q_ref, s_ref, f"decode {M}x{N}x{K}")


def test_rmsnorm_fp8_decode_flat_kernel_under_cta_cap():
    """Under a CTA cap too small for one cluster per feature tile the flat split-K kernel runs;
    both decode kernels give the oracle's codes on the same inputs."""
    M, N, K = 24, 4096, 768
    X, W, b, Z, g = _rms_case(M, N, K, True, seed=5)
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), f64(b), f64(Z), f64(g), 1e-6)
    for cap in (0, 24, 16):  # 32 feature tiles: one cluster each needs 32 SMs or more
        fl.set_max_ctas(cap)
        ws = fl.rmsnorm_fp8_workspace(M, N, K)
        q, s = _rms_run(X, W, b, Z, g, workspace=ws)
        assert_fp8_close(q, s, q_ref, s_ref, f"cap {cap}")
        _assert_ws_reset(ws, M, N)
    fl.set_max_ctas(0)


def test_rmsnorm_fp8_workspace_reuse_and_few_ctas():
    # the kernels leave the workspace counters at zero: back-to-back calls agree
    for M in (300, 24):
        X, W, b, Z, g = _rms_case(M, 2048, 384, True, seed=3)
        ws = fl.rmsnorm_fp8_workspace(M, 2048, 384)
        if M > 32:
            fl.set_max_ctas(8)  # 2048 / 256 = 8 tiles per row block: the smallest grid allowed
        q1, s1 = _rms_run(X, W, b, Z, g, workspace=ws)
        q2, s2 = _rms_run(X, W, b, Z, g, workspace=ws)
        fl.set_max_ctas(0)
        assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
        _assert_ws_reset(ws, M, 2048)
        q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), f64(b), f64(Z), f64(g), 1e-6)
        assert_fp8_close(q1, s1, q_ref, s_ref, f"reuse M={M}")


@pytest.mark.parametrize("graph", [False, True])
def test_rmsnorm_fp8_decode_back_to_back_shared_workspace(graph):
    """Decode calls launched back to back (programmatic dependent launches: each may start
    while the previous one finishes) over three operand sets sharing one workspace, eagerly
    and inside a CUDA graph: every call's output matches its own oracle result."""
    M, N, K = 32, 2048, 1024
    sets = [_rms_case(M, N, K, bias, seed=sd) for sd, bias in ((11, True), (12, False), (13, True))]
    dev = [tuple(None if a is None else dev_bf16(a) for a in c) for c in sets]
    ws = fl.rmsnorm_fp8_workspace(M, N, K)
    order = [0, 1, 2, 0, 2, 1, 1, 0]
    outs = [(torch.empty((M, N), dtype=torch.uint8, device="cuda"), torch.empty(M, dtype=torch.float32, device="cuda"))
            for _ in order]

    def run():
        for (Yq, rs), j in zip(outs, order):
            X, W, b, Z, g = dev[j]
            fl.fused_linear_residual_rmsnorm_fp8(X, W, b, Z, g, 1e-6, Yq=Yq, row_scale=rs, workspace=ws)

    if graph:
        run()  # warm-up outside capture (module load, attributes)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            run()
        for Yq, rs in outs:
            Yq.zero_()
            rs.zero_()
        gr.replay()
        gr.replay()
    else:
        run()
    torch.cuda.synchronize()
    refs = [oracle.rmsnorm_fp8(f64(X), f64(W), None if b is None else f64(b), f64(Z), f64(g), 1e-6)
            for X, W, b, Z, g in sets]
    for i, ((Yq, rs), j) in enumerate(zip(outs, order)):
        q_ref, s_ref, _ = refs[j]
        assert_fp8_close(Yq.cpu().numpy(), rs.cpu().numpy().astype(np.float64), q_ref, s_ref, f"call {i} (set {j})")
    _assert_ws_reset(ws, M, N)


def test_rmsnorm_fp8_decode_workspace_shared_across_shapes_and_kernels():
    """One workspace serves decode calls of different widths (so different numbers of feature
    tiles, whose per-tile statistics share the same records) and of both decode kernels (the
    flat one under a CTA cap), in an order where a stale record of an earlier call sits where the
    next call looks: every call's codes and scales match its own oracle result."""
    M, K = 24, 512
    cases = {N: _rms_case(M, N, K, True, seed=20 + N // 1024) for N in (4096, 2048, 3072)}
    refs = {N: oracle.rmsnorm_fp8(f64(X), f64(W), f64(b), f64(Z), f64(g), 1e-6) for N, (X, W, b, Z, g) in cases.items()}
    fl.set_max_ctas(16)
    size = max(fl.rmsnorm_fp8_workspace_bytes(M, N, K) for N in cases)
    fl.set_max_ctas(0)
    size = max([size] + [fl.rmsnorm_fp8_workspace_bytes(M, N, K) for N in cases])
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for N, cap in ((4096, 0), (2048, 0), (4096, 0), (3072, 16), (2048, 0), (4096, 16), (3072, 0), (4096, 0)):
        fl.set_max_ctas(cap)
        X, W, b, Z, g = cases[N]
        q, s = _rms_run(X, W, b, Z, g, workspace=ws)
        q_ref, s_ref, _ = refs[N]
        assert_fp8_close(q, s, q_ref, s_ref, f"N={N} cap={cap}")
        assert fl.check_device_status(ws) == fl.FL_OK
        _assert_ws_reset(ws, M, N)
    fl.set_max_ctas(0)


def test_rmsnorm_fp8_prefill_full_workload_sampled():
    w = syn.WORKLOADS["rmsnorm_fp8_prefill_8192x4096x14336"]
    ops = syn.make_operands(w)
    q, s = _rms_run(ops["X"], ops["W"], None, ops["Z"], ops["gamma"])
    rows = sample_rows(w.M)
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(ops["X"][rows]), f64(ops["W"]), None, f64(ops["Z"][rows]),
                                         f64(ops["gamma"]), w.eps)
    assert_fp8_close(q[rows], s[rows], q_ref, s_ref, "prefill full")


def test_rmsnorm_fp8_decode_full_workload():
    w = syn.WORKLOADS["rmsnorm_fp8_decode_32x4096x14336"]
    ops = syn.make_operands(w)
    q, s = _rms_run(ops["X"], ops["W"], None, ops["Z"], ops["gamma"])
    # h_out on the same launch configuration: the whole residual stream against the oracle's h
    _, _, h = fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(ops["X"]), dev_bf16(ops["W"]), None, dev_bf16(ops["Z"]),
                                                   dev_bf16(ops["gamma"]), w.eps, h_out=True)
    assert_bf16_close(host(h), oracle.linear(f64(ops["X"]), f64(ops["W"])) + f64(ops["Z"]), "decode full h_out")
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(ops["X"]), f64(ops["W"]), None, f64(ops["Z"]), f64(ops["gamma"]),
                                         w.eps)
    assert_fp8_close(q, s, q_ref, s_ref, "decode full")


@pytest.mark.parametrize("M,N,K,bias,pairing,cap", [
    (300, 1024, 520, True, True, 0), (300, 1024, 520, True, False, 0),  # prefill, both CTA modes
    (129, 1000, 256, False, True, 0),                                     # ragged rows and columns
    (32, 4096, 1024, True, True, 0), (17, 1000, 320, True, True, 0),     # cluster decode kernel
    (24, 4096, 768, True, True, 16)])                                     # flat decode kernel (CTA cap)
def test_rmsnorm_fp8_h_out(M, N, K, bias, pairing, cap):
    """h_out = X W^T + b + Z (the residual stream after the add) in bf16 against the oracle's h,
    with Z (and so h_out) at a row pitch wider than N; the codes and scales are those of the call
    without h_out, bit for bit."""
    fl.set_cta_pairing(pairing)
    fl.set_max_ctas(cap)
    X, W, b, Z, g = _rms_case(M, N, K, bias, seed=4)
    pitch = -(-N // 8) * 8 + 24
    Zd = torch.zeros((M, pitch), dtype=torch.bfloat16, device="cuda")[:, :N]
    Zd.copy_(dev_bf16(Z))
    dX, dW, db, dg = dev_bf16(X), dev_bf16(W), None if b is None else dev_bf16(b), dev_bf16(g)
    ws = fl.rmsnorm_fp8_workspace(M, N, K)
    q, s, h = fl.fused_linear_residual_rmsnorm_fp8(dX, dW, db, Zd, dg, 1e-6, workspace=ws, h_out=True)
    q2, s2 = fl.fused_linear_residual_rmsnorm_fp8(dX, dW, db, Zd, dg, 1e-6, workspace=ws)
    assert fl.check_device_status(ws) == fl.FL_OK
    assert h.stride(0) == pitch
    h_ref = oracle.linear(f64(X), f64(W), None if b is None else f64(b)) + f64(Z)
    assert_bf16_close(host(h), h_ref, f"h_out {M}x{N}x{K}")
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None if b is None else f64(b), f64(Z), f64(g), 1e-6)
    assert_fp8_close(q.cpu().numpy(), s.cpu().numpy().astype(np.float64), q_ref, s_ref, f"h_out codes {M}x{N}x{K}")
    assert torch.equal(q, q2) and torch.equal(s, s2)


def test_rmsnorm_fp8_h_out_rejects_overlap_with_z():
    M, N, K = 64, 256, 64
    X, W, b, Z, g = _rms_case(M, N, K, False)
    dZ = dev_bf16(Z)
    with pytest.raises(fl.FusedLinearError) as e:
        fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(X), dev_bf16(W), None, dZ, dev_bf16(g), 1e-6, h_out=dZ)
    assert e.value.status == fl.FL_ERR_INVALID_ARG


@pytest.mark.parametrize("cap", [8, 0])
def test_linear_decode_several_launches(cap):
    """More tiles than fit at once (two CTAs per SM) run as several launches of equal shares of the
    tiles: under a cap of 8 SMs (16 tiles per launch) and on the whole device (304 on 152 SMs).  GELU
    40 / 320 tiles, SwiGLU 47 / 313, QKV 48 / 384 head tiles, QKV + FP8 K/V 40 / 320."""
    fl.set_max_ctas(cap)
    big = cap == 0
    M, K = 3, 136
    N = 40960 if big else 5000
    X = _draw((M, K), syn.STREAM_X, seed=11)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=11)
    b = _draw((N,), syn.STREAM_B, 0.3, seed=11)
    Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), dev_bf16(b), mode="tanh")
    assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), f64(b), oracle.GELU_TANH), f"gelu launches N={N}")
    Nsw = 20000 if big else 3000
    Wg, Wu = _draw((Nsw, K), syn.STREAM_W, K ** -0.5, seed=12), _draw((Nsw, K), syn.STREAM_WUP, K ** -0.5, seed=12)
    Y = fl.fused_swiglu(dev_bf16(X), dev_bf16(Wg), dev_bf16(Wu), None, None)
    assert_bf16_close(host(Y), oracle.swiglu(f64(X), f64(Wg), f64(Wu), None, None), f"swiglu launches N={Nsw}")
    D = 128
    H = 128 if big else 16
    Wq = _draw((3 * H * D, K), syn.STREAM_W, K ** -0.5, seed=13)
    q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, head_dim=D, seq_len=7)
    assert_bf16_close(host(torch.cat([q, k, v], 1)), _qkv_ref(X, Wq, None, H, D, np.arange(M) % 7),
                      f"qkv launches H={H}")
    H, Hkv = (256, 32) if big else (32, 4)
    Wq = _draw(((H + 2 * Hkv) * D, K), syn.STREAM_W, K ** -0.5, seed=14)
    pos = np.array([5, 900, 77], dtype=np.int32)
    out = fl.fused_qkv_rope_fp8kv(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, n_kv_heads=Hkv, head_dim=D,
                                  positions=torch.from_numpy(pos).cuda())
    _check_kv_fp8(out, oracle.qkv_rope_kv_fp8(f64(X), f64(Wq), None, H, Hkv, D, 1e4, pos), f"fp8kv launches H={H}")


@pytest.mark.parametrize("name", ["gelu_decode_32x16384x4096", "qkv_decode_32x12288x4096",
                                  "qkv_fp8kv_decode_32x6144x4096", "swiglu_decode_32x14336x4096"])
def test_linear_decode_full_workloads(name):
    """The decode rows of bench.py at full size, in the launch shapes bench.py times (one CTA per
    tile; clusters of 3 and of 4 at two per SM; one CTA per tile at two per SM for SwiGLU's 224
    tiles), against the oracle on every output."""
    w = syn.WORKLOADS[name]
    ops = syn.make_operands(w)
    d = {k: dev_bf16(v) for k, v in ops.items()}
    if w.kind == "gelu_tanh":
        Y = fl.fused_linear_gelu(d["X"], d["W"], d.get("b"), mode="tanh")
        ref = oracle.linear_gelu(f64(ops["X"]), f64(ops["W"]), f64(ops["b"]) if "b" in ops else None,
                                 oracle.GELU_TANH)
        assert_bf16_close(host(Y), ref, name)
    elif w.kind == "qkv_rope":
        q, k, v = fl.fused_qkv_rope(d["X"], d["W"], None, n_heads=w.n_heads, head_dim=w.head_dim,
                                    seq_len=w.seq_len, theta=w.theta)
        ref = _qkv_ref(ops["X"], ops["W"], None, w.n_heads, w.head_dim, np.arange(w.M) % w.seq_len, w.theta)
        assert_bf16_close(host(torch.cat([q, k, v], 1)), ref, name)
    elif w.kind == "qkv_fp8kv":
        out = fl.fused_qkv_rope_fp8kv(d["X"], d["W"], None, n_heads=w.n_heads, n_kv_heads=w.n_kv_heads,
                                      head_dim=w.head_dim, seq_len=w.seq_len, theta=w.theta)
        ref = oracle.qkv_rope_kv_fp8(f64(ops["X"]), f64(ops["W"]), None, w.n_heads, w.n_kv_heads, w.head_dim,
                                     w.theta, np.arange(w.M) % w.seq_len)
        _check_kv_fp8(out, ref, name)
    else:
        Y = fl.fused_swiglu(d["X"], d["Wgate"], d["Wup"], None, None)
        assert_bf16_close(host(Y), oracle.swiglu(f64(ops["X"]), f64(ops["Wgate"]), f64(ops["Wup"]), None, None), name)


WS_STATUS = 256  # every workspace starts with its 256-byte status record; the counters follow


def _poison_counter(ws, M, N):
    """Sets a counter the kernels wait on to 100, which never equals its target, so the
    wait runs out: prefill counters[0] (row block 0's arrivals), decode counters[N / 128]
    (the grid-wide count of finished feature tiles)."""
    i = WS_STATUS + (4 * (N // 128) if M <= 32 else 0)
    ws[i:i + 4] = torch.tensor([100, 0, 0, 0], dtype=torch.uint8)


@pytest.mark.parametrize("M,N,cap", [(256, 1024, 0), (16, 1024, 4), (16, 4096, 0)])
def test_rmsnorm_fp8_wait_timeout_reports_status(M, N, cap):
    # A counter that never reaches its target makes the exchange wait run out:
    # the kernel records FL_ERR_TIMEOUT, drains and returns; the context stays usable.
    # (M = 16: under a cap of 4 CTAs N = 1024 runs the flat decode kernel, N = 4096 the cluster
    # one; both keep their grid-wide count at counters[N / 128].)
    K = 512
    fl.set_max_ctas(cap)
    X, W, b, Z, g = _rms_case(M, N, K, False)
    ws = fl.rmsnorm_fp8_workspace(M, N, K)
    _poison_counter(ws, M, N)
    fl.set_wait_timeout_ns(50_000_000)
    _rms_run(X, W, b, Z, g, workspace=ws)
    assert fl.check_device_status(ws) == fl.FL_ERR_TIMEOUT
    assert fl.device_status() == fl.FL_OK  # recorded in the workspace, not the device-wide word
    fl.set_wait_timeout_ns(0)
    ws.zero_()
    q, s = _rms_run(X, W, b, Z, g, workspace=ws)
    assert fl.device_status() == fl.FL_OK
    fl.set_max_ctas(0)
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None, f64(Z), f64(g), 1e-6)
    assert_fp8_close(q, s, q_ref, s_ref, "after timeout")


@pytest.mark.parametrize("M", [256, 16])
def test_timeout_on_one_stream_is_invisible_to_another(M):
    """Stream A runs on a workspace with a counter poisoned on the host and a short wait limit:
    its call records FL_ERR_TIMEOUT in A's workspace.  Stream B, with its own workspace and the
    default limit, runs the same problem meanwhile: B's status stays FL_OK and its output is
    the oracle's.  Neither the device-wide word nor B's record sees A's failure."""
    N, K = 1024, 512
    X, W, b, Z, g = _rms_case(M, N, K, False, seed=7)
    dX, dW, dZ, dg = dev_bf16(X), dev_bf16(W), dev_bf16(Z), dev_bf16(g)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    wa, wb = fl.rmsnorm_fp8_workspace(M, N, K), fl.rmsnorm_fp8_workspace(M, N, K)
    _poison_counter(wa, M, N)
    torch.cuda.synchronize()
    fl.set_wait_timeout_ns(50_000_000)
    with torch.cuda.stream(sa):
        fl.fused_linear_residual_rmsnorm_fp8(dX, dW, None, dZ, dg, 1e-6, workspace=wa, stream=sa)
    fl.set_wait_timeout_ns(0)
    with torch.cuda.stream(sb):
        qb, sbs = fl.fused_linear_residual_rmsnorm_fp8(dX, dW, None, dZ, dg, 1e-6, workspace=wb, stream=sb)
    assert fl.check_device_status(wb, stream=sb) == fl.FL_OK
    assert fl.check_device_status(wa, stream=sa) == fl.FL_ERR_TIMEOUT
    assert fl.check_device_status(wa, stream=sa) == fl.FL_OK  # the check cleared the record
    assert fl.device_status() == fl.FL_OK
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None, f64(Z), f64(g), 1e-6)
    assert_fp8_close(qb.cpu().numpy(), sbs.cpu().numpy().astype(np.float64), q_ref, s_ref, "stream B")


def test_argument_errors_on_device():
    X = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    Z = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(fl.FusedLinearError) as e:
        fl.fused_linear_residual_rmsnorm_fp8(X, W, None, Z, g, workspace=small)
    assert e.value.status == fl.FL_ERR_WORKSPACE
    with pytest.raises(fl.FusedLinearError) as e:
        fl.fused_qkv_rope(X, torch.zeros((3 * 64, 64), dtype=torch.bfloat16, device="cuda"), n_heads=1,
                          head_dim=64)
    assert e.value.status == fl.FL_ERR_UNSUPPORTED


# ------------------------------------------------------------------ GEMM -> residual -> RMSNorm -> GEMM
@pytest.mark.parametrize("pairing", [True, False])
def test_rms_chain_small(pairing):
    fl.set_cta_pairing(pairing)
    M, N, K, N2 = 300, 512, 200, 384
    X = _draw((M, K), syn.STREAM_X)
    W0 = _draw((N, K), syn.STREAM_W, K ** -0.5)
    b0 = _draw((N,), syn.STREAM_B, 0.02)
    Z = _draw((M, N), syn.STREAM_Z)
    g = _draw((N,), syn.STREAM_GAMMA, 0.1, 1.0)
    W1 = _draw((N2, N), syn.STREAM_W2, N ** -0.5)
    b1 = _draw((N2,), syn.STREAM_BUP, 0.02)
    H2, H1, part = fl.fused_linear_residual_gamma(dev_bf16(X), dev_bf16(W0), dev_bf16(b0), dev_bf16(Z), dev_bf16(g))
    Y = fl.fused_linear_rms_rowscale(H2, dev_bf16(W1), dev_bf16(b1), part, N, 1e-6)
    y_ref, h1_ref = oracle.residual_rmsnorm_linear(f64(X), f64(W0), f64(b0), f64(Z), f64(g), 1e-6, f64(W1), f64(b1))
    assert_bf16_close(host(H1), h1_ref, "h1 (residual stream)")
    assert_bf16_close(host(H2), h1_ref * f64(g), "h2 = h1 * gamma")
    tiles = np.stack([np.sum(h1_ref[:, j * 256:(j + 1) * 256] ** 2, axis=1) for j in range(2)])
    assert np.allclose(part.cpu().numpy(), tiles, rtol=1e-4, atol=1e-3), "per-tile sums of squares"
    assert_bf16_close(host(Y), y_ref, "y = RMSNorm(h1) W1 + b1")


@pytest.mark.parametrize("decode", [True, False])
@pytest.mark.parametrize("M,N,K,N2,store_h1,bias", [(32, 4096, 4096, 1024, True, False), (7, 384, 2048, 640, False, True),
                                                    (1, 1000, 512, 264, True, True), (3, 2048, 8192, 4096, True, False),
                                                    (20, 6144, 1024, 2048, False, False)])
def test_rms_chain_decode_shapes(decode, M, N, K, N2, store_h1, bias):
    """Decode shapes of both chain steps (step 1 finished by whole tokens, its 256-column sums of h1^2
    added from two 128-feature tiles onto zeroed entries; step 2 by features; N = 384 leaves the last
    entry one tile, N = 1000 ends inside a tile), and the GEMM kernel on the same shapes with the decode
    path off; two calls give the same bits."""
    fl.set_linear_decode(decode)
    try:
        X = _draw((M, K), syn.STREAM_X, seed=M + 5)
        W0 = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=M + 5)
        b0 = _draw((N,), syn.STREAM_B, 0.02, seed=M + 5) if bias else None
        Z = _draw((M, N), syn.STREAM_Z, seed=M + 5)
        g = _draw((N,), syn.STREAM_GAMMA, 0.1, 1.0, seed=M + 5)
        W1 = _draw((N2, N), syn.STREAM_W2, N ** -0.5, seed=M + 5)
        for kind, n_out, k_in in ((fl.DECODE_RESID_GAMMA, N, K), (fl.DECODE_ROWSCALE, N2, N)):
            plan = fl.linear_decode_shape(kind, M, n_out, k_in)
            assert (plan[0] > 0) == decode, (kind, plan)
        outs = []
        for _ in range(2):
            H2, H1, part = fl.fused_linear_residual_gamma(dev_bf16(X), dev_bf16(W0), None if b0 is None else dev_bf16(b0),
                                                          dev_bf16(Z), dev_bf16(g), store_h1=store_h1)
            Y = fl.fused_linear_rms_rowscale(H2, dev_bf16(W1), None, part, N, 1e-6)
            outs.append([t.clone() for t in (H2, part, Y) + ((H1,) if store_h1 else ())])
        for a, c in zip(*outs):
            assert torch.equal(a, c), "two calls differ"
        y_ref, h1_ref = oracle.residual_rmsnorm_linear(f64(X), f64(W0), None if b0 is None else f64(b0), f64(Z), f64(g),
                                                       1e-6, f64(W1), None)
        what = f"chain decode={decode} {M}x{N}x{K} -> {N2}"
        if store_h1:
            assert_bf16_close(host(H1), h1_ref, what + ": h1")
        assert_bf16_close(host(H2), h1_ref * f64(g), what + ": h2")
        tiles = np.stack([np.sum(h1_ref[:, j * 256:(j + 1) * 256] ** 2, axis=1) for j in range(-(-N // 256))])
        assert np.allclose(part.cpu().numpy(), tiles, rtol=1e-4, atol=1e-3), what + ": per-tile sums of squares"
        assert_bf16_close(host(Y), y_ref, what + ": y")
    finally:
        fl.set_linear_decode(True)


def test_rms_chain_full_workload_sampled():
    w = syn.WORKLOADS["rms_chain_8192x4096x4096_to_14336"]
    ops = syn.make_operands(w)
    H2, _, part = fl.fused_linear_residual_gamma(dev_bf16(ops["X"]), dev_bf16(ops["W"]), None, dev_bf16(ops["Z"]),
                                                 dev_bf16(ops["gamma"]), store_h1=False)
    Y = fl.fused_linear_rms_rowscale(H2, dev_bf16(ops["W2"]), None, part, w.N, w.eps)
    rows = sample_rows(w.M)
    y_ref, _ = oracle.residual_rmsnorm_linear(f64(ops["X"][rows]), f64(ops["W"]), None, f64(ops["Z"][rows]),
                                              f64(ops["gamma"]), w.eps, f64(ops["W2"]))
    assert_bf16_close(host(Y[torch.from_numpy(rows).cuda()]), y_ref, "rms chain full")


# ------------------------------------------------------------------ LM-head cross-entropy
@pytest.mark.parametrize("pairing", [True, False])
def test_cross_entropy_small_with_logits(pairing):
    fl.set_cta_pairing(pairing)
    M, V, K = 300, 1000, 200
    X = _draw((M, K), syn.STREAM_X)
    W = _draw((V, K), syn.STREAM_W, K ** -0.5)
    b = _draw((V,), syn.STREAM_B, 0.5)
    lab = syn.draw_labels(0, syn.STREAM_LABEL, M, V)
    lab[5], lab[17] = -100, V  # ignored row, label outside the vocabulary
    ws = fl.cross_entropy_workspace(M, V)
    for _ in range(2):  # the workspace counters are reset by the kernel
        loss, logits = fl.fused_linear_cross_entropy(dev_bf16(X), dev_bf16(W), dev_bf16(b),
                                                     torch.from_numpy(lab).cuda(), store_logits=True, workspace=ws)
        ref = oracle.linear_cross_entropy(f64(X), f64(W), f64(b), lab)
        _assert_loss_close(loss.cpu().numpy().astype(np.float64), ref, "ce small")
        assert_bf16_close(host(logits), oracle.linear(f64(X), f64(W), f64(b)), "logits")
    assert torch.count_nonzero(ws[:512]) == 0


def test_cross_entropy_full_workload_sampled():
    w = syn.WORKLOADS["lm_head_ce_8192x32768x4096"]
    ops = syn.make_operands(w)
    lab = syn.make_labels(w)
    loss, _ = fl.fused_linear_cross_entropy(dev_bf16(ops["X"]), dev_bf16(ops["W"]), None,
                                            torch.from_numpy(lab).cuda())
    rows = sample_rows(w.M)
    ref = oracle.linear_cross_entropy(f64(ops["X"][rows]), f64(ops["W"]), None, lab[rows])
    _assert_loss_close(loss.cpu().numpy()[rows].astype(np.float64), ref, "ce full")


# ------------------------------------------------------------------ block-scaled quantised write-back
def _quant_decoders():
    e2m1 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    return {"value_fp8": lambda c: oracle.e4m3_decode(c),
            "value_4bit": lambda c: e2m1[c],
            "scale": lambda c: oracle.e4m3_decode(c)}


def _check_quant(fmt, Yq, S, X, W, b, what, inv_smooth=None):
    q_ref, s_ref, y_ref = oracle.linear_quant(f64(X), f64(W), None if b is None else f64(b), fmt,
                                              inv_smooth=None if inv_smooth is None else inv_smooth.astype(np.float64))
    d = _quant_decoders()
    dec = {"scale": d["scale"]}
    if fmt == fl.QUANT_FP8_1X128:
        dec["value"] = d["value_fp8"]
    elif fmt == fl.QUANT_INT4_G32:
        dec["value"] = lambda c: np.where(c & 8, c.astype(np.int32) - 16, c).astype(np.float64)
    else:
        dec["value"] = d["value_4bit"]
    assert_quant_close(fmt, Yq.cpu().numpy(), S.cpu().numpy(), q_ref, s_ref, y_ref, dec, what)


@pytest.mark.parametrize("pairing", [True, False])
@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (1, 64, 40), (257, 1024, 136)])
def test_quant_small(fmt, pairing, M, N, K):
    fl.set_cta_pairing(pairing)
    X = _draw((M, K), syn.STREAM_X)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5)
    b = _draw((N,), syn.STREAM_B, 0.5)
    X[M // 2] = 0  # with no bias below, an all-zero row: scale 0, codes 0
    for bias in (b, None):
        Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), None if bias is None else dev_bf16(bias), fmt)
        _check_quant(fmt, Yq, S, X, W, bias, f"quant fmt {fmt} {M}x{N}x{K} bias={bias is not None}")
    if M > 2:
        assert torch.count_nonzero(Yq[M // 2]) == 0 and torch.count_nonzero(S[M // 2]) == 0


@pytest.mark.parametrize("pairing", [True, False])
@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (257, 1024, 136), (1, 64, 40)])
def test_quant_smoothing_small(fmt, pairing, M, N, K):
    """Step 3 of the quantised write-back: the per-column inverse smoothing factor multiplies the
    output before the block maxima; codes and scales against the oracle with the same factors."""
    fl.set_cta_pairing(pairing)
    X = _draw((M, K), syn.STREAM_X)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5)
    b = _draw((N,), syn.STREAM_B, 0.5)
    inv = syn.draw_inv_smooth(0, N)
    Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), dev_bf16(b), fmt, inv_smooth=torch.from_numpy(inv).cuda())
    _check_quant(fmt, Yq, S, X, W, b, f"smoothed quant fmt {fmt} {M}x{N}x{K}", inv_smooth=inv)


@pytest.mark.parametrize("decode", [True, False])
@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K,smooth", [(32, 4096, 1024, False), (7, 1000, 4096, True), (1, 16384, 256, True),
                                          (20, 6144, 2048, False), (3, 384, 8192, True)])
def test_quant_decode_shapes(decode, fmt, M, N, K, smooth):
    """Decode shapes of the block-scaled write-back (tiles of 128 features finished by whole tokens, on
    every launch shape these sizes pick: clusters of 4 at two CTAs per SM, clusters of 8, one CTA per
    tile at two per SM for 128 tiles; N = 1000 and 384 end inside a tile), with and without the
    smoothing factor, and the GEMM kernel on the same shapes with the decode path off; an all-zero
    token gets scale 0 and zero codes."""
    fl.set_linear_decode(decode)
    try:
        X = _draw((M, K), syn.STREAM_X, seed=M + 3)
        W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=M + 3)
        b = _draw((N,), syn.STREAM_B, 0.5, seed=M + 3) if not smooth else None
        if M > 2:
            X[M // 2] = 0
        inv = syn.draw_inv_smooth(M, N) if smooth else None
        plan = fl.linear_decode_shape(fl.DECODE_QUANT, M, N, K)
        assert (plan[0] > 0) == decode, plan
        Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), None if b is None else dev_bf16(b), fmt,
                                      inv_smooth=None if inv is None else torch.from_numpy(inv).cuda())
        _check_quant(fmt, Yq, S, X, W, b, f"quant decode={decode} fmt {fmt} {M}x{N}x{K} smooth {smooth} plan {plan}",
                     inv_smooth=inv)
        if M > 2 and b is None:
            assert torch.count_nonzero(Yq[M // 2]) == 0 and torch.count_nonzero(S[M // 2]) == 0
    finally:
        fl.set_linear_decode(True)


def test_quant_smoothing_of_ones_is_bit_identical():
    M, N, K = 257, 1024, 136
    X = dev_bf16(_draw((M, K), syn.STREAM_X))
    W = dev_bf16(_draw((N, K), syn.STREAM_W, K ** -0.5))
    ones = torch.ones(N, dtype=torch.float32, device="cuda")
    for fmt in (0, 1, 2):
        a = fl.fused_linear_quant(X, W, None, fmt)
        c = fl.fused_linear_quant(X, W, None, fmt, inv_smooth=ones)
        assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_quant_rejects_odd_n_for_4bit_and_bad_format():
    X = dev_bf16(_draw((8, 16), syn.STREAM_X))
    W = dev_bf16(_draw((33, 16), syn.STREAM_W))
    Yq = torch.empty((8, 32), dtype=torch.uint8, device="cuda")
    S = torch.empty((8, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(fl.FusedLinearError) as e:
        fl.fused_linear_quant(X, W, None, fl.QUANT_INT4_G32, Yq=Yq[:, :16], scales=S)
    assert e.value.status == fl.FL_ERR_UNSUPPORTED
    st = fl.load().fused_linear_quant(None, None, None, None, None, None, 8, 32, 16, 16, 16, 32, 4, 7, None)
    assert st == fl.FL_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["quant_fp8_1x128_8192x16384x4096", "quant_int4_g32_8192x16384x4096",
                                  "quant_nvfp4_g16_8192x16384x4096", "quant_fp8_1x128_smooth_8192x16384x4096",
                                  "quant_fp8_1x128_decode_32x16384x4096"])
def test_quant_full_workload_sampled(name):
    w = syn.WORKLOADS[name]
    fmt = {"fp8_1x128": 0, "int4_g32": 1, "nvfp4_g16": 2}[w.quant]
    ops = syn.make_operands(w)
    inv = ops.get("inv_smooth")
    Yq, S = fl.fused_linear_quant(dev_bf16(ops["X"]), dev_bf16(ops["W"]), dev_bf16(ops["b"]), fmt,
                                  inv_smooth=None if inv is None else torch.from_numpy(inv).cuda())
    rows = sample_rows(w.M) if w.M > 32 else np.arange(w.M)  # the decode shape: every output
    _check_quant(fmt, Yq[rows], S[rows], ops["X"][rows], ops["W"], ops["b"], name, inv_smooth=inv)


# ------------------------------------------------------------------ QKV + RoPE with an FP8 K/V cache
@pytest.mark.parametrize("pairing", [True, False])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (2, 2)])
def test_qkv_fp8kv_small(pairing, H, Hkv):
    fl.set_cta_pairing(pairing)
    M, K, D = 300, 200, 128
    X = _draw((M, K), syn.STREAM_X)
    Wq = _draw(((H + 2 * Hkv) * D, K), syn.STREAM_W, K ** -0.5)
    bq = _draw(((H + 2 * Hkv) * D,), syn.STREAM_B, 0.5)
    X[7] = 0  # without bias, row 7's K and V heads are all zero -> scale 0, codes 0
    pos = np.random.default_rng(2).integers(0, 8192, size=M).astype(np.int32)
    for bias in (bq, None):
        out = fl.fused_qkv_rope_fp8kv(dev_bf16(X), dev_bf16(Wq), None if bias is None else dev_bf16(bias), n_heads=H,
                                      n_kv_heads=Hkv, head_dim=D, positions=torch.from_numpy(pos).cuda())
        ref = oracle.qkv_rope_kv_fp8(f64(X), f64(Wq), None if bias is None else f64(bias), H, Hkv, D, 1e4, pos)
        _check_kv_fp8(out, ref, f"qkv fp8kv H={H} Hkv={Hkv} bias={bias is not None}")
    assert torch.count_nonzero(out[1][7]) == 0 and torch.count_nonzero(out[4][7]) == 0
    if H == Hkv:  # with as many kv heads as query heads, Q matches the bf16 entry point bit for bit
        q, _, _ = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, head_dim=D,
                                    positions=torch.from_numpy(pos).cuda())
        assert torch.equal(q, out[0])


@pytest.mark.parametrize("decode", [True, False])
@pytest.mark.parametrize("M,H,Hkv,K", [(32, 4, 2, 1024), (7, 32, 8, 4096), (3, 64, 8, 4096), (20, 2, 2, 200),
                                       (5, 16, 4, 2048), (2, 8, 2, 8192), (2, 128, 16, 256)])
def test_qkv_fp8kv_decode_shapes(decode, M, H, Hkv, K):
    """Decode shapes of the FP8 K/V form (one CTA per head tile; clusters of 4 and of 3 at two CTAs
    per SM, the 3 with uneven shares of the head, so its max spans the cluster; clusters of 2 and of
    8; one CTA per tile at two per SM for 160 tiles), and the GEMM kernel on the same shapes with the
    decode path off."""
    fl.set_linear_decode(decode)
    try:
        D = 128
        X = _draw((M, K), syn.STREAM_X, seed=M + 1)
        Wq = _draw(((H + 2 * Hkv) * D, K), syn.STREAM_W, K ** -0.5, seed=M + 1)
        bq = _draw(((H + 2 * Hkv) * D,), syn.STREAM_B, 0.5, seed=M + 1)
        zero = M // 2
        X[zero] = 0  # without bias this token's K and V heads are all zero -> scale 0, codes 0
        pos = np.random.default_rng(M).integers(0, 1 << 20, size=M).astype(np.int32)
        for bias in (bq, None):
            out = fl.fused_qkv_rope_fp8kv(dev_bf16(X), dev_bf16(Wq), None if bias is None else dev_bf16(bias),
                                          n_heads=H, n_kv_heads=Hkv, head_dim=D,
                                          positions=torch.from_numpy(pos).cuda())
            ref = oracle.qkv_rope_kv_fp8(f64(X), f64(Wq), None if bias is None else f64(bias), H, Hkv, D, 1e4, pos)
            _check_kv_fp8(out, ref, f"qkv fp8kv decode={decode} M={M} H={H} Hkv={Hkv} bias={bias is not None}")
        assert torch.count_nonzero(out[1][zero]) == 0 and torch.count_nonzero(out[4][zero]) == 0
    finally:
        fl.set_linear_decode(True)


def test_qkv_fp8kv_rejects_odd_heads():
    X = dev_bf16(_draw((8, 64), syn.STREAM_X))
    W = dev_bf16(_draw(((2 + 2) * 128, 64), syn.STREAM_W))
    with pytest.raises(fl.FusedLinearError) as e:
        fl.fused_qkv_rope_fp8kv(X, W, None, n_heads=2, n_kv_heads=1, head_dim=128)
    assert e.value.status == fl.FL_ERR_UNSUPPORTED


def test_qkv_fp8kv_full_workload_sampled():
    w = syn.WORKLOADS["qkv_fp8kv_8192x6144x4096"]
    ops = syn.make_operands(w)
    out = fl.fused_qkv_rope_fp8kv(dev_bf16(ops["X"]), dev_bf16(ops["W"]), None, n_heads=w.n_heads,
                                  n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, seq_len=w.seq_len, theta=w.theta)
    rows = sample_rows(w.M)
    ri = torch.from_numpy(rows).cuda()
    ref = oracle.qkv_rope_kv_fp8(f64(ops["X"][rows]), f64(ops["W"]), None, w.n_heads, w.n_kv_heads, w.head_dim,
                                 w.theta, rows % w.seq_len)
    _check_kv_fp8(tuple(t[ri] for t in out), ref, "qkv fp8kv full")


# ------------------------------------------------------------------ backward epilogues (dgrad, W as stored)
@pytest.mark.parametrize("pairing", [True, False])
@pytest.mark.parametrize("mode", ["tanh", "erf"])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (1, 72, 40), (257, 1024, 136)])
def test_dgrad_gelu_small(mode, pairing, M, N, K):
    fl.set_cta_pairing(pairing)
    dZ = _draw((M, K), syn.STREAM_X)
    W = _draw((K, N), syn.STREAM_W, K ** -0.5)
    H = _draw((M, N), syn.STREAM_Z, 2.0)
    dH = fl.fused_dgrad_gelu(dev_bf16(dZ), dev_bf16(W), dev_bf16(H), mode=mode)
    m = oracle.GELU_TANH if mode == "tanh" else oracle.GELU_ERF
    assert_bf16_close(host(dH), oracle.dgrad_gelu(f64(dZ), f64(W), f64(H), m), f"dgrad gelu {mode} {M}x{N}x{K}")


def test_dgrad_gelu_strided_and_k_zero():
    M, N, K = 130, 264, 72
    dZ = _draw((M, K + 8), syn.STREAM_X)
    W = _draw((K, N + 16), syn.STREAM_W, K ** -0.5)
    H = _draw((M, N + 24), syn.STREAM_Z, 2.0)
    out = torch.zeros((M, N + 40), dtype=torch.bfloat16, device="cuda")
    fl.fused_dgrad_gelu(dev_bf16(dZ)[:, :K], dev_bf16(W)[:, :N], dev_bf16(H)[:, :N], mode="erf", dH=out[:, :N])
    ref = oracle.dgrad_gelu(f64(dZ[:, :K]), f64(W[:, :N]), f64(H[:, :N]), oracle.GELU_ERF)
    assert_bf16_close(host(out[:, :N]), ref, "strided")
    assert torch.count_nonzero(out[:, N:]) == 0
    z = fl.fused_dgrad_gelu(torch.empty((M, 0), dtype=torch.bfloat16, device="cuda"),
                            torch.empty((0, N), dtype=torch.bfloat16, device="cuda"), dev_bf16(H)[:, :N])
    assert torch.count_nonzero(z) == 0  # K = 0: the gradient is zero


@pytest.mark.parametrize("pairing", [True, False])
@pytest.mark.parametrize("M,N,K", [(300, 264, 200), (1, 64, 40), (257, 768, 136)])
def test_swiglu_bwd_small(pairing, M, N, K):
    fl.set_cta_pairing(pairing)
    dO = _draw((M, K), syn.STREAM_X)
    Wd = _draw((K, N), syn.STREAM_W, K ** -0.5)
    G = _draw((M, N), syn.STREAM_Z, 3.0)
    U = _draw((M, N), syn.STREAM_GAMMA)
    out = fl.fused_swiglu_bwd(dev_bf16(dO), dev_bf16(Wd), dev_bf16(G), dev_bf16(U))
    assert tuple(out.shape) == (M, 2 * N)
    ref = oracle.swiglu_bwd(f64(dO), f64(Wd), f64(G), f64(U))
    assert_bf16_close(host(out), ref, f"swiglu bwd {M}x{N}x{K}")


@pytest.mark.parametrize("name", ["gelu_bwd_8192x16384x4096", "swiglu_bwd_8192x14336x4096"])
def test_backward_full_workload_sampled(name):
    w = syn.WORKLOADS[name]
    ops = syn.make_operands(w)
    rows = sample_rows(w.M)
    if w.kind == "gelu_bwd":
        out = fl.fused_dgrad_gelu(dev_bf16(ops["dZ"]), dev_bf16(ops["W"]), dev_bf16(ops["H"]), mode="tanh")
        ref = oracle.dgrad_gelu(f64(ops["dZ"][rows]), f64(ops["W"]), f64(ops["H"][rows]), oracle.GELU_TANH)
    else:
        out = fl.fused_swiglu_bwd(dev_bf16(ops["dO"]), dev_bf16(ops["Wd"]), dev_bf16(ops["G"]), dev_bf16(ops["U"]))
        ref = oracle.swiglu_bwd(f64(ops["dO"][rows]), f64(ops["Wd"]), f64(ops["G"][rows]), f64(ops["U"][rows]))
    assert_bf16_close(host(out[torch.from_numpy(rows).cuda()]), ref, name)


# ------------------------------------------------------------------ host-buffer pipeline
@pytest.mark.parametrize("M,N,K,bias", [(300, 520, 200, True), (1024, 4096, 512, False), (5, 8, 8, True),
                                        (1024, 256, 64, False)])
def test_linear_gelu_host_pipeline(M, N, K, bias):
    """Host buffers in and out, row and column blocks overlapped (3 x 3, 4 x 8, 1 x 1 and 4 x 1
    blocks): the same values as the device entry point bit for bit (same kernel, same
    accumulation order), and the oracle."""
    X = _draw((M, K), syn.STREAM_X)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5)
    b = _draw((N,), syn.STREAM_B, 0.5) if bias else None

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    Xh, Wh = pinned(X), pinned(W)
    bh = pinned(b) if bias else None
    buf = fl.linear_gelu_host_buffer(M, N, K)
    for _ in range(2):  # the buffer and the library's streams are reused
        Yh = fl.fused_linear_gelu_host(Xh, Wh, bh, mode="tanh", dev_buf=buf)
        torch.cuda.current_stream().synchronize()
        Yd = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), dev_bf16(b) if bias else None, mode="tanh")
        assert torch.equal(Yh, Yd.cpu())
    assert_bf16_close(host(Yh), oracle.linear_gelu(f64(X), f64(W), f64(b) if bias else None, oracle.GELU_TANH),
                      f"host pipeline {M}x{N}x{K}")


# ------------------------------------------------------------------ CUDA graphs
def test_graph_capture_of_every_entry_point_matches_eager():
    """One call of each kind captured in a CUDA graph (cooperative and cluster launches,
    workspace counters reset by the kernels) replays bit-identically to eager execution:
    every reduction merges in a fixed order."""
    M, N, K = 300, 512, 192
    X = dev_bf16(_draw((M, K), syn.STREAM_X))
    W = dev_bf16(_draw((N, K), syn.STREAM_W, K ** -0.5))
    b = dev_bf16(_draw((N,), syn.STREAM_B, 0.5))
    Z = dev_bf16(_draw((M, N), syn.STREAM_Z))
    g = dev_bf16(_draw((N,), syn.STREAM_GAMMA, 0.1, 1.0))
    Wt = dev_bf16(_draw((K, N), syn.STREAM_W2, K ** -0.5))           # [K, N] as stored, for the dgrad
    W1 = dev_bf16(_draw((256, N), syn.STREAM_W2, N ** -0.5, seed=1))  # second GEMM of the chain
    Wq = dev_bf16(_draw((3 * 256, K), syn.STREAM_WUP, K ** -0.5))   # 2 heads of 128
    Xd = X[:16].contiguous()
    Zd = dev_bf16(_draw((16, 4096), syn.STREAM_Z, seed=2))
    Wd = dev_bf16(_draw((4096, K), syn.STREAM_W, K ** -0.5, seed=2))
    gd = dev_bf16(_draw((4096,), syn.STREAM_GAMMA, 0.1, 1.0, seed=2))
    lab = torch.from_numpy(syn.draw_labels(0, syn.STREAM_LABEL, M, N)).cuda()
    Xf, Wf = X.float(), W.float()
    ws_p = fl.rmsnorm_fp8_workspace(M, N, K)
    ws_d = fl.rmsnorm_fp8_workspace(16, 4096, K)
    ws_c = fl.cross_entropy_workspace(M, N)
    parts = torch.empty((fl.rms_partials_per_row(N), M), dtype=torch.float32, device="cuda")

    def run():
        outs = [fl.fused_linear_gelu(X, W, b, mode="tanh"),
                *fl.fused_qkv_rope(X, Wq, None, n_heads=2, head_dim=128, seq_len=64),
                fl.fused_swiglu(X, W, W),
                *fl.fused_linear_residual_rmsnorm_fp8(X, W, b, Z, g, 1e-6, workspace=ws_p),
                *fl.fused_linear_residual_rmsnorm_fp8(Xd, Wd, None, Zd, gd, 1e-6, workspace=ws_d)]
        h2, _, _ = fl.fused_linear_residual_gamma(X, W, b, Z, g, store_h1=False, rms_partials=parts)
        outs.append(fl.fused_linear_rms_rowscale(h2, W1, None, parts, N, 1e-6))
        outs.append(fl.fused_linear_cross_entropy(X, W, None, lab, workspace=ws_c)[0])
        outs += list(fl.fused_linear_quant(X, W, b, fl.QUANT_NVFP4_G16))
        outs.append(fl.fused_dgrad_gelu(X, Wt, Z, mode="erf"))
        outs.append(fl.fused_linear_gelu(Xf, Wf, None, mode="erf"))
        return outs

    eager = [t.clone() for t in run()]
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        captured = run()
    for _ in range(2):
        for t in captured:
            t.zero_()
        gr.replay()
        torch.cuda.synchronize()
        for i, (a, c) in enumerate(zip(eager, captured)):
            assert torch.equal(a, c), f"output {i} differs after replay"
    assert torch.count_nonzero(ws_p[:256]) == 0 and torch.count_nonzero(ws_c[:256]) == 0


def test_every_entry_point_is_deterministic_across_calls():
    """Each entry point called twice on the same inputs, with other work in between, gives
    bit-identical outputs at shapes that span several waves of the persistent grid (and, for decode,
    both decode kernels): no reduction depends on scheduling or arrival order."""
    M, N, K = 2048, 4096, 1024
    X = dev_bf16(_draw((M, K), syn.STREAM_X, seed=11))
    W = dev_bf16(_draw((N, K), syn.STREAM_W, K ** -0.5, seed=11))
    b = dev_bf16(_draw((N,), syn.STREAM_B, 0.5, seed=11))
    Z = dev_bf16(_draw((M, N), syn.STREAM_Z, seed=11))
    g = dev_bf16(_draw((N,), syn.STREAM_GAMMA, 0.1, 1.0, seed=11))
    Wt = dev_bf16(_draw((K, N), syn.STREAM_W2, K ** -0.5, seed=11))    # [K, N] as stored (dgrad)
    G = dev_bf16(_draw((M, N), syn.STREAM_WUP, seed=12))
    Wq = dev_bf16(_draw((2 * 2048, K), syn.STREAM_WUP, K ** -0.5, seed=11))  # GQA 16 / 8 heads of 128
    Xd = X[:32].contiguous()
    ws_p = fl.rmsnorm_fp8_workspace(M, N, K)
    ws_c = fl.cross_entropy_workspace(M, N)
    lab = torch.from_numpy(syn.draw_labels(11, syn.STREAM_LABEL, M, N)).cuda()
    calls = {
        "gelu": lambda: [fl.fused_linear_gelu(X, W, b, mode="tanh")],
        "qkv": lambda: list(fl.fused_qkv_rope(X, Wq[:3 * 1024], None, n_heads=8, head_dim=128, seq_len=512)),
        "qkv_fp8kv": lambda: list(fl.fused_qkv_rope_fp8kv(X, Wq, None, n_heads=16, n_kv_heads=8, head_dim=128,
                                                          seq_len=512)),
        "swiglu": lambda: [fl.fused_swiglu(X, W, W)],
        "rmsnorm_prefill": lambda: list(fl.fused_linear_residual_rmsnorm_fp8(X, W, b, Z, g, 1e-6, workspace=ws_p)),
        "rmsnorm_decode": lambda: list(fl.fused_linear_residual_rmsnorm_fp8(Xd, W, b, Z[:32].contiguous(), g, 1e-6)),
        "cross_entropy": lambda: list(fl.fused_linear_cross_entropy(X, W, b, lab, workspace=ws_c))[:1],
        "quant_fp8": lambda: list(fl.fused_linear_quant(X, W, b, fl.QUANT_FP8_1X128)),
        "quant_int4": lambda: list(fl.fused_linear_quant(X, W, b, fl.QUANT_INT4_G32)),
        "dgrad_gelu": lambda: [fl.fused_dgrad_gelu(X, Wt, Z, mode="tanh")],
        "swiglu_bwd": lambda: [fl.fused_swiglu_bwd(X, Wt, G, Z)],
    }
    first = {k: [t.clone() for t in f()] for k, f in calls.items()}
    fl.set_max_ctas(24)  # decode on the flat split-K kernel (32 feature tiles), the GEMMs on fewer CTAs
    capped = {k: [t.clone() for t in calls[k]()] for k in ("rmsnorm_decode", "gelu", "swiglu_bwd")}
    for i, (a, c) in enumerate(zip(capped["rmsnorm_decode"], calls["rmsnorm_decode"]())):
        assert torch.equal(a, c), f"flat decode kernel: output {i} differs between two calls"
    fl.set_max_ctas(0)
    for k, f in reversed(list(calls.items())):  # the second pass in another order
        again = f()
        for i, (a, c) in enumerate(zip(first[k], again)):
            assert torch.equal(a, c), f"{k}: output {i} differs between two calls"
    for k in ("gelu", "swiglu_bwd"):  # the tile walk changes with the grid, the arithmetic does not
        for i, (a, c) in enumerate(zip(first[k], capped[k])):
            assert torch.equal(a, c), f"{k}: output {i} differs under a smaller grid"
    torch.cuda.synchronize()
    assert fl.device_status() == fl.FL_OK


# ------------------------------------------------------------------ random shapes, streams, threads
def _rand_shapes(seed, count, m_max=600, n_max=1200, k_max=700):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        M = int(rng.integers(1, m_max))
        N = int(rng.integers(1, n_max // 8)) * 8      # 16-byte row pitches in bf16
        K = int(rng.integers(1, k_max // 8)) * 8
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("pairing", [True, False])
def test_random_shapes_gelu_swiglu_quant_dgrad(pairing):
    """Seeded random shapes (ragged in M, N and K) for four epilogues, against the oracle."""
    fl.set_cta_pairing(pairing)
    for i, (M, N, K) in enumerate(_rand_shapes(7 + pairing, 6)):
        X = _draw((M, K), syn.STREAM_X, seed=i)
        W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=i)
        b = _draw((N,), syn.STREAM_B, 0.3, seed=i)
        mode = "tanh" if i % 2 else "erf"
        Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), dev_bf16(b), mode=mode)
        m = oracle.GELU_TANH if mode == "tanh" else oracle.GELU_ERF
        assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), f64(b), m), f"random gelu {M}x{N}x{K}")
        Wu = _draw((N, K), syn.STREAM_WUP, K ** -0.5, seed=i)
        Ys = fl.fused_swiglu(dev_bf16(X), dev_bf16(W), dev_bf16(Wu))
        assert_bf16_close(host(Ys), oracle.swiglu(f64(X), f64(W), f64(Wu)), f"random swiglu {M}x{N}x{K}")
        if N % 16 == 0:
            fmt = i % 3
            Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), dev_bf16(b), fmt)
            q_ref, s_ref, y_ref = oracle.linear_quant(f64(X), f64(W), f64(b), fmt)
            e2m1 = np.array([oracle.e2m1_decode(c) for c in range(16)])
            dec = {"scale": oracle.e4m3_decode,
                   "value": (oracle.e4m3_decode if fmt == 0 else
                             (lambda c: np.where(c & 8, c.astype(np.int32) - 16, c).astype(np.float64)) if fmt == 1 else
                             (lambda c: e2m1[c]))}
            assert_quant_close(fmt, Yq.cpu().numpy(), S.cpu().numpy(), q_ref, s_ref, y_ref, dec,
                               f"random quant {fmt} {M}x{N}x{K}")
        Wt = _draw((K, N), syn.STREAM_W2, K ** -0.5, seed=i)
        H = _draw((M, N), syn.STREAM_Z, 2.0, seed=i)
        dH = fl.fused_dgrad_gelu(dev_bf16(X), dev_bf16(Wt), dev_bf16(H), mode=mode)
        assert_bf16_close(host(dH), oracle.dgrad_gelu(f64(X), f64(Wt), f64(H), m), f"random dgrad {M}x{N}x{K}")


def test_random_shapes_rmsnorm_and_cross_entropy():
    for i, (M, N, K) in enumerate(_rand_shapes(11, 6, n_max=2000)):
        X, W, b, Z, g = _rms_case(M, N, K, i % 2 == 0, seed=i)
        q, s = _rms_run(X, W, b, Z, g)
        q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None if b is None else f64(b), f64(Z), f64(g), 1e-6)
        assert_fp8_close(q, s, q_ref, s_ref, f"random rmsnorm {M}x{N}x{K}")
        Md = int(np.random.default_rng(i).integers(1, 33))  # decode shape
        q, s = _rms_run(X[:Md], W, b, Z[:Md], g)
        q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X[:Md]), f64(W), None if b is None else f64(b), f64(Z[:Md]),
                                             f64(g), 1e-6)
        assert_fp8_close(q, s, q_ref, s_ref, f"random rmsnorm decode {Md}x{N}x{K}")
        lab = syn.draw_labels(i, syn.STREAM_LABEL, M, N)
        loss, _ = fl.fused_linear_cross_entropy(dev_bf16(X), dev_bf16(W), None, torch.from_numpy(lab).cuda())
        _assert_loss_close(loss.cpu().numpy().astype(np.float64),
                           oracle.linear_cross_entropy(f64(X), f64(W), None, lab), f"random ce {M}x{N}x{K}")


def test_descriptor_cache_follows_pointer_and_shape_changes():
    """Decode-shaped GELU calls (which encode their tensor maps on every call): a repeated call
    hits the descriptor cache and encodes nothing; new pointers and a new shape are new keys and
    encode again; new contents in the same buffers are read fresh; every result matches the
    oracle, and with the cache off the results are bit-identical."""
    fl.set_descriptor_cache(True)
    M, K = 16, 512
    host_sets, dev_sets = [], []
    for seed, N in ((1, 2048), (2, 2048), (3, 1024)):
        X, W = _draw((M, K), syn.STREAM_X, seed=seed), _draw((N, K), syn.STREAM_W, K ** -0.5, seed=seed)
        host_sets.append((X, W))
        dev_sets.append((dev_bf16(X), dev_bf16(W)))

    def run(i):
        return fl.fused_linear_gelu(dev_sets[i][0], dev_sets[i][1], None, mode="tanh")

    def check(y, i, what):
        X, W = host_sets[i]
        assert_bf16_close(host(y), oracle.linear_gelu(f64(X), f64(W), None, oracle.GELU_TANH), what)

    h0, m0 = fl.descriptor_cache_stats()
    y = run(0)
    h1, m1 = fl.descriptor_cache_stats()
    assert m1 > m0
    check(y, 0, "first call")
    y = run(0)
    h2, m2 = fl.descriptor_cache_stats()
    assert m2 == m1 and h2 > h1, "the repeated call should hit the cache"
    check(y, 0, "cached call")
    y1 = run(1)
    _, m3 = fl.descriptor_cache_stats()
    assert m3 > m2, "new pointers must encode new maps"
    check(y1, 1, "new pointers")
    y = run(2)
    _, m4 = fl.descriptor_cache_stats()
    assert m4 > m3, "a new shape must encode new maps"
    check(y, 2, "new shape")
    dev_sets[0][0].copy_(dev_sets[1][0])
    dev_sets[0][1].copy_(dev_sets[1][1])
    y = run(0)
    check(y, 1, "same buffers, new contents")
    fl.set_descriptor_cache(False)
    try:
        assert torch.equal(run(1), y1)
    finally:
        fl.set_descriptor_cache(True)


def test_two_streams_interleaved():
    """Launches alternating between two streams (each with its own workspaces) give the same
    results as on the default stream."""
    M, N, K = 300, 1024, 256
    X = dev_bf16(_draw((M, K), syn.STREAM_X))
    W = dev_bf16(_draw((N, K), syn.STREAM_W, K ** -0.5))
    Z = dev_bf16(_draw((M, N), syn.STREAM_Z))
    g = dev_bf16(_draw((N,), syn.STREAM_GAMMA, 0.1, 1.0))
    ref_gelu = fl.fused_linear_gelu(X, W, None).clone()
    ref_q, ref_s = [t.clone() for t in fl.fused_linear_residual_rmsnorm_fp8(X, W, None, Z, g, 1e-6)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ws = [fl.rmsnorm_fp8_workspace(M, N, K) for _ in streams]
    outs = []
    for it in range(6):
        k = it % 2
        with torch.cuda.stream(streams[k]):
            outs.append((fl.fused_linear_gelu(X, W, None, stream=streams[k]),
                         fl.fused_linear_residual_rmsnorm_fp8(X, W, None, Z, g, 1e-6, workspace=ws[k],
                                                              stream=streams[k])))
    torch.cuda.synchronize()
    for y, (q, s) in outs:
        assert torch.equal(y, ref_gelu) and torch.equal(q, ref_q) and torch.equal(s, ref_s)


def test_host_threads_on_separate_streams():
    """Four host threads, each with its own stream and workspace, call the library concurrently
    (the ctypes calls release the interpreter lock): every result matches the single-thread one."""
    import threading
    M, N, K = 200, 768, 192
    X = dev_bf16(_draw((M, K), syn.STREAM_X))
    W = dev_bf16(_draw((N, K), syn.STREAM_W, K ** -0.5))
    Z = dev_bf16(_draw((M, N), syn.STREAM_Z))
    g = dev_bf16(_draw((N,), syn.STREAM_GAMMA, 0.1, 1.0))
    lab = torch.from_numpy(syn.draw_labels(0, syn.STREAM_LABEL, M, N)).cuda()
    ref = (fl.fused_linear_gelu(X, W, None, mode="erf").clone(),
           *[t.clone() for t in fl.fused_linear_residual_rmsnorm_fp8(X, W, None, Z, g, 1e-6)],
           fl.fused_linear_cross_entropy(X, W, None, lab)[0].clone())
    torch.cuda.synchronize()
    errors = []

    def worker(tid):
        try:
            st = torch.cuda.Stream()
            ws = fl.rmsnorm_fp8_workspace(M, N, K)
            wc = fl.cross_entropy_workspace(M, N)
            with torch.cuda.stream(st):
                for _ in range(5):
                    y = fl.fused_linear_gelu(X, W, None, mode="erf", stream=st)
                    q, s = fl.fused_linear_residual_rmsnorm_fp8(X, W, None, Z, g, 1e-6, workspace=ws, stream=st)
                    loss, _ = fl.fused_linear_cross_entropy(X, W, None, lab, workspace=wc, stream=st)
                    st.synchronize()
                    for a, b2 in zip(ref, (y, q, s, loss)):
                        if not torch.equal(a, b2):
                            errors.append(f"thread {tid}: result differs")
        except Exception as e:  # reported below
            errors.append(f"thread {tid}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]


def test_default_outputs_accept_ragged_widths():
    """Outputs the binding allocates get 16-byte row pitches, so widths that are not a multiple of
    the 16-byte element count work: N = 300 (bf16) and N = 1000 (E4M3).  Inputs keep the rule
    (the residual here is given a padded pitch)."""
    M, K = 130, 64
    X = _draw((M, K), syn.STREAM_X)
    for N in (300, 1000):
        W = _draw((N, K), syn.STREAM_W, K ** -0.5)
        Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), None, mode="tanh")
        assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), None, oracle.GELU_TANH), f"ragged gelu N={N}")
        Z = _draw((M, N), syn.STREAM_Z)
        g = _draw((N,), syn.STREAM_GAMMA, 0.1, 1.0)
        Zd = torch.zeros((M, -(-N // 8) * 8), dtype=torch.bfloat16, device="cuda")[:, :N]  # inputs: 16-byte pitch
        Zd.copy_(dev_bf16(Z))
        q, s = fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(X), dev_bf16(W), None, Zd, dev_bf16(g), 1e-6)
        q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None, f64(Z), f64(g), 1e-6)
        assert_fp8_close(q.cpu().numpy(), s.cpu().numpy().astype(np.float64), q_ref, s_ref, f"ragged rmsnorm N={N}")
