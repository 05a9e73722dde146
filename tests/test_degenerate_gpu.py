"""Degenerate inputs and range edges the method defines, on the GPU, through the C ABI, against the
fp64 oracle: rows, heads and blocks whose maximum is zero (scale 0 and zero codes), K = 0 (the Linear
output is the bias alone), empty problems (M = 0 or N = 0) for every entry point (nothing is
written), NVFP4 block scales at both ends of E4M3, and RoPE at the largest accepted positions."""
import numpy as np
import pytest
import torch

import gemm_epilogue_tcgen05_gb300 as fl
import oracle
import synthetic as syn
from parity_utils import (assert_bf16_close, assert_fp8_close, assert_quant_close, dev_bf16, f64, host,
                          check_kv_fp8, ordered_e4m3, ordered_nibble, qkv_ref, unpack_nibbles)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    fl.set_max_ctas(0)
    fl.set_cta_pairing(True)
    yield
    fl.set_max_ctas(0)
    fl.set_cta_pairing(True)
    assert fl.device_status() == fl.FL_OK


def _draw(shape, stream, std=1.0, mean=0.0, seed=0):
    return syn.draw(seed, stream, shape, mean, std, "bf16")


@pytest.mark.parametrize("M,N,K,cap", [(300, 1024, 256, 0), (24, 4096, 512, 0), (24, 4096, 512, 16)])
def test_rmsnorm_fp8_zero_row_gets_zero_scale_and_codes(M, N, K, cap):
    """A row whose h = X W^T + Z is all zero has maximum 0: scale 0 and all codes 0 (prefill, the
    cluster decode kernel and, under a CTA cap, the flat one); the other rows are the oracle's."""
    fl.set_max_ctas(cap)
    X = _draw((M, K), syn.STREAM_X, seed=8)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=8)
    Z = _draw((M, N), syn.STREAM_Z, seed=8)
    g = _draw((N,), syn.STREAM_GAMMA, 0.1, 1.0, seed=8)
    g[1::3] ^= 0x8000  # a third of gamma negative (bf16 sign bit): a zero row must still code as +0
    zr = [0, M // 2, M - 1]
    X[zr] = 0
    Z[zr] = 0
    q, s = fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(X), dev_bf16(W), None, dev_bf16(Z), dev_bf16(g), 1e-6,
                                                workspace=fl.rmsnorm_fp8_workspace(M, N, K))
    q, s = q.cpu().numpy(), s.cpu().numpy().astype(np.float64)
    assert not q[zr].any() and not s[zr].any()
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(X), f64(W), None, f64(Z), f64(g), 1e-6)
    assert_fp8_close(q, s, q_ref, s_ref, f"zero rows {M}x{N}x{K} cap {cap}")


@pytest.mark.parametrize("M", [40, 5])
def test_rmsnorm_fp8_and_h_out_with_k_zero(M):
    """K = 0: h = b + Z; codes, scales and h_out against the oracle."""
    N = 512
    b = _draw((N,), syn.STREAM_B, 0.5, seed=9)
    Z = _draw((M, N), syn.STREAM_Z, seed=9)
    g = _draw((N,), syn.STREAM_GAMMA, 0.1, 1.0, seed=9)
    Xe = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    We = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    q, s, h = fl.fused_linear_residual_rmsnorm_fp8(Xe, We, dev_bf16(b), dev_bf16(Z), dev_bf16(g), 1e-6, h_out=True)
    h_ref = f64(b)[None, :] + f64(Z)
    assert_bf16_close(host(h), h_ref, f"h_out K=0 M={M}")
    q_ref, s_ref, _ = oracle.rmsnorm_fp8(np.zeros((M, 0)), np.zeros((N, 0)), f64(b), f64(Z), f64(g), 1e-6)
    assert_fp8_close(q.cpu().numpy(), s.cpu().numpy().astype(np.float64), q_ref, s_ref, f"K=0 M={M}")


@pytest.mark.parametrize("M", [257, 7])
def test_qkv_fp8kv_zero_token_gets_zero_scales_and_codes(M):
    """A token whose projection is all zero (zero input row, no bias) has head maxima 0: every K and
    V scale 0 and every code 0, prefill and decode."""
    H, Hkv, D, K = 4, 2, 128, 256
    X = _draw((M, K), syn.STREAM_X, seed=10)
    X[[0, M - 1]] = 0
    Wq = _draw(((H + 2 * Hkv) * D, K), syn.STREAM_W, K ** -0.5, seed=10)
    Q, Kq, Vq, ks, vs = fl.fused_qkv_rope_fp8kv(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, n_kv_heads=Hkv,
                                                head_dim=D, seq_len=64)
    for t in (Kq, Vq, ks, vs, Q):
        assert torch.count_nonzero(t[0]) == 0 and torch.count_nonzero(t[M - 1]) == 0
    ref = oracle.qkv_rope_kv_fp8(f64(X), f64(Wq), None, H, Hkv, D, 10000.0, np.arange(M) % 64)
    assert_fp8_close(Kq.cpu().numpy(), ks.cpu().numpy().astype(np.float64), ref["kq"], ref["ks"], f"K M={M}")
    assert_fp8_close(Vq.cpu().numpy(), vs.cpu().numpy().astype(np.float64), ref["vq"], ref["vs"], f"V M={M}")
    assert_bf16_close(host(Q), ref["q"], f"Q M={M}")


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_quant_smoothing_zero_factors_give_zero_blocks(fmt):
    """Inverse smoothing factors that are zero over a whole block make that block's maximum 0: scale
    0 and zero codes; partly zero blocks keep the oracle's scale and codes."""
    M, N, K = 130, 512, 96
    X = _draw((M, K), syn.STREAM_X, seed=11)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=11)
    b = _draw((N,), syn.STREAM_B, 0.5, seed=11)
    inv = syn.draw_inv_smooth(11, N)
    bs = {0: 128, 1: 32, 2: 16}[fmt]
    inv[:bs] = 0.0          # the first block of every row: all zero
    inv[bs + 3:bs + 7] = 0  # part of the second block
    Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), dev_bf16(b), fmt, inv_smooth=torch.from_numpy(inv).cuda())
    Yq, S = Yq.cpu().numpy(), S.cpu().numpy()
    assert not S[:, 0].any()
    assert not Yq[:, :bs if fmt == 0 else bs // 2].any()
    q_ref, s_ref, y_ref = oracle.linear_quant(f64(X), f64(W), f64(b), fmt, inv_smooth=inv.astype(np.float64))
    e2m1 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    dec = {"scale": lambda c: oracle.e4m3_decode(c)}
    dec["value"] = (lambda c: oracle.e4m3_decode(c)) if fmt == 0 else (
        (lambda c: np.where(c & 8, c.astype(np.int32) - 16, c).astype(np.float64)) if fmt == 1 else (lambda c: e2m1[c]))
    assert_quant_close(fmt, Yq, S, q_ref, s_ref, y_ref, dec, f"zero smoothing block fmt {fmt}")


def test_every_entry_point_accepts_empty_problems():
    """M = 0 (or N = 0 where the call has one) returns FL_OK and writes nothing."""
    dev = "cuda"
    lib = fl.load()
    sentinel = torch.full((64,), 7, dtype=torch.uint8, device=dev)
    p = sentinel.data_ptr()
    a = None
    # M = 0 through the C ABI, with real (untouched) output pointers
    st = [
        lib.fused_linear_gelu(a, a, a, p, 0, 64, 64, 64, 64, 64, fl.FL_BF16, fl.FL_GELU_TANH, None),
        lib.fused_swiglu(a, a, a, a, a, p, 0, 64, 64, 64, 64, 64, None),
        lib.fused_linear_quant(a, a, a, a, p, p, 0, 64, 64, 64, 64, 64, 1, 0, None),
        lib.fused_dgrad_gelu(a, a, a, p, 0, 64, 64, 64, 64, 64, 64, fl.FL_GELU_TANH, None),
        lib.fused_swiglu_bwd(a, a, a, a, p, 0, 64, 64, 64, 64, 64, 128, None),
        lib.fused_linear_residual_rmsnorm_fp8(a, a, a, a, a, 1e-6, p, p, p, 0, 64, 64, 64, 64, 64, 64, a, 0, None),
        lib.fused_linear_residual_rmsnorm_fp8(a, a, a, a, a, 1e-6, p, p, p, 8, 0, 64, 64, 64, 64, 64, a, 0, None),
        lib.fused_linear_cross_entropy(a, a, a, a, p, a, 0, 64, 64, 64, 64, 0, a, 0, None),
        lib.fused_qkv_rope(a, a, a, p, p, p, a, 0, 64, 2, 128, 16, 1e4, 64, 64, 256, None),
    ]
    assert st == [fl.FL_OK] * len(st), st
    torch.cuda.synchronize()
    assert torch.all(sentinel == 7)


def test_nvfp4_scale_saturates_and_underflows_like_the_oracle():
    """NVFP4's block scale is itself an E4M3 byte, e4m3(max / 6).  Inverse smoothing factors from
    1e-7 to 1e7 across the 16-column blocks push it through both ends of E4M3: a block whose
    max / 6 rounds to 0 gets scale 0 and zero codes, and a block whose max / 6 exceeds 448 gets the
    largest scale and codes saturated at +-6.  Scale codes and value codes against the oracle."""
    M, N, K = 48, 512, 128
    X = _draw((M, K), syn.STREAM_X, seed=12)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=12)
    nb = N // 16
    inv = np.repeat((10.0 ** (-7.0 + 14.0 * np.arange(nb) / (nb - 1))).astype(np.float32), 16)
    Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), None, 2, inv_smooth=torch.from_numpy(inv).cuda())
    Yq, S = Yq.cpu().numpy(), S.cpu().numpy()
    q_ref, s_ref, _ = oracle.linear_quant(f64(X), f64(W), None, 2, inv_smooth=inv.astype(np.float64))
    s_ref = s_ref.astype(np.uint8)
    assert (s_ref == 0).sum() >= 4 * M and (s_ref == 0x7E).sum() >= 4 * M, "both ends of E4M3 are reached"
    ds = np.abs(ordered_e4m3(S) - ordered_e4m3(s_ref))
    assert ds.max() <= 1 and np.mean(ds != 0) < 0.02, "scale codes"
    assert np.array_equal(S == 0, s_ref == 0) and np.array_equal(S == 0x7E, s_ref == 0x7E), "saturated / zero scales"
    codes, ref = unpack_nibbles(Yq, N), unpack_nibbles(q_ref, N)
    blk = np.arange(N) // 16
    assert not codes[(S == 0)[:, blk]].any(), "a zero scale gives zero codes"
    sat = (S == 0x7E)[:, blk]
    assert np.mean((codes[sat] & 7) == 7) > 0.5, "saturated blocks hold mostly +-6"
    d = np.abs(ordered_nibble(codes, 2) - ordered_nibble(ref, 2))
    same = (ds == 0)[:, blk]
    assert d[same].max(initial=0) <= 1 and np.mean(d != 0) < 0.02, "value codes"


@pytest.mark.parametrize("M,decode", [(300, False), (24, True), (24, False)])
def test_rope_at_the_top_of_the_position_range(M, decode):
    """Positions just below 2^24, the largest the entry points accept, where the rotation angle of the
    lowest pair reaches 1.7e7 rad and its reduction decides the result: QKV + RoPE and its FP8 K/V
    form (prefill, the decode kernels, and the GEMM kernel on the decode shape) against the oracle."""
    fl.set_linear_decode(decode)
    try:
        H, Hkv, D, K = 4, 2, 128, 256
        X = _draw((M, K), syn.STREAM_X, seed=13)
        pos = ((1 << 24) - 1 - np.random.default_rng(13).integers(0, 4096, size=M)).astype(np.int32)
        pos[0] = (1 << 24) - 1
        Wq = _draw((3 * H * D, K), syn.STREAM_W, K ** -0.5, seed=13)
        q, k, v = fl.fused_qkv_rope(dev_bf16(X), dev_bf16(Wq), None, n_heads=H, head_dim=D,
                                    positions=torch.from_numpy(pos).cuda())
        assert_bf16_close(host(torch.cat([q, k, v], 1)), qkv_ref(X, Wq, None, H, D, pos), f"qkv top positions M={M}")
        W8 = _draw(((H + 2 * Hkv) * D, K), syn.STREAM_W, K ** -0.5, seed=14)
        out = fl.fused_qkv_rope_fp8kv(dev_bf16(X), dev_bf16(W8), None, n_heads=H, n_kv_heads=Hkv, head_dim=D,
                                      positions=torch.from_numpy(pos).cuda())
        check_kv_fp8(out, oracle.qkv_rope_kv_fp8(f64(X), f64(W8), None, H, Hkv, D, 1e4, pos),
                     f"qkv fp8 kv top positions M={M}")
    finally:
        fl.set_linear_decode(True)
