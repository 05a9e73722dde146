"""A seeded random sweep over every computing entry point, on the GPU, against the fp64 oracle.

Each iteration draws one problem shape (a decode shape, M <= 32, two times in five, else up to 600
rows; N and K ragged multiples of 8), a CTA cap (none three times in four, else 1 to the SM count),
CTA pairing on or off and the decode kernels on or off, then runs the shape through GELU (bf16, and
now and then the fp32 3xTF32 form), SwiGLU, the block-scaled write-back (a random format, with or
without the inverse smoothing factor), the GELU dgrad, the SwiGLU backward, residual + RMSNorm +
FP8 (with or without h_out; the workspace reset afterwards), the LM-head cross-entropy (every
seventh label ignored), the deferred-scale chain, QKV + RoPE (explicit or implied positions) and its
grouped-query FP8 K/V form.  Every failure of a block is collected before the block fails, so one
run names every case that went wrong.  The tolerances are the parity tests' own.
"""
import numpy as np
import pytest
import torch

import gemm_epilogue_tcgen05_gb300 as fl
import oracle
import synthetic as syn
from parity_utils import (assert_bf16_close, assert_f32_close, assert_fp8_close, assert_loss_close, assert_quant_close,
                          assert_ws_reset, check_kv_fp8, dev_bf16, dev_f32, f64, host, qkv_ref, rms_case)

pytestmark = pytest.mark.gpu

ITERATIONS_PER_BLOCK = 10
E2M1 = np.array([oracle.e2m1_decode(c) for c in range(16)])


@pytest.fixture(autouse=True)
def _defaults():
    yield
    fl.set_max_ctas(0)
    fl.set_cta_pairing(True)
    fl.set_linear_decode(True)
    assert fl.device_status() == fl.FL_OK


def _draw(shape, stream, std=1.0, mean=0.0, seed=0, dtype="bf16"):
    return syn.draw(seed, stream, shape, mean, std, dtype)


def _quant_decoders(fmt):
    return {"scale": oracle.e4m3_decode,
            "value": (oracle.e4m3_decode if fmt == 0 else
                      (lambda c: np.where(c & 8, c.astype(np.int32) - 16, c).astype(np.float64)) if fmt == 1 else
                      (lambda c: E2M1[c]))}


def _iteration(s: int, sms: int, fails: list):
    rng = np.random.default_rng(s)
    cap = int(rng.choice([0, 0, 0, int(rng.integers(1, sms + 1))]))
    pairing = bool(rng.integers(0, 2))
    decode_on = bool(rng.integers(0, 4) != 0)
    fl.set_max_ctas(cap)
    fl.set_cta_pairing(pairing)
    fl.set_linear_decode(decode_on)
    M = int(rng.integers(1, 33)) if rng.integers(0, 5) < 2 else int(rng.integers(33, 600))
    N = int(rng.integers(1, 320)) * 8
    K = int(rng.integers(1, 190)) * 8
    tag = f"seed {s} cap {cap} pairing {int(pairing)} decode {int(decode_on)} {M}x{N}x{K}"

    def case(name, fn):
        try:
            fn()
            st = fl.device_status()
            assert st == fl.FL_OK, f"device status {st}"
        except Exception as e:  # noqa: BLE001 -- every failure of the block is reported together
            fails.append(f"{name} {tag}: {e!r}"[:400])

    X = _draw((M, K), syn.STREAM_X, seed=s)
    W = _draw((N, K), syn.STREAM_W, K ** -0.5, seed=s)
    b = _draw((N,), syn.STREAM_B, 0.3, seed=s) if rng.integers(0, 2) else None
    fb = None if b is None else f64(b)
    db = None if b is None else dev_bf16(b)
    mode = "tanh" if rng.integers(0, 2) else "erf"
    m = oracle.GELU_TANH if mode == "tanh" else oracle.GELU_ERF

    def gelu():
        Y = fl.fused_linear_gelu(dev_bf16(X), dev_bf16(W), db, mode=mode)
        assert_bf16_close(host(Y), oracle.linear_gelu(f64(X), f64(W), fb, m), "gelu")
    case("gelu", gelu)

    if rng.integers(0, 3) == 0:
        def gelu_f32():
            Mf, Nf, Kf = min(M, 200), min(N, 512), min(K, 256)
            Xf = _draw((Mf, Kf), syn.STREAM_X, seed=s, dtype="f32")
            Wf = _draw((Nf, Kf), syn.STREAM_W, Kf ** -0.5, seed=s, dtype="f32")
            Y = fl.fused_linear_gelu(dev_f32(Xf), dev_f32(Wf), None, mode=mode)
            assert_f32_close(host(Y), oracle.linear_gelu(f64(Xf, "f32"), f64(Wf, "f32"), None, m), "gelu fp32")
        case("gelu fp32", gelu_f32)

    Wu = _draw((N, K), syn.STREAM_WUP, K ** -0.5, seed=s)
    bu = _draw((N,), syn.STREAM_BUP, 0.3, seed=s) if b is not None else None

    def swiglu():
        Y = fl.fused_swiglu(dev_bf16(X), dev_bf16(W), dev_bf16(Wu), db, None if bu is None else dev_bf16(bu))
        assert_bf16_close(host(Y), oracle.swiglu(f64(X), f64(W), f64(Wu), fb, None if bu is None else f64(bu)),
                          "swiglu")
    case("swiglu", swiglu)

    if N % 16 == 0:
        fmt = int(rng.integers(0, 3))
        inv = syn.draw_inv_smooth(s, N) if rng.integers(0, 2) else None

        def quant():
            Yq, S = fl.fused_linear_quant(dev_bf16(X), dev_bf16(W), db, fmt,
                                          inv_smooth=None if inv is None else torch.from_numpy(inv).cuda())
            q_ref, s_ref, y_ref = oracle.linear_quant(f64(X), f64(W), fb, fmt,
                                                      inv_smooth=None if inv is None else inv.astype(np.float64))
            assert_quant_close(fmt, Yq.cpu().numpy(), S.cpu().numpy(), q_ref, s_ref, y_ref, _quant_decoders(fmt),
                               f"quant {fmt} smoothing {inv is not None}")
        case(f"quant {fmt}", quant)

    def dgrad():
        Wt = _draw((K, N), syn.STREAM_W2, K ** -0.5, seed=s)
        H = _draw((M, N), syn.STREAM_Z, 2.0, seed=s)
        dH = fl.fused_dgrad_gelu(dev_bf16(X), dev_bf16(Wt), dev_bf16(H), mode=mode)
        assert_bf16_close(host(dH), oracle.dgrad_gelu(f64(X), f64(Wt), f64(H), m), "dgrad")
    case("dgrad gelu", dgrad)

    def swiglu_bwd():
        Wd = _draw((K, N), syn.STREAM_W, K ** -0.5, seed=s)
        G = _draw((M, N), syn.STREAM_Z, 3.0, seed=s)
        U = _draw((M, N), syn.STREAM_GAMMA, seed=s)
        out = fl.fused_swiglu_bwd(dev_bf16(X), dev_bf16(Wd), dev_bf16(G), dev_bf16(U))
        assert_bf16_close(host(out), oracle.swiglu_bwd(f64(X), f64(Wd), f64(G), f64(U)), "swiglu bwd")
    case("swiglu bwd", swiglu_bwd)

    want_h = bool(rng.integers(0, 2))
    Xr, Wr, br, Z, g = rms_case(M, N, K, b is not None, seed=s)
    fbr = None if br is None else f64(br)

    def rmsnorm():
        ws = fl.rmsnorm_fp8_workspace(M, N, K)
        out = fl.fused_linear_residual_rmsnorm_fp8(dev_bf16(Xr), dev_bf16(Wr), None if br is None else dev_bf16(br),
                                                   dev_bf16(Z), dev_bf16(g), 1e-6, workspace=ws,
                                                   h_out=True if want_h else None)
        q_ref, s_ref, _ = oracle.rmsnorm_fp8(f64(Xr), f64(Wr), fbr, f64(Z), f64(g), 1e-6)
        assert_fp8_close(out[0].cpu().numpy(), out[1].cpu().numpy().astype(np.float64), q_ref, s_ref, "rmsnorm")
        if want_h:
            assert_bf16_close(host(out[2]), oracle.linear(f64(Xr), f64(Wr), fbr) + f64(Z), "rmsnorm h_out")
        assert_ws_reset(ws, M, N)
        assert fl.check_device_status(ws) == fl.FL_OK
    case("rmsnorm fp8", rmsnorm)

    def cross_entropy():
        lab = syn.draw_labels(s, syn.STREAM_LABEL, M, N)
        lab[::7] = -1
        loss, _ = fl.fused_linear_cross_entropy(dev_bf16(X), dev_bf16(W), db, torch.from_numpy(lab).cuda())
        assert_loss_close(loss.cpu().numpy().astype(np.float64), oracle.linear_cross_entropy(f64(X), f64(W), fb, lab),
                          "cross-entropy")
    case("cross-entropy", cross_entropy)

    N2 = int(rng.integers(1, 200)) * 8

    def chain():
        W1 = _draw((N2, N), syn.STREAM_W2, N ** -0.5, seed=s)
        H2, H1, part = fl.fused_linear_residual_gamma(dev_bf16(Xr), dev_bf16(Wr),
                                                      None if br is None else dev_bf16(br), dev_bf16(Z), dev_bf16(g))
        Y = fl.fused_linear_rms_rowscale(H2, dev_bf16(W1), None, part, N, 1e-6)
        y_ref, h1_ref = oracle.residual_rmsnorm_linear(f64(Xr), f64(Wr), fbr, f64(Z), f64(g), 1e-6, f64(W1), None)
        assert_bf16_close(host(H1), h1_ref, "chain h1")
        assert_bf16_close(host(Y), y_ref, "chain y")
    case(f"chain to {N2}", chain)

    H = 2 * int(rng.integers(1, 5))  # n_heads * 128 must be a multiple of 256
    Kq = int(rng.integers(1, 100)) * 8
    use_pos = bool(rng.integers(0, 2))
    Xq = _draw((M, Kq), syn.STREAM_X, seed=s)

    def qkv():
        Wq = _draw((3 * H * 128, Kq), syn.STREAM_W, Kq ** -0.5, seed=s)
        bq = _draw((3 * H * 128,), syn.STREAM_B, 0.02, seed=s) if b is not None else None
        pos = rng.integers(0, 1 << 16, size=M).astype(np.int32) if use_pos else np.arange(M) % 37
        q, k, v = fl.fused_qkv_rope(dev_bf16(Xq), dev_bf16(Wq), None if bq is None else dev_bf16(bq), n_heads=H,
                                    head_dim=128, seq_len=37,
                                    positions=torch.from_numpy(pos).cuda() if use_pos else None)
        assert_bf16_close(host(torch.cat([q, k, v], 1)), qkv_ref(Xq, Wq, bq, H, 128, pos), "qkv rope")
    case(f"qkv rope {H} heads K {Kq}", qkv)

    Hkv = int(rng.choice([2, 4, 8]))
    Hq = Hkv * int(rng.choice([1, 2, 4]))

    def qkv_fp8kv():
        Wq = _draw(((Hq + 2 * Hkv) * 128, Kq), syn.STREAM_W, Kq ** -0.5, seed=s + 1)
        bq = _draw(((Hq + 2 * Hkv) * 128,), syn.STREAM_B, 0.5, seed=s + 1) if b is not None else None
        pos = rng.integers(0, 1 << 20, size=M).astype(np.int32)
        out = fl.fused_qkv_rope_fp8kv(dev_bf16(Xq), dev_bf16(Wq), None if bq is None else dev_bf16(bq), n_heads=Hq,
                                      n_kv_heads=Hkv, head_dim=128, positions=torch.from_numpy(pos).cuda())
        ref = oracle.qkv_rope_kv_fp8(f64(Xq), f64(Wq), None if bq is None else f64(bq), Hq, Hkv, 128, 1e4, pos)
        check_kv_fp8(out, ref, "qkv fp8 kv")
    case(f"qkv fp8 kv {Hq}/{Hkv} heads K {Kq}", qkv_fp8kv)


@pytest.mark.parametrize("block", range(4))
def test_random_sweep(block):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fails = []
    for it in range(ITERATIONS_PER_BLOCK):
        _iteration(7000 + block * ITERATIONS_PER_BLOCK + it, sms, fails)
        torch.cuda.empty_cache()
    assert not fails, f"{len(fails)} failing cases:\n" + "\n".join(fails)
