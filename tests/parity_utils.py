"""Shared helpers for the GPU parity tests: moving generator output to the
device, reading results back, and the tolerance checks (bf16 outputs:
|gpu - ref| <= 2e-2 + 1e-2 |ref|; fp32 outputs: |gpu - ref| <= 1e-4; FP8
codes: ordered-code distance <= 1; per-row scales: relative error <= 1e-3;
block-scaled codes: see ``assert_quant_close``)."""
import numpy as np
import torch

import oracle
import synthetic as syn

BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL = 1e-4
SCALE_RTOL = 1e-3

# Error statistics of every comparison, printed as a table at the end of a test session
# (tol_used: the largest error as a fraction of the allowed one).
REPORT = []


def _record(kind: str, what: str, n: int, **stats):
    REPORT.append({"kind": kind, "what": what, "n": int(n), **{k: float(v) for k, v in stats.items()}})


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def f64(a: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    return syn.to_f64(a, dtype)


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_bf16_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(gpu - ref)
    _record("bf16", what, err.size, max_abs=err.max(initial=0),
            tol_used=(err / (BF16_ATOL + BF16_RTOL * np.abs(ref))).max(initial=0))
    bad = err > BF16_ATOL + BF16_RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside 2e-2+1e-2|ref|; "
                           f"max abs err {err.max():.4g} at {np.unravel_index(np.argmax(err), err.shape)}")
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"


def assert_f32_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(gpu - ref)
    _record("fp32", what, err.size, max_abs=err.max(initial=0), tol_used=err.max(initial=0) / F32_ATOL)
    assert err.max() <= F32_ATOL, f"{what}: max abs err {err.max():.3g} > 1e-4"


def ordered_e4m3(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def assert_fp8_close(codes: np.ndarray, scale: np.ndarray, q_ref: np.ndarray, s_ref: np.ndarray, what=""):
    d = np.abs(ordered_e4m3(codes) - ordered_e4m3(q_ref))
    _record("e4m3", what, d.size, max_code_dist=d.max(initial=0), frac_codes_differ=np.mean(d != 0),
            scale_max_rel=(np.abs(scale - s_ref) / np.maximum(np.abs(s_ref), 1e-30)).max(initial=0))
    assert d.max() <= 1, f"{what}: code distance {d.max()} at {np.unravel_index(np.argmax(d), d.shape)}"
    rel = np.abs(scale - s_ref) / np.maximum(np.abs(s_ref), 1e-30)
    assert rel.max() <= SCALE_RTOL, f"{what}: scale rel err {rel.max():.3g}"
    # fraction of codes that differ at all stays small (rounding-boundary cases only)
    assert np.mean(d != 0) < 0.02, f"{what}: {np.mean(d != 0):.3%} of codes differ"


def sample_rows(M: int, seed: int = 0) -> np.ndarray:
    """Rows of a full-size workload to compare: one random row in every 32-row slice, so every
    128-row block, both halves of every 256-row pair tile and the rows of every epilogue warp of
    every tile are checked (256 rows at M = 8192), plus the edges of the first blocks and the last
    row."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, 127, 128, 129, 255, 256, M - 1}
    rows |= {s + int(rng.integers(0, min(32, M - s))) for s in range(0, M, 32)}
    return np.array(sorted(r for r in rows if 0 <= r < M), dtype=np.int64)


def ordered_nibble(codes: np.ndarray, fmt: int) -> np.ndarray:
    """4-bit codes (already unpacked) as integers ordered like the values they encode."""
    c = codes.astype(np.int32) & 15
    if fmt == 1:  # two's complement INT4
        return np.where(c & 8, c - 16, c)
    return np.where(c & 8, -(c & 7), c & 7)  # E2M1: sign bit, then a monotone magnitude index


def unpack_nibbles(packed: np.ndarray, n: int) -> np.ndarray:
    """[rows, ceil(n/2)] bytes -> [rows, n] nibbles; column 2j is the low nibble of byte j."""
    out = np.empty((packed.shape[0], 2 * packed.shape[1]), dtype=np.uint8)
    out[:, 0::2] = packed & 15
    out[:, 1::2] = packed >> 4
    return out[:, :n]


def assert_quant_close(fmt: int, codes, scales, q_ref, s_ref, y_ref, decode, what=""):
    """Block-scaled output against the oracle.

    Scales: fp32 scales within 1e-3 relative; NVFP4's E4M3 scale codes within one
    code step and equal for at least 98% of the blocks.  Codes: in blocks whose
    scale code agrees, within one code step of the oracle's, and equal for at
    least 98% of all values.  Every value, dequantised with the kernel's own
    scale, lies within half the format's largest gap of the exact output
    (``decode`` maps codes to the values they stand for).
    """
    n = y_ref.shape[1]
    bs = {0: 128, 1: 32, 2: 16}[fmt]
    blk = np.arange(n) // bs
    if fmt == 0:
        oc, orf = ordered_e4m3(codes), ordered_e4m3(q_ref)
        same_scale = np.ones(scales.shape, dtype=bool)
        s_val = scales.astype(np.float64)
    else:
        oc = ordered_nibble(unpack_nibbles(codes, n), fmt)
        orf = ordered_nibble(unpack_nibbles(q_ref, n), fmt)
        if fmt == 2:
            ds = np.abs(ordered_e4m3(scales) - ordered_e4m3(s_ref.astype(np.uint8)))
            assert ds.max() <= 1, f"{what}: scale code distance {ds.max()}"
            assert np.mean(ds != 0) < 0.02, f"{what}: {np.mean(ds != 0):.3%} of scale codes differ"
            same_scale = ds == 0
            s_val = decode["scale"](scales)
        else:
            same_scale = np.ones(scales.shape, dtype=bool)
            s_val = scales.astype(np.float64)
    if fmt != 2:
        rel = np.abs(s_val - s_ref) / np.maximum(np.abs(s_ref), 1e-30)
        assert rel.max() <= SCALE_RTOL, f"{what}: scale rel err {rel.max():.3g}"
    d = np.abs(oc - orf)
    _record({0: "fp8 1x128", 1: "int4 g32", 2: "nvfp4 g16"}[fmt], what, d.size, max_code_dist=d.max(initial=0),
            frac_codes_differ=np.mean(d != 0))
    mask = same_scale[:, blk]
    assert d[mask].max(initial=0) <= 1, f"{what}: code distance {d[mask].max()}"
    assert np.mean(d != 0) < 0.02, f"{what}: {np.mean(d != 0):.3%} of codes differ"
    deq = decode["value"](codes if fmt == 0 else unpack_nibbles(codes, n)) * s_val[:, blk]
    half_gap = {0: None, 1: 0.5, 2: 1.0}[fmt]
    if fmt == 0:  # E4M3: relative half-step 2^-4, subnormal half-step 2^-10 (times the scale)
        bound = 2.0 ** -4 * np.abs(y_ref) + 2.0 ** -10 * s_val[:, blk]
    else:
        bound = half_gap * s_val[:, blk]
    err = np.abs(deq - y_ref)
    slack = 1e-5 * np.abs(y_ref).max(initial=0) + 1e-12
    assert np.all(err <= bound + slack), f"{what}: dequantised error {np.max(err - bound):.3g} over the bound"


# ------------------------------------------------------------------ cases and checks shared by the GPU test files
def rms_case(M: int, N: int, K: int, bias: bool, seed: int = 0):
    """Seeded operands of a residual + RMSNorm + FP8 call: X, W, b (or None), Z, gamma."""
    X = syn.draw(seed, syn.STREAM_X, (M, K), 0.0, 1.0, "bf16")
    W = syn.draw(seed, syn.STREAM_W, (N, K), 0.0, K ** -0.5, "bf16")
    b = syn.draw(seed, syn.STREAM_B, (N,), 0.0, 0.02, "bf16") if bias else None
    Z = syn.draw(seed, syn.STREAM_Z, (M, N), 0.0, 1.0, "bf16")
    g = syn.draw(seed, syn.STREAM_GAMMA, (N,), 1.0, 0.1, "bf16")
    return X, W, b, Z, g


def qkv_ref(X, Wq, bq, H, D, pos, theta=10000.0):
    """The oracle's QKV + RoPE output [Q | K | V] for bf16 host operands."""
    return oracle.qkv_rope(f64(X), f64(Wq), None if bq is None else f64(bq), H, D, theta, pos)


def assert_loss_close(got, ref, what):
    """The fp32 loss within the fp32 output bound, max |gpu - oracle| <= 1e-4 (recorded)."""
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), f"{what}: NaN pattern differs"
    assert_f32_close(got[~nan], ref[~nan], f"{what}: loss")


def check_kv_fp8(out, ref, what):
    """Q in bf16, and the K and V codes and scales of the FP8 cache form, against the oracle; the
    dequantised K and V also within half an E4M3 step of the exact values."""
    Q, Kq, Vq, ks, vs = out
    assert_bf16_close(host(Q), ref["q"], f"{what}: Q")
    hd = 128
    for codes, scale, r_codes, r_scale, exact, nm in ((Kq, ks, ref["kq"], ref["ks"], ref["kv"][:, :Kq.shape[1]], "K"),
                                                      (Vq, vs, ref["vq"], ref["vs"], ref["kv"][:, Kq.shape[1]:], "V")):
        c, s = codes.cpu().numpy(), scale.cpu().numpy().astype(np.float64)
        assert_fp8_close(c, s, r_codes, r_scale, f"{what}: {nm}")
        heads = np.arange(c.shape[1]) // hd
        deq = oracle.e4m3_decode(c) * s[:, heads]
        bound = 2.0 ** -4 * np.abs(exact) + 2.0 ** -10 * s[:, heads] + 1e-5 * np.abs(exact).max()
        assert np.all(np.abs(deq - exact) <= bound), f"{what}: {nm} dequantised outside the E4M3 half-step"


def assert_ws_reset(ws, M, N):
    """After a call the workspace's status words and the counters the kernels wait on are zero
    again (the decode kernels' epoch word, at byte 128 of the status area, counts calls)."""
    assert torch.count_nonzero(ws[:32]) == 0, "status record set"
    n = 4 * (-(-N // 128) + 2) if M <= 32 else 8 * -(-M // 128)
    assert torch.count_nonzero(ws[256:256 + n]) == 0, "counters not reset"
