"""Shared helpers for the GPU parity tests: moving generator output to the
device, reading results back, and the tolerance checks (bf16 outputs:
|gpu - ref| <= 2e-2 + 1e-2 |ref|; fp32 outputs: |gpu - ref| <= 1e-4; FP8
codes: ordered-code distance <= 1; per-row scales: relative error <= 1e-3)."""
import numpy as np
import torch

import synthetic as syn

BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL = 1e-4
SCALE_RTOL = 1e-3


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
    bad = err > BF16_ATOL + BF16_RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside 2e-2+1e-2|ref|; "
                           f"max abs err {err.max():.4g} at {np.unravel_index(np.argmax(err), err.shape)}")
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"


def assert_f32_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(gpu - ref)
    assert err.max() <= F32_ATOL, f"{what}: max abs err {err.max():.3g} > 1e-4"


def ordered_e4m3(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def assert_fp8_close(codes: np.ndarray, scale: np.ndarray, q_ref: np.ndarray, s_ref: np.ndarray, what=""):
    d = np.abs(ordered_e4m3(codes) - ordered_e4m3(q_ref))
    assert d.max() <= 1, f"{what}: code distance {d.max()} at {np.unravel_index(np.argmax(d), d.shape)}"
    rel = np.abs(scale - s_ref) / np.maximum(np.abs(s_ref), 1e-30)
    assert rel.max() <= SCALE_RTOL, f"{what}: scale rel err {rel.max():.3g}"
    # fraction of codes that differ at all stays small (rounding-boundary cases only)
    assert np.mean(d != 0) < 0.02, f"{what}: {np.mean(d != 0):.3%} of codes differ"


def sample_rows(M: int, extra: int = 4, seed: int = 0) -> np.ndarray:
    """Rows that cover tile edges (first/last of 128-row blocks) plus a few random ones."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, 127, 128, M - 1, M // 2, min(M - 1, 129)}
    rows |= set(rng.integers(0, M, size=extra).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < M), dtype=np.int64)
