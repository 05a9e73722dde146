#!/usr/bin/env python
"""Benchmark of the fused Linear + epilogue library on GB300.

One step = one call of the headline workload, Linear + bias + GELU(tanh) at
M=8192, N=16384, K=4096 in bf16 (fp32 accumulate), with inputs resident in
HBM and L2 flushed (a 256 MiB write) before every timed launch.  Each launch
is timed with CUDA events on the stream it is launched on.  `value` is
TFLOP/s over all ranks (2*M*N*K per step per rank); `e2e` repeats the
measurement with the inputs copied from pinned host memory and the output
copied back inside the timed region.  The other fused workloads of the hot
path are measured the same way and reported under `rows` (TFLOP/s, or HBM
GB/s for the decode shape).

`--impl reference` times the fp64 CPU oracle on a bounded row sample of the
same workload instead (rank 0 only).

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one rank per GPU; ranks run independent replicas of
the workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

HEADLINE = "gelu_tanh_8192x16384x4096"
DECODE = "rmsnorm_fp8_decode_32x4096x14336"  # the decode half of the metric (HBM GB/s)
METRIC = "fused GEMM+epilogue TFLOP/s & % bf16 tensor peak; decode-shape HBM GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------- environment
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS, "source": "fallback"}


# Vendor figures for context beside the measured peaks: dense bf16 tensor rate and HBM3e bandwidth.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and with whitespace runs collapsed, so that a change
    to comments alone keeps the hash (string and character literals are kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the library's source code (comments and layout excluded): the key under which the
    committed ncu traffic figures are looked up."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_epilogue_tcgen05_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == want and parts[1] == workload:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples (100 ms) of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        with open(self.out.name) as f:
            rows = [[c.strip() for c in line.split(",")] for line in f if line.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Largest value of x over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank; the job took the slowest rank's time."""
    return world * units_per_rank / seconds_max


# ----------------------------------------------------------------------------- byte model
def _nbytes(shape, dt: str) -> int:
    return math.prod(shape) * (2 if dt == "bf16" else 4)


def operand_bytes(w) -> dict:
    """Bytes of every input of one call, each read once (weights included)."""
    out = {name: _nbytes(shape, dt) for name, _, shape, _, _, dt in syn.operand_specs(w)}
    if w.smooth:
        out["inv_smooth"] = 4 * w.N
    if w.kind == "cross_entropy":
        out["labels"] = 4 * w.M
    return out


def output_bytes(w, store_h: bool = False) -> dict:
    """Bytes of every output of one call, each written once.  store_h: the RMSNorm call also writes
    h_out, and the chain's first GEMM also writes H1 (the residual stream after the add)."""
    M, N = w.M, w.N
    if w.kind in ("gelu_tanh", "gelu_erf", "swiglu", "gelu_bwd"):
        return {"Y": 2 * M * N}
    if w.kind == "swiglu_bwd":
        return {"dGU": 2 * M * 2 * N}
    if w.kind == "qkv_rope":
        dm = w.n_heads * w.head_dim
        return {"Q": 2 * M * dm, "K": 2 * M * dm, "V": 2 * M * dm}
    if w.kind == "qkv_fp8kv":
        dq, dkv = w.n_heads * w.head_dim, w.n_kv_heads * w.head_dim
        return {"Q": 2 * M * dq, "Kq": M * dkv, "Vq": M * dkv, "k_scale": 4 * M * w.n_kv_heads,
                "v_scale": 4 * M * w.n_kv_heads}
    if w.kind == "cross_entropy":
        return {"loss": 4 * M}
    if w.kind == "quant":
        bs = {"fp8_1x128": 128, "int4_g32": 32, "nvfp4_g16": 16}[w.quant]
        codes = M * N if w.quant == "fp8_1x128" else M * (N // 2)
        return {"codes": codes, "scales": M * -(-N // bs) * (1 if w.quant == "nvfp4_g16" else 4)}
    if w.kind == "rms_chain":
        # H2 is written by the first GEMM and read back by the second (counted as its output traffic)
        out = {"H2_write": 2 * M * N, "H2_read": 2 * M * N, "Y": 2 * M * w.N2}
        if store_h:
            out["H1"] = 2 * M * N
        return out
    out = {"Yq": M * N, "row_scale": 4 * M}  # residual + RMSNorm + FP8
    if store_h:
        out["h_out"] = 2 * M * N
    return out


def algorithmic_bytes(w, store_h: bool = False) -> float:
    """The roofline numerator of an HBM-bound call: each operand read once, each output written once."""
    return float(sum(operand_bytes(w).values()) + sum(output_bytes(w, store_h).values()))


def unfused_activation_bytes(w) -> dict:
    """Activation bytes per call that the unfused sequence moves between the GEMM and its consumer,
    in the accounting of the end-to-end ledger of "GEMM Epilogue 完全拆解" (§端到端账本): weights,
    the first GEMM's input and the last output are left out, since both forms move them alike.
      chain (output projection -> residual -> RMSNorm -> gate/up GEMM): the projection writes d;
        the residual add reads d + d and writes d; RMSNorm reads d and gamma (d, counted per token
        as the page does) and writes d; the next GEMM reads d: 3d written + 5d read;
      SwiGLU: the GEMM writes gate and up (2 d_ff), the elementwise kernel reads them and writes
        d_ff: 5 d_ff."""
    if w.kind == "rms_chain":
        return {"written": 3 * 2 * w.M * w.N, "read": 5 * 2 * w.M * w.N}
    if w.kind == "swiglu":
        return {"written": 3 * 2 * w.M * w.N, "read": 2 * 2 * w.M * w.N}
    raise ValueError(f"no unfused ledger for {w.kind}")


def fused_activation_bytes(w, store_h: bool = True) -> dict:
    """The same ledger for the fused kernels: chain, the first epilogue reads the residual (d) and
    writes H2 (d) and H1 (d, the residual stream kept for the next block), the second GEMM reads H2
    (d): 4d; SwiGLU: only its d_ff output leaves the epilogue."""
    if w.kind == "rms_chain":
        out = output_bytes(w, store_h)
        return {"written": out["H2_write"] + out.get("H1", 0), "read": operand_bytes(w)["Z"] + out["H2_read"]}
    if w.kind == "swiglu":
        return {"written": output_bytes(w)["Y"], "read": 0}
    raise ValueError(f"no fused ledger for {w.kind}")


# ----------------------------------------------------------------------------- workloads
def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def dev_operand(a):
    """A host operand on the device: bf16 bit patterns (uint16) as bf16, fp32 as fp32."""
    if a.dtype == np.float32:
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dev_bf16(a)


class Case:
    """Device operands of one workload plus the call that runs it through the C ABI."""

    def __init__(self, name: str):
        import gemm_epilogue_tcgen05_gb300 as fl
        self.fl = fl
        self.w = syn.WORKLOADS[name]
        self.name = name
        self.host = syn.make_operands(self.w)
        self.dev = {k: dev_operand(v) for k, v in self.host.items()}
        w = self.w
        d = self.dev
        if w.kind in ("gelu_tanh", "gelu_erf"):
            self.out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
            self.flops = 2.0 * w.M * w.N * w.K
        elif w.kind == "qkv_rope":
            dm = w.n_heads * w.head_dim
            self.out = tuple(torch.empty((w.M, dm), dtype=torch.bfloat16, device="cuda") for _ in range(3))
            self.flops = 2.0 * w.M * w.N * w.K
        elif w.kind == "qkv_fp8kv":
            dq, dkv = w.n_heads * w.head_dim, w.n_kv_heads * w.head_dim
            self.out = (torch.empty((w.M, dq), dtype=torch.bfloat16, device="cuda"),
                        torch.empty((w.M, dkv), dtype=torch.uint8, device="cuda"),
                        torch.empty((w.M, dkv), dtype=torch.uint8, device="cuda"),
                        torch.empty((w.M, w.n_kv_heads), dtype=torch.float32, device="cuda"),
                        torch.empty((w.M, w.n_kv_heads), dtype=torch.float32, device="cuda"))
            self.flops = 2.0 * w.M * w.N * w.K
        elif w.kind == "swiglu":
            self.out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
            self.flops = 2.0 * w.M * (2 * w.N) * w.K
        elif w.kind == "cross_entropy":
            self.labels = torch.from_numpy(syn.make_labels(w)).cuda()
            self.out = torch.empty(w.M, dtype=torch.float32, device="cuda")
            self.ws = fl.cross_entropy_workspace(w.M, w.N)
            self.flops = 2.0 * w.M * w.N * w.K
        elif w.kind in ("gelu_bwd", "swiglu_bwd"):
            width = w.N if w.kind == "gelu_bwd" else 2 * w.N
            self.out = torch.empty((w.M, width), dtype=torch.bfloat16, device="cuda")
            self.flops = 2.0 * w.M * w.N * w.K
        elif w.kind == "quant":
            self.fmt = QUANT_FMT[w.quant]
            bs = fl.QUANT_BLOCK[self.fmt]
            qbytes = w.N if self.fmt == fl.QUANT_FP8_1X128 else w.N // 2
            sdt = torch.uint8 if self.fmt == fl.QUANT_NVFP4_G16 else torch.float32
            self.out = (torch.empty((w.M, qbytes), dtype=torch.uint8, device="cuda"),
                        torch.empty((w.M, -(-w.N // bs)), dtype=sdt, device="cuda"))
            self.flops = 2.0 * w.M * w.N * w.K
        elif w.kind == "rms_chain":
            self.h2 = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
            self.part = torch.empty((fl.rms_partials_per_row(w.N), w.M), dtype=torch.float32, device="cuda")
            self.out = torch.empty((w.M, w.N2), dtype=torch.bfloat16, device="cuda")
            self.flops = 2.0 * w.M * w.N * w.K + 2.0 * w.M * w.N2 * w.N
        else:
            self.out = (torch.empty((w.M, w.N), dtype=torch.uint8, device="cuda"),
                        torch.empty(w.M, dtype=torch.float32, device="cuda"))
            self.ws = fl.rmsnorm_fp8_workspace(w.M, w.N, w.K)
            self.flops = 2.0 * w.M * w.N * w.K
        self.bytes = algorithmic_bytes(w)
        # decode shapes (32 tokens): the weight stream bounds them
        self.hbm_bound = w.M <= 32 and w.kind in ("rmsnorm_fp8", "gelu_tanh", "qkv_rope", "qkv_fp8kv", "swiglu", "quant")

    def run(self, stream=None, d=None, out=None, ws=None):
        """One call; `d`, `out` and `ws` replace the case's own operands, outputs and workspace."""
        fl, w = self.fl, self.w
        d = self.dev if d is None else d
        out = self.out if out is None else out
        ws = getattr(self, "ws", None) if ws is None else ws
        if w.kind in ("gelu_tanh", "gelu_erf"):
            fl.fused_linear_gelu(d["X"], d["W"], d.get("b"), Y=out,
                                 mode="tanh" if w.kind == "gelu_tanh" else "erf", stream=stream)
        elif w.kind == "qkv_rope":
            fl.fused_qkv_rope(d["X"], d["W"], d.get("b"), n_heads=w.n_heads, head_dim=w.head_dim,
                              seq_len=w.seq_len, theta=w.theta, out=out, stream=stream)
        elif w.kind == "qkv_fp8kv":
            fl.fused_qkv_rope_fp8kv(d["X"], d["W"], d.get("b"), n_heads=w.n_heads, n_kv_heads=w.n_kv_heads,
                                    head_dim=w.head_dim, seq_len=w.seq_len, theta=w.theta, out=out, stream=stream)
        elif w.kind == "swiglu":
            fl.fused_swiglu(d["X"], d["Wgate"], d["Wup"], d.get("bgate"), d.get("bup"), Y=out, stream=stream)
        elif w.kind == "cross_entropy":
            fl.fused_linear_cross_entropy(d["X"], d["W"], d.get("b"), self.labels, loss=out, workspace=self.ws,
                                          stream=stream)
        elif w.kind == "gelu_bwd":
            fl.fused_dgrad_gelu(d["dZ"], d["W"], d["H"], mode="tanh", dH=out, stream=stream)
        elif w.kind == "swiglu_bwd":
            fl.fused_swiglu_bwd(d["dO"], d["Wd"], d["G"], d["U"], dGU=out, stream=stream)
        elif w.kind == "quant":
            fl.fused_linear_quant(d["X"], d["W"], d.get("b"), self.fmt, Yq=out[0], scales=out[1],
                                  inv_smooth=d.get("inv_smooth"), stream=stream)
        elif w.kind == "rms_chain":
            fl.fused_linear_residual_gamma(d["X"], d["W"], d.get("b"), d["Z"], d["gamma"], store_h1=False, H2=self.h2,
                                           rms_partials=self.part, stream=stream)
            fl.fused_linear_rms_rowscale(self.h2, d["W2"], None, self.part, w.N, w.eps, Y=out, stream=stream)
        else:
            fl.fused_linear_residual_rmsnorm_fp8(d["X"], d["W"], d.get("b"), d["Z"], d["gamma"], w.eps,
                                                 Yq=out[0], row_scale=out[1], workspace=ws, stream=stream)

    def outputs(self):
        return self.out if isinstance(self.out, tuple) else (self.out,)

    def status(self, ws=None) -> int:
        """Device-side failures of the calls so far: the workspace's record and the device-wide word."""
        ws = getattr(self, "ws", None) if ws is None else ws
        st = self.fl.check_device_status(ws) if ws is not None else self.fl.FL_OK
        dev = self.fl.device_status()
        return st if st != self.fl.FL_OK else dev


def time_device(case: Case, steps: int, warmup: int, flush: torch.Tensor, barrier):
    """Per-launch CUDA-event times (ms) with an L2 flush before every launch."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        case.run(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        case.run(stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    torch.cuda.synchronize()
    if case.status() != case.fl.FL_OK:
        raise RuntimeError(f"{case.name}: device-side failure reported")
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], wall


def unfused_fn(case: Case, d=None):
    """The same computation as separate torch / cuBLAS kernels (comparison baseline, not our path);
    `d` replaces the case's own operands."""
    import torch.nn.functional as F
    w = case.w
    d = case.dev if d is None else d
    if w.kind in ("gelu_tanh", "gelu_erf"):
        approx = "tanh" if w.kind == "gelu_tanh" else "none"
        return lambda: F.gelu(F.linear(d["X"], d["W"], d.get("b")), approximate=approx)
    if w.kind == "qkv_rope":
        dm, hd = w.n_heads * w.head_dim, w.head_dim
        pos = torch.arange(w.M, device="cuda") % w.seq_len
        inv = w.theta ** (-torch.arange(0, hd, 2, device="cuda", dtype=torch.float32) / hd)
        ang = pos[:, None].float() * inv[None, :]
        cos, sin = ang.cos().repeat(1, w.n_heads), ang.sin().repeat(1, w.n_heads)

        def rope(t):
            t = t.float()
            x0, x1 = t[:, 0::2], t[:, 1::2]
            return torch.stack((x0 * cos - x1 * sin, x0 * sin + x1 * cos), dim=-1).reshape(t.shape).to(torch.bfloat16)

        def fn():
            h = F.linear(d["X"], d["W"])
            return rope(h[:, :dm]), rope(h[:, dm:2 * dm]), h[:, 2 * dm:].contiguous()
        return fn
    if w.kind == "qkv_fp8kv":
        dq, dkv, hd = w.n_heads * w.head_dim, w.n_kv_heads * w.head_dim, w.head_dim
        pos = torch.arange(w.M, device="cuda") % w.seq_len
        inv = w.theta ** (-torch.arange(0, hd, 2, device="cuda", dtype=torch.float32) / hd)
        ang = pos[:, None].float() * inv[None, :]
        cos_q, sin_q = ang.cos().repeat(1, w.n_heads), ang.sin().repeat(1, w.n_heads)
        cos_k, sin_k = ang.cos().repeat(1, w.n_kv_heads), ang.sin().repeat(1, w.n_kv_heads)

        def rot(t, c, s):
            x0, x1 = t[:, 0::2], t[:, 1::2]
            return torch.stack((x0 * c - x1 * s, x0 * s + x1 * c), dim=-1).reshape(t.shape)

        def fp8_heads(t):
            g = t.view(w.M, -1, hd)
            sc = g.abs().amax(dim=2, keepdim=True) / 448.0
            return (g / torch.where(sc > 0, sc, 1.0)).to(torch.float8_e4m3fn).view(w.M, -1), sc.view(w.M, -1)

        def fn_kv():
            h = F.linear(d["X"], d["W"]).float()
            q = rot(h[:, :dq], cos_q, sin_q).to(torch.bfloat16)
            return (q,) + fp8_heads(rot(h[:, dq:dq + dkv], cos_k, sin_k)) + fp8_heads(h[:, dq + dkv:])
        return fn_kv
    if w.kind == "swiglu":
        return lambda: F.silu(F.linear(d["X"], d["Wgate"])) * F.linear(d["X"], d["Wup"])
    if w.kind == "cross_entropy":
        return lambda: F.cross_entropy(F.linear(d["X"], d["W"]).float(), case.labels.long(), reduction="none")
    if w.kind == "gelu_bwd":
        return lambda: torch.ops.aten.gelu_backward(d["dZ"] @ d["W"], d["H"], approximate="tanh")
    if w.kind == "swiglu_bwd":
        def swiglu_bwd():
            dy = (d["dO"] @ d["Wd"]).float()
            g, u = d["G"].float(), d["U"].float()
            s = torch.sigmoid(g)
            return torch.stack((dy * u * s * (1 + g * (1 - s)), dy * g * s), dim=-1).reshape(w.M, -1).bfloat16()
        return swiglu_bwd
    if w.kind == "quant":
        if "inv_smooth" in d:
            return lambda: unfused_quant(F.linear(d["X"], d["W"], d.get("b")).float() * d["inv_smooth"], case.fmt)
        return lambda: unfused_quant(F.linear(d["X"], d["W"], d.get("b")).float(), case.fmt)
    if w.kind == "rms_chain":
        return lambda: F.linear(F.rms_norm(F.linear(d["X"], d["W"]) + d["Z"], (w.N,), weight=d["gamma"], eps=w.eps),
                                d["W2"])

    def rms():
        h = F.linear(d["X"], d["W"]).float() + d["Z"].float()
        y = F.rms_norm(h, (w.N,), weight=d["gamma"].float(), eps=w.eps)
        s = y.abs().amax(dim=1) / 448.0
        return (y / s[:, None]).to(torch.float8_e4m3fn), s
    return rms


QUANT_FMT = {"fp8_1x128": 0, "int4_g32": 1, "nvfp4_g16": 2}
_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def unfused_quant(y: torch.Tensor, fmt: int):
    """Block-scaled quantisation as separate torch kernels after the GEMM (comparison baseline only)."""
    M, N = y.shape
    bs = {0: 128, 1: 32, 2: 16}[fmt]
    g = y.view(M, N // bs, bs)
    amax = g.abs().amax(dim=2, keepdim=True)
    if fmt == 0:
        s = amax / 448.0
        return (g / torch.where(s > 0, s, 1.0)).to(torch.float8_e4m3fn).view(M, N), s.view(M, -1)
    if fmt == 1:
        s = amax / 7.0
        q = torch.clamp(torch.round(g / torch.where(s > 0, s, 1.0)), -7, 7).to(torch.int8).view(M, N)
        packed = (q[:, 0::2] & 15) | ((q[:, 1::2] & 15) << 4)
        return packed.to(torch.uint8), s.view(M, -1)
    sc = (amax / 6.0).to(torch.float8_e4m3fn)
    v = g / torch.where(sc.float() > 0, sc.float(), 1.0)
    mag = torch.bucketize(v.abs(), torch.tensor(_E2M1_MIDPOINTS, device=y.device)).to(torch.uint8)
    code = (mag | ((v < 0).to(torch.uint8) << 3)).view(M, N)
    return code[:, 0::2] | (code[:, 1::2] << 4), sc.view(M, -1)


def time_fn(fn, steps: int, warmup: int, flush: torch.Tensor):
    """CUDA-event time (ms) of a callable with an L2 flush before each timed call."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))


def standin_kernel(nbytes: int = 8 << 20):
    """A few-microsecond kernel that is not a decode call: an in-place scale of an 8 MiB bf16
    buffer (torch's elementwise kernel, 16 MiB of traffic), standing in for the other work a
    decode step puts between two calls of the same layer kind."""
    buf = torch.ones(nbytes // 2, dtype=torch.bfloat16, device="cuda")
    return lambda: buf.mul_(1.0)


def time_graph_rotating(case: Case, calls: int = 20, copies: int = 3, replays: int = 20, mode: str = "fused",
                        between=None):
    """Per-call time (ms) of `calls` back-to-back calls captured in one CUDA graph, cycling through
    `copies` separate copies of every operand (together larger than L2, so each call reads its
    operands from HBM), as a decode loop would issue them.
    mode "fused": the library call; "unfused": the torch/cuBLAS sequence of the same workload.
    between: an optional callable enqueued after every call (the interleaved measurement)."""
    import gemm_epilogue_tcgen05_gb300 as fl
    w = case.w
    sets = [case.dev] + [{k: v.clone() for k, v in case.dev.items()} for _ in range(copies - 1)]
    outs = [case.outputs()] + [tuple(torch.empty_like(t) for t in case.outputs()) for _ in range(copies - 1)]
    single = not isinstance(case.out, tuple)
    wss = [getattr(case, "ws", None)] + [fl.rmsnorm_fp8_workspace(w.M, w.N, w.K) if w.kind == "rmsnorm_fp8" else None
                                         for _ in range(copies - 1)]
    unf = [unfused_fn(case, d) for d in sets] if mode == "unfused" else None

    def seq(stream):
        for i in range(calls):
            if unf is not None:
                unf[i % copies]()
            else:
                o = outs[i % copies]
                case.run(stream, d=sets[i % copies], out=o[0] if single else o, ws=wss[i % copies])
            if between is not None:
                between()

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        seq(stream)  # warm-up outside the capture
    torch.cuda.synchronize()
    kind = "graph"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            seq(stream)
        run = g.replay
    except Exception:  # noqa: BLE001 - capture unsupported: fall back to plain back-to-back launches
        kind = "stream"
        torch.cuda.synchronize()

        def run():
            with torch.cuda.stream(stream):
                seq(stream)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(replays):
        run()
    e.record()
    torch.cuda.synchronize()
    if any(case.status(ws) != fl.FL_OK for ws in wss):
        raise RuntimeError("decode graph: device-side failure reported")
    return s.elapsed_time(e) / (replays * calls), kind


def time_graph_standin(between, calls: int = 20, replays: int = 20) -> float:
    """Per-call time (ms) of the stand-in kernel alone, captured and replayed like the decode graphs."""
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(calls):
            between()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            between()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(replays):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / (replays * calls)


def host_enqueue_us(case: Case, calls: int = 200) -> dict:
    """Host time to enqueue one decode call, through the C ABI directly (the arguments marshalled
    once beforehand) and through the Python binding, with the tensor-map descriptor cache on and
    off.  The calls run on the GPU meanwhile; the host never waits inside the timed loop."""
    import ctypes
    fl, w, d = case.fl, case.w, case.dev
    lib = fl.load()
    P = ctypes.c_void_p
    q, rs = case.out
    ws = case.ws
    stream = torch.cuda.current_stream()
    args = (P(d["X"].data_ptr()), P(d["W"].data_ptr()), None, P(d["Z"].data_ptr()), P(d["gamma"].data_ptr()),
            ctypes.c_float(w.eps), P(q.data_ptr()), P(rs.data_ptr()), None, w.M, w.N, w.K, d["X"].stride(0),
            d["W"].stride(0), d["Z"].stride(0), q.stride(0), P(ws.data_ptr()), ws.numel(), P(stream.cuda_stream))
    out = {}
    for cache in (True, False):
        fl.set_descriptor_cache(cache)
        for label, fn in (("c_abi", lambda: lib.fused_linear_residual_rmsnorm_fp8(*args)), ("python", case.run)):
            for _ in range(20):
                fn()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(3):
                t0 = time.perf_counter()
                for _ in range(calls):
                    fn()
                best = min(best, (time.perf_counter() - t0) / calls * 1e6)
                torch.cuda.synchronize()
            out[f"{label}_us_{'cached' if cache else 'uncached'}"] = best
    fl.set_descriptor_cache(True)
    if case.status() != fl.FL_OK:
        raise RuntimeError("host enqueue timing: device-side failure reported")
    out["what"] = (f"host wall time per call of {calls} back-to-back enqueues (best of 3), "
                   "validation + tensor-map encodes (or cache hits) + launch")
    return out


def time_e2e(case: Case, steps: int, warmup: int, barrier):
    """Per-step time (ms) of the public host-buffer call: pinned host inputs in, GEMM + epilogue,
    host output out, every step (fused_linear_gelu_host overlaps the copies with the GEMM)."""
    fl, w = case.fl, case.w
    stream = torch.cuda.current_stream()

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    Xh, Wh = pinned(case.host["X"]), pinned(case.host["W"])
    bh = pinned(case.host["b"]) if "b" in case.host else None
    Yh = torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory()
    buf = fl.linear_gelu_host_buffer(w.M, w.N, w.K)
    h2d = sum(t.numel() * t.element_size() for t in (Xh, Wh, bh) if t is not None)
    d2h = Yh.numel() * Yh.element_size()
    mode = "tanh" if w.kind == "gelu_tanh" else "erf"

    def step():
        fl.fused_linear_gelu_host(Xh, Wh, bh, Y=Yh, mode=mode, dev_buf=buf, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    del buf
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_inputs(w, rows: int) -> dict:
    """The first `rows` rows of the workload's operands (weights whole), as exact fp64 arrays."""
    ops = syn.make_operands(w, rows=(0, rows))
    return {k: syn.to_f64(v, w.dtype) for k, v in ops.items()}


def first_rows(f: dict, rows: int) -> dict:
    """The same operands cut to their first `rows` rows."""
    return {k: (v[:rows] if k in syn.ROW_OPERANDS else v) for k, v in f.items()}


def oracle_sample(w, rows: int, f: dict | None = None):
    """Oracle on the first `rows` rows of the workload (all output columns); returns seconds.
    `f` (from oracle_inputs, at least `rows` rows) saves regenerating the operands."""
    import oracle
    f = oracle_inputs(w, rows) if f is None else first_rows(f, rows)
    t0 = time.perf_counter()
    if w.kind in ("gelu_tanh", "gelu_erf"):
        oracle.linear_gelu(f["X"], f["W"], f.get("b"), oracle.GELU_TANH if w.kind == "gelu_tanh"
                           else oracle.GELU_ERF)
    elif w.kind == "qkv_rope":
        oracle.qkv_rope(f["X"], f["W"], f.get("b"), w.n_heads, w.head_dim, w.theta, np.arange(rows) % w.seq_len)
    elif w.kind == "swiglu":
        oracle.swiglu(f["X"], f["Wgate"], f["Wup"], f.get("bgate"), f.get("bup"))
    elif w.kind == "gelu_bwd":
        oracle.dgrad_gelu(f["dZ"], f["W"], f["H"], oracle.GELU_TANH)
    elif w.kind == "swiglu_bwd":
        oracle.swiglu_bwd(f["dO"], f["Wd"], f["G"], f["U"])
    elif w.kind == "qkv_fp8kv":
        oracle.qkv_rope_kv_fp8(f["X"], f["W"], f.get("b"), w.n_heads, w.n_kv_heads, w.head_dim, w.theta,
                               np.arange(rows) % w.seq_len)
    elif w.kind == "quant":
        oracle.linear_quant(f["X"], f["W"], f.get("b"), QUANT_FMT[w.quant], inv_smooth=f.get("inv_smooth"))
    elif w.kind == "cross_entropy":
        oracle.linear_cross_entropy(f["X"], f["W"], f.get("b"), syn.make_labels(w)[:rows])
    elif w.kind == "rms_chain":
        oracle.residual_rmsnorm_linear(f["X"], f["W"], f.get("b"), f["Z"], f["gamma"], w.eps, f["W2"])
    else:
        oracle.rmsnorm_fp8(f["X"], f["W"], f.get("b"), f["Z"], f["gamma"], w.eps)
    return time.perf_counter() - t0


def cpu_baseline(name: str, target_s: float = 10.0):
    import oracle
    w = syn.WORKLOADS[name]
    t1 = oracle_sample(w, 1)
    rows = int(max(1, min(w.M, math.floor(target_s / max(t1, 1e-6)))))
    secs = oracle_sample(w, rows) if rows > 1 else t1
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} of {w.M} rows of {name}, all {w.N} output columns, fp64 ({secs:.2f} s)"}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", default="all", choices=["all", "none"],
                    help="also measure the other fused workloads of the hot path")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(syn.WORKLOADS),
                    help="workload timed as the step (default: the headline); used for profiling runs")
    ap.add_argument("--no-cooperative", action="store_true",
                    help="launch the RMSNorm prefill kernel without the cooperative attribute (same grid); "
                         "for kernel profilers that refuse cooperative launches of clusters")
    ap.add_argument("--unfused", action="store_true",
                    help="with --workload: time the unfused torch/cuBLAS sequence of that workload instead "
                         "(comparison baseline); one extra call runs inside the NVTX range 'unfused_step'")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = dist.barrier
    else:
        dist = None

        def barrier():
            return None

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        barrier()
        __graft_entry__.build()

    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    if args.no_cooperative:
        import gemm_epilogue_tcgen05_gb300 as fl
        fl.set_cooperative_launch(False)
    if args.unfused:
        return unfused_workload(args, world, rank, local, dist)
    if args.workload != HEADLINE:
        return single_workload(args, world, rank, local, barrier, dist)
    head = Case(HEADLINE)
    with ClockSampler(local) as clk:
        times, wall = time_device(head, args.steps, args.warmup, flush, barrier)
    clocks = clk.summary()
    ms = statistics.mean(times)
    ms_max = max_over_ranks(ms, dist, "cuda")
    value = job_rate(head.flops, world, ms_max * 1e-3) / 1e12
    kernel_tflops = head.flops / (ms * 1e-3) / 1e12
    traffic = recorded_traffic(HEADLINE)
    # A long timed region that runs power-capped is compared with the sustained
    # measured peak; an unthrottled one with the burst peak.  Both fractions are reported.
    capped = "sw_power_cap" in clocks.get("reasons", []) or (
        clocks.get("sm_mhz") and clocks.get("sm_max_mhz") and clocks["sm_mhz"] < 0.93 * clocks["sm_max_mhz"])
    peak = pk["bf16_tflops_sustained"] if capped else pk["bf16_tflops"]
    which = "sustained (timed region ran power-capped)" if capped else "burst"
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": kernel_tflops / peak, "traffic": traffic,
                "peak_source": f"bf16 {which}, {'of measured' if pk['source'] == 'measured' else 'of fallback'}",
                "frac_of_burst_peak": kernel_tflops / pk["bf16_tflops"],
                "frac_of_nominal": kernel_tflops / NOMINAL_BF16_TFLOPS, "nominal": NOMINAL_BF16_TFLOPS,
                "algorithmic_bytes": head.bytes, "traffic_unit": "bytes per launch (ncu dram read + write)"}
    head_unfused = time_fn(unfused_fn(head), 20, 3, flush)
    e_times, h2d, d2h = time_e2e(head, max(3, min(args.steps, 100) // 2), 2, barrier)
    e_ms = max_over_ranks(statistics.mean(e_times), dist, "cuda")
    e2e = {"value": job_rate(head.flops, world, e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}
    del head

    rows = []
    decode = None
    standin = standin_ms = None
    if args.rows == "all":
        for name in ("qkv_rope_8192x12288x4096", "qkv_fp8kv_8192x6144x4096", "swiglu_8192x14336x4096", "rmsnorm_fp8_prefill_8192x4096x14336",
                     "rmsnorm_fp8_decode_32x4096x14336", "gelu_decode_32x16384x4096", "qkv_decode_32x12288x4096",
                     "qkv_fp8kv_decode_32x6144x4096", "swiglu_decode_32x14336x4096",
                     "quant_fp8_1x128_decode_32x16384x4096", "rms_chain_8192x4096x4096_to_14336",
                     "lm_head_ce_8192x32768x4096", "gelu_bwd_8192x16384x4096", "swiglu_bwd_8192x14336x4096",
                     "quant_fp8_1x128_8192x16384x4096",
                     "quant_int4_g32_8192x16384x4096", "quant_nvfp4_g16_8192x16384x4096",
                     "quant_fp8_1x128_smooth_8192x16384x4096"):
            c = Case(name)
            row_steps = min(args.steps, 200)
            ts, _ = time_device(c, row_steps, args.warmup, flush, barrier)
            m = statistics.mean(ts)
            unf = time_fn(unfused_fn(c), max(5, row_steps // 10), 3, flush)
            if c.hbm_bound:
                ach = c.bytes / (m * 1e-3) / 1e9
                g_ms, g_kind = time_graph_rotating(c)
                g_ach = c.bytes / (g_ms * 1e-3) / 1e9
                u_ms, _ = time_graph_rotating(c, mode="unfused")
                row = {"workload": name, "value": g_ach, "unit": "GB/s", "us_per_call": g_ms * 1e3,
                       "timing": f"{g_kind} of 20 back-to-back calls over 3 rotating operand copies (> L2)",
                       "single_launch": {"us": m * 1e3, "GB/s": ach, "frac": ach / pk["hbm_gbs"],
                                         "timing": "one launch, L2 flushed before it"},
                       "roofline": {"bound": "hbm", "achieved": g_ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                    "frac": g_ach / pk["hbm_gbs"], "traffic": recorded_traffic(name),
                                    "frac_of_nominal": g_ach / NOMINAL_HBM_GBS,
                                    "algorithmic_bytes": c.bytes},
                       "unfused_torch_us": u_ms * 1e3, "speedup_vs_unfused": u_ms / g_ms,
                       "unfused_timing": "the same graph form (20 calls, 3 rotating copies)",
                       "unfused_single_launch_us": unf * 1e3, "speedup_vs_unfused_single_launch": unf / m}
                # the same calls with a different kernel between each two (a decode step's real order)
                if standin is None:
                    standin = standin_kernel()
                    standin_ms = time_graph_standin(standin)
                i_ms, _ = time_graph_rotating(c, between=standin)
                per = i_ms - standin_ms
                i_ach = c.bytes / (per * 1e-3) / 1e9
                row["interleaved"] = {"us_per_call": per * 1e3, "GB/s": i_ach, "frac": i_ach / pk["hbm_gbs"],
                                      "us_per_pair": i_ms * 1e3, "standin_us": standin_ms * 1e3,
                                      "timing": "graph of 20 (call, stand-in kernel) pairs over 3 rotating operand "
                                                "copies, minus a graph of 20 stand-ins; stand-in: in-place scale "
                                                "of an 8 MiB bf16 buffer"}
                if name == DECODE:
                    decode = {"workload": name, "GB/s": g_ach, "frac": g_ach / pk["hbm_gbs"],
                              "us_per_call": g_ms * 1e3, "timing": row["timing"],
                              "interleaved": row["interleaved"],
                              "single_launch": row["single_launch"], "peak_gbs": pk["hbm_gbs"],
                              "host_enqueue": host_enqueue_us(c)}
                rows.append(row)
            else:
                ach = c.flops / (m * 1e-3) / 1e12
                rows.append({"workload": name, "value": ach, "unit": "TFLOP/s", "ms_per_launch": m,
                             "roofline": {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                                          "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"],
                                          "frac_of_nominal": ach / NOMINAL_BF16_TFLOPS,
                                          "traffic": recorded_traffic(name), "algorithmic_bytes": c.bytes},
                             "unfused_torch_ms": unf, "speedup_vs_unfused": unf / m})
                if c.w.kind in ("rms_chain", "swiglu"):
                    one = syn.scaled(c.w, M=1)
                    rows[-1]["activation_bytes_per_token"] = {
                        "fused": sum(fused_activation_bytes(one, store_h=False).values()),
                        "unfused": sum(unfused_activation_bytes(one).values()),
                        "what": "activation traffic between the GEMM and its consumer per token, weights and "
                                "the first input / last output excluded (the end-to-end ledger's accounting)"}
            del c
            torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded splitmix64/Box-Muller, bf16)",
        "config": {"workload": HEADLINE, "M": 8192, "N": 16384, "K": 4096, "epilogue": "bias + GELU(tanh)",
                   "l2": "256 MiB flush before every timed launch; inputs larger than L2",
                   "parallelism": f"replicas x{world} (rows are independent; no collective)"},
        "roofline": roofline, "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks,
        "unfused_baseline": {"ms_per_step": head_unfused, "speedup": head_unfused / ms,
                             "what": "torch F.gelu(F.linear(X, W, b), approximate='tanh'): cuBLAS GEMM + separate GELU"},
        "decode": decode, "rows": rows, "wall_s_timed_region": wall,
        # numbers the source pages print, for context only (other hardware, other kernels)
        "pages_context": {
            "unfused_layernorm_gelu_8x4096x4096_fp16_a100_ms": 0.5,
            "fused_layernorm_gelu_speedup": "about 2x (LayerNorm + GeLU fusion page)",
            "linear_gelu_fusion_speedup": "1.2-2x in general (Triton Linear + Attention fusion page)",
            "non_gemm_share_h100": "non-negligible, no figure (GEMM epilogue page, on CODA)"},
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(HEADLINE)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def single_workload(args, world, rank, local, barrier, dist):
    """Times one non-headline workload alone (profiling aid); prints one JSON line."""
    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    c = Case(args.workload)
    with ClockSampler(local) as clk:
        ts, _ = time_device(c, args.steps, args.warmup, flush, barrier)
    m = statistics.mean(ts)
    if c.hbm_bound:
        val, unit, pkv = c.bytes / (m * 1e-3) / 1e9, "GB/s", pk["hbm_gbs"]
    else:
        val, unit, pkv = c.flops / (m * 1e-3) / 1e12, "TFLOP/s", pk["bf16_tflops"]
    line = {"metric": METRIC, "value": world * val, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": m, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": {"workload": args.workload},
            "roofline": {"bound": "hbm" if c.hbm_bound else "tensor", "achieved": val, "peak": pkv,
                         "unit": unit, "frac": val / pkv, "traffic": recorded_traffic(args.workload)},
            "gpu_launches": args.steps, "clocks": clk.summary()}
    if c.hbm_bound:
        # decode shapes: also back to back, as a decode loop issues them
        g_ms, g_kind = time_graph_rotating(c)
        g_ach = c.bytes / (g_ms * 1e-3) / 1e9
        line["back_to_back"] = {"us_per_call": g_ms * 1e3, "GB/s": g_ach, "frac": g_ach / pkv,
                                "timing": f"{g_kind} of 20 back-to-back calls over 3 rotating operand copies (> L2)"}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def unfused_workload(args, world, rank, local, dist):
    """The unfused torch/cuBLAS sequence of one workload, timed like the fused kernel; one more call
    runs inside the NVTX range 'unfused_step' so a profiler can capture exactly its kernels."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    c = Case(args.workload)
    fn = unfused_fn(c)
    with ClockSampler(local) as clk:
        m = time_fn(fn, args.steps, args.warmup, flush)
    flush.zero_()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("unfused_step")
    fn()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if c.hbm_bound:
        val, unit = c.bytes / (m * 1e-3) / 1e9, "GB/s"
    else:
        val, unit = c.flops / (m * 1e-3) / 1e12, "TFLOP/s"
    line = {"impl": "unfused_torch", "metric": METRIC, "value": world * val, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload}, "clocks": clk.summary()}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def reference_arm(args, world, rank):
    """The fp64 CPU oracle on bounded samples of the headline workload (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    syn.build()
    w = syn.WORKLOADS[HEADLINE]
    f1 = oracle_inputs(w, 1)
    t1 = min(oracle_sample(w, 1, f1) for _ in range(3))
    per_step_target = 8.0 if args.steps <= 10 else 80.0 / args.steps
    rows = int(max(1, min(w.M, math.floor(per_step_target / max(t1, 1e-6)))))
    # operands generated once (the timed region is the oracle call alone); warm-up on one row
    f = oracle_inputs(w, rows)
    for _ in range(args.warmup):
        oracle_sample(w, 1, f)
    secs = [oracle_sample(w, rows, f) for _ in range(args.steps)]
    s = statistics.mean(secs)
    value = 2.0 * rows * w.N * w.K / s / 1e12
    sample = f"{rows} of {w.M} rows of {HEADLINE} per step, all {w.N} output columns, fp64"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE, "M": 8192, "N": 16384, "K": 4096},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
