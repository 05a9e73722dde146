"""The benchmark's byte accounting against the per-token ledgers printed on
"GEMM Epilogue 完全拆解: 推理内核的最后一公里" (pinghaoyang.com.cn), §端到端账本 and
§一个瓦片的字节账 (values in tests/golden/byte_ledger.txt).

The benchmark's roofline numerators come from ``bench.algorithmic_bytes`` and
its parts (``operand_bytes``, ``output_bytes``) and from the ledgers of the
fused and unfused activation traffic; here each is evaluated at M = 1 and
M = 2 tokens and the difference (the per-token bytes) is compared with the
number the page prints.  No GPU is needed.
"""
import os

import bench
import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "byte_ledger.txt")


def _ledger():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, d, dff, nbytes = line.split()
                out[key] = (int(d), int(dff), int(nbytes))
    return out


def _per_token(fn, w, **kw):
    """fn(w at 2 tokens) - fn(w at 1 token), summed over the returned parts."""
    two, one = fn(syn.scaled(w, M=2), **kw), fn(syn.scaled(w, M=1), **kw)
    if isinstance(two, dict):
        return sum(two.values()) - sum(one.values())
    return two - one


def test_output_projection_rmsnorm_gate_up_ledger():
    """Unfused: 3d written + 5d read = 8d elements, 64 KiB per token at d = 4096; fused (the
    deferred-r chain keeping the residual stream): about 4d, 32 KiB."""
    g = _ledger()
    d = g["oproj_rmsnorm_gateup_unfused"][0]
    w = syn.scaled(syn.WORKLOADS["rms_chain_8192x4096x4096_to_14336"], N=d, K=d)
    assert _per_token(bench.unfused_activation_bytes, w) == g["oproj_rmsnorm_gateup_unfused"][2]
    assert _per_token(bench.fused_activation_bytes, w, store_h=True) == g["oproj_rmsnorm_gateup_fused"][2]
    # the timed chain (no H1 copy) moves one d less per token than the ledger's fused form
    assert _per_token(bench.fused_activation_bytes, w, store_h=False) == g["oproj_rmsnorm_gateup_fused"][2] - 2 * d
    # and the whole-call numerator adds exactly the first GEMM's input row and the output row
    per_call = _per_token(bench.algorithmic_bytes, w)
    assert per_call == 2 * d + (2 * d + 2 * 2 * d) + 2 * w.N2


def test_swiglu_unfused_ledger():
    """SwiGLU's two paths unfused: write 2 d_ff, read 2 d_ff, write d_ff = 5 d_ff elements, about
    107 KiB per token at d_ff ~ 10922; fused, only the d_ff output leaves the epilogue."""
    d_ff, nbytes = _ledger()["swiglu_unfused_extra"][1:]
    w = syn.scaled(syn.WORKLOADS["swiglu_8192x14336x4096"], N=d_ff)
    assert _per_token(bench.unfused_activation_bytes, w) == nbytes
    assert _per_token(bench.fused_activation_bytes, w) == 2 * d_ff
    assert _per_token(bench.output_bytes, w) == 2 * d_ff


def test_kv_writeback_ledger():
    """K/V write-back per token and layer with H = 8 kv heads of D = 128: 4096 bytes in bf16, 2048
    in FP8 (plus one fp32 scale per head, which the page leaves out), 128 / 64 KiB over 32 layers."""
    g = _ledger()
    hd = g["kv_writeback_fp8_per_layer"][0]  # H * D
    fp8 = syn.WORKLOADS["qkv_fp8kv_8192x6144x4096"]
    assert fp8.n_kv_heads * fp8.head_dim == hd
    out2, out1 = bench.output_bytes(syn.scaled(fp8, M=2)), bench.output_bytes(syn.scaled(fp8, M=1))
    kv = (out2["Kq"] + out2["Vq"]) - (out1["Kq"] + out1["Vq"])
    assert kv == g["kv_writeback_fp8_per_layer"][2]
    assert 32 * kv == g["kv_writeback_fp8_32_layers"][2]
    scales = (out2["k_scale"] + out2["v_scale"]) - (out1["k_scale"] + out1["v_scale"])
    assert scales == 2 * 4 * fp8.n_kv_heads
    # the bf16 form: the multi-head QKV call with as many heads as the cache has kv heads
    bf = syn.scaled(syn.WORKLOADS["qkv_rope_8192x12288x4096"], n_heads=fp8.n_kv_heads, N=3 * hd)
    b2, b1 = bench.output_bytes(syn.scaled(bf, M=2)), bench.output_bytes(syn.scaled(bf, M=1))
    kv16 = (b2["K"] + b2["V"]) - (b1["K"] + b1["V"])
    assert kv16 == g["kv_writeback_bf16_per_layer"][2]
    assert 32 * kv16 == g["kv_writeback_bf16_32_layers"][2]


def test_numerators_of_the_decode_rows():
    """The HBM-bound rows' numerators: the weights dominate, read once (RMSNorm decode 118.76 MB)."""
    w = syn.WORKLOADS["rmsnorm_fp8_decode_32x4096x14336"]
    assert round(bench.algorithmic_bytes(w) / 1e6, 2) == 118.76
    assert bench.operand_bytes(w)["W"] == 2 * 4096 * 14336
