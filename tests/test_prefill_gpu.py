"""Prefill parity on the GPU: the CUDA kernels (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library, sampled_rows

pytestmark = pytest.mark.gpu


def _run(q, k, v, causal, out_dtype, scale=None):
    cga = library()
    dev = device()
    o, lse = cga.prefill(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                         out_dtype=out_dtype, return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    return o, lse


# ------------------------------------------------------------------ fp32 CUDA-core kernel

@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", [
    (1, 1, 1, 128, 64, True),     # configured: B1 H1 S128 D64 causal
    (1, 12, 12, 512, 64, False),  # configured: B1 H12 S512 D64, both mask settings
    (1, 12, 12, 512, 64, True),
    (2, 4, 2, 1, 64, True), (1, 2, 1, 2, 64, True), (1, 2, 2, 63, 64, False),
    (2, 4, 2, 65, 64, True), (1, 3, 1, 129, 128, True), (1, 2, 1, 300, 128, False),
])
def test_prefill_f32(B, Hq, Hkv, S, D, causal):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "f32", seed=0)
    o, lse = _run(q, k, v, causal, torch.float32)
    o_ref, lse_ref = oracle.prefill(q, k, v, causal, 1 / math.sqrt(D))
    check_out(o, o_ref, "f32", f"f32 prefill {B},{Hq},{Hkv},{S},{D},{causal}")
    check_lse(lse, lse_ref, "f32 prefill lse")


# ------------------------------------------------------------------ bf16 tensor-core kernel

SMALL_BF16 = [
    # B, Hq, Hkv, S, causal, q_mult
    (1, 1, 1, 1, True, 1.0), (1, 2, 1, 2, False, 1.0), (1, 2, 2, 127, True, 1.0),
    (1, 2, 2, 128, False, 1.0), (2, 4, 2, 129, True, 1.0), (1, 4, 1, 255, False, 3.0),
    (1, 2, 2, 256, True, 1.0), (2, 2, 1, 300, True, 3.0), (1, 8, 2, 640, False, 1.0),
    (1, 3, 3, 1000, True, 1.0),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,causal,q_mult", SMALL_BF16)
def test_prefill_bf16_small(B, Hq, Hkv, S, causal, q_mult):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, 128, "bf16", q_mult, seed=0)
    o_ref, lse_ref = oracle.prefill(q, k, v, causal, 1 / math.sqrt(128))
    tag = f"bf16 prefill {B},{Hq},{Hkv},{S},{causal},{q_mult}"
    o32, lse = _run(q, k, v, causal, torch.float32)
    check_out(o32, o_ref, "bf16_pre", tag + " fp32 out")
    check_lse(lse, lse_ref, tag + " lse")
    o16, lse16 = _run(q, k, v, causal, torch.bfloat16)
    check_out(o16, o_ref, "bf16", tag + " bf16 out")
    assert torch.equal(lse16, lse), "lse depends on the output dtype"


def test_prefill_bf16_c3_full():
    """Configured workload: B1 Hq8 Hkv2 S2048 D128, q x3 (peaky softmax), causal; every row."""
    cfg = workloads.CONFIGS["c3"]
    q, k, v = workloads.config_prefill_inputs(cfg)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, cfg.scale)
    o32, lse = _run(q, k, v, True, torch.float32)
    check_out(o32, o_ref, "bf16_pre", "c3 fp32 out")
    check_lse(lse, lse_ref, "c3 lse")
    o16, _ = _run(q, k, v, True, torch.bfloat16)
    check_out(o16, o_ref, "bf16", "c3 bf16 out")


@pytest.mark.parametrize("seed", [1, 2])
def test_prefill_bf16_c3_other_seeds(seed):
    """The configured B1 Hq8 Hkv2 S2048 q x3 causal workload drawn from two more seeds."""
    cfg = workloads.CONFIGS["c3"]
    q, k, v = workloads.config_prefill_inputs(cfg, seed=seed)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, cfg.scale)
    o32, lse = _run(q, k, v, True, torch.float32)
    check_out(o32, o_ref, "bf16_pre", f"c3 seed {seed} fp32 out")
    check_lse(lse, lse_ref, f"c3 seed {seed} lse")
    o16, _ = _run(q, k, v, True, torch.bfloat16)
    check_out(o16, o_ref, "bf16", f"c3 seed {seed} bf16 out")


def test_prefill_bf16_c3_noncausal_and_other_seed():
    q, k, v = workloads.prefill_inputs(1, 8, 2, 2048, 128, "bf16", 3.0, seed=7)
    o_ref, lse_ref = oracle.prefill(q, k, v, False, 1 / math.sqrt(128))
    o32, lse = _run(q, k, v, False, torch.float32)
    check_out(o32, o_ref, "bf16_pre", "c3 non-causal seed 7")
    check_lse(lse, lse_ref, "c3 non-causal lse")


@pytest.mark.parametrize("name", ["c5a", "c5b"])
def test_prefill_bf16_long_context_sampled(name):
    """Configured long-context workloads at full size; rows sampled for the oracle (every 64th
    row and the last 128 rows of every head). Both the bf16 output (after the final rounding) and
    the fp32 output (before it, where the long rows' fp32 accumulation would show) are checked."""
    cfg = workloads.CONFIGS[name]
    q, k, v = workloads.config_prefill_inputs(cfg)
    rows = sampled_rows(cfg.B, cfg.Hq, cfg.S)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, cfg.scale, rows=rows)
    for out_dtype, kind in ((torch.bfloat16, "bf16"), (torch.float32, "bf16_pre")):
        o, lse = _run(q, k, v, True, out_dtype)
        idx = torch.as_tensor(rows, device=o.device)
        check_out(o.reshape(-1, cfg.D)[idx], o_ref, kind, f"{name} sampled rows {kind}")
        check_lse(lse.reshape(-1)[idx], lse_ref, f"{name} sampled lse {kind}")
        del o, lse


def test_prefill_deterministic():
    q, k, v = workloads.prefill_inputs(2, 4, 2, 700, 128, "bf16", seed=3)
    o1, l1 = _run(q, k, v, True, torch.bfloat16)
    o2, l2 = _run(q, k, v, True, torch.bfloat16)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_constant_keys_gpu():
    """All keys equal: causal row i is the mean of V[0..i] (closed form), on the GPU."""
    B, H, S, D = 1, 2, 384, 128
    q, _, v = workloads.prefill_inputs(B, H, H, S, D, "bf16", seed=5)
    k = torch.randn(D, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    k = k.expand(B, H, S, D).contiguous()
    o32, _ = _run(q, k, v, True, torch.float32)
    vd = v.double().numpy()
    ref = np.cumsum(vd, axis=2) / np.arange(1, S + 1)[:, None]
    check_out(o32, ref, "bf16_pre", "constant keys")


def test_prefill_decode_consistency():
    """The last row of causal prefill equals decode of that query against the same cache."""
    cga = library()
    dev = device()
    B, Hq, Hkv, S, D = 2, 8, 2, 777, 128
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=11)
    o, lse = _run(q, k, v, True, torch.float32)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
    od, lsed = cga.decode(q[:, :, -1].contiguous().to(dev), k.to(dev), v.to(dev), seqlens,
                          out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert (o[:, :, -1] - od).abs().max().item() <= 2 * 4e-3
    assert (lse[:, :, -1] - lsed).abs().max().item() <= 2e-4
