"""Padded variable-length batched prefill (tensor-core kernel, through the C ABI) against the fp64
oracle. Padding positions of k and v hold NaN, so any read of them would show."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, S, lens, seed, q_mult=1.0):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, 128, "bf16", q_mult, seed=seed)
    for b, L in enumerate(lens):
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("B,Hq,Hkv,S,lens,causal", [
    (3, 8, 2, 700, [700, 300, 0], True),
    (3, 8, 2, 700, [1, 255, 699], False),
    (2, 4, 4, 1000, [513, 1000], True),
    (4, 8, 2, 2048, [2048, 1500, 129, 1024], True),
])
def test_varlen_parity(B, Hq, Hkv, S, lens, causal):
    cga = library()
    dev = device()
    q, k, v, sl = _inputs(B, Hq, Hkv, S, lens, seed=S)
    o_ref, lse_ref = oracle.prefill_varlen(q, k, v, sl, causal, 1 / math.sqrt(128))
    tag = f"varlen {B},{Hq},{Hkv},{S},{lens},{causal}"
    o32, lse = cga.prefill_varlen(q.to(dev), k.to(dev), v.to(dev), sl.to(dev), causal=causal,
                                  out_dtype=torch.float32, return_lse=True)
    o16 = cga.prefill_varlen(q.to(dev), k.to(dev), v.to(dev), sl.to(dev), causal=causal)
    torch.cuda.synchronize()
    check_out(o32, o_ref, "bf16_pre", tag + " fp32 out")
    check_lse(lse, lse_ref, tag + " lse")
    check_out(o16, o_ref, "bf16", tag + " bf16 out")
    for b, L in enumerate(lens):
        assert torch.all(o16[b, :, L:] == 0), "padding rows must be zero"
    assert cga.device_status() == 0
