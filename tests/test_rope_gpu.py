"""Decode step with the new token's RoPE and cache store (through the C ABI) against the fp64
oracle on the same seeded inputs: fused into the stream kernel for batches up to 1024, a rope
kernel before the chunked decode above that."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import bf16_ulp, check_lse, check_out, device, library

pytestmark = pytest.mark.gpu


def _tables(max_len, D, base=10000.0):
    inv = base ** (-torch.arange(D // 2, dtype=torch.float64) * 2.0 / D)
    ang = torch.arange(max_len, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).float(), torch.sin(ang).float()


def _lens_1100():
    lens = torch.randint(0, 97, (1100,), generator=torch.Generator().manual_seed(9))
    lens[::11] = 0
    return lens.tolist()


@pytest.mark.parametrize("B,Hq,Hkv,D,max_len,lens", [
    (4, 8, 2, 128, 4096, [4096, 1, 1000, 2]),
    (32, 8, 2, 128, 4096, None),
    (3, 16, 2, 64, 700, [700, 350, 1]),
    (3, 12, 2, 128, 500, [500, 1, 250]),     # three query-head subgroups share each kv head
    (4, 8, 2, 128, 300, [0, 300, 17, 1]),    # an empty sequence stores nothing
    (1100, 8, 2, 128, 96, "b1100"),          # above 1024: rope kernel, then chunked decode
])
def test_decode_rope_parity(B, Hq, Hkv, D, max_len, lens):
    cga = library()
    dev = device()
    if lens == "b1100":
        lens = _lens_1100()
    q, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, D, max_len,
                                            "uniform" if lens is None else "explicit", seed=7,
                                            seqlens=lens)
    g = torch.Generator().manual_seed(8)
    kn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
    ct, st = _tables(max_len, D)
    # the new token's row holds NaN before the step: it must be overwritten before use
    for b in range(B):
        if int(sl[b]) > 0:
            kc[b, :, int(sl[b]) - 1] = float("nan")
            vc[b, :, int(sl[b]) - 1] = float("nan")
    o_ref, lse_ref, krow_ref = oracle.decode_rope(q, kn, vn, ct, st, kc, vc, sl, 1 / math.sqrt(D))
    kcd, vcd = kc.to(dev), vc.to(dev)
    o, lse = cga.decode_rope(q.to(dev), kn.to(dev), vn.to(dev), ct.to(dev), st.to(dev), kcd, vcd,
                             sl.to(dev), out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    tag = f"decode rope {B},{Hq},{Hkv},{D},{max_len}"
    check_out(o, o_ref, "bf16_pre", tag)
    check_lse(lse, lse_ref, tag + " lse")
    # the stored key row equals the oracle's rounding within one bf16 step, the value exactly
    kca, vca = kcd.cpu(), vcd.cpu()
    untouched = torch.ones((B, max_len), dtype=torch.bool)
    for b in range(B):
        p = int(sl[b]) - 1
        if p < 0:
            continue
        untouched[b, p] = False
        krow = kca[b, :, p].double().numpy()
        assert np.all(np.abs(krow - krow_ref[b]) <= bf16_ulp(krow_ref[b]) + 1e-30), "k row"
        assert torch.equal(vca[b, :, p], vn[b]), "v row"
    # every other cache row keeps its bits (NaN past each length included)
    for before, after in ((kc, kca), (vc, vca)):
        same = before.view(torch.int16) == after.view(torch.int16)
        assert bool(same.all(dim=-1).permute(0, 2, 1)[untouched].all()), "other cache rows changed"
    assert cga.device_status() == 0
