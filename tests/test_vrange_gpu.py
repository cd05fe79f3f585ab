"""The tensor-core paths (prefill, chunk against a cache, padded varlen; head dim 64 and 128)
over the whole bf16 range of V, against the fp64 oracle.

The P V product runs in fp16, whose range is far narrower than bf16's, so every (batch, kv head)
slab of V is scaled by a power of two before the conversion and O is scaled back. These tests
scale V by c from 1e-6 to 1e5 (one slab tiny and another huge in the same call, too) and check
the scale-covariant bounds: O is linear in V, so for V = c * V0 the contract's absolute bounds
become 4e-3 * c. The value-scale sweep follows the pages' test method ("Agent-written Triton
ops", step 2: inputs across magnitudes, because small values underflow and large ones overflow).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library

pytestmark = pytest.mark.gpu

SCALES = [1e-6, 1e-3, 1e3, 1e5]


def _scaled(v, c):
    """V * c, rounded once to bf16 (the oracle reads the same rounded values)."""
    return (v.float() * c).to(torch.bfloat16)


def _prefill(q, k, v, causal, out_dtype):
    cga = library()
    dev = device()
    o, lse = cga.prefill(q.to(dev), k.to(dev), v.to(dev), causal=causal, out_dtype=out_dtype,
                         return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    return o, lse


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("c", SCALES)
def test_prefill_v_scaled(D, c):
    # two row blocks and a ragged tail; GQA group 2
    q, k, v = workloads.prefill_inputs(1, 4, 2, 300, D, "bf16", seed=21)
    v = _scaled(v, c)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(D))
    tag = f"prefill D{D} V x {c:g}"
    o32, lse = _prefill(q, k, v, True, torch.float32)
    check_out(o32, o_ref, "bf16_pre", tag + " fp32 out", scale=c)
    check_lse(lse, lse_ref, tag + " lse")
    o16, _ = _prefill(q, k, v, True, torch.bfloat16)
    check_out(o16, o_ref, "bf16", tag + " bf16 out", scale=c)


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_split_slabs_of_opposite_magnitude(D):
    """One kv head's V near 1e-6, the other's near 1e5, in one call whose small grid splits the
    keys (partials scaled per slab before the merge). The bound uses each head's own scale."""
    Hq, Hkv, S = 8, 2, 2048
    q, k, v = workloads.prefill_inputs(1, Hq, Hkv, S, D, "bf16", 3.0, seed=22)
    cs = [1e-6, 1e5]
    v = torch.cat([_scaled(v[:, g:g + 1], cs[g]) for g in range(Hkv)], dim=1)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(D))
    o32, lse = _prefill(q, k, v, True, torch.float32)
    G = Hq // Hkv
    for g in range(Hkv):
        hs = slice(g * G, (g + 1) * G)
        check_out(o32[:, hs], o_ref[:, hs], "bf16_pre", f"D{D} kv head {g} x {cs[g]:g}",
                  scale=cs[g])
    check_lse(lse, lse_ref, f"D{D} mixed lse")


def test_prefill_single_large_value():
    """A standard-normal V with one element of 1e6: rows that see that key are dominated by it.
    The fp16 probability of that key carries a relative rounding error of at most 2^-11, so the
    bound for row i is 4e-3 + 2^-10 * sum_j p_ij |v_j| (the oracle on |V| gives that sum); rows
    that never see it keep the plain 4e-3."""
    q, k, v = workloads.prefill_inputs(1, 2, 1, 200, 128, "bf16", seed=9)
    v[0, 0, 150, 3] = 1.0e6
    o_ref, _ = oracle.prefill(q, k, v, True, 1 / math.sqrt(128))
    o_abs, _ = oracle.prefill(q, k, v.abs(), True, 1 / math.sqrt(128))
    o32, _ = _prefill(q, k, v, True, torch.float32)
    err = np.abs(o32.double().cpu().numpy() - o_ref)
    bound = 4e-3 + 2.0 ** -10 * o_abs
    assert (err <= bound).all(), f"max err / bound {np.max(err / bound):.3f}"
    check_out(o32[:, :, :150], o_ref[:, :, :150], "bf16_pre", "rows before the large value")


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("c", [1e-6, 1e5])
def test_chunk_v_scaled(D, c):
    """Chunk against a cache (rows past each length are NaN, never counted in the scale)."""
    B, Hq, Hkv, Sq, max_len, lens = 2, 8, 2, 64, 700, [650, 300]
    g = torch.Generator().manual_seed(23)
    q = torch.randn((B, Hq, Sq, D), generator=g).to(torch.bfloat16)
    _, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, D, max_len, "explicit", seed=24,
                                            seqlens=lens)
    vc = _scaled(vc, c)
    o_ref, lse_ref = oracle.chunk(q, kc, vc, sl, 1 / math.sqrt(D), True)
    cga = library()
    dev = device()
    o, lse = cga.chunk(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), causal=True,
                       out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    check_out(o, o_ref, "bf16_pre", f"chunk D{D} V x {c:g}", scale=c)
    check_lse(lse, lse_ref, f"chunk D{D} lse")


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("c", [1e-6, 1e5])
def test_varlen_v_scaled(D, c):
    """Padded batch (padding of k and v is NaN)."""
    B, Hq, Hkv, S, lens = 3, 8, 2, 300, [300, 129, 1]
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=25)
    v = _scaled(v, c)
    for b, L in enumerate(lens):
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    o_ref, lse_ref = oracle.prefill_varlen(q, k, v, sl, True, 1 / math.sqrt(D))
    cga = library()
    dev = device()
    o, lse = cga.prefill_varlen(q.to(dev), k.to(dev), v.to(dev), sl.to(dev), causal=True,
                                out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    check_out(o, o_ref, "bf16_pre", f"varlen D{D} V x {c:g}", scale=c)
    check_lse(lse, lse_ref, f"varlen D{D} lse")


def test_on_chip_conversion_v_scaled():
    """Caches whose fp16 copy of V would exceed the 1 GiB copy limit (B64 Hkv8, 8320 rows): V is
    converted on chip in the attention kernel, with the same per-slab scale. Sequence 5's kv
    head 1 holds a value of 1e6 and sequence 7's V is scaled to about 1e-6."""
    dev = device()
    B, Hq, Hkv, Sq, max_len = 64, 8, 8, 64, 8320
    g = torch.Generator().manual_seed(41)
    lens = torch.full((B,), 256, dtype=torch.int32)
    kc = torch.zeros((B, Hkv, max_len, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kh = torch.randn((B, Hkv, 256, 128), generator=g).to(torch.bfloat16)
    vh = torch.randn((B, Hkv, 256, 128), generator=g).to(torch.bfloat16)
    vh[5, 1] = _scaled(vh[5, 1], 1e3)
    vh[5, 1, 250, 7] = 1.0e6
    vh[7] = _scaled(vh[7], 1e-6)
    kc[:, :, :256] = kh.to(dev)
    vc[:, :, :256] = vh.to(dev)
    q = torch.randn((B, Hq, Sq, 128), generator=g).to(torch.bfloat16)
    cga = library()
    o, lse = cga.chunk(q.to(dev), kc, vc, lens.to(dev), causal=True, out_dtype=torch.float32,
                       return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    o_ref, lse_ref = oracle.chunk(q, kh, vh, lens, 1 / math.sqrt(128), True)
    o_abs, _ = oracle.chunk(q, kh, vh.abs(), lens, 1 / math.sqrt(128), True)
    o = o.double().cpu().numpy()
    err = np.abs(o - o_ref)
    # scale-covariant bound per sequence (1e-6 for sequence 7), P-rounding bound where the 1e6
    # value and the x1e3 slab enter
    c = np.ones(B)
    c[7] = 1e-6
    bound = 4e-3 * c[:, None, None, None] + 2.0 ** -10 * o_abs
    assert (err <= bound).all(), f"max err / bound {np.max(err / bound):.3f}"
    check_lse(lse, lse_ref, "on-chip lse")
