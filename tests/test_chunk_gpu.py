"""A chunk of new queries against a KV cache (tensor-core kernel, through the C ABI) against the
fp64 oracle on the same seeded inputs. Cache rows beyond each length are NaN."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library, sampled_rows

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Sq, max_len, lens, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Sq, 128), generator=g).to(torch.bfloat16)
    _, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, 128, max_len, "explicit", seed=seed + 1,
                                            seqlens=lens)
    return q, kc, vc, sl


def _run(q, kc, vc, sl, causal, out_dtype):
    cga = library()
    dev = device()
    o, lse = cga.chunk(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), causal=causal,
                       out_dtype=out_dtype, return_lse=True)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,Sq,max_len,lens,causal", [
    (3, 8, 2, 1, 700, [700, 1, 300], True),
    (3, 8, 2, 5, 700, [700, 5, 129], True),
    (2, 8, 2, 128, 1024, [1024, 300], True),
    (2, 4, 4, 200, 900, [899, 200], True),
    (2, 8, 2, 300, 1000, [1000, 450], False),
    (2, 8, 1, 257, 640, [640, 100], True),   # second sequence shorter than the chunk
])
def test_chunk_parity(B, Hq, Hkv, Sq, max_len, lens, causal):
    q, kc, vc, sl = _inputs(B, Hq, Hkv, Sq, max_len, lens, seed=Sq)
    o_ref, lse_ref = oracle.chunk(q, kc, vc, sl, 1 / math.sqrt(128), causal)
    tag = f"chunk {B},{Hq},{Hkv},{Sq},{max_len},{lens},{causal}"
    o32, lse = _run(q, kc, vc, sl, causal, torch.float32)
    check_out(o32, o_ref, "bf16_pre", tag + " fp32 out")
    check_lse(lse, lse_ref, tag + " lse")
    o16, _ = _run(q, kc, vc, sl, causal, torch.bfloat16)
    check_out(o16, o_ref, "bf16", tag + " bf16 out")
    assert library().device_status() == 0


def test_chunk_of_whole_sequence_is_prefill():
    """seqlens = Sq = max_len: the chunk is plain causal prefill (both match the oracle; plain
    prefill of this small grid also splits its keys, so the two are close, not bit-equal)."""
    cga = library()
    dev = device()
    q, k, v = workloads.prefill_inputs(2, 8, 2, 700, 128, "bf16", seed=4)
    o_p, l_p = cga.prefill(q.to(dev), k.to(dev), v.to(dev), causal=True, return_lse=True,
                           out_dtype=torch.float32)
    sl = torch.tensor([700, 700], dtype=torch.int32)
    o_c, l_c = _run(q, k, v, sl, True, torch.float32)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(128))
    check_out(o_c, o_ref, "bf16_pre", "chunk = prefill")
    check_lse(l_c, lse_ref, "chunk = prefill lse")
    assert (o_c - o_p).abs().max().item() <= 2 * 4e-3
    assert (l_c - l_p).abs().max().item() <= 2e-4


def test_chunk_of_one_matches_decode():
    cga = library()
    dev = device()
    q, kc, vc, sl = _inputs(4, 8, 2, 1, 2048, [2048, 1000, 17, 1], seed=9)
    o_c, l_c = _run(q, kc, vc, sl, True, torch.float32)
    o_d, l_d = cga.decode(q[:, :, 0].contiguous().to(dev), kc.to(dev), vc.to(dev), sl.to(dev),
                          out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert (o_c[:, :, 0] - o_d).abs().max().item() <= 2 * 4e-3
    assert (l_c[:, :, 0] - l_d).abs().max().item() <= 2e-4


def test_chunk_long_cache_sampled():
    """B4 Sq512 against caches of 8192 (lengths 512..8192): rows sampled for the oracle."""
    lens = [8192, 4096, 513, 6000]
    q, kc, vc, sl = _inputs(4, 8, 2, 512, 8192, lens, seed=21)
    o16, lse = _run(q, kc, vc, sl, True, torch.bfloat16)
    rows = sampled_rows(4, 8, 512, every=16, tail=16)
    # oracle on the sampled rows: chunk with all rows, then pick (the oracle is per row anyway)
    o_ref, lse_ref = oracle.chunk(q, kc, vc, sl, 1 / math.sqrt(128), True)
    o_ref = o_ref.reshape(-1, 128)[rows]
    lse_ref = lse_ref.reshape(-1)[rows]
    idx = torch.as_tensor(rows, device=o16.device)
    check_out(o16.reshape(-1, 128)[idx], o_ref, "bf16", "long chunk sampled")
    check_lse(lse.reshape(-1)[idx], lse_ref, "long chunk lse")


def test_chunk_length_above_cache_is_clamped_and_flagged():
    cga = library()
    q, kc, vc, _ = _inputs(2, 8, 2, 64, 256, [256, 256], seed=3)
    sl = torch.tensor([256, 999], dtype=torch.int32)
    cga.device_status()
    o, _ = _run(q, kc, vc, sl, True, torch.float32)
    assert cga.device_status() & cga.ATTN_DEV_SEQLEN_CLAMPED
    o_ref, _ = oracle.chunk(q, kc, vc, torch.tensor([256, 256], dtype=torch.int32),
                            1 / math.sqrt(128), True)
    check_out(o, o_ref, "bf16_pre", "clamped chunk")


def test_chunk_cache_above_copy_limit_converts_on_chip():
    """Caches whose fp16 copy of V would exceed the library's 1 GiB limit (B64 Hkv8, 8320 rows of
    D128): the attention kernel converts V on chip instead. Only the rows below each length are
    written; the rest of both caches is uninitialised device memory, which must not leak in."""
    dev = device()
    B, Hq, Hkv, Sq, max_len = 64, 8, 8, 64, 8320
    assert B * Hkv * max_len * 128 * 2 > (1 << 30)
    g = torch.Generator().manual_seed(31)
    lens = torch.randint(1, 300, (B,), generator=g, dtype=torch.int32)
    lens[0] = 299
    lens[1] = 1
    kc = torch.empty((B, Hkv, max_len, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kh = torch.randn((B, Hkv, 300, 128), generator=g).to(torch.bfloat16)
    vh = torch.randn((B, Hkv, 300, 128), generator=g).to(torch.bfloat16)
    for b in range(B):
        L = int(lens[b])
        kc[b, :, :L] = kh[b, :, :L].to(dev)
        vc[b, :, :L] = vh[b, :, :L].to(dev)
    q = torch.randn((B, Hq, Sq, 128), generator=g).to(torch.bfloat16)
    cga = library()
    o, lse = cga.chunk(q.to(dev), kc, vc, lens.to(dev), causal=True, out_dtype=torch.float32,
                       return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    # the oracle sees the written rows only (every length is below 300)
    o_ref, lse_ref = oracle.chunk(q, kh, vh, lens, 1 / math.sqrt(128), True)
    check_out(o, o_ref, "bf16_pre", "large-cache chunk")
    check_lse(lse, lse_ref, "large-cache chunk lse")
