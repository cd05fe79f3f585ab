"""Head dim 64 on the tensor-core prefill kernel, and operands read and written in place through
strides ([B, S, H, D] tensors, q/k/v as head slices of one fused projection output), against
the fp64 oracle on the same seeded inputs (the oracle sees the plain [B, H, S, D] copies)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library, sampled_rows

pytestmark = pytest.mark.gpu


def _run(q, k, v, causal, out_dtype, out=None):
    cga = library()
    o, lse = cga.prefill(q, k, v, causal=causal, out_dtype=out_dtype, return_lse=True, out=out)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    return o, lse


# ------------------------------------------------------------------ head dim 64, bf16

D64 = [
    # B, Hq, Hkv, S, causal, q_mult
    (1, 1, 1, 1, True, 1.0), (1, 2, 1, 63, False, 1.0), (2, 4, 2, 129, True, 1.0),
    (1, 4, 1, 255, False, 3.0), (1, 12, 12, 512, True, 1.0), (1, 12, 12, 512, False, 1.0),
    (2, 2, 1, 300, True, 3.0), (1, 8, 2, 2048, True, 3.0),   # small grids: pair-mode blocks
]


@pytest.mark.parametrize("B,Hq,Hkv,S,causal,q_mult", D64)
def test_prefill_bf16_d64(B, Hq, Hkv, S, causal, q_mult):
    dev = device()
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, 64, "bf16", q_mult, seed=1)
    o_ref, lse_ref = oracle.prefill(q, k, v, causal, 1 / math.sqrt(64))
    tag = f"d64 prefill {B},{Hq},{Hkv},{S},{causal},{q_mult}"
    o32, lse = _run(q.to(dev), k.to(dev), v.to(dev), causal, torch.float32)
    check_out(o32, o_ref, "bf16_pre", tag + " fp32 out")
    check_lse(lse, lse_ref, tag + " lse")
    o16, lse16 = _run(q.to(dev), k.to(dev), v.to(dev), causal, torch.bfloat16)
    check_out(o16, o_ref, "bf16", tag + " bf16 out")
    assert torch.equal(lse16, lse)


# Head dim 64 on grids several waves deep: many heads (a group of 10 query heads per kv head),
# short ragged sequences, a peaky softmax, and a longer batch checked on sampled rows.
D64_MANY_HEADS = [
    # B, Hq, Hkv, S, causal, q_mult
    (4, 40, 8, 600, True, 1.0),
    (4, 40, 8, 600, False, 1.0),
    (2, 56, 8, 1100, True, 3.0),
    (1, 160, 16, 1024, True, 1.0),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,causal,q_mult", D64_MANY_HEADS)
def test_prefill_bf16_d64_many_heads(B, Hq, Hkv, S, causal, q_mult):
    test_prefill_bf16_d64(B, Hq, Hkv, S, causal, q_mult)


def test_prefill_bf16_d64_batch4_sampled():
    dev = device()
    B, Hq, Hkv, S = 4, 8, 2, 8192
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, 64, "bf16", seed=9)
    rows = sampled_rows(B, Hq, S)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(64), rows=rows)
    idx = torch.as_tensor(rows, device=dev)
    for dt, kind in ((torch.float32, "bf16_pre"), (torch.bfloat16, "bf16")):
        o, lse = _run(q.to(dev), k.to(dev), v.to(dev), True, dt)
        check_out(o.reshape(-1, 64)[idx], o_ref, kind, f"d64 B4 S8192 {dt}")
        check_lse(lse.reshape(-1)[idx], lse_ref, "d64 B4 S8192 lse")


def test_prefill_bf16_d64_long_sampled():
    dev = device()
    B, Hq, Hkv, S = 2, 8, 2, 8192
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, 64, "bf16", seed=2)
    o16, lse = _run(q.to(dev), k.to(dev), v.to(dev), True, torch.bfloat16)
    rows = sampled_rows(B, Hq, S)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(64), rows=rows)
    idx = torch.as_tensor(rows, device=dev)
    check_out(o16.reshape(-1, 64)[idx], o_ref, "bf16", "d64 S8192 sampled rows")
    check_lse(lse.reshape(-1)[idx], lse_ref, "d64 S8192 sampled lse")


def test_chunk_and_varlen_d64():
    cga = library()
    dev = device()
    # chunk: 3 sequences, 200 new queries against caches of 700 rows (NaN past each length)
    q, kc, vc, sl = workloads.decode_inputs(3, 8, 2, 64, 700, "explicit", seed=3,
                                            seqlens=[700, 200, 450])
    qc = workloads.prefill_inputs(3, 8, 2, 200, 64, "bf16", seed=4)[0]
    o_ref, lse_ref = oracle.chunk(qc, kc, vc, sl, 1 / math.sqrt(64), True)
    o, lse = cga.chunk(qc.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), out_dtype=torch.float32,
                       return_lse=True)
    torch.cuda.synchronize()
    check_out(o, o_ref, "bf16_pre", "d64 chunk")
    check_lse(lse, lse_ref, "d64 chunk lse")
    # varlen: padded batch, padding positions of k and v NaN
    q, k, v = workloads.prefill_inputs(3, 4, 2, 600, 64, "bf16", seed=5)
    lens = [600, 1, 333]
    for b, L in enumerate(lens):
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    o_ref, lse_ref = oracle.prefill_varlen(q, k, v, sl, True, 1 / math.sqrt(64))
    o, lse = cga.prefill_varlen(q.to(dev), k.to(dev), v.to(dev), sl.to(dev),
                                out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    check_out(o, o_ref, "bf16_pre", "d64 varlen")
    check_lse(lse, lse_ref, "d64 varlen lse")
    assert cga.device_status() == 0


# ------------------------------------------------------------------ strided operands


def _bshd(t, dev):
    """A [B,S,H,D] device copy of the [B,H,S,D] tensor t, returned as its [B,H,S,D] view."""
    return t.transpose(1, 2).contiguous().to(dev).transpose(1, 2)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", [
    (2, 8, 2, 300, 128, True), (1, 4, 4, 1000, 128, False), (2, 8, 2, 700, 64, True),
    (1, 8, 2, 2048, 128, True),   # pair-mode blocks write through the strides
    (4, 40, 8, 600, 64, True),    # head dim 64, many heads
])
def test_prefill_bshd_layout(B, Hq, Hkv, S, D, causal):
    dev = device()
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=6)
    o_ref, lse_ref = oracle.prefill(q, k, v, causal, 1 / math.sqrt(D))
    qv, kv, vv = _bshd(q, dev), _bshd(k, dev), _bshd(v, dev)
    assert not qv.is_contiguous()
    for dt, kind in ((torch.float32, "bf16_pre"), (torch.bfloat16, "bf16")):
        o_store = torch.full((B, S, Hq, D), float("nan"), dtype=dt, device=dev)
        o, lse = _run(qv, kv, vv, causal, dt, out=o_store.transpose(1, 2))
        assert o.data_ptr() == o_store.data_ptr()
        check_out(o_store.transpose(1, 2), o_ref, kind, f"bshd {B},{Hq},{Hkv},{S},{D} {dt}")
        check_lse(lse, lse_ref, "bshd lse")


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", [
    (2, 8, 2, 513, 128, True), (1, 16, 2, 256, 64, False), (3, 6, 2, 129, 128, True),
    (2, 80, 8, 1024, 64, True),   # head dim 64, many heads
])
def test_prefill_fused_qkv(B, Hq, Hkv, S, D, causal):
    """q, k, v as head slices of one [B, S, Hq + 2 Hkv, D] projection output; O written into a
    [B, S, Hq, D] buffer (the hidden layout) in place."""
    dev = device()
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=7)
    o_ref, lse_ref = oracle.prefill(q, k, v, causal, 1 / math.sqrt(D))
    qkv = torch.cat([q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2)], dim=2)
    qkv = qkv.contiguous().to(dev)
    qv = qkv[:, :, :Hq].transpose(1, 2)
    kv = qkv[:, :, Hq:Hq + Hkv].transpose(1, 2)
    vv = qkv[:, :, Hq + Hkv:].transpose(1, 2)
    before = qkv.clone()
    o_store = torch.full((B, S, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    _, lse = _run(qv, kv, vv, causal, torch.bfloat16, out=o_store.transpose(1, 2))
    check_out(o_store.transpose(1, 2), o_ref, "bf16", f"fused qkv {B},{Hq},{Hkv},{S},{D}")
    check_lse(lse, lse_ref, "fused qkv lse")
    assert torch.equal(qkv, before), "inputs were modified"


@pytest.mark.parametrize("B,Hq,Hkv,S,D", [(2, 8, 2, 1000, 128), (4, 40, 8, 600, 64)])
def test_strided_equals_contiguous_bitwise(B, Hq, Hkv, S, D):
    """The same values through the strided entry and the contiguous one give identical bits."""
    dev = device()
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=8)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = _run(qd, kd, vd, True, torch.bfloat16)
    o2, l2 = _run(_bshd(q, dev), _bshd(k, dev), _bshd(v, dev), True, torch.bfloat16)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_chunk_strided_caches_bitwise_equal_contiguous():
    """A chunk against caches stored [B, max_len, Hkv, D] (passed as transposed views), q as a
    [B, Sq, Hq, D] view and O written into a [B, Sq, Hq, D] buffer: the oracle's result, and the
    same bits as the contiguous call."""
    cga = library()
    dev = device()
    B, Hq, Hkv, Sq, max_len = 3, 8, 2, 200, 700
    q, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, 128, max_len, "explicit", seed=13,
                                            seqlens=[700, 200, 450])
    qc = workloads.prefill_inputs(B, Hq, Hkv, Sq, 128, "bf16", seed=14)[0]
    o_ref, lse_ref = oracle.chunk(qc, kc, vc, sl, 1 / math.sqrt(128), True)
    kv_, vv_, qv_ = _bshd(kc, dev), _bshd(vc, dev), _bshd(qc, dev)
    assert not kv_.is_contiguous()
    o_store = torch.full((B, Sq, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    o, lse = cga.chunk(qv_, kv_, vv_, sl.to(dev), out=o_store.transpose(1, 2),
                       out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    check_out(o_store.transpose(1, 2), o_ref, "bf16_pre", "strided chunk")
    check_lse(lse, lse_ref, "strided chunk lse")
    o2, l2 = cga.chunk(qc.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), out_dtype=torch.float32,
                       return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o_store.transpose(1, 2), o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("D", [128, 64])
def test_varlen_from_fused_qkv(D):
    """A padded batch read as head slices of one [B, S, Hq + 2 Hkv, D] projection output (K and V
    NaN past each length), O written into a [B, S, Hq, D] buffer, against the oracle."""
    dev = device()
    B, Hq, Hkv, S = 3, 8, 2, 600
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=15)
    lens = [600, 1, 333]
    for b, L in enumerate(lens):
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    o_ref, lse_ref = oracle.prefill_varlen(q, k, v, sl, True, 1 / math.sqrt(D))
    qkv = torch.cat([q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2)], dim=2)
    qkv = qkv.contiguous().to(dev)
    qv = qkv[:, :, :Hq].transpose(1, 2)
    kv = qkv[:, :, Hq:Hq + Hkv].transpose(1, 2)
    vv = qkv[:, :, Hq + Hkv:].transpose(1, 2)
    o_store = torch.full((B, S, Hq, D), float("nan"), dtype=torch.float32, device=dev)
    cga = library()
    _, lse = cga.prefill_varlen(qv, kv, vv, sl.to(dev), out=o_store.transpose(1, 2),
                                out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    check_out(o_store.transpose(1, 2), o_ref, "bf16_pre", f"fused-qkv varlen D{D}")
    check_lse(lse, lse_ref, f"fused-qkv varlen D{D} lse")


@pytest.mark.parametrize("D", [128, 64])
def test_key_split_sampled(D):
    """B1 Hq8 S6144: between one and two waves of two-tile blocks, where the planner splits the
    late row blocks' key tiles into segments and a second kernel merges them. Rows sampled
    (every 64th and the last 128 of each head: the split row blocks are the late ones)."""
    dev = device()
    B, Hq, Hkv, S = 1, 8, 2, 6144
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", 3.0, seed=9)
    rows = sampled_rows(B, Hq, S)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(D), rows=rows)
    idx = torch.as_tensor(rows, device=dev)
    for dt, kind in ((torch.float32, "bf16_pre"), (torch.bfloat16, "bf16")):
        o, lse = _run(q.to(dev), k.to(dev), v.to(dev), True, dt)
        check_out(o.reshape(-1, D)[idx], o_ref, kind, f"split S6144 D{D} {kind}")
        check_lse(lse.reshape(-1)[idx], lse_ref, f"split S6144 D{D} lse")
    # the merge kernel writes through the output's strides: a [B, S, Hq, D] buffer gives the
    # same bits as the contiguous output
    o1, l1 = _run(q.to(dev), k.to(dev), v.to(dev), True, torch.bfloat16)
    o_store = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=dev)
    _, l2 = _run(_bshd(q, dev), _bshd(k, dev), _bshd(v, dev), True, torch.bfloat16,
                 out=o_store.transpose(1, 2))
    assert torch.equal(o1, o_store.transpose(1, 2)) and torch.equal(l1, l2)
