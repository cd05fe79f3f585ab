"""Prefill with a caller-owned workspace (attn_prefill_ws): every arrangement of its scratch
gives the oracle's result, and prefill and decode calls with their own workspaces run
concurrently on two streams. Reusing buffers allocated once, instead of sharing one library
buffer, follows the pages' split buffers ("Hand-written Triton decoder" section 3.3)."""
import math

import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library

pytestmark = pytest.mark.gpu


def _ws(nbytes, dev):
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=dev)


def test_prefill_ws_full_equals_library_scratch_and_oracle():
    cga = library()
    dev = device()
    cfg = workloads.CONFIGS["c3"]
    q, k, v = [t.to(dev) for t in workloads.config_prefill_inputs(cfg)]
    need = cga.attn_prefill_workspace_bytes(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.D, 1)
    assert need > cfg.B * cfg.Hkv * cfg.S * cfg.D * 2  # at least the fp16 copy of V
    ws = _ws(need, dev)
    o1, l1 = cga.prefill(q, k, v, causal=True, out_dtype=torch.float32, return_lse=True,
                         workspace=ws)
    o2, l2 = cga.prefill(q, k, v, causal=True, out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle.prefill(*[t.cpu() for t in (q, k, v)], True, cfg.scale)
    check_out(o1, o_ref, "bf16_pre", "c3 with caller workspace")
    check_lse(l1, lse_ref, "c3 with caller workspace lse")
    assert cga.device_status() == 0


def test_prefill_ws_smaller_workspaces_fall_back_with_the_same_results():
    """A workspace without room for the split, or without room for the fp16 copy of V either
    (V converted on chip), still gives the oracle's result; less than the V scale area is
    rejected before anything is launched."""
    cga = library()
    dev = device()
    B, Hq, Hkv, S, D = 1, 8, 2, 2048, 128
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", 3.0, seed=31)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(D))
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    full = cga.attn_prefill_workspace_bytes(B, S, Hq, Hkv, D, 1)
    v16 = B * Hkv * S * D * 2
    small = 4096  # the V scale area of this shape is a few hundred bytes
    for nbytes, what in ((full - 1, "no split"), (small + v16, "copy only"), (small, "on chip")):
        ws = _ws(nbytes, dev)
        o, lse = cga.prefill(q, k, v, causal=True, out_dtype=torch.float32, return_lse=True,
                             workspace=ws)
        torch.cuda.synchronize()
        check_out(o, o_ref, "bf16_pre", what)
        check_lse(lse, lse_ref, what + " lse")
    o = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=dev)
    ws = _ws(16, dev)
    rc = cga.attn_prefill_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, B, S,
                             Hq, Hkv, D, 1 / math.sqrt(D), 1, cga.ATTN_BF16, ws.data_ptr(), 16,
                             torch.cuda.current_stream().cuda_stream)
    assert rc == cga.ATTN_ERR_WORKSPACE
    assert cga.device_status() == 0


def test_prefill_and_decode_on_two_streams_with_own_workspaces():
    cga = library()
    dev = device()
    B, Hq, Hkv, S, D = 2, 8, 2, 1500, 128
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=32)
    o_ref, lse_ref = oracle.prefill(q, k, v, True, 1 / math.sqrt(D))
    dcfg = workloads.CONFIGS["c4b"]
    dq, dkc, dvc, dsl = workloads.config_decode_inputs(dcfg, seed=33)
    od_ref, lsed_ref = oracle.decode(dq, dkc, dvc, dsl, dcfg.scale)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    dq, dkc, dvc, dsl = dq.to(dev), dkc.to(dev), dvc.to(dev), dsl.to(dev)
    ws_p1 = _ws(cga.attn_prefill_workspace_bytes(B, S, Hq, Hkv, D, 1), dev)
    ws_p2 = _ws(cga.attn_prefill_workspace_bytes(B, S, Hq, Hkv, D, 1), dev)
    ws_d = _ws(cga.attn_decode_workspace_bytes(dcfg.B, dcfg.Hq, dcfg.Hkv, dcfg.D,
                                               dcfg.max_len), dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    outs = []
    for rep in range(3):
        with torch.cuda.stream(s1):
            op, lp = cga.prefill(q, k, v, causal=True, out_dtype=torch.float32,
                                 return_lse=True, workspace=ws_p1)
        with torch.cuda.stream(s2):
            od, ld = cga.decode(dq, dkc, dvc, dsl, out_dtype=torch.float32, return_lse=True,
                                workspace=ws_d)
            op2 = cga.prefill(q, k, v, causal=True, out_dtype=torch.float32, workspace=ws_p2)
        outs.append((op, lp, od, ld, op2))
    torch.cuda.synchronize()
    for op, lp, od, ld, op2 in outs:
        check_out(op, o_ref, "bf16_pre", "prefill on stream 1")
        check_lse(lp, lse_ref, "prefill on stream 1 lse")
        check_out(od, od_ref, "bf16_pre", "decode on stream 2")
        check_lse(ld, lsed_ref, "decode on stream 2 lse")
        assert torch.equal(op, op2)
    assert cga.device_status() == 0
