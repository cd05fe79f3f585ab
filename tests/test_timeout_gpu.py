"""The failure path of the pipeline waits, made to run on the GPU without a fault.

Every wait of the prefill and decode pipelines is bounded; when one runs out the block sets
ATTN_DEV_WAIT_TIMEOUT, lets the copies and tensor-core work it already started finish, and returns
without writing its results. attn_debug_set_wait_limit lowers the bound to a cycle, so the first
wait that is not already satisfied gives up (nothing hangs and nothing faults: every barrier the
block waits on still completes, and the drain waits for it). The next call with the normal bound
must be correct, which shows the context and the library's state survived."""
import math

import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library

pytestmark = pytest.mark.gpu


def _calls(cga, dev):
    """(name, fn) pairs covering the kernels with pipeline waits: prefill split + fp16 copy,
    unsplit prefill with V converted on chip (a workspace that holds only the V scale area),
    the stream decode, the chunked decode (above 1024 sequences) and a head-dim-64 prefill. The decode caches are
    large (1.1 GB each call) so that their pipelines wait on device memory, not on L2."""
    q, k, v = [t.to(dev) for t in workloads.prefill_inputs(1, 8, 2, 2048, 128, "bf16", seed=51)]
    small_ws = torch.empty(4096, dtype=torch.uint8, device=dev)
    dq, dkc, dvc, dsl = [t.to(dev) for t in
                         workloads.decode_inputs(32, 8, 2, 128, 32768, "full", seed=52)]
    bq, bkc, bvc, bsl = [t.to(dev) for t in
                         workloads.decode_inputs(1100, 2, 1, 128, 2048, "full", seed=53)]
    # head dim 64, many heads (a grid several waves deep)
    q4, k4, v4 = [t.to(dev) for t in workloads.prefill_inputs(2, 80, 8, 1024, 64, "bf16",
                                                              seed=54)]
    return [
        ("prefill split", lambda: cga.prefill(q, k, v, causal=True, out_dtype=torch.float32,
                                              return_lse=True)),
        ("prefill on chip", lambda: cga.prefill(q, k, v, causal=True, out_dtype=torch.float32,
                                                return_lse=True, workspace=small_ws)),
        ("decode", lambda: cga.decode(dq, dkc, dvc, dsl, out_dtype=torch.float32,
                                      return_lse=True)),
        ("decode chunked", lambda: cga.decode(bq, bkc, bvc, bsl, out_dtype=torch.float32,
                                              return_lse=True)),
        ("prefill d64", lambda: cga.prefill(q4, k4, v4, causal=True,
                                                       out_dtype=torch.float32,
                                                       return_lse=True)),
    ], (q, k, v), (dq, dkc, dvc, dsl), (bq, bkc, bvc, bsl), (q4, k4, v4)


def test_wait_timeout_is_reported_and_the_next_call_is_correct():
    cga = library()
    dev = device()
    calls, pre, dec, big, pre4 = _calls(cga, dev)
    for _, fn in calls:  # first use: scratch sized, kernels loaded, with the normal bound
        fn()
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    try:
        assert cga.attn_debug_set_wait_limit(1) == cga.ATTN_OK
        for name, fn in calls:
            flush.zero_()  # the call's inputs come from device memory, not L2
            fn()
            torch.cuda.synchronize()
            st = cga.device_status()
            # A wait's first probe may itself block for a while (the hardware may suspend the
            # thread until the phase completes), so a wait only runs out when its copy takes
            # longer than that. The chunked decode's short pipelines (8 stages a warp) usually
            # find every copy landed; it runs here under the short bound all the same.
            if name != "decode chunked":
                assert st & cga.ATTN_DEV_WAIT_TIMEOUT, f"{name}: no wait ran out (status {st})"
            assert st & ~cga.ATTN_DEV_WAIT_TIMEOUT == 0, f"{name}: status {st}"
    finally:
        assert cga.attn_debug_set_wait_limit(0) == cga.ATTN_OK
    results = [fn() for _, fn in calls]
    torch.cuda.synchronize()
    assert cga.device_status() == 0
    o_ref, lse_ref = oracle.prefill(*[t.cpu() for t in pre], True, 1 / math.sqrt(128))
    for (o, lse), what in zip(results[:2], ("prefill split", "prefill on chip")):
        check_out(o, o_ref, "bf16_pre", what + " after the timeouts")
        check_lse(lse, lse_ref, what + " lse after the timeouts")
    od_ref, lsed_ref = oracle.decode(*[t.cpu() for t in dec], 1 / math.sqrt(128))
    check_out(results[2][0], od_ref, "bf16_pre", "decode after the timeouts")
    check_lse(results[2][1], lsed_ref, "decode lse after the timeouts")
    ob_ref, lseb_ref = oracle.decode(*[t.cpu() for t in big], 1 / math.sqrt(128))
    check_out(results[3][0], ob_ref, "bf16_pre", "chunked decode after the timeouts")
    check_lse(results[3][1], lseb_ref, "chunked decode lse after the timeouts")
    o4_ref, lse4_ref = oracle.prefill(*[t.cpu() for t in pre4], True, 1 / math.sqrt(64))
    check_out(results[4][0], o4_ref, "bf16_pre", "d64 prefill after the timeouts")
    check_lse(results[4][1], lse4_ref, "d64 prefill lse after the timeouts")
