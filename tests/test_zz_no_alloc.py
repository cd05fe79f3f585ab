"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all: a memory manager that owns every byte of the device,
a process whose allocator is frozen after start-up, a plug-in handed tensors but no allocator.
For them the library has one decode entry point that allocates nothing; its scratch is a fixed
array inside the library. These tests call it through the C ABI, twice in a row with different
inputs, and compare with the regular decode entry point. The file is named so that pytest
collects it last.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import TOL_BF16_PRE, device, library

pytestmark = pytest.mark.gpu


def _noalloc(cga, q, kc, vc, sl, out_dtype):
    B, Hq, D = q.shape
    Hkv, max_len = kc.shape[1], kc.shape[2]
    o = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    out_t = cga.ATTN_F32 if out_dtype == torch.float32 else cga.ATTN_BF16
    rc = cga.attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, D, max_len,
                                 1.0 / math.sqrt(D), out_t,
                                 torch.cuda.current_stream(q.device).cuda_stream)
    assert rc == cga.ATTN_OK, cga.attn_status_string(rc)
    return o, lse


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_regular_decode_two_calls(out_dtype):
    cga = library()
    dev = device()
    cases = [
        workloads.config_decode_inputs(workloads.CONFIGS["c4b"]),
        workloads.decode_inputs(5, 8, 2, 128, 1500, "explicit", seed=3,
                                seqlens=[1500, 1, 700, 0, 33]),
    ]
    for n, (q, kc, vc, sl) in enumerate(cases):
        q, kc, vc, sl = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
        o, lse = _noalloc(cga, q, kc, vc, sl, out_dtype)
        o_ref, lse_ref = cga.decode(q, kc, vc, sl, out_dtype=out_dtype, return_lse=True)
        torch.cuda.synchronize()
        diff = (o.double() - o_ref.double()).abs().max().item()
        assert diff <= TOL_BF16_PRE, f"call {n}: max |noalloc - decode| = {diff}"
        lmask = torch.isfinite(lse_ref)
        assert torch.equal(torch.isfinite(lse), lmask)
        assert (lse[lmask] - lse_ref[lmask]).abs().max().item() <= 1e-4
    assert cga.device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    cga = library()
    dev = device()
    B, Hq, Hkv, D, max_len = 64, 32, 8, 128, 8192
    need = cga.attn_decode_workspace_bytes(B, Hq, Hkv, D, max_len)
    assert need > cga._lib.ATTN_DECODE_NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device=dev)  # never read: rejected on the host
    rc = cga.attn_decode_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(),
                                 t.data_ptr(), None, B, Hq, Hkv, D, max_len, 0.1, cga.ATTN_F32,
                                 None)
    assert rc == cga.ATTN_ERR_WORKSPACE
