"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all: a memory manager that owns every byte of the device,
a process whose allocator is frozen after start-up, a plug-in handed tensors but no allocator.
For them the library has one decode entry point that allocates nothing; its scratch is a fixed
array inside the library. These tests call it through the C ABI, twice in a row with different
inputs, and check it against the fp64 oracle and against the regular decode entry point; a
fresh process checks that calls leave the device's free memory unchanged. The file is named so
that pytest collects it last.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


CASES = [
    # the configured batched decode (B32, Hq8/Hkv2, D128, lengths U[256, 4096]): full grid
    lambda: workloads.config_decode_inputs(workloads.CONFIGS["c4b"]),
    # ragged lengths including 0 and 1
    lambda: workloads.decode_inputs(5, 8, 2, 128, 1500, "explicit", seed=3,
                                    seqlens=[1500, 1, 700, 0, 33]),
    # a group of 8 query heads per kv head at D = 128: fewer warps than the full grid
    lambda: workloads.decode_inputs(4, 16, 2, 128, 2048, "explicit", seed=4,
                                    seqlens=[2048, 1, 1000, 0]),
    # above 1024 sequences: the chunked kernel, whose partials fit the array here
    lambda: workloads.decode_inputs(1100, 2, 1, 64, 64, "uniform", seed=5),
]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_oracle_two_calls_in_a_row(out_dtype):
    cga = library()
    dev = device()
    kind = "bf16_pre" if out_dtype == torch.float32 else "bf16"
    for n, make in enumerate(CASES):
        q, kc, vc, sl = make()
        D = q.shape[-1]
        o_ref, lse_ref = oracle.decode(q, kc, vc, sl, 1 / math.sqrt(D))
        dq, dkc, dvc, dsl = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
        for rep in range(2):
            o, lse = _noalloc(cga, dq, dkc, dvc, dsl, out_dtype)
            torch.cuda.synchronize()
            check_out(o, o_ref, kind, f"case {n} call {rep}")
            check_lse(lse, lse_ref, f"case {n} call {rep} lse")
    assert cga.device_status() == 0


def test_noalloc_equals_regular_decode_on_the_full_grid():
    """Where the array holds the full grid's partials the two entry points run the same kernels
    on the same split: identical bits."""
    cga = library()
    dev = device()
    for make in CASES[:2]:
        q, kc, vc, sl = [t.to(dev) for t in make()]
        o, lse = _noalloc(cga, q, kc, vc, sl, torch.bfloat16)
        o_ref, lse_ref = cga.decode(q, kc, vc, sl, return_lse=True)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, lse_ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    cga = library()
    dev = device()
    t = torch.empty(16, dtype=torch.bfloat16, device=dev)  # never read: rejected on the host
    for B, Hq, Hkv, D, max_len in [(1024, 16, 2, 128, 4096),   # B * Hq above the array's rows
                                   (2000, 8, 2, 128, 4096)]:   # chunked partials too large
        rc = cga.attn_decode_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(),
                                     t.data_ptr(), None, B, Hq, Hkv, D, max_len, 0.1,
                                     cga.ATTN_F32, None)
        assert rc == cga.ATTN_ERR_WORKSPACE


_FRESH_PROCESS = r"""
import math, sys
sys.path.insert(0, sys.argv[1])
import torch
import workloads
import causal_gqa_attention_gb300 as cga
from causal_gqa_attention_gb300 import build
build.build()
cga.load_library()
dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
inputs = []
for B, Hq, Hkv, D, L in [(32, 8, 2, 128, 4096), (4, 16, 2, 128, 2048), (7, 4, 4, 64, 3000)]:
    q, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, D, L, "uniform", seed=B)
    q, kc, vc, sl = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    inputs.append((q, kc, vc, sl, o, lse, B, Hq, Hkv, D, L))
def call(a):
    q, kc, vc, sl, o, lse, B, Hq, Hkv, D, L = a
    rc = cga.attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, D, L,
                                 1.0 / math.sqrt(D), cga.ATTN_F32,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == cga.ATTN_OK, rc
ob = torch.empty((inputs[0][6], inputs[0][7], inputs[0][9]), dtype=torch.bfloat16, device=dev)
# the first call of each shape loads the library's device code (the module holds the fixed
# array) and looks up the array's address; after that no call may change the free memory
for a in inputs:
    call(a)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info(dev)[0]
for rep in range(3):
    for a in inputs:
        call(a)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info(dev)[0]
assert free1 == free0, (free0, free1)
# control: the regular decode grows its library-owned buffer on first use, which shows up
q, kc, vc, sl, o, lse, B, Hq, Hkv, D, L = inputs[0]
cga.decode(q, kc, vc, sl, out=ob)
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info(dev)[0]
assert free2 < free1, (free1, free2)
print("noalloc free memory unchanged:", free0, free1)
"""


def test_noalloc_leaves_free_memory_unchanged_in_a_fresh_process():
    device()
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS, ROOT], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "free memory unchanged" in r.stdout
