"""Decode parity on the GPU: split-KV kernel + merge kernel (through the C ABI) against the
fp64 oracle on the same seeded inputs. Cache rows beyond each length are NaN."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_lse, check_out, device, library

pytestmark = pytest.mark.gpu


def _run(q, kc, vc, sl, out_dtype, **kw):
    cga = library()
    dev = device()
    o, lse = cga.decode(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), out_dtype=out_dtype,
                        return_lse=True, **kw)
    torch.cuda.synchronize()
    return o, lse


def _check(q, kc, vc, sl, tag, **kw):
    D = q.shape[-1]
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl, 1 / math.sqrt(D))
    o32, lse = _run(q, kc, vc, sl, torch.float32, **kw)
    check_out(o32, o_ref, "bf16_pre", tag + " fp32 out")
    check_lse(lse, lse_ref, tag + " lse")
    o16, _ = _run(q, kc, vc, sl, torch.bfloat16, **kw)
    check_out(o16, o_ref, "bf16", tag + " bf16 out")
    import causal_gqa_attention_gb300 as cga

    assert cga.device_status() == 0


@pytest.mark.parametrize("name", ["c4a", "c4b"])
def test_decode_configured(name):
    cfg = workloads.CONFIGS[name]
    q, kc, vc, sl = workloads.config_decode_inputs(cfg)
    _check(q, kc, vc, sl, name)


@pytest.mark.parametrize("seed", [1, 2])
def test_decode_batched_other_seeds(seed):
    """The configured batched decode (B32, lengths U[256, 4096]) drawn from two more seeds."""
    cfg = workloads.CONFIGS["c4b"]
    q, kc, vc, sl = workloads.config_decode_inputs(cfg, seed=seed)
    _check(q, kc, vc, sl, f"c4b seed {seed}")


@pytest.mark.parametrize("B,Hq,Hkv,D,max_len,lens", [
    (4, 8, 2, 128, 300, [1, 31, 32, 33]),
    (3, 8, 2, 128, 4096, [255, 256, 4096]),
    (2, 4, 4, 128, 1000, [999, 517]),        # no grouping (G = 1)
    (2, 16, 2, 128, 700, [700, 123]),        # G = 8
    (2, 6, 2, 128, 200, [200, 65]),          # G = 3 (one head per block)
    (3, 8, 2, 64, 513, [513, 64, 2]),        # D = 64
    (1, 8, 1, 128, 40000, [40000]),          # long context, one sequence over every warp
    (40, 8, 2, 128, 300, None),              # many short sequences per warp slice
    (2, 4, 2, 128, 300, [300, 17]),          # G = 2: two heads per stream
    (2, 12, 2, 64, 400, [400, 255]),         # G = 6: two heads per stream, three streams
    (2, 32, 2, 128, 600, [600, 37]),         # G = 16: eight heads per stream, two streams
    (2, 24, 2, 128, 500, [499, 250]),        # G = 12: four heads per stream, three streams
    (2, 10, 2, 128, 300, [300, 1]),          # G = 5: one head per stream, five streams
])
def test_decode_shapes(B, Hq, Hkv, D, max_len, lens):
    if lens is None:  # lengths 0..max_len, including empty sequences
        lens = torch.randint(0, max_len + 1, (B,), generator=torch.Generator().manual_seed(5))
        lens[::7] = 0
        lens = lens.tolist()
    q, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, D, max_len, "explicit", seed=1,
                                            seqlens=lens)
    _check(q, kc, vc, sl, f"decode {B},{Hq},{Hkv},{D},{max_len},{lens}")


def test_decode_empty_sequence():
    q, kc, vc, sl = workloads.decode_inputs(3, 8, 2, 128, 64, "explicit", seed=2,
                                            seqlens=[0, 5, 0])
    o, lse = _run(q, kc, vc, sl, torch.float32)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl, 1 / math.sqrt(128))
    check_out(o[1:2], o_ref[1:2], "bf16_pre", "empty-batch neighbour")


def test_decode_caller_workspace_and_determinism():
    """A caller workspace and the library-owned scratch run the same split and merge kernels:
    both agree with the oracle, and each gives identical bits on every call (the merge combines
    a stream's pieces in a fixed order)."""
    cga = library()
    dev = device()
    cfg = workloads.CONFIGS["c4b"]
    q, kc, vc, sl = workloads.config_decode_inputs(cfg)
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl, cfg.scale)
    nbytes = cga.attn_decode_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.max_len)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for kw in ({"workspace": ws}, {}):
        runs = [_run(q, kc, vc, sl, torch.float32, **kw) for _ in range(3)]
        for o, lse in runs[1:]:
            assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])
        check_out(runs[0][0], o_ref, "bf16_pre", f"c4b {list(kw)}")
        check_lse(runs[0][1], lse_ref, f"c4b lse {list(kw)}")
    small = torch.empty(nbytes - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(cga.AttnError) as ei:
        _run(q, kc, vc, sl, torch.bfloat16, workspace=small)
    assert ei.value.code == cga.ATTN_ERR_WORKSPACE


def test_decode_seqlen_above_max_len_is_clamped_and_flagged():
    cga = library()
    q, kc, vc, _ = workloads.decode_inputs(2, 8, 2, 128, 96, "full", seed=4)
    sl = torch.tensor([96, 500], dtype=torch.int32)
    cga.device_status()  # clear
    o, _ = _run(q, kc, vc, sl, torch.float32)
    assert cga.device_status() & cga.ATTN_DEV_SEQLEN_CLAMPED
    o_ref, _ = oracle.decode(q, kc, vc, torch.tensor([96, 96], dtype=torch.int32),
                             1 / math.sqrt(128))
    check_out(o, o_ref, "bf16_pre", "clamped length")


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (32, 2, 64), (3, 1, 128)])
def test_decode_large_batch_chunked_path(Hq, Hkv, D):
    """Batches above 1024 use the chunked split kernel (groups of 4, 16 and 3 query heads)."""
    B = 1100
    lens = torch.randint(1, 97, (B,), generator=torch.Generator().manual_seed(6))
    lens[::13] = 0
    q, kc, vc, sl = workloads.decode_inputs(B, Hq, Hkv, D, 96, "explicit", seed=2,
                                            seqlens=lens.tolist())
    _check(q, kc, vc, sl, f"decode B1100 Hq{Hq} Hkv{Hkv} D{D}")
