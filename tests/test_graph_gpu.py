"""The library under CUDA graph capture: every entry point records into a graph without host
synchronisation or allocation (after the scratch is sized outside the capture), and replays
give bit-identical results to eager calls on the same inputs, with new inputs copied into the
captured buffers between replays."""
import math

import pytest
import torch

import workloads
from parity import device, library

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm up fn on a side stream, then capture it; returns the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("B,Hq,Hkv,S,D", [(1, 8, 2, 2048, 128), (2, 8, 2, 3000, 128),
                                          (1, 8, 2, 2048, 64)])
def test_prefill_graph_replay(B, Hq, Hkv, S, D):
    cga = library()
    dev = device()
    q, k, v = [t.to(dev) for t in workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=1)]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    g = _capture(lambda: cga.prefill(q, k, v, causal=True, out=o, lse=lse, return_lse=True))
    for seed in (2, 3):
        nq, nk, nv = [t.to(dev) for t in workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16",
                                                                  seed=seed)]
        q.copy_(nq), k.copy_(nk), v.copy_(nv)
        g.replay()
        torch.cuda.synchronize()
        oe, le = cga.prefill(nq, nk, nv, causal=True, return_lse=True)
        torch.cuda.synchronize()
        assert torch.equal(o, oe) and torch.equal(lse, le), f"replay differs (seed {seed})"
    assert cga.device_status() == 0


def test_decode_and_rope_graph_replay():
    cga = library()
    dev = device()
    cfg = workloads.CONFIGS["c4b"]
    q, kc, vc, sl = [t.to(dev) for t in workloads.config_decode_inputs(cfg, nan_fill=False)]
    B, Hq, Hkv, D, L = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.max_len
    assert cga.attn_reserve_workspace(B, Hq, Hkv, D, L) == 0
    o = torch.empty_like(q)
    g = _capture(lambda: cga.decode(q, kc, vc, sl, out=o))
    nq = torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    q.copy_(nq.to(dev))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, cga.decode(q, kc, vc, sl))
    # decode with RoPE: the replay rewrites the same cache rows with the same values
    gen = torch.Generator().manual_seed(6)
    kn = torch.randn((B, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
    vn = torch.randn((B, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
    inv = 10000.0 ** (-torch.arange(D // 2, dtype=torch.float64) * 2 / D)
    ang = torch.arange(L, dtype=torch.float64)[:, None] * inv[None, :]
    ct, st = ang.cos().float().to(dev), ang.sin().float().to(dev)
    o2 = torch.empty_like(q)
    g2 = _capture(lambda: cga.decode_rope(q, kn, vn, ct, st, kc, vc, sl, out=o2))
    kc_after, vc_after = kc.clone(), vc.clone()
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(kc, kc_after) and torch.equal(vc, vc_after)
    assert torch.equal(o2, cga.decode_rope(q, kn, vn, ct, st, kc, vc, sl))
    assert cga.device_status() == 0


def test_chunk_and_varlen_graph_replay():
    cga = library()
    dev = device()
    _, kc, vc, sl = [t.to(dev) for t in workloads.decode_inputs(4, 8, 2, 128, 1500, "explicit",
                                                                seed=7,
                                                                seqlens=[1500, 700, 64, 1000],
                                                                nan_fill=False)]
    q = workloads.prefill_inputs(4, 8, 2, 64, 128, "bf16", seed=8)[0].to(dev)
    o = torch.empty_like(q)
    g = _capture(lambda: cga.chunk(q, kc, vc, sl, out=o))
    q.copy_(workloads.prefill_inputs(4, 8, 2, 64, 128, "bf16", seed=9)[0].to(dev))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, cga.chunk(q, kc, vc, sl))
    qv, kv, vv = [t.to(dev) for t in workloads.prefill_inputs(3, 8, 2, 900, 128, "bf16", seed=10)]
    lens = torch.tensor([900, 1, 450], dtype=torch.int32, device=dev)
    ov = torch.empty_like(qv)
    g2 = _capture(lambda: cga.prefill_varlen(qv, kv, vv, lens, out=ov))
    lens.copy_(torch.tensor([300, 900, 0], dtype=torch.int32))
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(ov, cga.prefill_varlen(qv, kv, vv, lens))
    assert cga.device_status() == 0


def test_prefill_captured_before_scratch_grows_matches_eager():
    """A prefill captured with no warm-up, larger than any scratch the process has grown so far
    (V of B8 Hkv8 S8192 D128: 134 MB as fp16): the captured call cannot grow the scratch, so it
    converts V on chip; the eager call afterwards grows it and takes the fp16 copy. Both give
    the same bits."""
    cga = library()
    dev = device()
    B, Hq, Hkv, S, D = 8, 8, 8, 8192, 128
    g = torch.Generator(device=dev).manual_seed(12)
    q = torch.randn((B, Hq, S, D), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((B, Hkv, S, D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B, Hkv, S, D), generator=g, device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        cga.prefill(q, k, v, causal=True, out=o, lse=lse, return_lse=True)
    graph.replay()
    torch.cuda.synchronize()
    oe, le = cga.prefill(q, k, v, causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o, oe) and torch.equal(lse, le)
    assert cga.device_status() == 0
