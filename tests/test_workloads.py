"""Seeded input generators and work accounting (no GPU)."""
import os

import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split()
            out[k] = int(v)
    return out


def test_traffic_and_contraction_sizes_match_page_table():
    g = _golden("fusion_traffic_one_head_s512_d64.txt")
    t = workloads.unfused_intermediate_bytes(512, 64, heads=12, elem=4)
    assert t["S"] == g["s_matrix_bytes"] and t["P"] == g["p_matrix_bytes"]
    assert t["O"] == g["o_matrix_bytes"]
    assert 12 * t["S"] == g["twelve_head_s_bytes"]
    # flops = 2 per multiply-add, two contractions
    assert workloads.prefill_flops(1, 1, 512, 64, False) == 2 * (g["qk_multiply_adds"]
                                                                 + g["pv_multiply_adds"])


def test_causal_pairs():
    assert workloads.prefill_pairs(4, True) == 10 and workloads.prefill_pairs(4, False) == 16
    # configured work: B1 Hq8 S2048 D128 causal = 8.594 GFLOP
    assert workloads.prefill_flops(1, 8, 2048, 128, True) == 4 * 8 * 128 * 2048 * 2049 // 2


def test_inputs_are_seeded_and_rounded():
    q1, k1, v1 = workloads.prefill_inputs(1, 2, 1, 9, 8, "bf16", 3.0, seed=0)
    q2, k2, v2 = workloads.prefill_inputs(1, 2, 1, 9, 8, "bf16", 3.0, seed=0)
    assert q1.dtype == torch.bfloat16 and torch.equal(q1, q2) and torch.equal(v1, v2)
    g = torch.Generator("cpu").manual_seed(0)
    q = torch.randn((1, 2, 9, 8), generator=g) * 3.0
    assert torch.equal(q1, q.to(torch.bfloat16))
    q3, _, _ = workloads.prefill_inputs(1, 2, 1, 9, 8, "bf16", 3.0, seed=1)
    assert not torch.equal(q1, q3)


def test_decode_inputs_nan_beyond_length():
    q, kc, vc, sl = workloads.decode_inputs(4, 4, 2, 16, 300, "uniform", seed=0)
    assert sl.dtype == torch.int32 and sl.min() >= 256 and sl.max() <= 300
    for b in range(4):
        L = int(sl[b])
        assert torch.isnan(kc[b, :, L:].float()).all() and torch.isnan(vc[b, :, L:].float()).all()
        assert torch.isfinite(kc[b, :, :L].float()).all()
    cfg = workloads.CONFIGS["c4b"]
    _, _, _, sl = workloads.config_decode_inputs(cfg)
    assert sl.shape == (32,) and 256 <= int(sl.min()) and int(sl.max()) <= 4096
    nbytes = workloads.decode_bytes(sl.tolist(), 8, 2, 128)
    assert nbytes == int(sl.sum()) * 2 * 128 * 2 * 2 + 2 * 32 * 8 * 128 * 2
