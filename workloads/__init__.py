"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module draws random inputs and counts algorithmic work. It holds none of the attention
arithmetic: both the CUDA path and the oracle receive the tensors made here.

Input recipe (every config):
  * ``torch.Generator('cpu').manual_seed(seed)``, seed 0 unless a test says otherwise;
  * draw order: per-sequence lengths (batched decode only: ``randint(256, 4097)``, both ends
    inclusive), then q, k, v as standard-normal fp32 in [B, H, S, D] order (decode: q [B,Hq,D],
    k/v caches [B,Hkv,max_len,D]);
  * q is multiplied by ``q_mult`` in fp32 (3 for the peaky-softmax config), then every tensor
    is rounded once to the compute dtype (bf16 round-to-nearest-even, or kept fp32);
  * decode caches: rows at or beyond a sequence's length are set to NaN, so any read of them
    would poison the result.

Shapes follow the pages: 12 heads, head dim 64, S 128..2048 ("Attention three-op fusion",
xdnf.cn/news/349386, section 5.1) and Hq 8 / Hkv 2 / head dim 128 / contexts up to 32768
("Hand-written Triton decoder", m.nlpx.cn/news/28229, section 2.1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    dtype: str  # "f32" or "bf16"
    causal: tuple = (True,)
    q_mult: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    max_len: int
    lens: str = "full"  # "full": every sequence is max_len long; "uniform": randint(256, max_len]
    dtype: str = "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


CONFIGS = {
    "c1": PrefillConfig("c1_b1_h1_s128_d64_f32_causal", 1, 1, 1, 128, 64, "f32", (True,)),
    "c2": PrefillConfig("c2_b1_h12_s512_d64_f32", 1, 12, 12, 512, 64, "f32", (False, True)),
    "c3": PrefillConfig("c3_b1_hq8_hkv2_s2048_d128_bf16_causal_qx3", 1, 8, 2, 2048, 128, "bf16",
                        (True,), 3.0),
    "c4a": DecodeConfig("c4a_decode_b1_l4096_hq8_hkv2_d128_bf16", 1, 8, 2, 128, 4096, "full"),
    "c4b": DecodeConfig("c4b_decode_b32_l256to4096_hq8_hkv2_d128_bf16", 32, 8, 2, 128, 4096,
                        "uniform"),
    "c5a": PrefillConfig("c5a_b1_hq8_hkv2_s32768_d128_bf16_causal", 1, 8, 2, 32768, 128, "bf16"),
    "c5b": PrefillConfig("c5b_b8_hq8_hkv2_s8192_d128_bf16_causal", 8, 8, 2, 8192, 128, "bf16"),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def prefill_inputs(B, Hq, Hkv, S, D, dtype="bf16", q_mult=1.0, seed=0):
    """(q, k, v) CPU tensors: q [B,Hq,S,D], k/v [B,Hkv,S,D] in ``dtype``."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((B, Hq, S, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, S, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, S, D), generator=g, dtype=torch.float32)
    if q_mult != 1.0:
        q = q * q_mult
    dt = torch_dtype(dtype)
    return q.to(dt), k.to(dt), v.to(dt)


def decode_lengths(B, max_len, lens="uniform", g=None, lo=256):
    if lens == "full":
        return torch.full((B,), max_len, dtype=torch.int32)
    if lens == "uniform":
        return torch.randint(min(lo, max_len), max_len + 1, (B,), generator=g, dtype=torch.int32)
    raise ValueError(lens)


def decode_inputs(B, Hq, Hkv, D, max_len, lens="uniform", dtype="bf16", seed=0, seqlens=None,
                  nan_fill=True):
    """(q [B,Hq,D], kcache, vcache [B,Hkv,max_len,D], seqlens int32 [B]) on the CPU.

    ``seqlens`` overrides the drawn lengths (still drawn first so the stream is unchanged)."""
    g = torch.Generator("cpu").manual_seed(seed)
    drawn = decode_lengths(B, max_len, lens, g) if lens != "explicit" else None
    sl = torch.as_tensor(seqlens, dtype=torch.int32) if seqlens is not None else drawn
    q = torch.randn((B, Hq, D), generator=g, dtype=torch.float32)
    kc = torch.randn((B, Hkv, max_len, D), generator=g, dtype=torch.float32)
    vc = torch.randn((B, Hkv, max_len, D), generator=g, dtype=torch.float32)
    if nan_fill:
        pos = torch.arange(max_len).view(1, 1, max_len, 1)
        dead = pos >= sl.view(B, 1, 1, 1).long()
        kc = kc.masked_fill(dead, float("nan"))
        vc = vc.masked_fill(dead, float("nan"))
    dt = torch_dtype(dtype)
    return q.to(dt), kc.to(dt), vc.to(dt), sl


def config_prefill_inputs(cfg: PrefillConfig, seed=0):
    return prefill_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.S, cfg.D, cfg.dtype, cfg.q_mult, seed)


def config_decode_inputs(cfg: DecodeConfig, seed=0, nan_fill=True):
    return decode_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.max_len, cfg.lens, cfg.dtype, seed,
                         nan_fill=nan_fill)


# ---------------------------------------------------------------- algorithmic work accounting

def prefill_pairs(S: int, causal: bool) -> int:
    """(query, key) pairs scored per head: S^2, or S(S+1)/2 with the causal mask."""
    return S * (S + 1) // 2 if causal else S * S


def prefill_flops(B, Hq, S, D, causal) -> int:
    """Two contractions (Q K^T and P V), 2 flops per multiply-add, D per pair each."""
    return 4 * B * Hq * D * prefill_pairs(S, causal)


def decode_bytes(seqlens, Hq, Hkv, D, elem=2, lse=False) -> int:
    """Bytes a decode step must move: every valid K and V row once, q in, o out (+ fp32 LSE)."""
    total_len = int(sum(int(x) for x in seqlens))
    B = len(seqlens)
    kv = total_len * Hkv * D * elem * 2
    qo = 2 * B * Hq * D * elem
    return kv + qo + (4 * B * Hq if lse else 0)


def unfused_intermediate_bytes(S: int, D: int, heads: int, elem: int = 4) -> dict:
    """Traffic of the separate three-kernel chain the fused kernel removes: S and P (S x S each)
    written once and read once, O (S x D) written once; per head and for ``heads`` heads."""
    s_bytes = S * S * elem
    per_head = 2 * s_bytes + 2 * s_bytes + S * D * elem
    return {"S": s_bytes, "P": s_bytes, "O": S * D * elem, "per_head": per_head,
            "all_heads": per_head * heads}
