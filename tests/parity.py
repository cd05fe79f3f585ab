"""Helpers shared by the GPU parity tests: the device, the library, and the acceptance checks.

Tolerances (from the contract of the library, written out here):
  * fp32 inputs and output:                    max |o - o_ref| <= 1e-5
  * bf16 inputs, fp32 output (before rounding): max |o - o_ref| <= 4e-3
  * bf16 inputs, bf16 output:                  |o - o_ref| <= ulp_bf16(o_ref) + 4e-3
  * LSE (natural log):                         max |lse - lse_ref| <= 1e-4
where ulp_bf16(x) = 2^(floor(log2 |x|) - 7), the spacing of bf16 numbers at x.

The bounds are stated for standard-normal inputs. O is linear in V, so for V = c * V0 (V0
standard normal) the absolute bounds scale with c: ``check_out(..., scale=c)`` multiplies the
4e-3 terms by c (the ulp term is already relative to o_ref). The LSE does not depend on V.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

TOL_F32 = 1e-5
TOL_BF16_PRE = 4e-3
TOL_BF16_ABS = 4e-3
TOL_LSE = 1e-4


def device() -> torch.device:
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    return torch.device("cuda", 0)


def library():
    from causal_gqa_attention_gb300 import build

    build.build()
    import causal_gqa_attention_gb300 as cga

    cga.load_library()
    return cga


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 7), 0.0)


def to64(t) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def check_out(o_gpu, o_ref, kind: str, what: str, scale: float = 1.0):
    """kind: 'f32' | 'bf16_pre' | 'bf16'. scale: the factor c of V = c * V0 (see above)."""
    o = to64(o_gpu)
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    if kind == "f32":
        bad = err > TOL_F32 * scale
    elif kind == "bf16_pre":
        bad = err > TOL_BF16_PRE * scale
    else:
        bad = err > bf16_ulp(o_ref) + TOL_BF16_ABS * scale
    if bad.any():
        idx = np.unravel_index(np.argmax(err), err.shape)
        pytest.fail(f"{what}: {int(bad.sum())} of {err.size} outside tolerance; max err "
                    f"{err.max():.3e} at {idx} (gpu {o[idx]:.6f}, ref {o_ref[idx]:.6f})")
    return float(err.max())


def check_lse(lse_gpu, lse_ref, what: str):
    l = to64(lse_gpu)
    assert l.shape == lse_ref.shape
    both_ninf = np.isneginf(l) & np.isneginf(lse_ref)
    with np.errstate(invalid="ignore"):  # -inf - -inf where both are empty rows
        err = np.where(both_ninf, 0.0, np.abs(l - lse_ref))
    assert np.isfinite(err).all(), f"{what}: non-finite lse error"
    assert err.max() <= TOL_LSE, f"{what}: lse max err {err.max():.3e}"
    return float(err.max())


def sampled_rows(B: int, H: int, S: int, every: int = 64, tail: int = 128) -> np.ndarray:
    """Flat row ids (b*H + h)*S + i: every `every`-th row and the last `tail` rows per head."""
    rows = np.unique(np.concatenate([np.arange(0, S, every), np.arange(max(0, S - tail), S)]))
    heads = np.arange(B * H, dtype=np.int64)[:, None] * S
    return (heads + rows[None, :]).reshape(-1)
