"""The C-ABI library without a GPU: it builds, loads, exports every symbol the header declares,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gqa_attn.h")


@pytest.fixture(scope="module")
def lib():
    from causal_gqa_attention_gb300 import _lib, build

    build.build()
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*[\s\*]+([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n.startswith("attn_")))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("attn_prefill", "attn_decode", "attn_prefill_ex", "attn_decode_ex"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from causal_gqa_attention_gb300 import _lib

    names = _declared_functions()
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"
    import causal_gqa_attention_gb300 as cga

    for n in names:
        assert callable(getattr(cga, n)), f"binding lacks {n}"


def test_debug_build_exports_the_same_symbols(lib):
    """The debug build (device-side index checks) is the same library with the checks compiled
    in: it builds without a GPU, exports every declared symbol and says it is the debug build."""
    from causal_gqa_attention_gb300 import _lib, build

    dbg = _lib.load(build.build(debug=True))
    for n in _declared_functions():
        assert hasattr(dbg, n), f"debug build lacks {n}"
    assert dbg.attn_debug_build() == 1
    assert lib.attn_debug_build() == 0


def test_status_strings_and_version(lib):
    assert lib.attn_version() >= 100
    assert lib.attn_status_string(0) == b"ok"
    for code in range(1, 7):
        assert lib.attn_status_string(code) not in (b"ok", b"unknown status")


A16 = 1 << 20  # a 16-byte aligned fake device address; never dereferenced (rejected before)


@pytest.mark.parametrize("args,code", [
    # q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, in, out
    ((0, A16, A16, A16, None, 1, 8, 2, 1, 128, 0.1, 1, 1, 1), 1),   # NULL q
    ((A16, A16, A16, A16, None, 0, 8, 2, 1, 128, 0.1, 1, 1, 1), 1),  # B = 0
    ((A16, A16, A16, A16, None, 1, 0, 2, 1, 128, 0.1, 1, 1, 1), 1),  # S = 0
    ((A16, A16, A16, A16, None, 1, 8, 3, 2, 128, 0.1, 1, 1, 1), 1),  # Hq % Hkv
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 128, 0.0, 1, 1, 1), 1),  # scale 0
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 128, float("nan"), 1, 1, 1), 1),
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 128, 0.1, 1, 7, 1), 1),  # bad dtype
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 96, 0.1, 1, 1, 1), 2),   # bf16 needs D in {64, 128}
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 32, 0.1, 1, 1, 1), 2),
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 96, 0.1, 1, 0, 0), 2),   # fp32 D = 96
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 64, 0.1, 1, 0, 1), 2),   # fp32 in, bf16 out
    ((A16 + 8, A16, A16, A16, None, 1, 8, 2, 1, 128, 0.1, 1, 1, 1), 3),  # misaligned q
    ((A16, A16, A16, A16, A16 + 2, 1, 8, 2, 1, 128, 0.1, 1, 1, 1), 3),  # misaligned lse
])
def test_prefill_rejects_on_host(lib, args, code):
    assert lib.attn_prefill_ex(*args, None) == code


def _ll3(a, b, c):
    return (ctypes.c_longlong * 3)(a, b, c)


# every case is rejected before any CUDA call (the pointers are never dereferenced)
@pytest.mark.parametrize("strides,code", [
    ((None, (8, 8, 8), (8, 8, 8), (8, 8, 8)), 1),                     # NULL stride array
    (((1024, 132, 8), (8, 8, 8), (8, 8, 8), (8, 8, 8)), 3),           # q token stride 264 B
    (((1024, 128, 8), (8, 8, 4), (8, 8, 8), (8, 8, 8)), 3),           # k head stride 8 B
    (((1024, 128, 8), (8, 8, 8), (0, 8, 8), (8, 8, 8)), 3),           # v batch stride 0
    (((1024, 128, 8), (8, 8, 8), (8, 8, 8), (8, 8, -8)), 3),          # negative o stride
    (((1024, 128, 8), (8, 8, 8), (8, 8, 8), (8, 1 << 40, 8)), 3),     # huge o stride
])
def test_prefill_strided_rejects_on_host(lib, strides, code):
    arrs = [None if st is None else _ll3(*st) for st in strides]
    assert lib.attn_prefill_strided(A16, A16, A16, A16, None, 1, 8, 2, 1, 64, *arrs, 0.1, 1, 1,
                                    None) == code


@pytest.mark.parametrize("strides,code", [
    ((None, (8, 8, 8), (8, 8, 8), (8, 8, 8)), 1),                     # NULL stride array
    (((1024, 132, 8), (8, 8, 8), (8, 8, 8), (8, 8, 8)), 3),           # q token stride 264 B
    (((1024, 128, 8), (8, 8, 4), (8, 8, 8), (8, 8, 8)), 3),           # cache head stride 8 B
    (((1024, 128, 8), (8, 8, 8), (0, 8, 8), (8, 8, 8)), 3),           # cache batch stride 0
    (((1024, 128, 8), (8, 8, 8), (8, 8, 8), (8, 8, -8)), 3),          # negative o stride
])
def test_chunk_and_varlen_strided_reject_on_host(lib, strides, code):
    arrs = [None if st is None else _ll3(*st) for st in strides]
    # q, kc, vc, seqlens, o, lse, B, Sq, Hq, Hkv, D, max_len, strides x4, scale, causal, out
    assert lib.attn_chunk_strided(A16, A16, A16, A16, A16, None, 1, 8, 2, 1, 64, 64, *arrs, 0.1,
                                  1, 1, None) == code
    # q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D, strides x4, scale, causal, out
    assert lib.attn_prefill_varlen_strided(A16, A16, A16, A16, A16, None, 1, 8, 2, 1, 64, *arrs,
                                           0.1, 1, 1, None) == code


def test_prefill_strided_fp32_out_stride(lib):
    # an o token stride of 6 fp32 elements (24 B) is not a 16-byte multiple
    ok = _ll3(1024, 128, 8)
    assert lib.attn_prefill_strided(A16, A16, A16, A16, None, 1, 8, 2, 1, 64, ok, ok, ok,
                                    _ll3(1024, 6, 8), 0.1, 1, 0, None) == 3
    # unsupported head dim before strides are looked at
    assert lib.attn_prefill_strided(A16, A16, A16, A16, None, 1, 8, 2, 1, 96, ok, ok, ok, ok,
                                    0.1, 1, 1, None) == 2


@pytest.mark.parametrize("args,code", [
    # q, kc, vc, seqlens, o, lse, B, Hq, Hkv, D, max_len, scale, ws, ws_bytes, out
    ((A16, A16, A16, None, A16, None, 2, 8, 2, 128, 64, 0.1, None, 0, 1), 1),  # NULL seqlens
    ((A16, A16, A16, A16, A16, None, 2, 8, 3, 128, 64, 0.1, None, 0, 1), 1),   # Hq % Hkv
    ((A16, A16, A16, A16, A16, None, 2, 8, 2, 128, 0, 0.1, None, 0, 1), 1),    # max_len 0
    ((A16, A16, A16, A16, A16, None, 2, 8, 2, 128, 64, -1.0, None, 0, 1), 1),  # scale < 0
    ((A16, A16, A16, A16, A16, None, 2, 8, 2, 96, 64, 0.1, None, 0, 1), 2),    # D = 96
    ((A16, A16 + 4, A16, A16, A16, None, 2, 8, 2, 128, 64, 0.1, None, 0, 1), 3),
    ((A16, A16, A16, A16, A16, None, 2, 8, 2, 128, 64, 0.1, A16, 16, 1), 4),   # ws too small
])
def test_decode_rejects_on_host(lib, args, code):
    assert lib.attn_decode_ex(*args, None) == code


def test_decode_split_plan(lib):
    # at least ~3 blocks per SM of a 152-SM part, chunks of 64..512 keys
    assert lib.attn_decode_chunk_len(32, 2, 4096) == 512
    assert lib.attn_decode_chunk_len(1, 2, 4096) == 64
    assert lib.attn_decode_chunk_len(1, 2, 0) == 0
    for B, Hkv, L in [(1, 1, 1), (3, 2, 100), (64, 8, 32768), (1, 2, 32768)]:
        c = lib.attn_decode_chunk_len(B, Hkv, L)
        assert 64 <= c <= 512 and c & (c - 1) == 0
    # batches up to 1024: stream kernel, partials for 1824 warp slices x 4 heads + one per
    # (sequence, head); larger batches: one partial per (sequence, head, chunk)
    ws = lib.attn_decode_workspace_bytes(32, 8, 2, 128, 4096)
    assert ws == (1824 * 4 + 32 * 8) * (128 * 4 + 8)
    B = 2000
    c = lib.attn_decode_chunk_len(B, 2, 4096)
    assert lib.attn_decode_workspace_bytes(B, 8, 2, 128, 4096) == B * 8 * (4096 // c) * (128 * 4 + 8)
    assert lib.attn_decode_workspace_bytes(2, 3, 2, 128, 10) == 0


@pytest.mark.parametrize("args,code", [
    # q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, out, ws, ws_bytes
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 128, 0.1, 1, 1, A16 + 16, 1 << 20), 3),  # ws not 256-B aligned
    ((A16, A16, A16, A16, None, 1, 8, 3, 2, 128, 0.1, 1, 1, A16, 1 << 20), 1),       # Hq % Hkv
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 96, 0.1, 1, 1, A16, 1 << 20), 2),        # D = 96
    ((A16, A16, A16, A16, None, 1, 8, 2, 1, 128, 0.1, 1, 5, A16, 1 << 20), 1),       # out dtype
])
def test_prefill_ws_rejects_on_host(lib, args, code):
    assert lib.attn_prefill_ws(*args, None) == code


def test_prefill_workspace_bytes_invalid(lib):
    # invalid shapes return 0 before any device query
    assert lib.attn_prefill_workspace_bytes(1, 8, 3, 2, 128, 1) == 0
    assert lib.attn_prefill_workspace_bytes(1, 8, 2, 1, 96, 1) == 0
    assert lib.attn_prefill_workspace_bytes(0, 8, 2, 1, 128, 1) == 0
