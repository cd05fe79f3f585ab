"""fp64 CPU oracle for the attention forward (prefill and decode, grouped-query heads).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers. The CUDA library under ``causal_gqa_attention_gb300`` does not
import this package, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over query rows); this module
compiles it with gcc on first use and marshals numpy arrays. Inputs of any float dtype
(including torch bf16 tensors) are widened exactly to float64 before the call.

Citations for each function are in ``oracle.c``. Summary:
  * ``prefill`` / ``decode``: S = Q K^T * scale, mask -> -inf, two-pass row softmax, O = P V,
    LSE = m + log l ("Attention three-op fusion", xdnf.cn/news/349386, sections 1.1, 3.2, 4.3;
    "CS336 Lecture 6", semidirectx.com, section 6; "triton-optimization" skill, section 3.5).
  * ``chunk``: Sq new queries against a cache, query i at position L_b - Sq + i ("Hand-written
    Triton decoder", m.nlpx.cn/news/28229, section 1.4; "Attention three-op fusion", section 4.3).
  * ``prefill_varlen``: a padded batch, padding rows see no key ("Attention three-op fusion",
    section 4.3).
  * ``rope`` / ``decode_rope``: rotate-half RoPE with cos/sin tables, the new key stored in the
    cache before attention ("triton-optimization" skill, section 3.4; "Hand-written Triton
    decoder", sections 1.2 and 2.2).
  * ``row_partial`` / ``merge`` / ``online_row``: the online-softmax recurrence and the merge
    of key-block partials ("Attention three-op fusion", sections 2.2, 2.3 and 4.4).
Every function is pinned to values the pages or the mathematics fix (tests/oracle_pins.py:
closed forms, brute force on tiny inputs, reductions of chunk and varlen to prefill and
decode, RoPE closed forms and composition, order-free merging).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (no fast-math: IEEE -inf is used)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.oracle_prefill_rows.restype = ctypes.c_int
    lib.oracle_prefill_rows.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                        _i64p, ctypes.c_int64, _dp, _dp, ctypes.c_int]
    lib.oracle_decode.restype = ctypes.c_int
    lib.oracle_decode.argtypes = [_dp, _dp, _dp, _i32p, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                  ctypes.c_int]
    lib.oracle_chunk.restype = ctypes.c_int
    lib.oracle_chunk.argtypes = [_dp, _dp, _dp, _i32p, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_prefill_varlen.restype = ctypes.c_int
    lib.oracle_prefill_varlen.argtypes = [_dp, _dp, _dp, _i32p, _dp, _dp, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_rope_rows.restype = None
    lib.oracle_rope_rows.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int]
    lib.oracle_row_partial.restype = None
    lib.oracle_row_partial.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                       _dp, _dp, _dp]
    lib.oracle_merge.restype = None
    lib.oracle_merge.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, _dp, _dp]
    lib.oracle_online_row.restype = None
    lib.oracle_online_row.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_int, _dp, _dp]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it if needed). ``path`` loads another build of the
    same source, e.g. a deliberately broken copy in a mutation test."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _f64(x) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array (torch tensors of any float dtype too)."""
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU without numpy bf16 support
        x = x.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def prefill(q, k, v, causal: bool, scale: float, rows=None, nthreads: int = 0, lib=None):
    """Attention forward for q [B,Hq,S,D], k/v [B,Hkv,S,D].

    Returns (o, lse): o [B,Hq,S,D] and lse [B,Hq,S] in float64, or, when ``rows`` (flat row ids
    (b*Hq + h)*S + i) is given, o [n,D] and lse [n] for those rows only."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, S, D) and v.shape == k.shape
    if rows is None:
        o = np.empty((B, Hq, S, D))
        lse = np.empty((B, Hq, S))
        rc = lib.oracle_prefill_rows(_p(q), _p(k), _p(v), B, S, Hq, Hkv, D, float(scale),
                                     int(bool(causal)), None, 0, _p(o), _p(lse), nthreads)
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.empty((r.size, D))
        lse = np.empty((r.size,))
        rc = lib.oracle_prefill_rows(_p(q), _p(k), _p(v), B, S, Hq, Hkv, D, float(scale),
                                     int(bool(causal)), r.ctypes.data_as(_i64p), r.size,
                                     _p(o), _p(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle_prefill_rows rejected its arguments")
    return o, lse


def decode(q, kcache, vcache, seqlens, scale: float, nthreads: int = 0, lib=None):
    """Single-token decode: q [B,Hq,D], caches [B,Hkv,max_len,D], seqlens [B] (int).

    Returns (o [B,Hq,D], lse [B,Hq]) in float64."""
    lib = lib or load()
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().to("cpu").numpy()
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    B, Hq, D = q.shape
    Hkv, max_len = kc.shape[1], kc.shape[2]
    assert kc.shape == (B, Hkv, max_len, D) and vc.shape == kc.shape and sl.shape == (B,)
    o = np.empty((B, Hq, D))
    lse = np.empty((B, Hq))
    rc = lib.oracle_decode(_p(q), _p(kc), _p(vc), sl.ctypes.data_as(_i32p), _p(o), _p(lse),
                           B, Hq, Hkv, D, max_len, float(scale), nthreads)
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return o, lse


def chunk(q, kcache, vcache, seqlens, scale: float, causal: bool = True, nthreads: int = 0,
          lib=None):
    """Sq new queries per sequence against a cache: q [B,Hq,Sq,D], caches [B,Hkv,max_len,D],
    seqlens [B]; query i of sequence b is at position seqlens[b] - Sq + i.
    Returns (o [B,Hq,Sq,D], lse [B,Hq,Sq]) in float64."""
    lib = lib or load()
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().to("cpu").numpy()
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    B, Hq, Sq, D = q.shape
    Hkv, max_len = kc.shape[1], kc.shape[2]
    assert kc.shape == (B, Hkv, max_len, D) and vc.shape == kc.shape and sl.shape == (B,)
    o = np.empty((B, Hq, Sq, D))
    lse = np.empty((B, Hq, Sq))
    rc = lib.oracle_chunk(_p(q), _p(kc), _p(vc), sl.ctypes.data_as(_i32p), _p(o), _p(lse), B, Sq,
                          Hq, Hkv, D, max_len, float(scale), int(bool(causal)), nthreads)
    if rc != 0:
        raise ValueError("oracle_chunk rejected its arguments")
    return o, lse


def prefill_varlen(q, k, v, seqlens, causal: bool, scale: float, nthreads: int = 0, lib=None):
    """Padded batch: q [B,Hq,S,D], k/v [B,Hkv,S,D], sequence b valid in its first seqlens[b]
    tokens; padding rows give O = 0, LSE = -inf. Returns (o, lse) in float64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().to("cpu").numpy()
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, S, D) and v.shape == k.shape and sl.shape == (B,)
    o = np.empty((B, Hq, S, D))
    lse = np.empty((B, Hq, S))
    rc = lib.oracle_prefill_varlen(_p(q), _p(k), _p(v), sl.ctypes.data_as(_i32p), _p(o), _p(lse),
                                   B, S, Hq, Hkv, D, float(scale), int(bool(causal)), nthreads)
    if rc != 0:
        raise ValueError("oracle_prefill_varlen rejected its arguments")
    return o, lse


def rope(x, cos_rows, sin_rows, lib=None):
    """Rotate-half RoPE of x [..., D] with per-row tables cos/sin [..., D/2] (same leading
    shape). fp64."""
    lib = lib or load()
    x = _f64(x)
    c = np.ascontiguousarray(np.broadcast_to(_f64(cos_rows), x.shape[:-1] + (x.shape[-1] // 2,)))
    sn = np.ascontiguousarray(np.broadcast_to(_f64(sin_rows), x.shape[:-1] + (x.shape[-1] // 2,)))
    out = np.empty_like(x)
    lib.oracle_rope_rows(_p(x), _p(c), _p(sn), _p(out), x.size // x.shape[-1], x.shape[-1])
    return out


def decode_rope(q, k_new, v_new, cos_tab, sin_tab, kcache, vcache, seqlens, scale: float,
                lib=None):
    """One decode step with the new token's RoPE and cache store: q [B,Hq,D] and k_new
    [B,Hkv,D] are rotated at position p = seqlens[b]-1 with tables cos/sin [max_len, D/2]; the
    rotated k (rounded to the cache's bf16) and v_new go to cache row p; then decode.
    Returns (o [B,Hq,D], lse [B,Hq], k_row [B,Hkv,D] as stored) in float64."""
    import torch

    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().to("cpu").numpy()
    sl = np.asarray(seqlens, dtype=np.int64)
    qd, kd = _f64(q), _f64(k_new)
    ct, st = _f64(cos_tab), _f64(sin_tab)
    B, Hq, D = qd.shape
    Hkv = kd.shape[1]
    pos = np.maximum(sl - 1, 0)
    q_rot = rope(qd, ct[pos][:, None, :], st[pos][:, None, :], lib=lib)
    k_rot = rope(kd, ct[pos][:, None, :], st[pos][:, None, :], lib=lib)
    k_store = torch.from_numpy(k_rot).to(torch.bfloat16).double().numpy()
    kc, vc = _f64(kcache).copy(), _f64(vcache).copy()
    for b in range(B):
        if sl[b] > 0:
            kc[b, :, pos[b]] = k_store[b]
            vc[b, :, pos[b]] = _f64(v_new)[b]
    o, lse = decode(q_rot, kc, vc, sl.astype(np.int32), scale, lib=lib)
    return o, lse, k_store


def row_partial(q_row, k_rows, v_rows, scale: float, lib=None):
    """Partial state (m, l, o_unnormalised[D]) of one query row over a block of keys."""
    lib = lib or load()
    q, k, v = _f64(q_row), _f64(k_rows), _f64(v_rows)
    n, D = k.shape
    m, l = ctypes.c_double(), ctypes.c_double()
    o = np.empty(D)
    lib.oracle_row_partial(_p(q), _p(k), _p(v), n, D, float(scale), ctypes.byref(m),
                           ctypes.byref(l), _p(o))
    return m.value, l.value, o


def merge(m, l, o_un, lib=None):
    """Merge block partials of one row (in the order given) -> (o [D], lse)."""
    lib = lib or load()
    m, l, o_un = _f64(m), _f64(l), _f64(o_un)
    nb, D = o_un.shape
    o = np.empty(D)
    lse = ctypes.c_double()
    lib.oracle_merge(_p(m), _p(l), _p(o_un), nb, D, _p(o), ctypes.byref(lse))
    return o, lse.value


def online_row(q_row, k_rows, v_rows, scale: float, block: int, lib=None):
    """The online-softmax recurrence over key blocks of size ``block`` -> (o [D], lse)."""
    lib = lib or load()
    q, k, v = _f64(q_row), _f64(k_rows), _f64(v_rows)
    n, D = k.shape
    o = np.empty(D)
    lse = ctypes.c_double()
    lib.oracle_online_row(_p(q), _p(k), _p(v), n, D, float(scale), int(block), _p(o),
                          ctypes.byref(lse))
    return o, lse.value
