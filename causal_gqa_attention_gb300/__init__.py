"""Fused causal GQA attention forward for GB300 (sm_103a): prefill and split-KV decode.

Two layers, both argument marshalling only (every step of the computation runs in the CUDA
library built from ``csrc/``):

* ``attn_prefill``, ``attn_prefill_ex``, ``attn_decode``, ``attn_decode_ex``, ... -- the C ABI of
  ``include/gqa_attn.h`` under the same names, taking raw device pointers (ints) and sizes;
  they return the C status code.
* ``prefill(q, k, v, ...)`` and ``decode(q, kcache, vcache, seqlens, ...)`` -- the same calls on
  torch CUDA tensors: shape/dtype checks, output allocation, the current torch stream; they
  raise ``AttnError`` on a non-zero status.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import math

from . import _lib
from ._lib import (ATTN_BF16, ATTN_DEV_INDEX_CHECK, ATTN_DEV_SEQLEN_CLAMPED, ATTN_DEV_WAIT_TIMEOUT,
                   ATTN_ERR_ALIGN,
                   ATTN_ERR_CUDA, ATTN_ERR_INVALID, ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED,
                   ATTN_ERR_WORKSPACE, ATTN_F32, ATTN_OK, AttnError)

__all__ = [
    "attn_prefill", "attn_prefill_ex", "attn_prefill_ws", "attn_prefill_workspace_bytes",
    "attn_reserve_workspace_bytes", "attn_prefill_strided", "attn_prefill_varlen",
    "attn_prefill_varlen_strided", "prefill_varlen", "attn_chunk", "attn_chunk_strided",
    "attn_decode", "attn_decode_ex",
    "attn_decode_noalloc", "chunk", "attn_decode_rope", "decode_rope",
    "attn_decode_workspace_bytes", "attn_decode_chunk_len", "attn_reserve_workspace",
    "attn_device_status", "attn_debug_set_wait_limit", "attn_status_string", "attn_version",
    "attn_debug_build", "prefill", "decode",
    "device_status", "AttnError", "ATTN_OK", "ATTN_ERR_INVALID", "ATTN_ERR_UNSUPPORTED",
    "ATTN_ERR_ALIGN", "ATTN_ERR_WORKSPACE", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_F32",
    "ATTN_BF16", "ATTN_DEV_SEQLEN_CLAMPED", "ATTN_DEV_WAIT_TIMEOUT", "ATTN_DEV_INDEX_CHECK",
    "load_library",
]


def load_library():
    return _lib.load()


# ------------------------------------------------------------------ C ABI, same names


def attn_prefill(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, stream):
    return _lib.load().attn_prefill(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, stream)


def attn_prefill_ex(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, in_dtype, out_dtype,
                    stream):
    return _lib.load().attn_prefill_ex(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal,
                                       in_dtype, out_dtype, stream)


def attn_prefill_ws(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, out_dtype, workspace,
                    workspace_bytes, stream):
    return _lib.load().attn_prefill_ws(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal,
                                       out_dtype, workspace, workspace_bytes, stream)


def attn_prefill_workspace_bytes(B, S, Hq, Hkv, D, causal):
    return _lib.load().attn_prefill_workspace_bytes(B, S, Hq, Hkv, D, causal)


def attn_reserve_workspace_bytes(nbytes):
    return _lib.load().attn_reserve_workspace_bytes(nbytes)


def attn_prefill_strided(q, k, v, o, lse, B, S, Hq, Hkv, D, q_strides, k_strides, v_strides,
                         o_strides, scale, causal, out_dtype, stream):
    return _lib.load().attn_prefill_strided(q, k, v, o, lse, B, S, Hq, Hkv, D, q_strides,
                                            k_strides, v_strides, o_strides, scale, causal,
                                            out_dtype, stream)


def attn_prefill_varlen(q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D, scale, causal, out_dtype,
                        stream):
    return _lib.load().attn_prefill_varlen(q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D, scale,
                                           causal, out_dtype, stream)


def attn_chunk(q, kcache, vcache, seqlens, o, lse, B, Sq, Hq, Hkv, D, max_len, scale, causal,
               out_dtype, stream):
    return _lib.load().attn_chunk(q, kcache, vcache, seqlens, o, lse, B, Sq, Hq, Hkv, D, max_len,
                                  scale, causal, out_dtype, stream)


def attn_chunk_strided(q, kcache, vcache, seqlens, o, lse, B, Sq, Hq, Hkv, D, max_len, q_strides,
                       k_strides, v_strides, o_strides, scale, causal, out_dtype, stream):
    return _lib.load().attn_chunk_strided(q, kcache, vcache, seqlens, o, lse, B, Sq, Hq, Hkv, D,
                                          max_len, q_strides, k_strides, v_strides, o_strides,
                                          scale, causal, out_dtype, stream)


def attn_prefill_varlen_strided(q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D, q_strides,
                                k_strides, v_strides, o_strides, scale, causal, out_dtype,
                                stream):
    return _lib.load().attn_prefill_varlen_strided(q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D,
                                                   q_strides, k_strides, v_strides, o_strides,
                                                   scale, causal, out_dtype, stream)


def attn_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, D, max_len, scale, stream):
    return _lib.load().attn_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, D, max_len, scale,
                                   stream)


def attn_decode_ex(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, D, max_len, scale, workspace,
                   workspace_bytes, out_dtype, stream):
    return _lib.load().attn_decode_ex(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, D, max_len,
                                      scale, workspace, workspace_bytes, out_dtype, stream)


def attn_decode_rope(q, k_new, v_new, cos_t, sin_t, kcache, vcache, seqlens, o, lse, B, Hq, Hkv,
                     D, max_len, scale, out_dtype, stream):
    return _lib.load().attn_decode_rope(q, k_new, v_new, cos_t, sin_t, kcache, vcache, seqlens, o,
                                        lse, B, Hq, Hkv, D, max_len, scale, out_dtype, stream)


def attn_decode_noalloc(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, D, max_len, scale,
                        out_dtype, stream):
    """Decode that allocates nothing: scratch is a fixed array inside the library (for callers
    that cannot call cudaMalloc). Raw pointers; returns the C status code."""
    return _lib.load().attn_decode_noalloc(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, D,
                                           max_len, scale, out_dtype, stream)


def attn_decode_workspace_bytes(B, Hq, Hkv, D, max_len):
    return _lib.load().attn_decode_workspace_bytes(B, Hq, Hkv, D, max_len)


def attn_decode_chunk_len(B, Hkv, max_len):
    return _lib.load().attn_decode_chunk_len(B, Hkv, max_len)


def attn_reserve_workspace(B, Hq, Hkv, D, max_len):
    return _lib.load().attn_reserve_workspace(B, Hq, Hkv, D, max_len)


def attn_debug_set_wait_limit(cycles):
    return _lib.load().attn_debug_set_wait_limit(cycles)


def attn_device_status(stream, status_ptr):
    return _lib.load().attn_device_status(stream, status_ptr)


def attn_status_string(code):
    return _lib.load().attn_status_string(code).decode()


def attn_version():
    return _lib.load().attn_version()


def attn_debug_build():
    return _lib.load().attn_debug_build()


# ------------------------------------------------------------------ torch tensor front end


def _torch():
    import torch

    return torch


def _stream_handle(device):
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_cuda(name, t, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _bshd_strides(t):
    """Element strides {batch, token, head} of a [B, H, S, D] view (head dim contiguous); a
    dimension of extent 1 gets a nominal stride (it is never stepped)."""
    import ctypes

    sb, sh, ss = t.stride(0), t.stride(1), t.stride(2)
    if t.shape[0] == 1:
        sb = 8
    if t.shape[1] == 1:
        sh = 8
    if t.shape[2] == 1:
        ss = 8
    return (ctypes.c_longlong * 3)(sb, ss, sh)


def _check_view(name, t, dtype):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError(f"{name} must be a 4-D view with a contiguous last dim")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def prefill(q, k, v, causal: bool = True, scale: float | None = None, out_dtype=None,
            return_lse: bool = False, out=None, lse=None, workspace=None):
    """Attention forward with q_len = kv_len.

    q [B,Hq,S,D], k/v [B,Hkv,S,D], all bf16 (tensor-core path, D in {64,128}) or all fp32 (fp32
    CUDA-core path, D in {64,128}). ``out_dtype`` defaults to the input dtype (bf16 inputs may
    ask for fp32 output: the result before the final rounding). Returns o, or (o, lse) with
    lse [B,Hq,S] fp32 (natural log).

    bf16 q, k, v (and ``out``) may be views with any strides as long as the head dim is
    contiguous, e.g. ``x.transpose(1, 2)`` of a [B,S,H,D] tensor, or head slices of a fused QKV
    projection output viewed as [B,S,Hq+2Hkv,D]: they are read and written in place.

    ``workspace``: optional uint8 CUDA tensor (contiguous bf16 operands only) used as the call's
    scratch instead of the library-owned buffer, so prefills on different streams can overlap;
    ``attn_prefill_workspace_bytes`` gives the size that holds everything."""
    torch = _torch()
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, S, D) or v.shape != k.shape:
        raise ValueError(f"k/v shape {tuple(k.shape)}/{tuple(v.shape)} do not match q {tuple(q.shape)}")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q/k/v must be bf16 or fp32")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, S, D), dtype=out_dtype, device=q.device)
    elif out.shape != (B, Hq, S, D):
        raise ValueError(f"out must be [B,Hq,S,D], got {tuple(out.shape)}")
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out_t = ATTN_BF16 if out_dtype == torch.bfloat16 else ATTN_F32
    views = (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype), ("out", out, out_dtype))
    if q.dtype == torch.bfloat16 and not all(t.is_contiguous() for _, t, _ in views):
        if workspace is not None:
            raise ValueError("a workspace needs contiguous q, k, v and out")
        for n, t, dt in views:
            _check_view(n, t, dt)
        with torch.cuda.device(q.device):
            rc = attn_prefill_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, Hq,
                                      Hkv, D, _bshd_strides(q), _bshd_strides(k),
                                      _bshd_strides(v), _bshd_strides(out), float(scale),
                                      int(bool(causal)), out_t, _stream_handle(q.device))
        _lib.check("attn_prefill_strided", rc)
        return (out, lse) if return_lse else out
    for n, t, dt in views:
        _check_cuda(n, t, dt)
    if workspace is not None:
        if q.dtype != torch.bfloat16:
            raise ValueError("a workspace applies to bf16 inputs only")
        _check_cuda("workspace", workspace)
        with torch.cuda.device(q.device):
            rc = attn_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, Hq, Hkv,
                                 D, float(scale), int(bool(causal)), out_t, workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_handle(q.device))
        _lib.check("attn_prefill_ws", rc)
        return (out, lse) if return_lse else out
    in_t = ATTN_BF16 if q.dtype == torch.bfloat16 else ATTN_F32
    with torch.cuda.device(q.device):
        rc = attn_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, Hq, Hkv, D,
                             float(scale), int(bool(causal)), in_t, out_t,
                             _stream_handle(q.device))
    _lib.check("attn_prefill_ex", rc)
    return (out, lse) if return_lse else out


def chunk(q, kcache, vcache, seqlens, causal: bool = True, scale: float | None = None,
          out_dtype=None, return_lse: bool = False, out=None, lse=None):
    """Sq new queries per sequence against a bf16 KV cache: q [B,Hq,Sq,D] bf16 (the last Sq
    tokens of each sequence, already in the cache), caches [B,Hkv,max_len,D] bf16, seqlens [B]
    int32 on the device. Query i of sequence b sits at position seqlens[b] - Sq + i.
    Returns o [B,Hq,Sq,D] (bf16 by default), or (o, lse [B,Hq,Sq]).

    q, the caches and ``out`` may be views with any strides whose head dim is contiguous, e.g.
    caches stored [B,max_len,Hkv,D] and passed as ``cache.transpose(1, 2)``."""
    torch = _torch()
    B, Hq, Sq, D = q.shape
    Hkv, max_len = kcache.shape[1], kcache.shape[2]
    if kcache.shape != (B, Hkv, max_len, D) or vcache.shape != kcache.shape:
        raise ValueError("cache shapes do not match q")
    _check_cuda("seqlens", seqlens, torch.int32)
    if seqlens.shape != (B,):
        raise ValueError("seqlens must be [B]")
    out_dtype = out_dtype or torch.bfloat16
    if out is None:
        out = torch.empty((B, Hq, Sq, D), dtype=out_dtype, device=q.device)
    elif out.shape != (B, Hq, Sq, D):
        raise ValueError(f"out must be [B,Hq,Sq,D], got {tuple(out.shape)}")
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out_t = ATTN_BF16 if out_dtype == torch.bfloat16 else ATTN_F32
    views = (("q", q, torch.bfloat16), ("kcache", kcache, torch.bfloat16),
             ("vcache", vcache, torch.bfloat16), ("out", out, out_dtype))
    if not all(t.is_contiguous() for _, t, _ in views):
        for n, t, dt in views:
            _check_view(n, t, dt)
        with torch.cuda.device(q.device):
            rc = attn_chunk_strided(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens),
                                    _ptr(out), _ptr(lse), B, Sq, Hq, Hkv, D, max_len,
                                    _bshd_strides(q), _bshd_strides(kcache),
                                    _bshd_strides(vcache), _bshd_strides(out), float(scale),
                                    int(bool(causal)), out_t, _stream_handle(q.device))
        _lib.check("attn_chunk_strided", rc)
        return (out, lse) if return_lse else out
    for n, t, dt in views:
        _check_cuda(n, t, dt)
    with torch.cuda.device(q.device):
        rc = attn_chunk(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(out), _ptr(lse),
                        B, Sq, Hq, Hkv, D, max_len, float(scale), int(bool(causal)), out_t,
                        _stream_handle(q.device))
    _lib.check("attn_chunk", rc)
    return (out, lse) if return_lse else out


def prefill_varlen(q, k, v, seqlens, causal: bool = True, scale: float | None = None,
                   out_dtype=None, return_lse: bool = False, out=None, lse=None):
    """Padded batch: q [B,Hq,S,D], k/v [B,Hkv,S,D] bf16, sequence b valid in its first seqlens[b]
    tokens (seqlens int32 on the device). Padding rows give o = 0 (lse = -inf).

    q, k, v and ``out`` may be views with any strides whose head dim is contiguous (e.g. head
    slices of a padded fused QKV projection output)."""
    torch = _torch()
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, S, D) or v.shape != k.shape:
        raise ValueError("k/v shapes do not match q")
    _check_cuda("seqlens", seqlens, torch.int32)
    if seqlens.shape != (B,):
        raise ValueError("seqlens must be [B]")
    out_dtype = out_dtype or torch.bfloat16
    if out is None:
        out = torch.empty((B, Hq, S, D), dtype=out_dtype, device=q.device)
    elif out.shape != (B, Hq, S, D):
        raise ValueError(f"out must be [B,Hq,S,D], got {tuple(out.shape)}")
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out_t = ATTN_BF16 if out_dtype == torch.bfloat16 else ATTN_F32
    views = (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
             ("out", out, out_dtype))
    if not all(t.is_contiguous() for _, t, _ in views):
        for n, t, dt in views:
            _check_view(n, t, dt)
        with torch.cuda.device(q.device):
            rc = attn_prefill_varlen_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(seqlens), _ptr(out),
                                             _ptr(lse), B, S, Hq, Hkv, D, _bshd_strides(q),
                                             _bshd_strides(k), _bshd_strides(v),
                                             _bshd_strides(out), float(scale),
                                             int(bool(causal)), out_t, _stream_handle(q.device))
        _lib.check("attn_prefill_varlen_strided", rc)
        return (out, lse) if return_lse else out
    for n, t, dt in views:
        _check_cuda(n, t, dt)
    with torch.cuda.device(q.device):
        rc = attn_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(seqlens), _ptr(out), _ptr(lse), B,
                                 S, Hq, Hkv, D, float(scale), int(bool(causal)), out_t,
                                 _stream_handle(q.device))
    _lib.check("attn_prefill_varlen", rc)
    return (out, lse) if return_lse else out


def decode(q, kcache, vcache, seqlens, scale: float | None = None, out_dtype=None,
           return_lse: bool = False, workspace=None, out=None, lse=None):
    """One query token per sequence: q [B,Hq,D] bf16, caches [B,Hkv,max_len,D] bf16, seqlens
    [B] int32 on the device. Returns o [B,Hq,D] (bf16 by default), or (o, lse [B,Hq]).

    ``workspace``: optional uint8 CUDA tensor of at least ``attn_decode_workspace_bytes``;
    without it the library-owned per-device buffer is used."""
    torch = _torch()
    B, Hq, D = q.shape
    Hkv, max_len = kcache.shape[1], kcache.shape[2]
    if kcache.shape != (B, Hkv, max_len, D) or vcache.shape != kcache.shape:
        raise ValueError("cache shapes do not match q")
    _check_cuda("q", q, torch.bfloat16)
    _check_cuda("kcache", kcache, torch.bfloat16)
    _check_cuda("vcache", vcache, torch.bfloat16)
    _check_cuda("seqlens", seqlens, torch.int32)
    if seqlens.shape != (B,):
        raise ValueError("seqlens must be [B]")
    out_dtype = out_dtype or torch.bfloat16
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    else:
        _check_cuda("out", out, out_dtype)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _check_cuda("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    out_t = ATTN_BF16 if out_dtype == torch.bfloat16 else ATTN_F32
    with torch.cuda.device(q.device):
        rc = attn_decode_ex(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(out),
                            _ptr(lse), B, Hq, Hkv, D, max_len, float(scale), ws_ptr, ws_bytes,
                            out_t, _stream_handle(q.device))
    _lib.check("attn_decode_ex", rc)
    return (out, lse) if return_lse else out


def decode_rope(q, k_new, v_new, cos_t, sin_t, kcache, vcache, seqlens,
                scale: float | None = None, out_dtype=None, return_lse: bool = False, out=None,
                lse=None):
    """Decode step with the new token's RoPE and cache store: q [B,Hq,D], k_new/v_new [B,Hkv,D]
    bf16 (not rotated), cos_t/sin_t [max_len, D/2] fp32, caches [B,Hkv,max_len,D] bf16 (row
    seqlens[b]-1 is written), seqlens [B] int32 (device, including the new token)."""
    torch = _torch()
    B, Hq, D = q.shape
    Hkv, max_len = kcache.shape[1], kcache.shape[2]
    if kcache.shape != (B, Hkv, max_len, D) or vcache.shape != kcache.shape:
        raise ValueError("cache shapes do not match q")
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    if cos_t.shape != (max_len, D // 2) or sin_t.shape != cos_t.shape:
        raise ValueError("cos/sin tables must be [max_len, D/2]")
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("kcache", kcache),
                 ("vcache", vcache)):
        _check_cuda(n, t, torch.bfloat16)
    _check_cuda("cos_t", cos_t, torch.float32)
    _check_cuda("sin_t", sin_t, torch.float32)
    _check_cuda("seqlens", seqlens, torch.int32)
    out_dtype = out_dtype or torch.bfloat16
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out_t = ATTN_BF16 if out_dtype == torch.bfloat16 else ATTN_F32
    with torch.cuda.device(q.device):
        rc = attn_decode_rope(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cos_t), _ptr(sin_t),
                              _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(out), _ptr(lse), B,
                              Hq, Hkv, D, max_len, float(scale), out_t, _stream_handle(q.device))
    _lib.check("attn_decode_rope", rc)
    return (out, lse) if return_lse else out


def device_status(device=None) -> int:
    """Synchronise the current stream, then read and clear the device status word."""
    import ctypes

    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    st = ctypes.c_uint(0)
    with torch.cuda.device(dev):
        rc = attn_device_status(_stream_handle(dev), ctypes.byref(st))
    _lib.check("attn_device_status", rc)
    return st.value
