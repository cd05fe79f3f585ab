"""ctypes declarations of the C ABI in ``include/gqa_attn.h`` (same names, same arguments).

Loading fails loudly when the CUDA library has not been built: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgqa_attn.so")
# the build with device-side index checks, used when GQA_ATTN_DEBUG=1 (built on first use)
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libgqa_attn_debug.so")

ATTN_OK = 0
ATTN_ERR_INVALID = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIGN = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_TIMEOUT = 6
ATTN_F32 = 0
ATTN_BF16 = 1
ATTN_DEV_SEQLEN_CLAMPED = 0x1
ATTN_DEV_WAIT_TIMEOUT = 0x2
ATTN_DEV_INDEX_CHECK = 0x4
ATTN_DECODE_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

# name -> (restype, argtypes); the order of the header
SIGNATURES = {
    "attn_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_prefill_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp]),
    "attn_prefill_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "attn_prefill_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz,
                             _vp]),
    "attn_prefill_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                                  _f, _i, _i, _vp]),
    "attn_prefill_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i,
                                 _vp]),
    "attn_chunk": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "attn_chunk_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                _vp, _vp, _f, _i, _i, _vp]),
    "attn_prefill_varlen_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                         _vp, _vp, _vp, _f, _i, _i, _vp]),
    "attn_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "attn_decode_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz, _i,
                            _vp]),
    "attn_decode_rope": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                              _i, _f, _i, _vp]),
    "attn_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "attn_decode_chunk_len": (_i, [_i, _i, _i]),
    "attn_reserve_workspace": (_i, [_i, _i, _i, _i, _i]),
    "attn_reserve_workspace_bytes": (_i, [_sz]),
    "attn_debug_set_wait_limit": (_i, [ctypes.c_longlong]),
    "attn_device_status": (_i, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "attn_status_string": (ctypes.c_char_p, [_i]),
    "attn_version": (_i, []),
    "attn_debug_build": (_i, []),
}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} (code {code})")


def debug_requested() -> bool:
    return os.environ.get("GQA_ATTN_DEBUG", "") == "1"


def load(path: str | None = None) -> ctypes.CDLL:
    """The loaded CUDA library. Raises if it has not been built (run ``build()``). With
    GQA_ATTN_DEBUG=1 in the environment this is the debug build (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if path is None and debug_requested():
                from causal_gqa_attention_gb300 import build as _build

                p = _build.build(debug=True)
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA library {p} is missing; build it with "
                    "causal_gqa_attention_gb300.build.build() (there is no fallback path)")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            if path is not None:
                return lib
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    try:
        return load().attn_status_string(code).decode()
    except RuntimeError:
        return f"status {code}"


def check(fn: str, code: int) -> None:
    if code != ATTN_OK:
        raise AttnError(fn, code)
