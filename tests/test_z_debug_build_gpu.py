"""The debug build of the library (device-side index checks, selected by GQA_ATTN_DEBUG=1):
the prefill, chunk, varlen, decode and RoPE-decode parity tests run against it in a child
process, and after each of them no index check may have failed (the conftest fixture reads the
device status word). The child builds the debug library on first use."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

FILES = ["tests/test_prefill_gpu.py", "tests/test_layout_gpu.py", "tests/test_chunk_gpu.py",
         "tests/test_varlen_gpu.py", "tests/test_decode_gpu.py", "tests/test_rope_gpu.py"]


def _child(args, timeout):
    env = dict(os.environ, GQA_ATTN_DEBUG="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=timeout)


@pytest.mark.gpu
def test_debug_build_is_the_one_loaded():
    r = _child(["-c", "import causal_gqa_attention_gb300 as c; "
                      "assert c.attn_debug_build() == 1; print('debug')"], 900)
    assert r.returncode == 0 and "debug" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.gpu
def test_parity_suites_pass_on_the_debug_build():
    r = _child(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *FILES], 1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
