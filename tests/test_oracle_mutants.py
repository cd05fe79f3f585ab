"""Mutation check of the oracle's pins (no GPU).

Each case plants one plausible mistake in a copy of the oracle's C source, builds it, and
requires that at least one pin fails on the broken copy. The committed oracle is untouched.
"""
import importlib.util
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("scale_dropped", "s[j] = scale * dot;\n    }\n    /* pass 1", "s[j] = dot;\n    }\n    /* pass 1"),
    ("partial_scale_dropped", "s[j] = scale * dot;\n        if (s[j] > m) m = s[j];",
     "s[j] = dot;\n        if (s[j] > m) m = s[j];"),
    ("causal_off_by_one", "vis[j] = causal ? (j <= i) : 1;", "vis[j] = causal ? (j < i) : 1;"),
    ("causal_wrong_side", "vis[j] = causal ? (j <= i) : 1;", "vis[j] = causal ? (j >= i) : 1;"),
    # "CS336 Lecture 6", exercise 3: a mask filled with 0 instead of -inf adds e^0 terms
    ("mask_fill_zero", "if (!visible[j]) { s[j] = -INFINITY; continue; }",
     "if (!visible[j]) { s[j] = 0.0; continue; }"),
    ("gqa_modulo_mapping", "const int g = h / G; /* contiguous", "const int g = h % Hkv; /*"),
    ("exp_sign_flipped", "s[j] = exp(s[j] - m); l += s[j];", "s[j] = exp(m - s[j]); l += s[j];"),
    ("scores_use_v", "for (int d = 0; d < D; ++d) dot += q[d] * kj[d];",
     "for (int d = 0; d < D; ++d) dot += q[d] * (v + (int64_t)j * kv_stride)[d];"),
    ("pv_uses_k", "const double *vj = v + (int64_t)j * kv_stride;",
     "const double *vj = k + (int64_t)j * kv_stride;"),
    ("no_normalisation", "double p = s[j] / l;", "double p = s[j];"),
    ("lse_missing_max", "*lse = m + log(l);\n}\n\nstatic", "*lse = log(l);\n}\n\nstatic"),
    ("row_max_skipped", "for (int j = 0; j < n_keys; ++j) if (s[j] > m) m = s[j];",
     "m = 0.0;"),
    ("decode_drops_newest", "for (int j = 0; j < L; ++j) vis[j] = 1;",
     "for (int j = 0; j < L; ++j) vis[j] = (j < L - 1);"),
    ("merge_weight_dropped", "L += l[i] * w;", "L += l[i];"),
    ("online_no_rescale", "l *= c;\n        for (int d = 0; d < D; ++d) acc[d] *= c;",
     "for (int d = 0; d < D; ++d) acc[d] *= c;"),
    ("partial_no_max", "double e = exp(s[j] - m);", "double e = exp(s[j]);"),
    ("chunk_offset_dropped", "const long long p = (long long)L - Sq + i;",
     "const long long p = (long long)i;"),
    ("varlen_padding_rows_live", "vis[j] = (i < L) && (causal ? (j <= i) : 1);",
     "vis[j] = (causal ? (j <= i) : 1);"),
    ("rope_sign_swapped", "o[d] = xr[d] * c[d] - xr[d + H] * sn[d];",
     "o[d] = xr[d] * c[d] + xr[d + H] * sn[d];"),
    ("rope_halves_mixed", "o[d + H] = xr[d] * sn[d] + xr[d + H] * c[d];",
     "o[d + H] = xr[d + H] * sn[d] + xr[d] * c[d];"),
    ("chunk_strict_causal", "vis[j] = causal ? ((long long)j <= p) : 1;",
     "vis[j] = causal ? ((long long)j < p) : 1;"),
]


def _run_pins(lib):
    failed = []
    have_mp = importlib.util.find_spec("mpmath") is not None
    for pin in oracle_pins.ALL_PINS:
        if pin is oracle_pins.pin_brute_force_tiny and not have_mp:
            continue
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique/found"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(old, new))
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib_{name}.so"))
    failed = _run_pins(oracle.load(so))
    assert failed, f"no pin caught mutant {name}"


def test_pins_pass_on_unmutated_copy(tmp_path):
    src = tmp_path / "oracle_copy.c"
    src.write_text(open(SRC).read())
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / "lib_copy.so"))
    assert _run_pins(oracle.load(so)) == []
