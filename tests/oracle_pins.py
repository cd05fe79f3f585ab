"""Pins of the fp64 oracle: facts that the mathematics or the pages fix, checked against an
oracle build passed in as ``lib``. Each ``pin_*`` function raises AssertionError on failure.

They run against the real oracle (tests/test_oracle_pins.py) and against deliberately broken
copies of it (tests/test_oracle_mutants.py), where at least one pin must fail.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

RNG_SEED = 1234


def _rng(off=0):
    return np.random.default_rng(RNG_SEED + off)


def _close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):  # inf - inf where both_inf (masked out) or a mutant
        err = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(err)), f"{what}: non-finite error"
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"{what}: max err {m} > {tol}"


# ---------------------------------------------------------------------------------- pins


def pin_rows_of_p_sum_to_one(lib):
    """With V = identity (D = S), O is P itself: every row sums to 1, entries are >= 0, and
    with the causal mask P[i, j] is exactly 0 for j > i."""
    for S, causal, (Hq, Hkv) in [(7, True, (2, 1)), (16, False, (3, 3)), (33, True, (4, 2))]:
        rng = _rng(S)
        Dk = 5
        q = rng.standard_normal((1, Hq, S, Dk))
        k = rng.standard_normal((1, Hkv, S, Dk))
        # pad q/k to D = S with zeros so that V = I fits the same head dim
        qp = np.zeros((1, Hq, S, S)); qp[..., :Dk] = q
        kp = np.zeros((1, Hkv, S, S)); kp[..., :Dk] = k
        v = np.broadcast_to(np.eye(S), (1, Hkv, S, S)).copy()
        P, _ = oracle.prefill(qp, kp, v, causal, 0.7, lib=lib)
        _close(P.sum(-1), np.ones((1, Hq, S)), 1e-12, "row sums")
        assert (P >= 0).all(), "negative probability"
        if causal:
            upper = np.triu(np.ones((S, S), dtype=bool), 1)
            assert np.all(P[..., upper] == 0.0), "masked key got weight"
            assert np.all(P[..., ~upper] > 0.0), "visible key got zero weight"


def pin_constant_keys_give_prefix_means(lib):
    """All keys equal -> uniform weights: causal O[i] = mean(V[0..i]), non-causal O[i] =
    mean(V); LSE[i] = s + ln(#visible)."""
    rng = _rng(1)
    B, Hq, Hkv, S, D = 2, 4, 2, 19, 6
    q = rng.standard_normal((B, Hq, S, D))
    krow = rng.standard_normal(D)
    k = np.broadcast_to(krow, (B, Hkv, S, D)).copy()
    v = rng.standard_normal((B, Hkv, S, D))
    scale = 0.37
    G = Hq // Hkv
    vg = np.repeat(v, G, axis=1)
    s = scale * np.einsum("bhsd,d->bhs", q, krow)
    o, lse = oracle.prefill(q, k, v, True, scale, lib=lib)
    cnt = np.arange(1, S + 1)
    _close(o, np.cumsum(vg, axis=2) / cnt[:, None], 1e-12, "causal prefix mean")
    _close(lse, s + np.log(cnt), 1e-12, "causal lse")
    o, lse = oracle.prefill(q, k, v, False, scale, lib=lib)
    _close(o, np.broadcast_to(vg.mean(axis=2, keepdims=True), o.shape), 1e-12, "mean")
    _close(lse, s + math.log(S), 1e-12, "non-causal lse")


def pin_single_key_returns_v(lib):
    """kv_len = 1: O = V[0] exactly and LSE = scale * q.k."""
    rng = _rng(2)
    q = rng.standard_normal((2, 4, 1, 8)); k = rng.standard_normal((2, 2, 1, 8))
    v = rng.standard_normal((2, 2, 1, 8))
    for causal in (True, False):
        o, lse = oracle.prefill(q, k, v, causal, 0.5, lib=lib)
        assert np.array_equal(o, np.repeat(v, 2, axis=1)), "O != V"
        _close(lse, 0.5 * np.einsum("bhsd,bhsd->bhs", q, np.repeat(k, 2, axis=1)), 1e-14, "lse")
    # decode with one cached token
    qd = rng.standard_normal((3, 4, 8)); kc = rng.standard_normal((3, 2, 5, 8))
    vc = rng.standard_normal((3, 2, 5, 8))
    o, lse = oracle.decode(qd, kc, vc, [1, 1, 1], 0.5, lib=lib)
    assert np.array_equal(o, np.repeat(vc[:, :, 0], 2, axis=1)), "decode O != V[0]"


def pin_two_keys_closed_form(lib):
    """Scores 0 and ln 3 give weights 1/4 and 3/4: O = (v0 + 3 v1) / 4, LSE = ln 4."""
    D = 4
    q = np.zeros((1, 1, 2, D)); q[0, 0, 1, 0] = 1.0
    k = np.zeros((1, 1, 2, D)); k[0, 0, 1, 0] = math.log(3.0) / 0.25
    v = np.array([[[[1.0, -2.0, 0.5, 4.0], [3.0, 2.0, -1.5, 0.0]]]])
    o, lse = oracle.prefill(q, k, v, True, 0.25, lib=lib)
    # row 0 sees key 0 only; row 1 sees scores (0, ln 3)
    _close(o[0, 0, 0], v[0, 0, 0], 0.0, "row 0")
    _close(o[0, 0, 1], (v[0, 0, 0] + 3 * v[0, 0, 1]) / 4, 1e-15, "row 1")
    _close(lse[0, 0], [0.0, math.log(4.0)], 1e-15, "lse")
    o, lse = oracle.prefill(q, k, v, False, 0.25, lib=lib)
    _close(o[0, 0, 0], (v[0, 0, 0] + v[0, 0, 1]) / 2, 1e-15, "non-causal row 0")


def pin_shift_invariance(lib):
    """Adding c to every score of a row (an extra dim: k[.., D] = 1, q[.., D] = c / scale)
    leaves O unchanged and adds c to LSE ("CS336 Lecture 6", exercise 3: softmax is
    unchanged by subtracting any constant)."""
    rng = _rng(3)
    B, Hq, Hkv, S, D = 1, 2, 1, 23, 7
    q = rng.standard_normal((B, Hq, S, D)); k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    scale = 0.6
    c = rng.uniform(-30, 30, size=(B, Hq, S))
    q2 = np.concatenate([q, (c / scale)[..., None]], axis=-1)
    k2 = np.concatenate([k, np.ones((B, Hkv, S, 1))], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, Hkv, S, 1))], axis=-1)
    for causal in (True, False):
        o, lse = oracle.prefill(q, k, v, causal, scale, lib=lib)
        o2, lse2 = oracle.prefill(q2, k2, v2, causal, scale, lib=lib)
        _close(o2[..., :D], o, 1e-12, "shifted O")
        _close(lse2, lse + c, 1e-11, "shifted lse")


def pin_gqa_equals_repeated_heads(lib):
    """GQA with contiguous groups equals multi-head attention on K/V heads repeated G times
    (kv head of query head h is h // G)."""
    rng = _rng(4)
    B, Hq, Hkv, S, D = 2, 6, 2, 13, 4
    q = rng.standard_normal((B, Hq, S, D)); k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    for causal in (True, False):
        o, lse = oracle.prefill(q, k, v, causal, 0.5, lib=lib)
        o2, lse2 = oracle.prefill(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), causal,
                                  0.5, lib=lib)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2), "GQA != repeated MHA"
    # decode: same mapping
    qd = rng.standard_normal((B, Hq, D)); kc = rng.standard_normal((B, Hkv, 9, D))
    vc = rng.standard_normal((B, Hkv, 9, D))
    o, _ = oracle.decode(qd, kc, vc, [9, 4], 0.5, lib=lib)
    o2, _ = oracle.decode(qd, np.repeat(kc, 3, axis=1), np.repeat(vc, 3, axis=1), [9, 4], 0.5,
                          lib=lib)
    assert np.array_equal(o, o2), "decode GQA != repeated MHA"


def _brute_row(qi, K, V, scale, n_vis):
    """Softmax written directly as exp(s_j) / sum_k exp(s_k) in 60-digit arithmetic (no max
    subtraction, no blocking): an independent restatement used on tiny inputs."""
    import mpmath

    mpmath.mp.dps = 60
    s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                         for a, b in zip(qi, K[j])) for j in range(n_vis)]
    e = [mpmath.exp(x) for x in s]
    den = mpmath.fsum(e)
    o = [float(mpmath.fsum(e[j] * mpmath.mpf(float(V[j][d])) for j in range(n_vis)) / den)
         for d in range(len(V[0]))]
    return o, float(mpmath.log(den))


def pin_brute_force_tiny(lib):
    """Tiny shapes against a 60-digit restatement of the textbook formula."""
    rng = _rng(5)
    for (B, Hq, Hkv, S, D, causal) in [(2, 4, 2, 5, 3, True), (1, 2, 2, 7, 4, False),
                                       (2, 3, 1, 6, 2, True)]:
        q = rng.standard_normal((B, Hq, S, D)) * 2
        k = rng.standard_normal((B, Hkv, S, D))
        v = rng.standard_normal((B, Hkv, S, D))
        scale = 1 / math.sqrt(D)
        o, lse = oracle.prefill(q, k, v, causal, scale, lib=lib)
        G = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                for i in range(S):
                    n = i + 1 if causal else S
                    ob, lb = _brute_row(q[b, h, i], k[b, h // G], v[b, h // G], scale, n)
                    _close(o[b, h, i], ob, 1e-13, f"brute O b{b} h{h} i{i}")
                    _close(lse[b, h, i], lb, 1e-13, f"brute lse b{b} h{h} i{i}")
    # decode rows too
    qd = rng.standard_normal((2, 4, 3)); kc = rng.standard_normal((2, 2, 6, 3))
    vc = rng.standard_normal((2, 2, 6, 3))
    lens = [6, 2]
    o, lse = oracle.decode(qd, kc, vc, lens, 0.8, lib=lib)
    for b in range(2):
        for h in range(4):
            ob, lb = _brute_row(qd[b, h], kc[b, h // 2], vc[b, h // 2], 0.8, lens[b])
            _close(o[b, h], ob, 1e-13, "brute decode O")
            _close(lse[b, h], lb, 1e-13, "brute decode lse")


def pin_merge_is_order_free(lib):
    """Block partials of a row, merged in any order, give the two-pass row ("Attention
    three-op fusion", section 2.2: merge order does not matter). Includes empty blocks."""
    rng = _rng(6)
    n, D, scale = 61, 9, 0.45
    qi = rng.standard_normal(D) * 3
    K = rng.standard_normal((n, D)); V = rng.standard_normal((n, D))
    o_ref, lse_ref = oracle.decode(qi[None, None], K[None, None], V[None, None], [n], scale,
                                   lib=lib)
    o_ref, lse_ref = o_ref[0], lse_ref[0]
    for trial in range(6):
        cuts = np.sort(rng.choice(np.arange(0, n + 1), size=5, replace=True))
        bounds = [0, *cuts.tolist(), n]
        parts = [oracle.row_partial(qi, K[a:b], V[a:b], scale, lib=lib)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        order = rng.permutation(len(parts))
        m = np.array([parts[i][0] for i in order]); l = np.array([parts[i][1] for i in order])
        o_un = np.stack([parts[i][2] for i in order])
        o, lse = oracle.merge(m, l, o_un, lib=lib)
        _close(o, o_ref[0], 1e-12, f"merged O trial {trial}")
        _close(lse, lse_ref[0], 1e-12, f"merged lse trial {trial}")
    # all-empty merge: O = 0, LSE = -inf
    o, lse = oracle.merge(np.array([-np.inf, -np.inf]), np.zeros(2), np.zeros((2, D)), lib=lib)
    assert np.all(o == 0) and lse == -np.inf, "empty merge"


def pin_online_equals_two_pass(lib):
    """The online recurrence over blocks of any size equals the two-pass softmax row
    ("Attention three-op fusion", section 2.2: one pass, numerically equivalent)."""
    rng = _rng(7)
    n, D, scale = 100, 8, 0.3
    qi = rng.standard_normal(D) * 4
    K = rng.standard_normal((n, D)); V = rng.standard_normal((n, D))
    o_ref, lse_ref = oracle.decode(qi[None, None], K[None, None], V[None, None], [n], scale,
                                   lib=lib)
    o_ref, lse_ref = o_ref[0], lse_ref[0]
    for block in (1, 3, 16, 64, 100, 257):
        o, lse = oracle.online_row(qi, K, V, scale, block, lib=lib)
        _close(o, o_ref[0], 1e-12, f"online O block {block}")
        _close(lse, lse_ref[0], 1e-12, f"online lse block {block}")


def pin_decode_is_last_prefill_row(lib):
    """Decode of the last query against the cache equals the last row of causal prefill;
    cache rows beyond the length (NaN here) are never read."""
    rng = _rng(8)
    B, Hq, Hkv, S, D = 2, 4, 2, 17, 6
    q = rng.standard_normal((B, Hq, S, D)); k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    o, lse = oracle.prefill(q, k, v, True, 0.4, lib=lib)
    max_len = S + 5
    kc = np.full((B, Hkv, max_len, D), np.nan); vc = np.full((B, Hkv, max_len, D), np.nan)
    kc[:, :, :S] = k; vc[:, :, :S] = v
    od, lsed = oracle.decode(q[:, :, -1], kc, vc, [S, S], 0.4, lib=lib)
    _close(od, o[:, :, -1], 1e-13, "decode vs prefill O")
    _close(lsed, lse[:, :, -1], 1e-13, "decode vs prefill lse")
    # a shorter sequence equals prefill of the truncated sequence (row L-1)
    L = 9
    od, lsed = oracle.decode(q[:, :, L - 1], kc, vc, [L, L], 0.4, lib=lib)
    o9, lse9 = oracle.prefill(q[:, :, :L], k[:, :, :L], v[:, :, :L], True, 0.4, lib=lib)
    _close(od, o9[:, :, -1], 1e-13, "short decode O")


def pin_empty_decode_row(lib):
    """A sequence of length 0 has no visible key: O = 0, LSE = -inf, no NaN."""
    rng = _rng(9)
    q = rng.standard_normal((2, 2, 4)); kc = rng.standard_normal((2, 1, 3, 4))
    vc = rng.standard_normal((2, 1, 3, 4))
    o, lse = oracle.decode(q, kc, vc, [0, 3], 1.0, lib=lib)
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf), "empty row"
    assert np.all(np.isfinite(o[1])) and np.all(np.isfinite(lse[1]))


def pin_hard_max_limit(lib):
    """When one score exceeds the others by far more than the fp64 exp range, the softmax is
    one-hot: O equals the V row of the largest score and LSE equals that score."""
    rng = _rng(10)
    S, D = 12, 5
    q = np.zeros((1, 1, S, D)); q[..., 0] = 1.0
    k = np.zeros((1, 1, S, D)); k[0, 0, :, 0] = rng.permutation(S) * 2000.0
    v = rng.standard_normal((1, 1, S, D))
    o, lse = oracle.prefill(q, k, v, False, 1.0, lib=lib)
    j = int(np.argmax(k[0, 0, :, 0]))
    assert np.all(o[0, 0] == v[0, 0, j]), "hard max O"
    _close(lse[0, 0], np.full(S, k[0, 0, j, 0]), 0.0, "hard max lse")


def pin_chunk_reduces_to_prefill_and_decode(lib):
    """A chunk of all L_b tokens is causal prefill of the sequence; a chunk of one token is
    decode; a chunk of the last c tokens equals the last c rows of prefill."""
    rng = _rng(11)
    B, Hq, Hkv, S, D = 2, 4, 2, 21, 5
    q = rng.standard_normal((B, Hq, S, D)); k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    o, lse = oracle.prefill(q, k, v, True, 0.45, lib=lib)
    max_len = S + 3
    kc = np.full((B, Hkv, max_len, D), np.nan); vc = np.full((B, Hkv, max_len, D), np.nan)
    kc[:, :, :S] = k; vc[:, :, :S] = v
    oc, lsec = oracle.chunk(q, kc, vc, [S, S], 0.45, True, lib=lib)
    _close(oc, o, 1e-13, "chunk = prefill O")
    _close(lsec, lse, 1e-13, "chunk = prefill lse")
    for c in (1, 4):
        oc, lsec = oracle.chunk(q[:, :, S - c:], kc, vc, [S, S], 0.45, True, lib=lib)
        _close(oc, o[:, :, S - c:], 1e-13, f"chunk of {c} = last prefill rows")
    od, lsed = oracle.decode(q[:, :, -1], kc, vc, [S, S], 0.45, lib=lib)
    oc, lsec = oracle.chunk(q[:, :, -1:], kc, vc, [S, S], 0.45, True, lib=lib)
    _close(oc[:, :, 0], od, 1e-13, "chunk of 1 = decode")
    # non-causal chunk: every query sees all L_b keys, as decode does
    oc, _ = oracle.chunk(q[:, :, :3], kc, vc, [S, 7], 0.45, False, lib=lib)
    for i in range(3):
        od, _ = oracle.decode(q[:, :, i], kc, vc, [S, 7], 0.45, lib=lib)
        _close(oc[:, :, i], od, 1e-13, "non-causal chunk = decode per query")
    # a query before the start of the sequence sees nothing
    oc, lsec = oracle.chunk(q[:, :, :4], kc, vc, [2, S], 0.45, True, lib=lib)
    assert np.all(oc[0, :, :2] == 0) and np.all(np.isneginf(lsec[0, :, :2]))


def pin_varlen_is_prefill_of_each_sequence(lib):
    """Each sequence of a padded batch equals prefill of its own valid tokens; padding rows are
    O = 0, LSE = -inf; full lengths give plain prefill."""
    rng = _rng(12)
    B, Hq, Hkv, S, D = 3, 4, 2, 17, 6
    q = rng.standard_normal((B, Hq, S, D)); k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    lens = [17, 9, 0]
    for causal in (True, False):
        o, lse = oracle.prefill_varlen(q, k, v, lens, causal, 0.4, lib=lib)
        for b, L in enumerate(lens):
            if L:
                ob, lb = oracle.prefill(q[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
                                        causal, 0.4, lib=lib)
                _close(o[b:b + 1, :, :L], ob, 1e-13, f"varlen seq {b}")
                _close(lse[b:b + 1, :, :L], lb, 1e-13, f"varlen lse {b}")
            assert np.all(o[b, :, L:] == 0) and np.all(np.isneginf(lse[b, :, L:])), "padding rows"
        of, lf = oracle.prefill_varlen(q, k, v, [S, S, S], causal, 0.4, lib=lib)
        op, lp = oracle.prefill(q, k, v, causal, 0.4, lib=lib)
        assert np.array_equal(of, op) and np.array_equal(lf, lp)


def _rope_tables(n_pos, D, base=10000.0):
    inv = base ** (-np.arange(D // 2) * 2.0 / D)
    ang = np.arange(n_pos)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def pin_rope_closed_forms(lib):
    """Rotate-half RoPE: a 2-D example worked by hand, norms preserved, identity at angle 0,
    and q.k depends only on the position difference for a real RoPE table."""
    th = 0.7
    out = oracle.rope(np.array([[1.0, 0.0], [0.0, 1.0]]), np.array([[math.cos(th)]] * 2),
                      np.array([[math.sin(th)]] * 2), lib=lib)
    _close(out, np.array([[math.cos(th), math.sin(th)], [-math.sin(th), math.cos(th)]]), 1e-15,
           "hand rotation")
    rng = _rng(13)
    D = 16
    x = rng.standard_normal((5, D))
    c, sn = _rope_tables(64, D)
    rx = oracle.rope(x, c[7], sn[7], lib=lib)
    _close(np.linalg.norm(rx, axis=-1), np.linalg.norm(x, axis=-1), 1e-12, "norm")
    _close(oracle.rope(x, np.ones(D // 2), np.zeros(D // 2), lib=lib), x, 0.0, "identity")
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    dots = [oracle.rope(q[None], c[p + 9], sn[p + 9], lib=lib)[0]
            @ oracle.rope(k[None], c[p], sn[p], lib=lib)[0] for p in (0, 5, 30)]
    _close(np.array(dots), np.full(3, dots[0]), 1e-12, "relative position")


def pin_decode_rope_composition(lib):
    """With identity tables the step is: store k_new, v_new at row L-1, then plain decode."""
    rng = _rng(14)
    B, Hq, Hkv, D, max_len = 2, 4, 2, 8, 12
    q = rng.standard_normal((B, Hq, D)); kn = rng.standard_normal((B, Hkv, D))
    vn = rng.standard_normal((B, Hkv, D))
    kc = rng.standard_normal((B, Hkv, max_len, D)); vc = rng.standard_normal((B, Hkv, max_len, D))
    ones, zeros = np.ones((max_len, D // 2)), np.zeros((max_len, D // 2))
    o, lse, kst = oracle.decode_rope(q, kn, vn, ones, zeros, kc, vc, [12, 5], 0.5, lib=lib)
    import torch
    kb = torch.from_numpy(kn).to(torch.bfloat16).double().numpy()
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[0, :, 11] = kb[0]; vc2[0, :, 11] = vn[0]
    kc2[1, :, 4] = kb[1]; vc2[1, :, 4] = vn[1]
    o2, lse2 = oracle.decode(q, kc2, vc2, [12, 5], 0.5, lib=lib)
    _close(o, o2, 1e-14, "rope step O"); _close(lse, lse2, 1e-14, "rope step lse")


ALL_PINS = [pin_rows_of_p_sum_to_one, pin_constant_keys_give_prefix_means,
            pin_single_key_returns_v, pin_two_keys_closed_form, pin_shift_invariance,
            pin_gqa_equals_repeated_heads, pin_brute_force_tiny, pin_merge_is_order_free,
            pin_online_equals_two_pass, pin_decode_is_last_prefill_row, pin_empty_decode_row,
            pin_hard_max_limit, pin_chunk_reduces_to_prefill_and_decode,
            pin_varlen_is_prefill_of_each_sequence, pin_rope_closed_forms,
            pin_decode_rope_composition]
