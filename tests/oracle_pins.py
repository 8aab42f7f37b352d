"""Pins for the fp64 oracle: checks against facts fixed by the pages and by the
mathematics, never against the oracle itself.

Each ``pin_*`` takes an oracle library handle (``lib``) and returns a list of
failure messages (empty = pass), so the same pins can be run against the real
oracle and against deliberately broken copies of it (see
``test_oracle_mutants.py``).

Formula pinned: attn = softmax(Q K^T / sqrt(d)) V over [b, h, s, d]
("flash-attn 实现 prefill 阶段", 问题分析); scale applied after the dot product
and natural exponent (flash-attention-minimal ``forward_kernel``); running
statistics start at m = -inf, l = 0, O = 0 (its host ``forward()``).
"""
from __future__ import annotations

import json
import math
import os

import mpmath
import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _textbook_mp(q, k, v, causal, scale, dps=40):
    """Softmax attention by the textbook formula in mpmath, exp without any
    max subtraction (inputs kept small), key j visible iff j <= i + sk - sq."""
    mpmath.mp.dps = dps
    b, h, sq, d = q.shape
    sk = k.shape[2]
    o = np.zeros((b, h, sq, d))
    lse = np.zeros((b, h, sq))
    for bi in range(b):
        for hi in range(h):
            for i in range(sq):
                vis = [j for j in range(sk) if (not causal) or j <= i + sk - sq]
                if not vis:
                    lse[bi, hi, i] = -math.inf
                    continue
                e = []
                for j in vis:
                    dot = mpmath.fsum(mpmath.mpf(float(q[bi, hi, i, c])) * mpmath.mpf(float(k[bi, hi, j, c]))
                                      for c in range(d))
                    e.append(mpmath.exp(dot * mpmath.mpf(scale)))
                z = mpmath.fsum(e)
                for c in range(d):
                    o[bi, hi, i, c] = float(mpmath.fsum(e[t] * mpmath.mpf(float(v[bi, hi, j, c]))
                                                        for t, j in enumerate(vis)) / z)
                lse[bi, hi, i] = float(mpmath.log(z))
    return o, lse


def _cmp(name, got, want, tol=TOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if got.shape != want.shape:
        return [f"{name}: shape {got.shape} != {want.shape}"]
    both_inf = np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(got - want))
    diff = np.where(np.isnan(diff), np.inf, diff)
    err = float(diff.max()) if diff.size else 0.0
    return [] if err <= tol else [f"{name}: max err {err:.3e} > {tol:.1e}"]


def _scale_of(s):
    if isinstance(s, (int, float)):
        return float(s)
    if s.startswith("ln"):
        return math.log(float(s[2:]))
    return float(s)


def _val(x):
    if isinstance(x, str):
        if x in ("-inf", "inf"):
            return float(x)
        return _scale_of(x)
    return float(x)


# ---------------------------------------------------------------- pins

def pin_worked_examples(lib):
    """Hand-derived examples stored in tests/golden/worked_examples.json."""
    fails = []
    with open(os.path.join(HERE, "golden", "worked_examples.json")) as f:
        data = json.load(f)
    for ex in data["examples"]:
        q = np.array(ex["q"], np.float64)[None, None]
        k = np.array(ex["k"], np.float64)[None, None]
        v = np.array(ex["v"], np.float64)[None, None]
        want_o = np.array(ex["o"], np.float64)[None, None]
        want_l = np.array([_val(x) for x in ex["lse"]])[None, None]
        for fn in ("def", "online"):
            if fn == "def":
                o, l = oracle.attn_fwd(q, k, v, ex["causal"], _scale_of(ex["scale"]), lib=lib)
            else:
                o, l = oracle.attn_fwd_online(q, k, v, ex["causal"], _scale_of(ex["scale"]), 2, lib=lib)
            fails += _cmp(f"{ex['name']}[{fn}].o", o, want_o)
            fails += _cmp(f"{ex['name']}[{fn}].lse", l, want_l)
    return fails


def pin_bruteforce(lib, shapes=None):
    """Tiny inputs against the textbook formula in 40-digit arithmetic."""
    fails = []
    shapes = shapes or [(sq, sk, d) for sq in (1, 2, 3, 5) for sk in (1, 2, 3, 5) for d in (1, 4)] \
        + [(3, 5, 64), (5, 3, 64), (5, 5, 64)]
    for t, (sq, sk, d) in enumerate(shapes):
        r = _rng(1000 + t)
        q = r.standard_normal((1, 2, sq, d))
        k = r.standard_normal((1, 2, sk, d))
        v = r.standard_normal((1, 2, sk, d))
        scale = 1.0 / math.sqrt(d) * (1.0 + 0.25 * t % 3)
        for causal in (False, True):
            want_o, want_l = _textbook_mp(q, k, v, causal, scale)
            o, l = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
            fails += _cmp(f"brute sq{sq} sk{sk} d{d} c{int(causal)} o", o, want_o)
            fails += _cmp(f"brute sq{sq} sk{sk} d{d} c{int(causal)} lse", l, want_l)
            o2, l2 = oracle.attn_fwd_online(q, k, v, causal, scale, 2, lib=lib)
            fails += _cmp(f"brute-online sq{sq} sk{sk} d{d} c{int(causal)} o", o2, want_o)
            fails += _cmp(f"brute-online sq{sq} sk{sk} d{d} c{int(causal)} lse", l2, want_l)
    return fails


def pin_rows_sum_to_one(lib):
    """With V = identity (d = sk), O[i, :] is the probability row P[i, :]:
    entries are >= 0, masked keys get exactly 0, and each row sums to 1."""
    fails = []
    for causal in (False, True):
        for sq, sk in ((7, 7), (5, 9), (9, 5)):
            r = _rng(sq * 31 + sk)
            q = r.standard_normal((1, 1, sq, sk)) * 3
            k = r.standard_normal((1, 1, sk, sk)) * 3
            v = np.eye(sk)[None, None]
            o, _ = oracle.attn_fwd(q, k, v, causal, 0.7, lib=lib)
            p = o[0, 0]
            for i in range(sq):
                vis = [j for j in range(sk) if (not causal) or j <= i + sk - sq]
                if not vis:
                    fails += _cmp(f"P-row-empty c{causal} {sq}x{sk} r{i}", p[i], np.zeros(sk))
                    continue
                if p[i].min() < 0:
                    fails.append(f"P negative c{causal} {sq}x{sk} r{i}")
                fails += _cmp(f"P-sum c{causal} {sq}x{sk} r{i}", p[i].sum(), 1.0)
                masked = [j for j in range(sk) if j not in vis]
                if masked and np.abs(p[i, masked]).max() != 0.0:
                    fails.append(f"P masked nonzero c{causal} {sq}x{sk} r{i}")
    return fails


def pin_identical_keys(lib):
    """All K rows equal k: O[i] is the mean of the visible V rows and
    LSE_i = scale*(q_i . k) + ln(#visible)."""
    fails = []
    sq, sk, d = 6, 6, 8
    r = _rng(5)
    q = r.standard_normal((1, 1, sq, d))
    krow = r.standard_normal(d)
    k = np.tile(krow, (sk, 1))[None, None]
    v = r.standard_normal((1, 1, sk, d))
    scale = 0.37
    for causal in (False, True):
        o, l = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
        for i in range(sq):
            n = (i + 1) if causal else sk
            fails += _cmp(f"same-k c{causal} O[{i}]", o[0, 0, i], v[0, 0, :n].mean(axis=0))
            fails += _cmp(f"same-k c{causal} LSE[{i}]", l[0, 0, i], scale * float(q[0, 0, i] @ krow) + math.log(n))
    return fails


def pin_zero_query_or_scale(lib):
    """Q = 0 (or scale = 0): uniform attention over the visible keys."""
    fails = []
    b, h, sq, sk, d = 2, 3, 4, 6, 5
    r = _rng(11)
    k = r.standard_normal((b, h, sk, d))
    v = r.standard_normal((b, h, sk, d))
    for causal in (False, True):
        for variant in ("q0", "s0"):
            q = np.zeros((b, h, sq, d)) if variant == "q0" else r.standard_normal((b, h, sq, d))
            scale = 0.5 if variant == "q0" else 0.0
            o, l = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
            for i in range(sq):
                n = min(sk, i + 1 + sk - sq) if causal else sk
                fails += _cmp(f"{variant} c{causal} O[{i}]", o[:, :, i], v[:, :, :n].mean(axis=2))
                fails += _cmp(f"{variant} c{causal} LSE[{i}]", l[:, :, i], np.full((b, h), math.log(n)))
    return fails


def pin_causal_row0(lib):
    """Causal, sq == sk: row 0 sees only key 0, so O[0] = V[0] and
    LSE_0 = scale * q_0 . k_0."""
    fails = []
    r = _rng(3)
    b, h, s, d = 2, 2, 9, 16
    q = r.standard_normal((b, h, s, d))
    k = r.standard_normal((b, h, s, d))
    v = r.standard_normal((b, h, s, d))
    o, l = oracle.attn_fwd(q, k, v, True, 0.25, lib=lib)
    fails += _cmp("row0 O", o[:, :, 0], v[:, :, 0])
    fails += _cmp("row0 LSE", l[:, :, 0], 0.25 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]))
    return fails


def pin_permutation(lib):
    """Non-causal: permuting K and V rows together changes nothing; permuting
    Q rows permutes O and LSE rows (both masks)."""
    fails = []
    r = _rng(21)
    b, h, sq, sk, d = 1, 2, 7, 11, 8
    q = r.standard_normal((b, h, sq, d))
    k = r.standard_normal((b, h, sk, d))
    v = r.standard_normal((b, h, sk, d))
    o, l = oracle.attn_fwd(q, k, v, False, 0.3, lib=lib)
    pk = r.permutation(sk)
    o2, l2 = oracle.attn_fwd(q, k[:, :, pk], v[:, :, pk], False, 0.3, lib=lib)
    fails += _cmp("perm-kv O", o2, o)
    fails += _cmp("perm-kv LSE", l2, l)
    pq = r.permutation(sq)
    o3, l3 = oracle.attn_fwd(q[:, :, pq], k, v, False, 0.3, lib=lib)
    fails += _cmp("perm-q O", o3, o[:, :, pq])
    fails += _cmp("perm-q LSE", l3, l[:, :, pq])
    return fails


def pin_shift(lib):
    """Adding the same constant c to every logit of a row leaves O unchanged
    and adds c to LSE.  The shift is made by an extra feature: Q' = [Q, 1],
    K' = [K, c/scale]; c = 1000 would overflow exp without the max shift."""
    fails = []
    r = _rng(9)
    b, h, sq, sk, d = 1, 2, 5, 7, 6
    q = r.standard_normal((b, h, sq, d))
    k = r.standard_normal((b, h, sk, d))
    v = r.standard_normal((b, h, sk, d))
    scale = 0.5
    for causal in (False, True):
        o, l = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
        for c in (3.0, 1000.0):
            q2 = np.concatenate([q, np.ones((b, h, sq, 1))], axis=-1)
            k2 = np.concatenate([k, np.full((b, h, sk, 1), c / scale)], axis=-1)
            v2 = np.concatenate([v, np.zeros((b, h, sk, 1))], axis=-1)
            o2, l2 = oracle.attn_fwd(q2, k2, v2, causal, scale, lib=lib)
            fails += _cmp(f"shift{c} c{causal} O", o2[..., :d], o, tol=1e-9)
            fails += _cmp(f"shift{c} c{causal} LSE", l2 - c, l, tol=1e-9)
    return fails


def pin_online_matches_definition(lib):
    """The tile recurrence equals the two-pass definition for tile sizes
    1, 7, 32, 128 (ragged last tiles included)."""
    fails = []
    r = _rng(33)
    b, h, sq, sk, d = 1, 2, 37, 150, 16
    q = r.standard_normal((b, h, sq, d)) * 3
    k = r.standard_normal((b, h, sk, d)) * 3
    v = r.standard_normal((b, h, sk, d))
    for causal in (False, True):
        o, l = oracle.attn_fwd(q, k, v, causal, 1 / 4, lib=lib)
        for bc in (1, 7, 32, 128):
            o2, l2 = oracle.attn_fwd_online(q, k, v, causal, 1 / 4, bc, lib=lib)
            fails += _cmp(f"online bc{bc} c{causal} O", o2, o)
            fails += _cmp(f"online bc{bc} c{causal} LSE", l2, l)
    return fails


def pin_head_rows(lib):
    """The row-subset entry gives the same rows as the full computation on a
    head chosen from a batch (checks head/row indexing of both)."""
    fails = []
    r = _rng(44)
    b, h, sq, sk, d = 2, 3, 13, 17, 8
    q = r.standard_normal((b, h, sq, d))
    k = r.standard_normal((b, h, sk, d))
    v = r.standard_normal((b, h, sk, d))
    for causal in (False, True):
        o, l = oracle.attn_fwd(q, k, v, causal, 0.4, lib=lib)
        rows = [0, 5, 12, 3]
        o2, l2 = oracle.attn_head_rows(q[1, 2], k[1, 2], v[1, 2], rows, causal, 0.4, lib=lib)
        fails += _cmp(f"rows c{causal} O", o2, o[1, 2, rows])
        fails += _cmp(f"rows c{causal} LSE", l2, l[1, 2, rows])
    return fails


def pin_empty(lib):
    """sk = 0: every row sees no key, so O = 0 and LSE = -inf."""
    fails = []
    q = _rng(1).standard_normal((1, 2, 3, 4))
    k = np.zeros((1, 2, 0, 4))
    v = np.zeros((1, 2, 0, 4))
    for causal in (False, True):
        for fn in ("def", "online"):
            if fn == "def":
                o, l = oracle.attn_fwd(q, k, v, causal, 1.0, lib=lib)
            else:
                o, l = oracle.attn_fwd_online(q, k, v, causal, 1.0, 4, lib=lib)
            fails += _cmp(f"empty[{fn}] c{causal} O", o, np.zeros_like(q))
            fails += _cmp(f"empty[{fn}] c{causal} LSE", l, np.full((1, 2, 3), -np.inf))
    return fails


ALL_PINS = [
    pin_worked_examples,
    pin_bruteforce,
    pin_rows_sum_to_one,
    pin_identical_keys,
    pin_zero_query_or_scale,
    pin_causal_row0,
    pin_permutation,
    pin_shift,
    pin_online_matches_definition,
    pin_head_rows,
    pin_empty,
]
