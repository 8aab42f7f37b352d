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


# ---------------------------------------------------------------- backward pins
#
# The gradients are pinned by the forward: dL/dQ, dL/dK, dL/dV of the scalar
# L = sum(O * dO) by central differences, in 40-digit arithmetic on tiny
# inputs (textbook softmax, nothing shared with the oracle) and in fp64 on
# the already-pinned forward oracle for larger ones; plus what the chain rule
# fixes without computing it (rows of dS sum to zero, so the key gradients
# sum to zero; rows of P sum to one, so the value gradients sum to the
# output gradients of the rows that see a key; identical keys or a zero
# scale make the query gradient vanish).


def _loss_mp(q, k, v, do, causal, scale):
    """L = sum_i sum_c O[i, c] dO[i, c] for one head, textbook softmax in
    mpmath (q, k, v, do: nested lists of mpf)."""
    sq, sk, d = len(q), len(k), len(k[0]) if k else 0
    total = mpmath.mpf(0)
    for i in range(sq):
        vis = [j for j in range(sk) if (not causal) or j <= i + sk - sq]
        if not vis:
            continue
        e = [mpmath.exp(scale * mpmath.fsum(q[i][c] * k[j][c] for c in range(d))) for j in vis]
        z = mpmath.fsum(e)
        for c in range(d):
            total += do[i][c] * mpmath.fsum(e[t] * v[j][c] for t, j in enumerate(vis)) / z
    return total


def pin_bwd_finite_difference_mp(lib):
    """Every entry of dQ, dK, dV on tiny inputs against central differences
    of the 40-digit textbook loss (step 1e-12: truncation ~1e-24)."""
    fails = []
    mpmath.mp.dps = 40
    hstep = mpmath.mpf("1e-12")
    for t, (sq, sk, d) in enumerate([(1, 1, 1), (2, 3, 2), (3, 2, 2), (3, 3, 1)]):
        r = _rng(7000 + t)
        q, k, v, do = (r.standard_normal(shape) for shape in ((sq, d), (sk, d), (sk, d), (sq, d)))
        scale = 0.7 + 0.1 * t
        for causal in (False, True):
            dq, dk, dv = oracle.attn_bwd(q[None, None], k[None, None], v[None, None], do[None, None],
                                         causal, scale, lib=lib)
            mp = [[[mpmath.mpf(float(x)) for x in row] for row in a] for a in (q, k, v, do)]
            sc = mpmath.mpf(scale)
            for which, got in ((0, dq[0, 0]), (1, dk[0, 0]), (2, dv[0, 0])):
                want = np.zeros_like(got)
                for (a, c) in np.ndindex(got.shape):
                    plus = [[row[:] for row in m] for m in mp]
                    minus = [[row[:] for row in m] for m in mp]
                    plus[which][a][c] += hstep
                    minus[which][a][c] -= hstep
                    want[a, c] = float((_loss_mp(*plus, causal, sc) - _loss_mp(*minus, causal, sc)) / (2 * hstep))
                fails += _cmp(f"bwd-fd-mp sq{sq} sk{sk} d{d} c{int(causal)} grad{which}", got, want, 1e-11)
    return fails


def pin_bwd_finite_difference_f64(lib):
    """Larger inputs (several heads, sq != sk both ways): sampled entries of
    every gradient against central differences of the fp64 forward oracle
    (step 1e-5: error ~1e-10)."""
    fails = []
    for t, (sq, sk, d) in enumerate([(6, 9, 5), (9, 6, 5), (8, 8, 16)]):
        r = _rng(7100 + t)
        q = r.standard_normal((1, 2, sq, d))
        k = r.standard_normal((1, 2, sk, d))
        v = r.standard_normal((1, 2, sk, d))
        do = r.standard_normal((1, 2, sq, d))
        scale = 1.0 / math.sqrt(d)
        for causal in (False, True):
            grads = oracle.attn_bwd(q, k, v, do, causal, scale, lib=lib)

            def loss(a, b, c):
                o, _ = oracle.attn_fwd(a, b, c, causal, scale, lib=lib)
                return float((o * do).sum())

            for which in range(3):
                base = (q, k, v)[which]
                for idx in [tuple(int(r.integers(0, n)) for n in base.shape) for _ in range(12)]:
                    h = 1e-5
                    args_p = [x.copy() for x in (q, k, v)]
                    args_m = [x.copy() for x in (q, k, v)]
                    args_p[which][idx] += h
                    args_m[which][idx] -= h
                    want = (loss(*args_p) - loss(*args_m)) / (2 * h)
                    got = grads[which][idx]
                    if not abs(got - want) <= 1e-7:
                        fails.append(f"bwd-fd-f64 sq{sq} sk{sk} c{int(causal)} grad{which}{idx}: "
                                     f"{got:.12f} vs {want:.12f}")
    return fails


def pin_bwd_sums(lib):
    """Sum over keys of dK is 0 (each row of dS sums to 0); sum over keys of
    dV is the sum of dO over the rows that see at least one key."""
    fails = []
    for t, (sq, sk, d) in enumerate([(5, 5, 4), (7, 4, 3), (4, 7, 3), (33, 40, 8)]):
        r = _rng(7200 + t)
        q, do = r.standard_normal((1, 2, sq, d)), r.standard_normal((1, 2, sq, d))
        k, v = r.standard_normal((1, 2, sk, d)), r.standard_normal((1, 2, sk, d))
        for causal in (False, True):
            _, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.8, lib=lib)
            sees = np.array([(not causal) or (i + sk - sq >= 0) for i in range(sq)])
            fails += _cmp(f"bwd-sum-dk sq{sq} sk{sk} c{int(causal)}", dk.sum(axis=2), np.zeros((1, 2, d)))
            fails += _cmp(f"bwd-sum-dv sq{sq} sk{sk} c{int(causal)}", dv.sum(axis=2),
                          do[:, :, sees].sum(axis=2))
    return fails


def pin_bwd_identical_keys_and_zero_scale(lib):
    """Identical key rows: the logits of a row are all equal whatever Q is,
    so dQ = 0.  Zero scale: dQ = dK = 0 and attention is uniform over the
    visible keys, so dV[j] = sum over rows i that see j of dO[i] / n_i."""
    fails = []
    r = _rng(7300)
    sq, sk, d = 6, 8, 4
    q, do = r.standard_normal((1, 1, sq, d)), r.standard_normal((1, 1, sq, d))
    k1 = np.repeat(r.standard_normal((1, 1, 1, d)), sk, axis=2)
    k, v = r.standard_normal((1, 1, sk, d)), r.standard_normal((1, 1, sk, d))
    for causal in (False, True):
        dq, _, _ = oracle.attn_bwd(q, k1, v, do, causal, 0.9, lib=lib)
        fails += _cmp(f"bwd-identical-keys c{int(causal)} dq", dq, np.zeros_like(dq))
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.0, lib=lib)
        fails += _cmp(f"bwd-scale0 c{int(causal)} dq", dq, np.zeros_like(dq))
        fails += _cmp(f"bwd-scale0 c{int(causal)} dk", dk, np.zeros_like(dk))
        want = np.zeros_like(dv)
        for i in range(sq):
            vis = [j for j in range(sk) if (not causal) or j <= i + sk - sq]
            for j in vis:
                want[0, 0, j] += do[0, 0, i] / len(vis)
        fails += _cmp(f"bwd-scale0 c{int(causal)} dv", dv, want)
    return fails


def pin_bwd_rows_cols_and_probs(lib):
    """The single-head row / key variants agree with the full gradients, and
    the probabilities reproduce the pinned forward (P V = O, rows sum to 1)."""
    fails = []
    r = _rng(7400)
    sq, sk, d = 37, 29, 6
    q, do = r.standard_normal((2, 2, sq, d)), r.standard_normal((2, 2, sq, d))
    k, v = r.standard_normal((2, 2, sk, d)), r.standard_normal((2, 2, sk, d))
    rows, cols = [0, 5, 17, 36], [0, 3, 19, 28]
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.6, lib=lib)
        dq_r = oracle.attn_bwd_dq_rows(q[1, 0], k[1, 0], v[1, 0], do[1, 0], rows, causal, 0.6, lib=lib)
        dk_c, dv_c = oracle.attn_bwd_dkv_cols(q[1, 0], k[1, 0], v[1, 0], do[1, 0], cols, causal, 0.6, lib=lib)
        fails += _cmp(f"bwd-rows c{int(causal)}", dq_r, dq[1, 0, rows])
        fails += _cmp(f"bwd-cols-dk c{int(causal)}", dk_c, dk[1, 0, cols])
        fails += _cmp(f"bwd-cols-dv c{int(causal)}", dv_c, dv[1, 0, cols])
        p = oracle.attn_probs(q, k, causal, 0.6, lib=lib)
        o, _ = oracle.attn_fwd(q, k, v, causal, 0.6, lib=lib)
        fails += _cmp(f"probs c{int(causal)} PV", np.einsum("bhij,bhjc->bhic", p, v), o)
        sees = np.array([(not causal) or (i + sk - sq >= 0) for i in range(sq)], np.float64)
        fails += _cmp(f"probs c{int(causal)} rows", p.sum(-1), np.broadcast_to(sees, p.shape[:3]))
    return fails


def pin_bwd_empty(lib):
    """No keys: dQ = 0 (and dK, dV are empty); no queries: dK = dV = 0."""
    fails = []
    r = _rng(7500)
    q, do = r.standard_normal((1, 2, 3, 4)), r.standard_normal((1, 2, 3, 4))
    k0 = np.zeros((1, 2, 0, 4))
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k0, k0, do, causal, 1.0, lib=lib)
        fails += _cmp(f"bwd-empty-k c{int(causal)} dq", dq, np.zeros_like(q))
        k, v = r.standard_normal((1, 2, 5, 4)), r.standard_normal((1, 2, 5, 4))
        q0 = np.zeros((1, 2, 0, 4))
        _, dk, dv = oracle.attn_bwd(q0, k, v, q0, causal, 1.0, lib=lib)
        fails += _cmp(f"bwd-empty-q c{int(causal)} dk", dk, np.zeros_like(k))
        fails += _cmp(f"bwd-empty-q c{int(causal)} dv", dv, np.zeros_like(v))
    return fails


# ---------------------------------------------------------------- KV cache

def _kvcache_textbook(q, kc, vc, lens, kn, vn, causal, scale):
    """The KV-cache reading written out in plain Python: copy the new rows
    in after each element's clamped length, then the textbook formula over
    the element's first L keys (mask bottom-right aligned to L)."""
    kc = np.array(kc, np.float64, copy=True)
    vc = np.array(vc, np.float64, copy=True)
    b, h, sq, d = q.shape
    cap = kc.shape[2]
    s_new = 0 if kn is None else kn.shape[2]
    o = np.zeros((b, h, sq, d))
    lse = np.zeros((b, h, sq))
    for e in range(b):
        l0 = min(max(int(lens[e]), 0), cap)
        for t in range(s_new):
            if l0 + t < cap:
                kc[e, :, l0 + t] = kn[e, :, t]
                vc[e, :, l0 + t] = vn[e, :, t]
        n = min(l0 + s_new, cap)
        oe, le = _textbook_mp(q[e:e + 1], kc[e:e + 1, :, :n], vc[e:e + 1, :, :n], causal, scale)
        o[e], lse[e] = oe[0], le[0]
    return o, lse, kc, vc


def pin_kvcache_bruteforce(lib):
    """Tiny KV-cache problems (lengths that fit, fill, overflow the cache,
    negative, beyond capacity, rows that see no key) against the reading
    written out in Python with 40-digit arithmetic."""
    fails = []
    cases = [  # (b, h, sq, cap, s_new, d, lens)
        (3, 2, 2, 7, 2, 4, [0, 3, 6]),
        (2, 1, 1, 5, 0, 3, [5, 2]),
        (2, 2, 3, 6, 1, 2, [-4, 9]),
        (1, 2, 4, 6, 1, 4, [1]),
        (2, 1, 2, 4, 3, 2, [2, 0]),
    ]
    for t, (b, h, sq, cap, s_new, d, lens) in enumerate(cases):
        r = _rng(4000 + t)
        q = r.standard_normal((b, h, sq, d))
        kc = r.standard_normal((b, h, cap, d))
        vc = r.standard_normal((b, h, cap, d))
        kn = r.standard_normal((b, h, s_new, d)) if s_new else None
        vn = r.standard_normal((b, h, s_new, d)) if s_new else None
        scale = 0.7 / math.sqrt(d)
        for causal in (False, True):
            want = _kvcache_textbook(q, kc, vc, lens, kn, vn, causal, scale)
            got = oracle.attn_fwd_kvcache(q, kc, vc, lens, kn, vn, causal, scale, lib=lib)
            for name, g, w in zip(("o", "lse", "k_cache", "v_cache"), got, want):
                fails += _cmp(f"kvcache case{t} c{int(causal)} {name}", g, w)
    return fails


def pin_kvcache_unused_slots(lib):
    """Cache slots past an element's valid length take no part: NaN there
    leaves the result equal to the one with zeros there."""
    fails = []
    r = _rng(4100)
    b, h, sq, cap, s_new, d = 3, 2, 3, 10, 2, 4
    lens = [0, 4, 8]
    q = r.standard_normal((b, h, sq, d))
    kc = r.standard_normal((b, h, cap, d))
    vc = r.standard_normal((b, h, cap, d))
    kn = r.standard_normal((b, h, s_new, d))
    vn = r.standard_normal((b, h, s_new, d))
    kz, vz, kx, vx = kc.copy(), vc.copy(), kc.copy(), vc.copy()
    for e, n in enumerate(lens):
        kz[e, :, n:], vz[e, :, n:] = 0.0, 0.0
        kx[e, :, n:], vx[e, :, n:] = np.nan, np.nan
    for causal in (False, True):
        oz, lz, _, _ = oracle.attn_fwd_kvcache(q, kz, vz, lens, kn, vn, causal, 0.5, lib=lib)
        ox, lx, _, _ = oracle.attn_fwd_kvcache(q, kx, vx, lens, kn, vn, causal, 0.5, lib=lib)
        fails += _cmp(f"kvcache-nan c{int(causal)} o", ox, oz, 0.0)
        fails += _cmp(f"kvcache-nan c{int(causal)} lse", lx, lz, 0.0)
    return fails


def pin_kvcache_decode_matches_prefill(lib):
    """Causal attention over a whole sequence, computed in one pass, equals
    feeding the sequence through the cache in chunks (each chunk's queries,
    keys and values appended, its rows attending to everything so far)."""
    fails = []
    r = _rng(4200)
    b, h, s, d, cap = 2, 2, 10, 8, 13
    q = r.standard_normal((b, h, s, d))
    k = r.standard_normal((b, h, s, d))
    v = r.standard_normal((b, h, s, d))
    full_o, full_l = oracle.attn_fwd(q, k, v, True, 0.4, lib=lib)
    kc = np.zeros((b, h, cap, d))
    vc = np.zeros((b, h, cap, d))
    a = 0
    for c in (1, 1, 3, 2, 1, 2):
        sl = slice(a, a + c)
        o, l, kc, vc = oracle.attn_fwd_kvcache(q[:, :, sl], kc, vc, [a] * b, k[:, :, sl], v[:, :, sl], True,
                                               0.4, lib=lib)
        fails += _cmp(f"kvcache-decode rows {a}..{a + c} o", o, full_o[:, :, sl])
        fails += _cmp(f"kvcache-decode rows {a}..{a + c} lse", l, full_l[:, :, sl])
        a += c
    fails += _cmp("kvcache-decode cache k", kc[:, :, :s], k, 0.0)
    fails += _cmp("kvcache-decode cache tail", kc[:, :, s:], np.zeros((b, h, cap - s, d)), 0.0)
    return fails


def pin_kvcache_paged(lib):
    """A paged cache is a re-indexing: the paged oracle with pages in order
    equals the dense KV-cache oracle on the same logical caches; shuffling
    the pool's pages (and the table with them) changes nothing; and each new
    row lands in page table[e, pos // page_size], row pos % page_size, read
    here directly from the pool."""
    fails = []
    r = _rng(4300)
    b, h, sq, d, ps, pages, s_new = 2, 2, 3, 4, 4, 3, 2
    lens = [5, 10]
    q = r.standard_normal((b, h, sq, d))
    kn = r.standard_normal((b, h, s_new, d))
    vn = r.standard_normal((b, h, s_new, d))
    num_pages = b * pages + 1
    kp = r.standard_normal((num_pages, ps, h, d))
    vp = r.standard_normal((num_pages, ps, h, d))
    table = np.arange(b * pages).reshape(b, pages)
    dense_k = kp[table].reshape(b, pages * ps, h, d).transpose(0, 2, 1, 3)
    dense_v = vp[table].reshape(b, pages * ps, h, d).transpose(0, 2, 1, 3)
    for causal in (False, True):
        o, l, kp2, vp2 = oracle.attn_fwd_kvcache_paged(q, kp, vp, table, lens, kn, vn, causal, 0.6, lib=lib)
        od, ld, kc, _ = oracle.attn_fwd_kvcache(q, dense_k, dense_v, lens, kn, vn, causal, 0.6, lib=lib)
        fails += _cmp(f"paged-identity c{int(causal)} o", o, od, 0.0)
        fails += _cmp(f"paged-identity c{int(causal)} lse", l, ld, 0.0)
        for e in range(b):
            for t in range(s_new):
                pos = lens[e] + t
                if pos >= pages * ps:
                    continue
                page, row = table[e, pos // ps], pos % ps
                fails += _cmp(f"paged write e{e} t{t}", kp2[page, row], kn[e, :, t], 0.0)
        perm = r.permutation(num_pages)   # pool page i moves to slot perm[i]
        kq = np.empty_like(kp)
        vq = np.empty_like(vp)
        kq[perm], vq[perm] = kp, vp
        o2, l2, _, _ = oracle.attn_fwd_kvcache_paged(q, kq, vq, perm[table], lens, kn, vn, causal, 0.6, lib=lib)
        fails += _cmp(f"paged-shuffled c{int(causal)} o", o2, o, 0.0)
        fails += _cmp(f"paged-shuffled c{int(causal)} lse", l2, l, 0.0)
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
    pin_bwd_finite_difference_mp,
    pin_bwd_finite_difference_f64,
    pin_bwd_sums,
    pin_bwd_identical_keys_and_zero_scale,
    pin_bwd_rows_cols_and_probs,
    pin_bwd_empty,
    pin_kvcache_bruteforce,
    pin_kvcache_unused_slots,
    pin_kvcache_decode_matches_prefill,
    pin_kvcache_paged,
]
