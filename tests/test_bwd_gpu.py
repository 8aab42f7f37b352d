"""Backward (attn_bwd) against the fp64 oracle's gradients, element by
element, under the per-element bound of ``bwd_parity`` (derived from the
kernel's roundings).  The kernel is given the oracle's O (rounded to the
input type) and LSE (fp32) as the forward outputs, so what is measured is
the backward alone; the full-size case also runs on the GPU forward's
outputs for the heads it does not check."""
import math

import numpy as np
import pytest
import torch

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import workloads as W
import oracle
from bwd_parity import bounds, check

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _draw(b, h, sq, sk, dtype, seed, qk_std=1.0, d=128):
    q, k, v = W.draw(b, h, sq, sk, d, dtype, seed, qk_std)
    do = W.draw_grad(b, h, sq, d, dtype, seed + 1000)
    return q, k, v, do


def _gpu_bwd(q, k, v, o, do, lse, causal, scale):
    dev = torch.device("cuda", 0)
    qd, kd, vd, od, dod = (t.to(dev) for t in (q, k, v, o, do))
    ld = lse.to(dev)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    af.attn_bwd(qd, kd, vd, od, dod, ld, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return tuple(t.float().cpu().double().numpy() for t in (dq, dk, dv))


def _fwd_outputs(q, k, v, causal, scale, dtype):
    """The forward's outputs as the backward takes them: the oracle's O
    rounded to the input type, LSE in fp32."""
    o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal, scale)
    return o_ref, lse_ref, torch.from_numpy(o_ref).to(DT[dtype]), torch.from_numpy(lse_ref).float()


def _check_all(q, k, v, do, causal, scale, dtype, what):
    o_ref, lse_ref, o_t, lse_t = _fwd_outputs(q, k, v, causal, scale, dtype)
    dq, dk, dv = _gpu_bwd(q, k, v, o_t, do, lse_t, causal, scale)
    qn, kn, vn, don = (t.double().numpy() for t in (q, k, v, do))
    dq_r, dk_r, dv_r = oracle.attn_bwd(qn, kn, vn, don, causal, scale)
    worst = {}
    for bi in range(q.shape[0]):
        for hi in range(q.shape[1]):
            bq, bk, bv = bounds(qn[bi, hi], kn[bi, hi], vn[bi, hi], don[bi, hi], o_ref[bi, hi], lse_ref[bi, hi],
                                dq_r[bi, hi], dk_r[bi, hi], dv_r[bi, hi], causal, scale, dtype)
            for name, got, ref, bd in (("dq", dq, dq_r, bq), ("dk", dk, dk_r, bk), ("dv", dv, dv_r, bv)):
                r, rel = check(f"{what} {name} ({bi},{hi})", got[bi, hi], ref[bi, hi], bd)
                worst[name] = max(worst.get(name, (0, 0)), (r, rel))
    print(what, {k: (round(a, 3), f"{b:.2e}") for k, (a, b) in worst.items()})
    return dq, dk, dv


SHAPES = [
    # b, h, sq, sk, dtype, causal, d
    (1, 2, 128, 128, "bf16", False, 128),
    (1, 2, 128, 128, "bf16", True, 128),
    (2, 3, 300, 300, "bf16", True, 128),      # ragged tail, several key blocks
    (1, 2, 257, 385, "fp16", False, 128),     # sq != sk, ragged both
    (1, 2, 385, 257, "fp16", True, 128),      # sq > sk: rows that see no key
    (1, 2, 257, 385, "bf16", True, 128),      # sq < sk, bottom-right causal
    (1, 1, 1, 1, "bf16", False, 128),
    (1, 1, 1, 200, "fp16", True, 128),
    (1, 2, 1000, 1000, "bf16", True, 128),
    (2, 2, 640, 640, "fp16", False, 128),
    # head dim 64: dQ = dS K with the queries on the lanes
    (1, 2, 128, 128, "bf16", False, 64),
    (2, 3, 300, 300, "bf16", True, 64),
    (1, 2, 257, 385, "fp16", False, 64),
    (1, 2, 385, 257, "fp16", True, 64),
    (1, 1, 1, 200, "bf16", True, 64),
    (2, 2, 1000, 1000, "bf16", False, 64),
]


@pytest.mark.parametrize("b,h,sq,sk,dtype,causal,d", SHAPES)
def test_bwd_matches_oracle(b, h, sq, sk, dtype, causal, d):
    q, k, v, do = _draw(b, h, sq, sk, dtype, 31000 + sq + 7 * sk + int(causal) + d, d=d)
    _check_all(q, k, v, do, causal, 1.0 / math.sqrt(d), dtype, f"b{b} h{h} sq{sq} sk{sk} {dtype} c{int(causal)} d{d}")


@pytest.mark.parametrize("scale", [0.0, -0.07, 0.3])
def test_bwd_scales(scale):
    q, k, v, do = _draw(1, 2, 200, 260, "bf16", 31500)
    _check_all(q, k, v, do, True, scale, "bf16", f"scale {scale}")


def test_bwd_large_logits():
    """Q, K ~ N(0, 9), as in the long benchmark problem."""
    q, k, v, do = _draw(1, 2, 512, 512, "bf16", 31600, qk_std=3.0)
    _check_all(q, k, v, do, True, 1.0 / math.sqrt(128), "bf16", "qk_std 3")


def test_bwd_empty():
    dev = torch.device("cuda", 0)
    q, k, v, do = _draw(1, 2, 64, 0, "bf16", 31700)
    o = torch.zeros_like(q)
    lse = torch.full((1, 2, 64), -math.inf)
    dq, dk, dv = _gpu_bwd(q, k, v, o, do, lse, True, 0.1)
    assert (dq == 0).all() and dk.size == 0 and dv.size == 0
    q, k, v, do = _draw(1, 2, 0, 64, "bf16", 31701)
    dq, dk, dv = _gpu_bwd(q, k, v, torch.zeros_like(q), do, torch.zeros((1, 2, 0)), False, 0.1)
    assert dq.size == 0 and (dk == 0).all() and (dv == 0).all()


def test_bwd_dk_dv_deterministic():
    """dK and dV are accumulated in one place each (bitwise repeatable); dQ
    is summed over key blocks with fp32 atomics, so only its value up to
    summation order repeats."""
    q, k, v, do = _draw(1, 2, 384, 384, "bf16", 31800)
    _, _, o_t, lse_t = _fwd_outputs(q, k, v, True, 0.09, "bf16")
    a = _gpu_bwd(q, k, v, o_t, do, lse_t, True, 0.09)
    b = _gpu_bwd(q, k, v, o_t, do, lse_t, True, 0.09)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.abs(a[0] - b[0]).max() <= 2.0 ** -7 * np.abs(a[0]).max()


@pytest.mark.parametrize("name", list(W.BWD))
def test_bwd_workload_sampled(name):
    """The benchmarked backward problems at full size.  All heads run with
    the GPU forward's O and LSE, except two sampled heads that get the
    oracle's; on those, sampled rows of dQ and sampled keys of dK, dV are
    checked against the oracle under the same bound."""
    bw = W.BWD[name]
    w = bw.w
    q, k, v = W.inputs(w)
    do = W.draw_grad(w.b, w.h, w.sq, w.d, w.dtype, bw.grad_seed)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = af.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    heads = W.sample_heads(w, n=2)
    rng = np.random.default_rng(5)
    n = 40
    rows = np.unique(np.concatenate([[0, w.sq - 1], rng.integers(0, w.sq, n)]))
    cols = np.unique(np.concatenate([[0, w.sk - 1], rng.integers(0, w.sk, n)]))
    ref = {}
    for bi, hi in heads:
        qn, kn, vn, don = (t[bi, hi].double().numpy() for t in (q, k, v, do))
        o_ref, lse_ref = oracle.attn_fwd(qn[None, None], kn[None, None], vn[None, None], w.causal, w.scale)
        o[bi, hi] = torch.from_numpy(o_ref[0, 0]).to(o.dtype).to(dev)
        lse[bi, hi] = torch.from_numpy(lse_ref[0, 0]).float().to(dev)
        dq_r = oracle.attn_bwd_dq_rows(qn, kn, vn, don, rows, w.causal, w.scale)
        dk_r, dv_r = oracle.attn_bwd_dkv_cols(qn, kn, vn, don, cols, w.causal, w.scale)
        ref[(bi, hi)] = (qn, kn, vn, don, o_ref[0, 0], lse_ref[0, 0], dq_r, dk_r, dv_r)
    dq, dk, dv = af.attn_bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    for (bi, hi), (qn, kn, vn, don, o_ref, lse_ref, dq_r, dk_r, dv_r) in ref.items():
        bq, bk, bv = bounds(qn, kn, vn, don, o_ref, lse_ref, dq_r, dk_r, dv_r, w.causal, w.scale, w.dtype,
                            rows=rows, cols=cols)
        got_q = dq[bi, hi].float().cpu().double().numpy()[rows]
        got_k = dk[bi, hi].float().cpu().double().numpy()[cols]
        got_v = dv[bi, hi].float().cpu().double().numpy()[cols]
        res = [check(f"{name} {nm} ({bi},{hi})", g, r, bd)
               for nm, g, r, bd in (("dq", got_q, dq_r, bq), ("dk", got_k, dk_r, bk), ("dv", got_v, dv_r, bv))]
        print(name, (bi, hi), [(round(a, 3), f"{b:.2e}") for a, b in res])
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()

