"""Packed variable-length backward (attn_bwd_varlen): every sequence against
the fp64 oracle's gradients under the bound of ``bwd_parity``, and against
the dense backward of that sequence alone (dK, dV bit for bit; dQ up to the
order of its fp32 sums)."""
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


def _case(lens_q, lens_k, h, d, dtype, causal, seed):
    q, k, v, cu_q, cu_k, dense = W.draw_varlen(lens_q, lens_k, h, d, dtype, seed)
    scale = 1.0 / math.sqrt(d)
    total_q = q.shape[0]
    g = torch.Generator().manual_seed(seed + 77)
    do = torch.randn(q.shape, generator=g).to(DT[dtype])
    # forward outputs from the oracle (O rounded to the type, LSE fp32), packed
    o = torch.zeros(q.shape, dtype=DT[dtype])
    lse = torch.full((h, total_q), -math.inf, dtype=torch.float32)
    refs = []
    for s, (qs, ks, vs) in enumerate(dense):
        a, b = int(cu_q[s]), int(cu_q[s + 1])
        o_s, l_s = oracle.attn_fwd(qs.double().numpy(), ks.double().numpy(), vs.double().numpy(), causal, scale)
        o[a:b] = torch.from_numpy(o_s[0].transpose(1, 0, 2)).to(DT[dtype])
        lse[:, a:b] = torch.from_numpy(l_s[0]).float()
        do_s = do[a:b].transpose(0, 1)[None].contiguous()
        grads = oracle.attn_bwd(qs.double().numpy(), ks.double().numpy(), vs.double().numpy(),
                                do_s.double().numpy(), causal, scale)
        refs.append((qs, ks, vs, do_s, o_s, l_s, grads))
    dev = torch.device("cuda", 0)
    args = [t.to(dev) for t in (q, k, v, o, do, lse)]
    dq = torch.full_like(args[0], float("nan"))
    dk = torch.full_like(args[1], float("nan"))
    dv = torch.full_like(args[2], float("nan"))
    af.attn_bwd_varlen(*args, cu_q.to(dev), cu_k.to(dev), max(lens_q), max(lens_k), causal=causal, scale=scale,
                       dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return q, k, v, o, do, lse, cu_q, cu_k, dq.cpu(), dk.cpu(), dv.cpu(), refs, scale


CASES = [
    # lens_q, lens_k, h, d, dtype, causal
    ([300, 17, 640, 129], [300, 17, 640, 129], 2, 128, "bf16", True),
    ([300, 17, 640, 129], [300, 17, 640, 129], 2, 128, "fp16", False),
    ([100, 0, 257, 5], [80, 33, 257, 0], 2, 128, "bf16", True),     # a sequence without queries, one without keys
    ([513, 64, 200], [513, 64, 200], 3, 64, "bf16", True),
    ([90, 400], [300, 40], 2, 64, "fp16", False),
]


@pytest.mark.parametrize("lens_q,lens_k,h,d,dtype,causal", CASES)
def test_varlen_bwd_matches_oracle_and_dense(lens_q, lens_k, h, d, dtype, causal):
    q, k, v, o, do, lse, cu_q, cu_k, dq, dk, dv, refs, scale = _case(lens_q, lens_k, h, d, dtype, causal,
                                                                      41000 + sum(lens_q) + d)
    dev = torch.device("cuda", 0)
    for s, (qs, ks, vs, do_s, o_s, l_s, (gq, gk, gv)) in enumerate(refs):
        a, b = int(cu_q[s]), int(cu_q[s + 1])
        c, e = int(cu_k[s]), int(cu_k[s + 1])
        got_q = dq[a:b].transpose(0, 1).float().double().numpy()
        got_k = dk[c:e].transpose(0, 1).float().double().numpy()
        got_v = dv[c:e].transpose(0, 1).float().double().numpy()
        for hi in range(h):
            bq, bk, bv = bounds(qs[0, hi].double().numpy(), ks[0, hi].double().numpy(), vs[0, hi].double().numpy(),
                                do_s[0, hi].double().numpy(), o_s[0, hi], l_s[0, hi], gq[0, hi], gk[0, hi], gv[0, hi],
                                causal, scale, dtype)
            check(f"seq{s} h{hi} dq", got_q[hi], gq[0, hi], bq)
            check(f"seq{s} h{hi} dk", got_k[hi], gk[0, hi], bk)
            check(f"seq{s} h{hi} dv", got_v[hi], gv[0, hi], bv)
        if b > a and e > c:
            # the dense backward of this sequence alone
            ddq, ddk, ddv = af.attn_bwd(qs.to(dev), ks.to(dev), vs.to(dev),
                                        o[a:b].transpose(0, 1)[None].contiguous().to(dev), do_s.to(dev),
                                        lse[:, a:b][None].contiguous().to(dev), causal=causal, scale=scale)
            torch.cuda.synchronize()
            assert torch.equal(ddk[0].cpu(), dk[c:e].transpose(0, 1)), f"seq{s}: dK differs from the dense backward"
            assert torch.equal(ddv[0].cpu(), dv[c:e].transpose(0, 1)), f"seq{s}: dV differs from the dense backward"
            tol = 2.0 ** -7 * float(ddq.abs().max()) + 1e-6
            assert float((ddq[0].cpu().float() - dq[a:b].transpose(0, 1).float()).abs().max()) <= tol


@pytest.mark.parametrize("name", list(W.BWD_VARLEN))
def test_bwd_varlen_workload_sampled(name):
    """The benchmarked packed backward at full size.  All planes run with the
    GPU forward's O and LSE, except two sampled (sequence, head) planes (the
    longest sequence and a seeded other one) that get the oracle's; on
    those, sampled query rows of dQ and sampled keys of dK, dV are checked
    against the oracle under the per-element bound."""
    bw = W.BWD_VARLEN[name]
    w = bw.w
    lens = w.lengths()
    q, k, v, cu_q, cu_k, dense = W.varlen_inputs(w)
    do = W.bwd_varlen_grad(bw)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod, cqd, ckd = (t.to(dev) for t in (q, k, v, do, cu_q, cu_k))
    mx = max(lens)
    o, lse = af.attn_fwd_varlen(qd, kd, vd, cqd, ckd, mx, mx, causal=w.causal, scale=w.scale)
    rng = np.random.default_rng(9)
    longest = int(np.argmax(lens))
    other = int(rng.integers(0, len(lens) - 1))
    other = other + 1 if other >= longest else other
    planes = [(longest, 0), (other, int(rng.integers(0, w.h)))]
    ref = {}
    for s, hi in planes:
        a, L = int(cu_q[s]), lens[s]
        qs, ks, vs = (t[0, hi].double().numpy() for t in dense[s])
        dos = do[a:a + L, hi].double().numpy()
        o_ref, lse_ref = oracle.attn_fwd(qs[None, None], ks[None, None], vs[None, None], w.causal, w.scale)
        o[a:a + L, hi] = torch.from_numpy(o_ref[0, 0]).to(o.dtype).to(dev)
        lse[hi, a:a + L] = torch.from_numpy(lse_ref[0, 0]).float().to(dev)
        rows = np.unique(np.concatenate([[0, L - 1], rng.integers(0, L, 40)]))
        cols = np.unique(np.concatenate([[0, L - 1], rng.integers(0, L, 40)]))
        dq_r = oracle.attn_bwd_dq_rows(qs, ks, vs, dos, rows, w.causal, w.scale)
        dk_r, dv_r = oracle.attn_bwd_dkv_cols(qs, ks, vs, dos, cols, w.causal, w.scale)
        ref[(s, hi)] = (qs, ks, vs, dos, o_ref[0, 0], lse_ref[0, 0], rows, cols, dq_r, dk_r, dv_r)
    dq, dk, dv = af.attn_bwd_varlen(qd, kd, vd, o, dod, lse, cqd, ckd, mx, mx, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    for (s, hi), (qs, ks, vs, dos, o_ref, lse_ref, rows, cols, dq_r, dk_r, dv_r) in ref.items():
        a = int(cu_q[s])
        bq, bk, bv = bounds(qs, ks, vs, dos, o_ref, lse_ref, dq_r, dk_r, dv_r, w.causal, w.scale, w.dtype,
                            rows=rows, cols=cols)
        ri = torch.as_tensor(a + rows, device=dev)
        ci = torch.as_tensor(a + cols, device=dev)
        got_q = dq[ri, hi].float().cpu().double().numpy()
        got_k = dk[ci, hi].float().cpu().double().numpy()
        got_v = dv[ci, hi].float().cpu().double().numpy()
        res = [check(f"{name} {nm} (seq {s}, head {hi})", g, r, bd)
               for nm, g, r, bd in (("dq", got_q, dq_r, bq), ("dk", got_k, dk_r, bk), ("dv", got_v, dv_r, bv))]
        print(name, (s, hi), [(round(x, 3), f"{y:.2e}") for x, y in res])
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [128, 64])
def test_varlen_nonfinite_neighbour_does_not_leak(causal, d):
    """Tiles that cross a sequence's end read the next sequence's tokens.
    With every input of the second sequence set to NaN, the first
    sequence's forward outputs and gradients must be those of a clean run
    (O, LSE, dK, dV bit for bit; dQ up to the order of its fp32 sums)."""
    lens = [300, 200]
    h = 2
    q, k, v, cu_q, cu_k, _ = W.draw_varlen(lens, lens, h, d, "bf16", 4242 + d)
    g = torch.Generator().manual_seed(4343)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    cq, ck = cu_q.to(dev), cu_k.to(dev)
    n0 = lens[0]

    def run(poison):
        qd, kd, vd, dod = (t.clone().to(dev) for t in (q, k, v, do))
        if poison:
            for t in (qd, kd, vd, dod):
                t[n0:] = float("nan")
        o, lse = af.attn_fwd_varlen(qd, kd, vd, cq, ck, max(lens), max(lens), causal=causal)
        if poison:
            o[n0:] = float("nan")
            lse[:, n0:] = float("nan")
        dq, dk, dv = af.attn_bwd_varlen(qd, kd, vd, o, dod, lse, cq, ck, max(lens), max(lens), causal=causal)
        torch.cuda.synchronize()
        return [t[:n0].cpu() for t in (o, dq, dk, dv)] + [lse[:, :n0].cpu()]

    clean = run(False)
    dirty = run(True)
    for name, a, b in zip(("o", "dq", "dk", "dv", "lse"), clean, dirty):
        assert torch.isfinite(b).all(), f"{name}: non-finite values leaked into the first sequence"
        if name == "dq":
            assert torch.allclose(a.float(), b.float(), rtol=1e-2, atol=1e-3), name
        else:
            assert torch.equal(a, b), f"{name} differs from the clean run"
