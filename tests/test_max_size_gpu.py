"""Problems with more than 2^32 elements per tensor, so that element offsets
of Q, K, V, O (and, in the backward, of dO, dQ, dK, dV and the fp32 dQ
accumulator) pass 2^31 and 2^32, where a 32-bit index would wrap.

Inputs are drawn on the device (``workloads.randn_device``, seeded); the
heads and sequences compared with the fp64 oracle are copied back to the
host: the first and the last, and those whose elements straddle 2^31 and
2^32.  Outputs start as NaN, so an element the kernels never write fails the
finiteness check over the whole tensor, and a write through a wrapped index
lands in a low head, which the checked first heads catch.  Each test holds
about 90 GB of device memory at its peak; the checked build runs the two
forwards first (the kernels' index checks report a violation instead of
making the access)."""
import math

import numpy as np
import pytest
import torch

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import workloads as W
from parity import compare
from bwd_parity import bounds, check
import oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _need_memory(gib):
    torch.cuda.empty_cache()  # blocks cached by earlier tests count as used
    free, _ = torch.cuda.mem_get_info(DEV)
    if free < gib * (1 << 30):
        pytest.skip(f"needs {gib} GiB of free device memory, {free / (1 << 30):.0f} GiB free")


def _host(t):
    return t.float().cpu().double().numpy()


# 2 x 52430 heads of 320 x 128: 4,295,065,600 elements per tensor; head
# 52428 straddles element 2^31 and head 104857 (batch 1, head 52427) element
# 2^32.  320 rows and keys: a ragged second unit and key tile.
DENSE = dict(b=2, h=52430, s=320, d=128, dtype="bf16", causal=True)
# about 1,060 sequences of 1 to 2048 tokens, 32 heads of 128: more than 2^20
# tokens, so element (token * 32 + head) * 128 passes 2^32; token 2^19 is
# element 2^31.
VARLEN = dict(n=1060, lo=1, hi=2048, seed=41010, h=32, d=128, dtype="bf16", causal=True)


def dense_forward():
    """The dense forward at more than 2^32 elements per tensor, checked on
    the boundary heads; returns the device tensors and the oracle's values
    for the checked heads."""
    b, h, s, d, dtype, causal = (DENSE[x] for x in ("b", "h", "s", "d", "dtype", "causal"))
    scale = 1.0 / math.sqrt(d)
    n = b * h * s * d
    assert n > 2 ** 32
    _need_memory(100)
    q = W.randn_device((b, h, s, d), dtype, 41001, DEV)
    k = W.randn_device((b, h, s, d), dtype, 41002, DEV)
    v = W.randn_device((b, h, s, d), dtype, 41003, DEV)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((b, h, s), float("nan"), dtype=torch.float32, device=DEV)
    af.attn_fwd(q, k, v, causal=causal, scale=scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and not torch.isnan(lse).any()
    heads = [(0, 0), (0, 52428), (0, h - 1), (1, 0), (1, 52427), (1, h - 1)]
    head_elems = s * d
    for bi, hi in heads:
        first = (bi * h + hi) * head_elems
        if (bi, hi) == (0, 52428):
            assert first < 2 ** 31 < first + head_elems
        if (bi, hi) == (1, 52427):
            assert first < 2 ** 32 < first + head_elems
    ref = {}
    for bi, hi in heads:
        qn, kn, vn = (_host(t[bi, hi]) for t in (q, k, v))
        o_ref, lse_ref = oracle.attn_fwd(qn[None, None], kn[None, None], vn[None, None], causal, scale)
        compare(_host(o[bi, hi])[None, None], lse[bi, hi].cpu().double().numpy()[None, None], o_ref, lse_ref, dtype,
                f"forward head ({bi},{hi})")
        ref[(bi, hi)] = (qn, kn, vn, o_ref[0, 0], lse_ref[0, 0])
    return q, k, v, o, lse, ref


def test_dense_forward_and_backward_past_2_32_elements():
    b, h, s, d, dtype, causal = (DENSE[x] for x in ("b", "h", "s", "d", "dtype", "causal"))
    scale = 1.0 / math.sqrt(d)
    q, k, v, o, lse, ref = dense_forward()
    # Backward on the GPU forward's O and LSE, except the checked heads,
    # which get the oracle's (the bound assumes O rounded from the exact one).
    do = W.randn_device((b, h, s, d), dtype, 41004, DEV)
    for (bi, hi), (_, _, _, o_ref, lse_ref) in ref.items():
        o[bi, hi] = torch.from_numpy(o_ref).to(o.dtype).to(DEV)
        lse[bi, hi] = torch.from_numpy(lse_ref).float().to(DEV)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    af.attn_bwd(q, k, v, o, do, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    for (bi, hi), (qn, kn, vn, o_ref, lse_ref) in ref.items():
        don = _host(do[bi, hi])
        dq_r, dk_r, dv_r = oracle.attn_bwd(qn[None, None], kn[None, None], vn[None, None], don[None, None], causal,
                                           scale)
        bq, bk, bv = bounds(qn, kn, vn, don, o_ref, lse_ref, dq_r[0, 0], dk_r[0, 0], dv_r[0, 0], causal, scale, dtype)
        for name, got, r, bd in (("dq", dq, dq_r, bq), ("dk", dk, dk_r, bk), ("dv", dv, dv_r, bv)):
            check(f"backward {name} ({bi},{hi})", _host(got[bi, hi]), r[0, 0], bd)
    del q, k, v, o, lse, do, dq, dk, dv
    torch.cuda.empty_cache()


def varlen_forward():
    """The packed forward at more than 2^32 elements per tensor, checked on
    the first and last sequences and those holding tokens 2^19 and 2^20;
    returns the device tensors, the offsets and the oracle's values."""
    h, d, dtype, causal = (VARLEN[x] for x in ("h", "d", "dtype", "causal"))
    scale = 1.0 / math.sqrt(d)
    lens = W.varlen_lengths(VARLEN["n"], VARLEN["lo"], VARLEN["hi"], VARLEN["seed"])
    total = sum(lens)
    assert total * h * d > 2 ** 32
    _need_memory(100)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)
    cu_d = cu.to(torch.int32).to(DEV)
    q = W.randn_device((total, h, d), dtype, 41011, DEV)
    k = W.randn_device((total, h, d), dtype, 41012, DEV)
    v = W.randn_device((total, h, d), dtype, 41013, DEV)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((h, total), float("nan"), dtype=torch.float32, device=DEV)
    af.attn_fwd_varlen(q, k, v, cu_d, cu_d, max(lens), max(lens), causal=causal, scale=scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and not torch.isnan(lse).any()
    starts = cu.tolist()

    def seq_of(tok):
        return int(np.searchsorted(np.asarray(starts), tok, side="right")) - 1

    seqs = sorted({0, seq_of(2 ** 19), seq_of(2 ** 20), len(lens) - 1})
    ref = {}
    for si in seqs:
        a, e = starts[si], starts[si + 1]
        qs, ks, vs = (_host(t[a:e]).transpose(1, 0, 2)[None] for t in (q, k, v))  # [1, h, len, d]
        o_ref, lse_ref = oracle.attn_fwd(qs, ks, vs, causal, scale)
        compare(_host(o[a:e]).transpose(1, 0, 2)[None], lse[:, a:e].cpu().double().numpy()[None], o_ref, lse_ref,
                dtype, f"varlen forward sequence {si} (tokens {a}..{e})")
        ref[si] = (qs[0], ks[0], vs[0], o_ref[0], lse_ref[0])
    return q, k, v, o, lse, lens, starts, cu_d, ref


def test_varlen_forward_and_backward_past_2_32_elements():
    h, d, dtype, causal = (VARLEN[x] for x in ("h", "d", "dtype", "causal"))
    scale = 1.0 / math.sqrt(d)
    q, k, v, o, lse, lens, starts, cu_d, ref = varlen_forward()
    total = q.shape[0]
    do = W.randn_device((total, h, d), dtype, 41014, DEV)
    for si, (_, _, _, o_ref, lse_ref) in ref.items():
        a, e = starts[si], starts[si + 1]
        o[a:e] = torch.from_numpy(o_ref.transpose(1, 0, 2).copy()).to(o.dtype).to(DEV)
        lse[:, a:e] = torch.from_numpy(lse_ref).float().to(DEV)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    af.attn_bwd_varlen(q, k, v, o, do, lse, cu_d, cu_d, max(lens), max(lens), causal=causal, scale=scale,
                       dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    for si, (qs, ks, vs, o_ref, lse_ref) in ref.items():
        a, e = starts[si], starts[si + 1]
        dos = _host(do[a:e]).transpose(1, 0, 2)  # [h, len, d]
        heads = [0, h - 1]  # every head of a straddling sequence crosses the boundary
        for hi in heads:
            dq_r, dk_r, dv_r = oracle.attn_bwd(qs[hi][None, None], ks[hi][None, None], vs[hi][None, None],
                                               dos[hi][None, None], causal, scale)
            bq, bk, bv = bounds(qs[hi], ks[hi], vs[hi], dos[hi], o_ref[hi], lse_ref[hi], dq_r[0, 0], dk_r[0, 0],
                                dv_r[0, 0], causal, scale, dtype)
            for name, got, r, bd in (("dq", dq, dq_r, bq), ("dk", dk, dk_r, bk), ("dv", dv, dv_r, bv)):
                check(f"varlen backward {name} sequence {si} head {hi}", _host(got[a:e, hi]), r[0, 0], bd)
    del q, k, v, o, lse, do, dq, dk, dv
    torch.cuda.empty_cache()


def test_long_sequence_forward_and_backward_sampled_rows():
    """Two heads of 2^17 tokens, causal: 1,024 key tiles for the last query
    block, row and key indices up to 2^17.  Sampled rows (the first, the
    last, the unit and tile boundaries and seeded others) of O, LSE and dQ
    against the oracle; the backward gets the oracle's O and LSE on those
    rows (the bound assumes them) and the forward's elsewhere."""
    b, h, s, d, dtype = 1, 2, 1 << 17, 128, "bf16"
    causal, scale = True, 1.0 / math.sqrt(d)
    q, k, v = W.draw(b, h, s, s, d, dtype, seed=41020)
    do = W.draw_grad(b, h, s, d, dtype, seed=41021)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = af.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(41022)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, s // 2 - 1, s // 2, s - 257, s - 256, s - 1],
                                     rng.integers(0, s, 16)]))
    ref = {}
    for hi in range(h):
        qn, kn, vn = (t[0, hi].double().numpy() for t in (q, k, v))
        o_r, lse_r = oracle.attn_head_rows(qn, kn, vn, rows, causal, scale)
        compare(o[0, hi].float().cpu().double().numpy()[rows], lse[0, hi].cpu().double().numpy()[rows], o_r, lse_r,
                dtype, f"forward rows of head {hi}")
        ri = torch.from_numpy(rows).to(DEV)
        o[0, hi, ri] = torch.from_numpy(o_r).to(o.dtype).to(DEV)
        lse[0, hi, ri] = torch.from_numpy(lse_r).float().to(DEV)
        ref[hi] = (qn, kn, vn)
    dq, dk, dv = af.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    for hi, (qn, kn, vn) in ref.items():
        don = do[0, hi].double().numpy()
        dq_r = oracle.attn_bwd_dq_rows(qn, kn, vn, don, rows, causal, scale)
        on = o[0, hi].float().cpu().double().numpy()
        ln = lse[0, hi].cpu().double().numpy()
        bq, _, _ = bounds(qn, kn, vn, don, on, ln, dq_r, np.zeros((0, d)), np.zeros((0, d)), causal, scale, dtype,
                          rows=rows, cols=np.zeros(0, dtype=np.int64))
        check(f"dq rows of head {hi}", dq[0, hi].float().cpu().double().numpy()[rows], dq_r, bq)
