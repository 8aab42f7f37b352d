"""Packed variable-length forward against the fp64 oracle, sequence by
sequence (each sequence is an independent attention problem)."""
import math
import zlib

import numpy as np
import pytest
import torch

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import workloads as W
from parity import compare
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # lens_q, lens_k (None = same as q), h, d, dtype, causal
    ([300, 1, 0, 513, 128, 1000], None, 2, 128, "bf16", True),
    ([300, 1, 0, 513, 128, 1000], None, 2, 128, "fp16", False),
    ([77, 256, 257], [400, 1024, 100], 3, 64, "bf16", True),     # sq != sk per sequence
    ([64, 2000], [5000, 31], 2, 128, "fp16", False),
    ([1] * 7, [4096] * 7, 4, 128, "bf16", True),                 # decode-like batch
    ([1500], None, 1, 64, "fp16", True),
]


def _check(lens_q, lens_k, h, d, dtype, causal, seed, qk_std=1.0):
    lens_k = lens_k or lens_q
    q, k, v, cu_q, cu_k, dense = W.draw_varlen(lens_q, lens_k, h, d, dtype, seed, qk_std)
    dev = torch.device("cuda", 0)
    o = torch.full_like(q, float("nan"), device=dev)
    lse = torch.full((h, q.shape[0]), float("nan"), dtype=torch.float32, device=dev)
    af.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev), max(lens_q), max(lens_k),
                       causal=causal, scale=1 / math.sqrt(d), o=o, lse=lse)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for s, (qs, ks, vs) in enumerate(dense):
        a, b = int(cu_q[s]), int(cu_q[s + 1])
        if a == b:
            continue
        o_ref, lse_ref = oracle.attn_fwd(qs.double().numpy(), ks.double().numpy(), vs.double().numpy(), causal,
                                         1 / math.sqrt(d))
        compare(o[a:b].transpose(1, 0, 2)[None], lse[:, a:b][None], o_ref, lse_ref, dtype, f"sequence {s}")


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{len(c[0])}seq_h{c[2]}_d{c[3]}_{c[4]}_c{int(c[5])}")
def test_varlen_matches_oracle(case):
    lens_q, lens_k, h, d, dtype, causal = case
    _check(lens_q, lens_k, h, d, dtype, causal, seed=zlib.crc32(repr(case).encode()))


def test_varlen_large_logits():
    _check([700, 1200], None, 2, 128, "bf16", True, seed=3, qk_std=3.0)


def test_varlen_matches_dense_for_equal_lengths():
    """All sequences of one length: the packed call equals the dense one."""
    q, k, v, cu_q, cu_k, dense = W.draw_varlen([384] * 3, [384] * 3, 2, 128, "bf16", 9)
    dev = torch.device("cuda", 0)
    o_v, l_v = af.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev), 384, 384, causal=True)
    qd = torch.cat([t[0] for t in dense], 0).to(dev)[None].reshape(3, 2, 384, 128)
    kd = torch.cat([t[1] for t in dense], 0).to(dev)[None].reshape(3, 2, 384, 128)
    vd = torch.cat([t[2] for t in dense], 0).to(dev)[None].reshape(3, 2, 384, 128)
    o_d, l_d = af.attn_fwd(qd.contiguous(), kd.contiguous(), vd.contiguous(), causal=True)
    torch.cuda.synchronize()
    o_v = o_v.reshape(3, 384, 2, 128).transpose(1, 2)
    assert torch.equal(o_v.cpu(), o_d.cpu())
    assert torch.equal(l_v.reshape(2, 3, 384).transpose(0, 1).cpu(), l_d.cpu())


@pytest.mark.parametrize("name", list(W.VARLEN))
def test_varlen_workload_full_size(name):
    """The benchmarked packed batch at full size; the shortest and the
    longest sequence and one more are compared with the oracle on two heads."""
    w = W.VARLEN[name]
    q, k, v, cu_q, cu_k, dense = W.varlen_inputs(w)
    lens = w.lengths()
    dev = torch.device("cuda", 0)
    o, lse = af.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev), max(lens), max(lens),
                                causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    assert np.isfinite(o).all()
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 5})
    for s in picks:
        a, b = int(cu_q[s]), int(cu_q[s + 1])
        qs, ks, vs = dense[s]
        for hh in (0, w.h - 1):
            o_ref, lse_ref = oracle.attn_fwd(qs[:, hh:hh + 1].double().numpy(), ks[:, hh:hh + 1].double().numpy(),
                                             vs[:, hh:hh + 1].double().numpy(), w.causal, w.scale)
            compare(o[a:b, hh][None, None], lse[hh, a:b][None, None], o_ref, lse_ref, w.dtype, f"seq {s} head {hh}")


def test_varlen_repeated_launches_reuse_the_schedule_counters():
    """Packed problems hand out work units through a device counter that each
    launch takes from a rotating set of 256 and leaves at zero.  300 launches
    of two alternating problems (so every counter is reused) must each give
    the first result of their problem bit for bit."""
    dev = torch.device("cuda", 0)
    probs = []
    for seed, lens in ((11, [700, 64, 1500]), (12, [300, 2049])):
        q, k, v, cu_q, cu_k, _ = W.draw_varlen(lens, lens, 4, 128, "bf16", seed)
        probs.append(((q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev)), max(lens)))
    ref = []
    for (q, k, v, cq, ck), mx in probs:
        o, lse = af.attn_fwd_varlen(q, k, v, cq, ck, mx, mx, causal=True)
        ref.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    outs = []
    for i in range(300):
        (q, k, v, cq, ck), mx = probs[i % 2]
        outs.append(af.attn_fwd_varlen(q, k, v, cq, ck, mx, mx, causal=True))
    torch.cuda.synchronize()
    for i, (o, lse) in enumerate(outs):
        assert torch.equal(o, ref[i % 2][0]) and torch.equal(lse, ref[i % 2][1]), f"launch {i} differs"


def test_varlen_concurrent_streams():
    """Packed forwards in flight on two streams at once take different
    schedule counters: each gives the result it gives alone."""
    dev = torch.device("cuda", 0)
    probs = []
    for seed, lens in ((21, [900, 333, 1200]), (22, [64, 2000, 17])):
        q, k, v, cu_q, cu_k, _ = W.draw_varlen(lens, lens, 8, 128, "bf16", seed)
        probs.append(((q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev)), max(lens)))
    ref = []
    for (q, k, v, cq, ck), mx in probs:
        o, lse = af.attn_fwd_varlen(q, k, v, cq, ck, mx, mx, causal=True)
        ref.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    outs = [[], []]
    for _ in range(20):
        for i, st in enumerate(streams):
            (q, k, v, cq, ck), mx = probs[i]
            with torch.cuda.stream(st):
                outs[i].append(af.attn_fwd_varlen(q, k, v, cq, ck, mx, mx, causal=True, stream=st))
    torch.cuda.synchronize()
    for i in range(2):
        for n, (o, lse) in enumerate(outs[i]):
            assert torch.equal(o, ref[i][0]) and torch.equal(lse, ref[i][1]), f"stream {i} launch {n} differs"
