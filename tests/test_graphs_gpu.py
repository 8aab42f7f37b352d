"""The entry points captured in CUDA graphs and replayed: the forward, the
packed forward (dynamic schedule: each replay reuses the captured
generation, one replay at a time) and the backward (prep, main and convert
kernels).  Replays read the inputs as they are at replay time: each replay
follows an in-place change of the inputs and is compared with an eager call
on the same inputs (the forward bit for bit; the backward's dK, dV bit for
bit and dQ, summed in another order, within a bound) and the forward with
the fp64 oracle.  The status word stays clean."""
import math

import numpy as np
import pytest
import torch

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import binding
from attention_forward_14_gb300 import workloads as W
from parity import compare
import oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _capture(fn):
    """Capture fn() on a side stream (after one eager call, which sets up the
    library's per-device state outside the capture)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    torch.cuda.synchronize()
    return g


def test_forward_graph_replays_follow_the_inputs():
    b, h, s, d = 2, 3, 700, 128
    q, k, v = (t.to(DEV) for t in W.draw(b, h, s, s, d, "bf16", seed=51))
    o = torch.empty_like(q)
    lse = torch.empty(b, h, s, dtype=torch.float32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    g = _capture(lambda st: af.attn_fwd(q, k, v, causal=True, scale=scale, o=o, lse=lse, stream=st))
    binding.status_clear()
    for rep in range(3):
        nq, nk, nv = W.draw(b, h, s, s, d, "bf16", seed=60 + rep)
        q.copy_(nq)
        k.copy_(nk)
        v.copy_(nv)
        g.replay()
        torch.cuda.synchronize()
        o_g, lse_g = o.clone(), lse.clone()
        o_e, lse_e = af.attn_fwd(q, k, v, causal=True, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e), f"replay {rep} differs from the eager call"
        o_ref, lse_ref = oracle.attn_fwd(nq.double().numpy(), nk.double().numpy(), nv.double().numpy(), True, scale)
        compare(o_g.float().cpu().double().numpy(), lse_g.cpu().double().numpy(), o_ref, lse_ref, "bf16",
                f"graph replay {rep}")
    assert binding.status()[0] == 0


def test_packed_forward_graph_replays_one_at_a_time():
    lens = [300, 1, 513, 128, 1000]
    h, d = 2, 64
    q, k, v, cu_q, cu_k, dense = W.draw_varlen(lens, lens, h, d, "fp16", seed=71)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    cq, ck = cu_q.to(DEV), cu_k.to(DEV)
    o = torch.empty_like(qd)
    lse = torch.empty(h, q.shape[0], dtype=torch.float32, device=DEV)
    g = _capture(lambda st: af.attn_fwd_varlen(qd, kd, vd, cq, ck, max(lens), max(lens), causal=True,
                                               o=o, lse=lse, stream=st))
    binding.status_clear()
    o_e, lse_e = af.attn_fwd_varlen(qd, kd, vd, cq, ck, max(lens), max(lens), causal=True)
    torch.cuda.synchronize()
    for rep in range(4):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_e) and torch.equal(lse, lse_e), f"replay {rep} differs from the eager call"
    assert binding.status()[0] == 0


def test_backward_graph_replays_follow_the_inputs():
    b, h, s, d = 1, 2, 640, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.to(DEV) for t in W.draw(b, h, s, s, d, "bf16", seed=81))
    do = W.draw_grad(b, h, s, d, "bf16", 82).to(DEV)
    o, lse = af.attn_fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(af.bwd_workspace_bytes(b, h, s, d), dtype=torch.uint8, device=DEV)
    g = _capture(lambda st: af.attn_bwd(q, k, v, o, do, lse, causal=True, scale=scale, dq=dq, dk=dk, dv=dv,
                                        workspace=ws, stream=st))
    binding.status_clear()
    for rep in range(3):
        do.copy_(W.draw_grad(b, h, s, d, "bf16", 90 + rep))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (dq, dk, dv)]
        ref = af.attn_bwd(q, k, v, o, do, lse, causal=True, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]), f"replay {rep}: dK / dV differ"
        # dQ: fp32 sums over key blocks in another order, then one rounding
        diff = (got[0].float() - ref[0].float()).abs().max().item()
        assert diff <= 2.0 ** -7 * ref[0].float().abs().max().item(), (rep, diff)
    assert binding.status()[0] == 0
