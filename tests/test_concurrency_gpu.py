"""Concurrent use of the library: host threads calling the forward at once
on their own streams with shapes of their own (the tensor-map cache and the
per-thread error message are shared state), and backward calls in flight on
two streams at once with a workspace each.  Every result is compared with a
result of the same call made alone."""
import math
import threading

import torch
import pytest

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import binding
from attention_forward_14_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def test_forward_from_several_host_threads():
    shapes = [(1, 2, 300, 300, 128, True), (2, 1, 513, 257, 64, False), (1, 3, 1000, 1000, 128, False),
              (1, 1, 129, 700, 64, True)]
    inputs = [tuple(t.to(DEV) for t in W.draw(b, h, sq, sk, d, "bf16", seed=100 + i))
              for i, (b, h, sq, sk, d, _) in enumerate(shapes)]
    alone = []
    for (b, h, sq, sk, d, causal), (q, k, v) in zip(shapes, inputs):
        alone.append(af.attn_fwd(q, k, v, causal=causal))
    torch.cuda.synchronize()
    results, errors = {}, []

    def worker(i):
        try:
            b, h, sq, sk, d, causal = shapes[i]
            q, k, v = inputs[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                outs = [af.attn_fwd(q, k, v, causal=causal, stream=st) for _ in range(20)]
            st.synchronize()
            results[i] = outs
        except Exception as e:  # reported below, in the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, outs in results.items():
        for o, lse in outs:
            assert torch.equal(o, alone[i][0]) and torch.equal(lse, alone[i][1]), f"shape {shapes[i]}"
    assert binding.status()[0] == 0


def test_backward_on_two_streams_at_once():
    """Two backward calls in flight at once, each with its own workspace (as
    the header requires): both equal the same calls made alone (dK, dV bit for
    bit; dQ up to the order of its fp32 sums)."""
    cases = [(1, 4, 1024, 1024, 128, True, 200), (2, 2, 700, 900, 64, False, 201)]
    runs = []
    for b, h, sq, sk, d, causal, seed in cases:
        q, k, v = (t.to(DEV) for t in W.draw(b, h, sq, sk, d, "bf16", seed=seed))
        do = W.draw_grad(b, h, sq, d, "bf16", seed + 50).to(DEV)
        o, lse = af.attn_fwd(q, k, v, causal=causal)
        ref = af.attn_bwd(q, k, v, o, do, lse, causal=causal)
        ws = torch.empty(af.bwd_workspace_bytes(b, h, sq, d), dtype=torch.uint8, device=DEV)
        runs.append((q, k, v, o, do, lse, causal, ref, ws))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    for rep in range(5):
        for i, (q, k, v, o, do, lse, causal, _, ws) in enumerate(runs):
            with torch.cuda.stream(streams[i]):
                outs[i].append(af.attn_bwd(q, k, v, o, do, lse, causal=causal, workspace=ws, stream=streams[i]))
        # the next launches on a stream may reuse its workspace only after this one
    torch.cuda.synchronize()
    for i, (*_, ref, _ws) in enumerate(runs):
        for dq, dk, dv in outs[i]:
            assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
            diff = (dq.float() - ref[0].float()).abs().max().item()
            assert diff <= 2.0 ** -7 * ref[0].float().abs().max().item(), diff
    assert binding.status()[0] == 0
