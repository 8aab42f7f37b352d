"""The dynamic schedule's counter slots (attn_fwd_varlen, attn_fwd_kvcache)
are tagged per launch: two launches in flight on one slot must be reported
in the status word, never share the counters silently.  The slot is forced
with the testing hook attn_fwd_sched_pin_slot.  Nothing here waits on
another launch inside a kernel: a launch that finds its slot held takes no
work and returns."""
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

SLOT = 17
COLLISION, SITE_SCHED_SLOT = 2, 11


def _kv_problem(b, h, sq, cap, lens, seed):
    dev = torch.device("cuda", 0)
    q, kc, vc = W.draw(b, h, sq, cap, 128, "bf16", seed)
    return (q, kc, vc), tuple(t.to(dev) for t in (q, kc, vc)), torch.tensor(lens, dtype=torch.int32, device=dev)


def _check_rows(o, lse, q, kc, vc, lens, rows, what):
    scale = 1 / math.sqrt(128)
    for bi in range(q.shape[0]):
        for hi in range(q.shape[1]):
            L = lens[bi]
            o_ref, lse_ref = oracle.attn_head_rows(q[bi, hi].double().numpy(), kc[bi, hi, :L].double().numpy(),
                                                   vc[bi, hi, :L].double().numpy(), rows, False, scale)
            compare(o[bi, hi][rows].float().cpu().double().numpy(), lse[bi, hi][rows].cpu().double().numpy(),
                    o_ref, lse_ref, "bf16", f"{what} ({bi},{hi})")


def _lib():
    lib = binding.load()
    binding.status_clear()
    return lib


def test_launches_in_flight_on_one_slot_report_a_collision():
    lib = _lib()
    try:
        assert lib.attn_fwd_sched_pin_slot(SLOT) == 0
        # A: one long unit (256 queries against 2^18 cached keys, about 3 ms)
        cap_a = 1 << 18
        (qa, ka, va), (qad, kad, vad), la = _kv_problem(1, 1, 256, cap_a, [cap_a], 31)
        # B: a small decoding step, enqueued on another stream while A runs
        (qb, kb, vb), (qbd, kbd, vbd), lb = _kv_problem(2, 2, 1, 640, [200, 639], 32)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        oa = torch.full_like(qad, float("nan"))
        lsea = torch.full(qad.shape[:3], float("nan"), dtype=torch.float32, device=qad.device)
        ob = torch.full_like(qbd, float("nan"))
        lseb = torch.full(qbd.shape[:3], float("nan"), dtype=torch.float32, device=qbd.device)
        torch.cuda.synchronize()
        af.attn_fwd_kvcache(qad, kad, vad, la, num_splits=1, o=oa, lse=lsea, stream=s1)
        af.attn_fwd_kvcache(qbd, kbd, vbd, lb, num_splits=1, o=ob, lse=lseb, stream=s2)
        torch.cuda.synchronize()
        code, _, _, site = binding.status()
        assert (code, site) == (COLLISION, SITE_SCHED_SLOT)
        # A owned the slot and is intact; B took no work (its outputs stay unwritten)
        _check_rows(oa, lsea, qa, ka, va, [cap_a], np.arange(0, 256, 9), "launch holding the slot")
        assert torch.isnan(ob.float()).all() and torch.isnan(lseb).all()
        # after the clear, the slot is free again and B runs correctly on it
        binding.status_clear()
        af.attn_fwd_kvcache(qbd, kbd, vbd, lb, num_splits=1, o=ob, lse=lseb)
        torch.cuda.synchronize()
        assert binding.status()[0] == 0
        _check_rows(ob, lseb, qb, kb, vb, [200, 639], np.array([0]), "after clear")
    finally:
        lib.attn_fwd_sched_pin_slot(-1)
        binding.status_clear()


def test_launches_one_after_another_share_a_slot_cleanly():
    """Launches on one slot that do not overlap (one stream) are not
    collisions: each frees the slot for the next."""
    lib = _lib()
    try:
        assert lib.attn_fwd_sched_pin_slot(SLOT) == 0
        (q, kc, vc), (qd, kd, vd), lens = _kv_problem(2, 2, 3, 700, [650, 100], 33)
        for _ in range(5):
            o, lse = af.attn_fwd_kvcache(qd, kd, vd, lens, num_splits=1)
        torch.cuda.synchronize()
        assert binding.status()[0] == 0
        _check_rows(o, lse, q, kc, vc, [650, 100], np.arange(3), "sequential on one slot")
    finally:
        lib.attn_fwd_sched_pin_slot(-1)
