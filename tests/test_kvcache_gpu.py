"""KV-cache forward (new rows written into the cache at each batch element's
length, then attention over the valid keys, split-KV or not) against the
fp64 oracle on seeded inputs.  Unused cache slots hold NaN throughout: none
of it may reach the result."""
import math
import zlib

import numpy as np
import pytest
import torch

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import binding
from attention_forward_14_gb300 import workloads as W
from parity import compare
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # b, h, sq, s_cache, s_new, d, dtype, causal, splits, cache lengths
    (4, 8, 1, 4096, 1, 128, "bf16", True, 1, (4095, 17, 0, 2048)),    # decode, one fills the cache
    (4, 8, 1, 4096, 1, 128, "bf16", True, 8, (4095, 17, 0, 2048)),    # the same, split-KV
    (3, 4, 1, 3000, 0, 64, "fp16", False, 4, (3000, 129, 1)),          # no new rows
    (2, 2, 5, 1000, 5, 128, "fp16", True, 3, (100, 997)),              # last rows dropped (full)
    (2, 2, 300, 700, 300, 128, "bf16", True, 1, (0, 400)),             # chunked prefill into a cache
    (2, 2, 300, 700, 300, 128, "bf16", True, 3, (0, 400)),             # the same, split-KV
    (2, 4, 40, 2000, 40, 64, "fp16", True, 5, (1960, 700)),            # speculative-decode-sized chunk, d = 64
    (2, 2, 64, 500, 0, 64, "bf16", True, 2, (10, -5)),                 # rows with no key, negative length
    (1, 2, 8, 256, 2, 128, "bf16", False, 2, (1000,)),                 # length beyond capacity: clamped
    (2, 3, 2, 130, 1, 64, "fp16", True, 2, (127, 128)),                # tail tiles of one key
    (3, 2, 1, 0, 0, 128, "bf16", False, 1, (0, 5, -1)),                # empty cache
]


def _draw_case(case):
    b, h, sq, cap, s_new, d, dt, causal, splits, lens = case
    seed = zlib.crc32(repr(case).encode())
    q, _, _ = W.draw(b, h, sq, 1, d, dt, seed=seed)
    _, kc, vc = W.draw(b, h, 1, cap, d, dt, seed=seed + 1)
    if s_new:
        _, kn, vn = W.draw(b, h, 1, s_new, d, dt, seed=seed + 2)
    else:
        kn = vn = None
    for e, n in enumerate(lens):  # unused slots: NaN
        start = min(max(n, 0), cap)
        kc[e, :, start:] = float("nan")
        vc[e, :, start:] = float("nan")
    return q, kc, vc, kn, vn


def _run(case, q, kc, vc, kn, vn, scale):
    b, h, sq, cap, s_new, d, dt, causal, splits, lens = case
    dev = torch.device("cuda", 0)
    kcd, vcd = kc.to(dev), vc.to(dev)
    seqlens = torch.tensor(lens, dtype=torch.int32, device=dev)
    o = torch.full((b, h, sq, d), float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full((b, h, sq), float("nan"), dtype=torch.float32, device=dev)
    af.attn_fwd_kvcache(q.to(dev), kcd, vcd, seqlens, kn.to(dev) if kn is not None else None,
                        vn.to(dev) if vn is not None else None, causal=causal, scale=scale,
                        num_splits=splits, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(seqlens.cpu(), torch.tensor(lens, dtype=torch.int32)), "cache_seqlens was modified"
    return (o.float().cpu().double().numpy(), lse.cpu().double().numpy(),
            kcd.float().cpu().double().numpy(), vcd.float().cpu().double().numpy())


def _np(t):
    return None if t is None else t.double().numpy()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c[:9])))
def test_kvcache_matches_oracle(case):
    b, h, sq, cap, s_new, d, dt, causal, splits, lens = case
    q, kc, vc, kn, vn = _draw_case(case)
    scale = 1 / math.sqrt(d)
    o, lse, kc_out, vc_out = _run(case, q, kc, vc, kn, vn, scale)
    o_ref, lse_ref, kc_ref, vc_ref = oracle.attn_fwd_kvcache(_np(q), _np(kc), _np(vc), list(lens), _np(kn),
                                                             _np(vn), causal, scale)
    compare(o, lse, o_ref, lse_ref, dt, f"kvcache {case}")
    # the cache write is a copy: bit-exact, NaN slots included
    assert np.array_equal(kc_out, kc_ref, equal_nan=True), "k_cache after the write differs"
    assert np.array_equal(vc_out, vc_ref, equal_nan=True), "v_cache after the write differs"


def test_kvcache_decode_loop_matches_causal_prefill():
    """Sixteen decode steps (one query, one new key/value each) reproduce the
    rows of one causal forward over the whole sequence, step by step."""
    b, h, s0, steps, d, cap = 2, 4, 1000, 16, 128, 1100
    scale = 1 / math.sqrt(d)
    q, k, v = W.draw(b, h, s0 + steps, s0 + steps, d, "bf16", seed=4242)
    o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), True, scale)
    dev = torch.device("cuda", 0)
    kc = torch.full((b, h, cap, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(kc, float("nan"))
    kc[:, :, :s0] = k[:, :, :s0].to(dev)
    vc[:, :, :s0] = v[:, :, :s0].to(dev)
    for t in range(s0, s0 + steps):
        seqlens = torch.full((b,), t, dtype=torch.int32, device=dev)
        sl = slice(t, t + 1)
        o, lse = af.attn_fwd_kvcache(q[:, :, sl].contiguous().to(dev), kc, vc, seqlens,
                                     k[:, :, sl].contiguous().to(dev), v[:, :, sl].contiguous().to(dev),
                                     causal=True, scale=scale, num_splits=3)
        torch.cuda.synchronize()
        compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref[:, :, sl], lse_ref[:, :, sl],
                "bf16", f"decode step {t}")
    assert torch.equal(kc[:, :, :s0 + steps].cpu(), k)


def test_kvcache_full_cache_equals_plain_forward():
    """Every element at full capacity, nothing new: the same bits as
    attn_fwd (the same kernel, the same tiles, only the lengths come from
    the device)."""
    dev = torch.device("cuda", 0)
    q, k, v = W.draw(2, 4, 300, 2000, 128, "fp16", seed=91)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    seqlens = torch.full((2,), 2000, dtype=torch.int32, device=dev)
    for causal in (False, True):
        o1, l1 = af.attn_fwd(qd, kd, vd, causal=causal)
        o2, l2 = af.attn_fwd_kvcache(qd, kd, vd, seqlens, causal=causal, num_splits=1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_kvcache_argument_errors():
    dev = torch.device("cuda", 0)
    q = torch.zeros((1, 1, 1, 64), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device=dev)
    seqlens = torch.zeros((1,), dtype=torch.int32, device=dev)
    with pytest.raises(binding.AttnError) as e:  # new rows inside the cache itself
        af.attn_fwd_kvcache(q, kc, kc.clone(), seqlens, kc[:, :, :1], kc[:, :, 1:2], num_splits=1)
    assert e.value.code == -2
    with pytest.raises(binding.AttnError) as e:  # more splits than key tiles
        af.attn_fwd_kvcache(q, kc, kc.clone(), seqlens, num_splits=3)
    assert e.value.code == -2


PAGED_CASES = [
    # b, h, sq, page_size, pages_per_seq, s_new, d, dtype, causal, splits, cache lengths
    (3, 4, 1, 128, 12, 1, 128, "bf16", True, 1, (1535, 300, 0)),     # decode; one element fills its pages
    (3, 4, 1, 256, 6, 1, 128, "bf16", True, 4, (1000, 17, 1400)),    # split-KV, 256-key pages
    (2, 2, 33, 128, 5, 33, 64, "fp16", True, 3, (100, 600)),          # a chunk of new tokens, d = 64
    (2, 3, 4, 384, 2, 0, 128, "fp16", False, 2, (700, 5)),           # no new rows, 3-tile pages
]


def _paged_case(case):
    b, h, sq, ps, pps, s_new, d, dt, causal, splits, lens = case
    seed = zlib.crc32(repr(case).encode())
    num_pages = b * pps + 3  # three pages no element uses
    q, _, _ = W.draw(b, h, sq, 1, d, dt, seed=seed)
    _, kp, vp = W.draw(1, num_pages * ps, 1, h, d, dt, seed=seed + 1)  # [1, num_pages*ps, h, d] as pool rows
    kp = kp.reshape(num_pages, ps, h, d).contiguous()
    vp = vp.reshape(num_pages, ps, h, d).contiguous()
    if s_new:
        _, kn, vn = W.draw(b, h, 1, s_new, d, dt, seed=seed + 2)
    else:
        kn = vn = None
    g = torch.Generator().manual_seed(seed + 3)
    table = torch.randperm(num_pages, generator=g)[: b * pps].reshape(b, pps).to(torch.int32)
    used = set(table.flatten().tolist())
    for pg in range(num_pages):  # pages no element uses: NaN
        if pg not in used:
            kp[pg] = float("nan")
            vp[pg] = float("nan")
    for e, n in enumerate(lens):  # rows past each element's length: NaN
        start = min(max(n, 0), ps * pps)
        for p in range(pps):
            lo = max(start - p * ps, 0)
            if lo < ps:
                kp[int(table[e, p]), lo:] = float("nan")
                vp[int(table[e, p]), lo:] = float("nan")
    return q, kp, vp, kn, vn, table


@pytest.mark.parametrize("case", PAGED_CASES, ids=lambda c: "_".join(map(str, c[:10])))
def test_kvcache_paged_matches_oracle(case):
    b, h, sq, ps, pps, s_new, d, dt, causal, splits, lens = case
    q, kp, vp, kn, vn, table = _paged_case(case)
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda", 0)
    kpd, vpd = kp.to(dev), vp.to(dev)
    o, lse = af.attn_fwd_kvcache_paged(q.to(dev), kpd, vpd, torch.tensor(lens, dtype=torch.int32, device=dev),
                                       table.to(dev), kn.to(dev) if kn is not None else None,
                                       vn.to(dev) if vn is not None else None, causal=causal, scale=scale,
                                       num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref, kp_ref, vp_ref = oracle.attn_fwd_kvcache_paged(_np(q), _np(kp), _np(vp), table.numpy(),
                                                                   list(lens), _np(kn), _np(vn), causal, scale)
    compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, dt, f"paged {case}")
    assert np.array_equal(kpd.float().cpu().double().numpy(), kp_ref, equal_nan=True), "k pool after the write"
    assert np.array_equal(vpd.float().cpu().double().numpy(), vp_ref, equal_nan=True), "v pool after the write"


@pytest.mark.parametrize("splits", [1, 3])
def test_kvcache_paged_equals_dense_cache(splits):
    """The same logical caches, once dense and once as shuffled 256-key
    pages: bit for bit the same outputs."""
    dev = torch.device("cuda", 0)
    b, h, d, ps, pps = 2, 4, 128, 256, 4
    cap = ps * pps
    q, kc, vc = W.draw(b, h, 2, cap, d, "bf16", seed=777)
    lens = torch.tensor([900, 333], dtype=torch.int32, device=dev)
    g = torch.Generator().manual_seed(778)
    table = torch.randperm(b * pps, generator=g).reshape(b, pps).to(torch.int32)
    kp = torch.empty((b * pps, ps, h, d), dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    for e in range(b):
        for p in range(pps):
            kp[table[e, p]] = kc[e, :, p * ps:(p + 1) * ps].transpose(0, 1)
            vp[table[e, p]] = vc[e, :, p * ps:(p + 1) * ps].transpose(0, 1)
    for causal in (False, True):
        o1, l1 = af.attn_fwd_kvcache(q.to(dev), kc.to(dev), vc.to(dev), lens, causal=causal, num_splits=splits)
        o2, l2 = af.attn_fwd_kvcache_paged(q.to(dev), kp.to(dev), vp.to(dev), lens, table.to(dev), causal=causal,
                                           num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
