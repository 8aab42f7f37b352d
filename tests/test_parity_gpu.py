"""GPU parity: the C-ABI forward (tcgen05 kernel) against the fp64 oracle on
seeded inputs.  Small problems are compared in full; the two largest
workloads are compared on whole sampled heads and on sampled rows of more
heads, at full size and in the launch configuration the benchmark times."""
import math
import zlib

import numpy as np
import pytest
import torch

from attention_forward_14_gb300 import workloads as W
from parity import check_full, check_heads, check_rows, compare, run_gpu
import oracle

pytestmark = pytest.mark.gpu


def _draw(b, h, sq, sk, d, dtype, seed, qk_std=1.0):
    return W.draw(b, h, sq, sk, d, dtype, seed, qk_std)


# Shapes that span several 256-row units and 128-key tiles, ragged tails,
# single rows/keys, sq != sk in both directions (bottom-right causal).
SHAPES = [
    (1, 1, 1, 1),
    (1, 2, 127, 127),
    (1, 1, 129, 129),
    (2, 3, 300, 300),
    (1, 2, 257, 513),
    (1, 1, 513, 100),
    (1, 1, 1, 1000),
    (1, 1, 1000, 1),
    (1, 2, 640, 384),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(shape, causal, dtype, d):
    b, h, sq, sk = shape
    q, k, v = _draw(b, h, sq, sk, d, dtype, seed=zlib.crc32(repr((shape, causal, dtype, d)).encode()))
    check_full(q, k, v, causal, 1.0 / math.sqrt(d), f"{shape} c{causal} {dtype} d{d}")


@pytest.mark.parametrize("name", W.ORDER[:3])
def test_workload_full(name):
    w = W.WORKLOADS[name]
    q, k, v = W.inputs(w)
    check_full(q, k, v, w.causal, w.scale, name)


@pytest.mark.parametrize("name", W.ORDER[3:])
def test_workload_sampled(name):
    """Full-size run; whole heads (first, last and seeded others) compared in
    full, plus seeded rows of further heads."""
    w = W.WORKLOADS[name]
    q, k, v = W.inputs(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    assert np.isfinite(o).all()
    n_full = 4 if w.sq <= 4096 else 2
    pairs = W.sample_heads(w, n=n_full + 4)
    check_heads(o, lse, q, k, v, w.causal, w.scale, pairs[:n_full], name)
    g = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, w.sq - 1],
                                     g.integers(0, w.sq, 48)]))
    check_rows(o, lse, q, k, v, w.causal, w.scale, pairs[n_full:], rows, name)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_large_logits_rescaling(dtype):
    """Q, K ~ N(0, 9): logits with std 9 move the running max many times."""
    q, k, v = _draw(1, 2, 1024, 1024, 128, dtype, seed=5, qk_std=3.0)
    for causal in (False, True):
        check_full(q, k, v, causal, 1 / math.sqrt(128), f"qk3 c{causal}")


@pytest.mark.parametrize("scale", [0.0, -0.3, 1.0])
def test_scale_values(scale):
    q, k, v = _draw(1, 2, 300, 400, 64, "bf16", seed=11)
    for causal in (False, True):
        check_full(q, k, v, causal, scale, f"scale {scale} c{causal}")


def test_zero_query_uniform():
    q, k, v = _draw(1, 1, 256, 256, 128, "fp16", seed=3)
    q.zero_()
    o, lse = run_gpu(q, k, v, False, 0.1)
    want = v.double().numpy().mean(axis=2, keepdims=True).repeat(256, axis=2)
    compare(o, lse, want, np.full((1, 1, 256), math.log(256)), "fp16", "Q=0")


def test_empty_keys_and_rows():
    import attention_forward_14_gb300 as af
    dev = torch.device("cuda", 0)
    q = torch.randn(1, 2, 5, 64, device=dev, dtype=torch.bfloat16)
    k = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 2, 5), float("nan"), device=dev)
    af.attn_fwd(q, k, k, causal=False, o=o, lse=lse)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()
    q0 = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    o0, l0 = af.attn_fwd(q0, q, q)
    assert o0.numel() == 0


def test_lse_optional_and_deterministic():
    import attention_forward_14_gb300 as af
    q, k, v = (t.cuda() for t in _draw(2, 4, 700, 700, 128, "bf16", seed=8))
    o1, l1 = af.attn_fwd(q, k, v, causal=True)
    o2, _ = af.attn_fwd(q, k, v, causal=True, return_lse=False)
    o3, l3 = af.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(o1, o3) and torch.equal(l1, l3)


def test_host_entry_point_matches_device_entry_point():
    import attention_forward_14_gb300 as af
    q, k, v = _draw(1, 4, 512, 512, 128, "bf16", seed=9)
    dev = torch.device("cuda", 0)
    od, ld = af.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    bufs = [torch.empty_like(t, device=dev) for t in (q, k, v, q)]
    lbuf = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    af.attn_fwd_host(qh, kh, vh, oh, lh, *bufs, lbuf, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())


@pytest.mark.parametrize("h,s", [(8, 8192), (7, 10000)])
def test_host_entry_point_pipelined_chunks(h, s):
    """Problems of 64 MB and more run as up to 8 chunks of heads with the
    copies overlapping the forward (h = 7: seven chunks of one head);
    every head's result is the device entry point's, bit for bit, on a
    caller stream that is not the default one."""
    import attention_forward_14_gb300 as af
    q, k, v = _draw(1, h, s, s, 128, "bf16", seed=19 + h)
    dev = torch.device("cuda", 0)
    od, ld = af.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.full_like(qh, float("nan")).pin_memory()
    lh = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    bufs = [torch.empty_like(t, device=dev) for t in (q, k, v, q)]
    lbuf = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(dev)
    af.attn_fwd_host(qh, kh, vh, oh, lh, *bufs, lbuf, causal=True, stream=st)
    st.synchronize()
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())


def test_watchdog_reports_instead_of_hanging():
    """One K/V load is withheld: every wait runs out after 50 ms, the kernel
    records where, frees its resources and returns; the context stays usable."""
    from attention_forward_14_gb300 import binding
    q, k, v = (t.cuda() for t in _draw(1, 1, 256, 256, 128, "bf16", seed=1))
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 256, device="cuda")
    code = binding.watchdog_selftest(q, k, v, o, lse, False, 0.1, withheld_load=1, timeout_ms=50)
    assert code != 0
    st = binding.status()
    # code 1 (a wait ran out) at one of the kernel's wait sites: loads,
    # MMA operands, S / P / O hand-offs, the unit ring, the O staging panel
    assert st[0] == 1 and 1 <= st[3] <= 13
    binding.status_clear()
    assert binding.status()[0] == 0
    # the GPU still computes correctly afterwards
    check_full(*_draw(1, 1, 256, 256, 128, "bf16", seed=2), False, 0.1, "after watchdog")
    assert binding.status()[0] == 0
