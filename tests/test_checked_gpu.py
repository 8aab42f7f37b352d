"""The checked build (libattn_fwd_checked.so: the same sources with every
computed index of the forward and backward compared with its bounds -- copy
coordinates, page lookups, thread-written O / LSE / split-partial / dK / dV
offsets, dQ reduce-add coordinates, decoded units, the tensor-memory
allocation and the shared-memory window) runs the small-shape parity suite,
the split-KV, packed, KV-cache, paged and e4m3 cases, the dense and packed
backward cases and the >2^32-element problems, each against the fp64 oracle
as in their own test files, with the status word read after every case: no
check may fire on valid inputs.  Its self-tests put one unit past the end
of a forward and of a backward problem and check that the bounds violation
is reported instead of used.  Nothing here faults: an index that fails its
check is not used."""
import math

import numpy as np
import pytest
import torch

from attention_forward_14_gb300 import binding
from attention_forward_14_gb300 import workloads as W

import test_bwd_gpu as BW
import test_fp8_gpu as F8
import test_kvcache_gpu as KV
import test_max_size_gpu as MS
import test_parity_gpu as P
import test_splitkv_gpu as SK
import test_varlen_bwd_gpu as VB
import test_varlen_gpu as VL

pytestmark = pytest.mark.gpu

BOUNDS, SITE_CHK_UNIT, SITE_BWD_CHK_UNIT = 3, 22, 42


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    """Route the binding through the checked build for this module."""
    from attention_forward_14_gb300.build import build
    build()
    saved = binding.load()
    checked = binding.load(binding.CHECKED_LIB_PATH)
    binding._lib = checked
    binding.status_clear()
    try:
        yield checked
    finally:
        binding._lib = saved


def _clean(what):
    code = binding.status()
    assert code[0] == 0, f"{what}: status {code}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", P.SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_checked_small_shapes(shape, causal, dtype, d):
    P.test_small_shapes(shape, causal, dtype, d)
    _clean(f"small {shape} c{causal} {dtype} d{d}")


@pytest.mark.parametrize("case", SK.CASES, ids=lambda c: "_".join(map(str, c)))
def test_checked_splitkv(case):
    SK.test_splitkv_matches_oracle(case)
    _clean(f"splitkv {case}")


@pytest.mark.parametrize("case", VL.CASES, ids=lambda c: f"{len(c[0])}seq_h{c[2]}_d{c[3]}_{c[4]}_c{int(c[5])}")
def test_checked_varlen(case):
    VL.test_varlen_matches_oracle(case)
    _clean(f"varlen {case}")


@pytest.mark.parametrize("case", KV.CASES, ids=lambda c: "_".join(map(str, c[:9])))
def test_checked_kvcache(case):
    KV.test_kvcache_matches_oracle(case)
    _clean(f"kvcache {case}")


@pytest.mark.parametrize("case", KV.PAGED_CASES, ids=lambda c: "_".join(map(str, c[:10])))
def test_checked_kvcache_paged(case):
    KV.test_kvcache_paged_matches_oracle(case)
    _clean(f"paged {case}")


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_checked_fp8(causal, d):
    F8._check(2, 3, 300, 300, causal, seed=17 + d, what=f"checked e4m3 c{causal} d{d}", d=d)
    _clean(f"e4m3 c{causal} d{d}")


@pytest.mark.parametrize("which", ["dense", "varlen"])
def test_checked_past_2_32_elements(which):
    """The >2^32-element problems, forward and backward: every computed
    offset of the larger tensors within its bounds (and the boundary heads
    correct)."""
    if which == "dense":
        MS.test_dense_forward_and_backward_past_2_32_elements()
    else:
        MS.test_varlen_forward_and_backward_past_2_32_elements()
    _clean(f"{which} forward and backward past 2^32 elements")
    torch.cuda.empty_cache()


@pytest.mark.parametrize("b,h,sq,sk,dtype,causal,d", BW.SHAPES)
def test_checked_bwd(b, h, sq, sk, dtype, causal, d):
    BW.test_bwd_matches_oracle(b, h, sq, sk, dtype, causal, d)
    _clean(f"backward b{b} h{h} sq{sq} sk{sk} {dtype} c{int(causal)} d{d}")


@pytest.mark.parametrize("lens_q,lens_k,h,d,dtype,causal", VB.CASES)
def test_checked_bwd_varlen(lens_q, lens_k, h, d, dtype, causal):
    VB.test_varlen_bwd_matches_oracle_and_dense(lens_q, lens_k, h, d, dtype, causal)
    _clean(f"packed backward {lens_q} {lens_k} h{h} d{d} {dtype} c{int(causal)}")


def test_checked_bwd_bounds_selftest_reports_instead_of_using():
    """One backward unit past the end of a 1-head problem: every warp role
    finds its index out of range before decoding it, the status says where,
    and the next call on the same context is correct and clean."""
    dev = torch.device("cuda", 0)
    q, k, v, do = BW._draw(1, 1, 256, 256, "bf16", 5, d=64)
    _, _, o, lse = BW._fwd_outputs(q, k, v, False, 0.125, "bf16")
    qd, kd, vd, od, dod = (t.to(dev) for t in (q, k, v, o, do))
    ld = lse.to(dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    nbytes = binding.bwd_workspace_bytes(1, 1, 256, 64)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    lib = binding.load()
    rc = lib.attn_bwd_bounds_selftest(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), dod.data_ptr(),
                                      ld.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 1, 1, 256, 256, 64,
                                      0.125, 1, ws.data_ptr(), nbytes, None)
    assert rc == BOUNDS, (rc, lib.attn_last_error())
    st = binding.status()
    assert st[0] == BOUNDS and st[3] == SITE_BWD_CHK_UNIT
    binding.status_clear()
    BW.test_bwd_matches_oracle(1, 2, 300, 300, "bf16", True, 64)
    _clean("after the backward bounds self-test")


def test_checked_bounds_selftest_reports_instead_of_using():
    """One unit past the end of a 1-head problem: its head plane is out of
    range; every warp role finds that before touching memory, the status says
    where, and the next call on the same context is correct and clean."""
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in W.draw(1, 1, 256, 256, 64, "bf16", seed=5))
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 256, device=dev)
    lib = binding.load()
    rc = lib.attn_fwd_bounds_selftest(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256,
                                      256, 64, 0.125, 1, None)
    assert rc == BOUNDS, (rc, lib.attn_last_error())
    st = binding.status()
    assert st[0] == BOUNDS and st[3] == SITE_CHK_UNIT
    binding.status_clear()
    P.check_full(*W.draw(1, 2, 300, 300, 64, "bf16", seed=6), False, 0.125, "after the bounds self-test")
    _clean("after the bounds self-test")


def test_checked_bwd_watchdog_reports_instead_of_hanging():
    """The first query-tile load of every CTA is withheld: the waits run out
    after 50 ms, the kernel records where, winds down and returns; the
    context stays usable and the next backward is correct."""
    dev = torch.device("cuda", 0)
    q, k, v, do = BW._draw(1, 2, 256, 256, "bf16", 31900)
    _, _, o, lse = BW._fwd_outputs(q, k, v, False, 0.1, "bf16")
    code = binding.bwd_watchdog_selftest(q.to(dev), k.to(dev), v.to(dev), o.to(dev), do.to(dev), lse.to(dev),
                                         False, 0.1, withheld_load=0, timeout_ms=50)
    assert code == 1
    st = binding.status()
    # code 1 (a wait ran out) at one of the backward's wait sites
    assert st[0] == 1 and 21 <= st[3] <= 38, st
    binding.status_clear()
    assert binding.status()[0] == 0
    BW._check_all(q, k, v, do, False, 0.1, "bf16", "after the backward watchdog")
    _clean("after the backward watchdog")
