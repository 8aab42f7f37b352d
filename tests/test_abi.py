"""The C-ABI library loads, exports every declared symbol and rejects bad
arguments before touching the GPU (CPU only: no compute calls)."""
import ctypes
import math
import os
import re

import pytest

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import binding
from attention_forward_14_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_fwd.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_expected_entry_points():
    assert set(declared_functions()) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.attn_version().decode().startswith("attn_fwd sm_103a")


def test_library_is_sm103a_only():
    from attention_forward_14_gb300 import build as b
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


BUF = ctypes.create_string_buffer(4096 + 512)
P = ctypes.addressof(BUF) + (-ctypes.addressof(BUF)) % 256  # 256-aligned host address


def call(lib, q=P, k=P, v=P, o=P, lse=None, b=1, h=1, sq=4, sk=4, d=64, causal=0, scale=0.125, dtype=1):
    rc = lib.attn_fwd(q, k, v, o, lse, b, h, sq, sk, d, causal, scale, dtype, None)
    return rc, lib.attn_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), -3), (dict(d=0), -3), (dict(d=256), -3),
    (dict(dtype=2), -4), (dict(dtype=-1), -4),
    (dict(b=-1), -2), (dict(sq=-3), -2), (dict(sk=-1), -2), (dict(sq=1 << 31), -2),
    (dict(b=1 << 16, h=1 << 16), -2),
    (dict(scale=math.nan), -5), (dict(scale=math.inf), -5),
    (dict(o=None), -1), (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1),
    (dict(q=P + 8), -6), (dict(o=P + 2), -6), (dict(lse=P + 2), -6),
])
def test_argument_errors(lib, kw, code):
    rc, msg = call(lib, **kw)
    assert rc == code, (rc, msg)
    assert msg


@pytest.mark.parametrize("kw", [dict(b=0), dict(h=0), dict(sq=0), dict(b=0, q=None, k=None, v=None, o=None)])
def test_empty_problem_is_ok_without_launch(lib, kw):
    rc, msg = call(lib, **kw)
    assert rc == 0 and msg == ""


def test_no_device_gives_error_not_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, msg = call(lib)
    assert rc in (-7, -8) and msg


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(af.AttnError):
        binding.load(str(tmp_path / "missing.so"))


def test_splitkv_workspace_size(lib):
    assert lib.attn_fwd_splitkv_workspace_bytes(2, 3, 5, 128, 4) == 4 * 2 * 3 * 5 * (128 + 2) * 4
    assert lib.attn_fwd_splitkv_workspace_bytes(2, 3, 5, 64, 1) == 0
    assert lib.attn_fwd_splitkv_workspace_bytes(2, 3, 5, 96, 4) == -2
    assert lib.attn_fwd_splitkv_workspace_bytes(2, 3, 5, 128, 0) == -2


@pytest.mark.parametrize("splits,ws,ws_bytes,code", [
    (0, P, 1 << 20, -2), (2000, P, 1 << 20, -2),
    (9, P, 1 << 20, -2),          # 1000 keys = 8 tiles of 128
    (4, None, 1 << 20, -1),       # missing workspace
    (4, P, 16, -2),               # too small
    (4, P + 8, 1 << 20, -6),      # misaligned
])
def test_splitkv_argument_errors(lib, splits, ws, ws_bytes, code):
    rc = lib.attn_fwd_splitkv(P, P, P, P, None, 1, 2, 3, 1000, 128, 0, 0.1, 1, splits, ws, ws_bytes, None)
    assert rc == code, (rc, lib.attn_last_error())


def call_bwd(lib, b=1, h=1, sq=4, sk=4, d=128, causal=0, scale=0.1, dtype=1, ws=P, ws_bytes=1 << 20, ptr=P):
    rc = lib.attn_bwd(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, b, h, sq, sk, d, causal, scale, dtype, ws, ws_bytes,
                      None)
    return rc, lib.attn_last_error().decode()


def test_bwd_rejects_bad_arguments(lib):
    assert call_bwd(lib, d=96)[0] == -3
    assert call_bwd(lib, dtype=7)[0] == -4
    assert call_bwd(lib, b=-1)[0] == -2
    assert call_bwd(lib, sq=(1 << 30) + 1)[0] == -2
    assert call_bwd(lib, scale=math.nan)[0] == -5
    assert call_bwd(lib, scale=math.inf)[0] == -5
    assert call_bwd(lib, ptr=None)[0] == -1
    assert call_bwd(lib, ptr=P + 4)[0] == -6
    rc, msg = call_bwd(lib, b=0)
    assert rc == 0, msg  # nothing to do


def test_bwd_workspace_bytes(lib):
    # fp32 dQ accumulator + two fp32 values per query row padded to 128 rows
    # + the scheduler's counter
    assert lib.attn_bwd_workspace_bytes(2, 3, 300, 128) == 6 * 300 * 128 * 4 + 2 * 6 * 384 * 4 + 256
    assert lib.attn_bwd_workspace_bytes(1, 1, 0, 128) == 256
    assert lib.attn_bwd_workspace_bytes(1, 1, 4, 96) == -3
    assert lib.attn_bwd_workspace_bytes(1, 1, 128, 64) == 128 * 64 * 4 + 2 * 128 * 4 + 256
    assert lib.attn_bwd_workspace_bytes(-1, 1, 4, 128) == -2


def call_kvcache(lib, kn=None, vn=None, seqlens=P, b=1, h=2, sq=1, cap=1000, s_new=0, d=128, splits=1,
                 ws=None, ws_bytes=0, cache=P):
    rc = lib.attn_fwd_kvcache(P, cache, cache, kn, vn, seqlens, P, None, b, h, sq, cap, s_new, d, 1, 0.1, 1,
                              splits, ws, ws_bytes, None)
    return rc, lib.attn_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(seqlens=None), -1),                       # no lengths
    (dict(seqlens=P + 2), -6),                      # misaligned lengths
    (dict(s_new=2), -1),                            # new rows announced, none given
    (dict(kn=P + 1024, s_new=1), -1),               # k_new without v_new
    (dict(s_new=-1), -2),
    (dict(splits=0), -2), (dict(splits=9), -2),     # 1000 keys = 8 tiles of 128
    (dict(splits=4), -1),                           # split-KV without a workspace
    (dict(kn=P, vn=P, s_new=1), -2),                # new rows overlap the cache
    (dict(kn=P + 8, vn=P + 8, s_new=1, cache=P + 2048), -6),  # misaligned new rows
    (dict(d=96), -3),
])
def test_kvcache_argument_errors(lib, kw, code):
    rc, msg = call_kvcache(lib, **kw)
    assert rc == code, (rc, msg)


def test_kvcache_nothing_to_do(lib):
    assert call_kvcache(lib, b=0, seqlens=None)[0] == 0
    assert call_kvcache(lib, h=0, seqlens=None)[0] == 0


def call_paged(lib, table=P, page_size=256, num_pages=8, pps=2, seqlens=P):
    rc = lib.attn_fwd_kvcache_paged(P, P, P, None, None, seqlens, table, P, None, 1, 2, 1, num_pages, page_size, pps,
                                    0, 128, 1, 0.1, 1, 1, None, 0, None)
    return rc, lib.attn_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(page_size=100), -2), (dict(page_size=0), -2), (dict(page_size=192), -2),
    (dict(num_pages=0), -2), (dict(pps=0), -2),
    (dict(num_pages=1 << 24, page_size=1 << 8), -2),   # pool above 2^31-1 tokens
    (dict(table=None), -1), (dict(table=P + 2), -6),
])
def test_kvcache_paged_argument_errors(lib, kw, code):
    rc, msg = call_paged(lib, **kw)
    assert rc == code, (rc, msg)


def test_noalloc_rejects_bad_head_dim_like_the_other_entry_points(lib):
    """A bad head dim is ATTN_ERR_HEADDIM from the no-alloc entry point too
    (its scratch-size check comes after the checks it shares with
    attn_fwd_splitkv), and absurd sizes are rejected without overflow."""
    rc = lib.attn_fwd_splitkv_noalloc(P, P, P, P, None, 1, 2, 3, 1000, 96, 0, 0.1, 1, 2, None)
    assert rc == -3, lib.attn_last_error()
    rc = lib.attn_fwd_splitkv_noalloc(P, P, P, P, None, 1 << 15, (1 << 16) - 1, 1 << 30, 1 << 30, 128, 0, 0.1, 1,
                                      1024, None)
    assert rc == -2 and "scratch" in lib.attn_last_error().decode()
    rc = lib.attn_fwd_splitkv_noalloc(P, P, P, P, None, 1, 2, 3, 1000, 128, 0, 0.1, 1, 0, None)
    assert rc == -2


def test_debug_status_and_slot_hook_without_device(lib):
    """attn_fwd_debug_status (the watchdog code alone) and the schedule-slot
    testing hook exist; without a GPU they return an error, not a crash, and
    the hook rejects slots outside -1..255 before looking for a device."""
    import torch
    assert lib.attn_fwd_sched_pin_slot(256) == -2
    assert lib.attn_fwd_sched_pin_slot(-2) == -2
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.attn_fwd_debug_status() in (-7, -8)
    assert lib.attn_fwd_sched_pin_slot(3) in (-7, -8)


def test_checked_library_exports_the_same_interface(lib):
    """The checked build (every computed index of the forward and backward
    bounds-checked) exports every declared symbol too; the bounds self-tests
    need it and the normal build says so."""
    checked = binding.load(binding.CHECKED_LIB_PATH)
    for name in declared_functions():
        assert hasattr(checked, name), name
    rc = lib.attn_fwd_bounds_selftest(P, P, P, P, None, 1, 1, 4, 4, 64, 0.1, 1, None)
    assert rc == -10 and "checked build" in lib.attn_last_error().decode()
    rc = lib.attn_bwd_bounds_selftest(P, P, P, P, P, P, P, P, P, 1, 1, 4, 4, 64, 0.1, 1, P, 1 << 20, None)
    assert rc == -10 and "checked build" in lib.attn_last_error().decode()
    rc = lib.attn_bwd_watchdog_selftest(P, P, P, P, P, P, P, P, P, 1, 1, 4, 4, 64, 0, 0.1, 1, P, 1 << 20, 0, 50, None)
    assert rc == -10 and "checked build" in lib.attn_last_error().decode()
