"""attn_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory (for example a plugin whose host program plans every
device allocation itself, or code that must not pay cudaMalloc's implicit
synchronisation).  It keeps its split partials in a fixed scratch array
inside the library instead of a caller workspace.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.  Each test builds its own inputs
and loads the library itself, so it passes alone in a fresh process as well
as after the other tests."""
import ctypes
import math

import pytest

from attention_forward_14_gb300 import binding
from attention_forward_14_gb300 import workloads as W

BF16 = 1


def _noalloc(lib, q, k, v, o, lse, causal, scale, splits):
    import torch
    b, h, sq, d = q.shape
    sk = k.shape[2]
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        b, h, sq, sk, d, int(causal), float(scale), BF16, int(splits),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Sizes whose partials do not fit the fixed scratch get ATTN_ERR_SHAPE and
    a message that says so, before anything reaches a GPU."""
    from attention_forward_14_gb300.build import build
    build()
    lib = binding.load()
    # 64 splits x 64 heads x 512 rows x (128 + 2) floats is far above 16 MiB
    rc = lib.attn_fwd_splitkv_noalloc(None, None, None, None, None, 1, 64, 512, 65536, 128, 0, 0.1, BF16, 64, None)
    assert rc == -2
    msg = lib.attn_last_error().decode()
    assert "scratch" in msg and "need" in msg


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_splitkv_on_two_calls_in_a_row():
    """Two consecutive calls (different inputs, one of them causal, so the
    second cannot pass on what the first left in the shared scratch) are
    checked element by element against the fp64 oracle on the same seeded
    inputs, within the bf16 tolerances of the parity tests (O max-abs 2e-2
    and rel-L2 1e-2, LSE 1e-3); they are also compared with
    attn_fwd_splitkv given its own workspace."""
    import torch
    from parity import compare
    import attention_forward_14_gb300 as af
    import oracle

    lib = binding.load()
    dev = torch.device("cuda", 0)
    b, h, sq, sk, d, splits = 2, 8, 3, 4096, 128, 8
    assert binding.splitkv_workspace_bytes(b, h, sq, d, splits) <= 16 * 1024 * 1024
    scale = 1.0 / math.sqrt(d)
    for call, (seed, causal) in enumerate(((101, False), (202, True))):
        qc, kc, vc = W.draw(b, h, sq, sk, d, "bf16", seed)
        q, k, v = (t.to(dev) for t in (qc, kc, vc))
        o = torch.full_like(q, float("nan"))
        lse = torch.full((b, h, sq), float("nan"), dtype=torch.float32, device=dev)
        rc = _noalloc(lib, q, k, v, o, lse, causal, scale, splits)
        assert rc == 0, lib.attn_last_error().decode()
        torch.cuda.synchronize()
        got_o, got_lse = o.float().cpu().double().numpy(), lse.cpu().double().numpy()
        o_ref, lse_ref = oracle.attn_fwd(qc.double().numpy(), kc.double().numpy(), vc.double().numpy(), causal,
                                         scale)
        compare(got_o, got_lse, o_ref, lse_ref, "bf16", f"no-alloc call {call + 1} against the oracle")
        o_sk, lse_sk = af.attn_fwd_splitkv(q, k, v, causal=causal, scale=scale, num_splits=splits)
        torch.cuda.synchronize()
        compare(got_o, got_lse, o_sk.float().cpu().double().numpy(), lse_sk.cpu().double().numpy(), "bf16",
                f"no-alloc call {call + 1} against attn_fwd_splitkv")
