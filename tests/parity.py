"""Helpers shared by the GPU parity tests: run the C-ABI forward on seeded
inputs and compare it with the fp64 oracle element by element.

Tolerances (fixed for this project): fp16 O max-abs <= 1e-2 and rel-L2 <=
5e-3; bf16 O max-abs <= 2e-2 and rel-L2 <= 1e-2; LSE max-abs <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import attention_forward_14_gb300 as af

TOL = {
    "fp16": dict(max_abs=1e-2, rel_l2=5e-3),
    "bf16": dict(max_abs=2e-2, rel_l2=1e-2),
}
LSE_TOL = 1e-3


def dtype_name(t: torch.dtype) -> str:
    return {torch.float16: "fp16", torch.bfloat16: "bf16"}[t]


def run_gpu(q, k, v, causal, scale, with_lse=True):
    """q/k/v CPU tensors -> (O, LSE) from the GPU as fp64 numpy.  Outputs are
    pre-filled with NaN so that an unwritten element fails the comparison."""
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    af.attn_fwd(qd, kd, vd, causal=causal, scale=scale, o=o, lse=lse)
    torch.cuda.synchronize()
    o_np = o.float().cpu().double().numpy()
    l_np = lse.cpu().double().numpy() if with_lse else None
    return o_np, l_np


def compare(o, lse, o_ref, lse_ref, dtype: str, what: str = ""):
    """Assert the tolerances above (O max-abs and rel-L2, LSE max-abs); returns the error figures."""
    tol = TOL[dtype]
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite O ({np.isnan(o).sum()} NaN)"
    diff = np.abs(o - o_ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    den = float(np.linalg.norm(o_ref))
    rel = float(np.linalg.norm(o - o_ref) / den) if den > 0 else float(np.linalg.norm(o - o_ref))
    res = dict(max_abs=max_abs, rel_l2=rel)
    assert max_abs <= tol["max_abs"], f"{what}: O max-abs {max_abs:.3e} > {tol['max_abs']}"
    assert rel <= tol["rel_l2"], f"{what}: O rel-L2 {rel:.3e} > {tol['rel_l2']}"
    if lse is not None:
        assert not np.isnan(lse).any(), f"{what}: NaN in LSE"
        inf_ref = np.isinf(lse_ref)
        assert (np.isinf(lse) == inf_ref).all(), f"{what}: LSE -inf pattern differs"
        if (~inf_ref).any():
            lerr = float(np.abs(lse[~inf_ref] - lse_ref[~inf_ref]).max())
            res["lse_max_abs"] = lerr
            assert lerr <= LSE_TOL, f"{what}: LSE max-abs {lerr:.3e} > {LSE_TOL}"
    return res


def check_full(q, k, v, causal, scale, what=""):
    """Whole problem against the oracle."""
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal, scale)
    return compare(o, lse, o_ref, lse_ref, dtype_name(q.dtype), what)


def check_heads(o, lse, q, k, v, causal, scale, pairs, what=""):
    """Given full GPU outputs, compare the listed (batch, head) pairs in full."""
    out = []
    for bi, hi in pairs:
        qh, kh, vh = (t[bi, hi].double().numpy()[None, None] for t in (q, k, v))
        o_ref, lse_ref = oracle.attn_fwd(qh, kh, vh, causal, scale)
        out.append(compare(o[bi, hi][None, None], lse[bi, hi][None, None], o_ref, lse_ref,
                           dtype_name(q.dtype), f"{what} head ({bi},{hi})"))
    return out


def check_rows(o, lse, q, k, v, causal, scale, pairs, rows, what=""):
    """Given full GPU outputs, compare selected rows of the listed heads."""
    out = []
    for bi, hi in pairs:
        o_ref, lse_ref = oracle.attn_head_rows(q[bi, hi].double().numpy(), k[bi, hi].double().numpy(),
                                               v[bi, hi].double().numpy(), rows, causal, scale)
        out.append(compare(o[bi, hi][rows], lse[bi, hi][rows], o_ref, lse_ref, dtype_name(q.dtype),
                           f"{what} rows of ({bi},{hi})"))
    return out
