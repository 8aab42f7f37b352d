"""Error bounds for the GPU backward against the fp64 oracle.

The bound is first order in the roundings the kernel makes, per element,
derived from its arithmetic (not tuned):
  u     unit roundoff of the input type (2^-8 bf16, 2^-11 fp16);
  eps   2^-16, a generous allowance for the fp32 arithmetic (ex2.approx,
        the fp32 LSE, fp32 accumulation of up to 2^16 terms);
  tiny  2^-25 for fp16 (half the subnormal spacing; bf16 has none).
The kernel computes, for key j and query i:
  P = exp2(s*scale*log2e - lse2)            |dP_hat - P| <= eps P
  D = dO_i . O_i with O rounded to the type   |dD| <= u a_i,  a_i = |dO_i|.|O_i|
  dP = dO_i . V_j in fp32                     |d dP| <= eps b_ij, b = |dO| |V|^T
  dS = round(scale round(P) (dP - D))        (P as rounded for dV, as in the kernel)
     => |d dS| <= scale P (u a_i + eps (b_ij + |dP - D|)) + (2u + eps) |scale dS| + tiny
  dV = round(sum_i round(P) dO_i)             <= (u + eps) P^T |dO| + u |dV| + tiny
  dK = round(sum_i dS Q_i)                    <= E^T |Q| + eps |scale dS|^T |Q| + u |dK| + tiny
  dQ = round(sum_j dS K_j) (fp32 accumulator) <= E |K|   + eps |scale dS| |K|   + u |dQ| + tiny
The test allows (1 + 1/8) x that per element (second-order terms), and
requires the L2 norm of the error to stay below the RMS of a uniform error
within the bound (||bound||_2 / sqrt(3)), which a systematic error spread
over many elements would exceed.
"""
from __future__ import annotations

import math

import numpy as np

U = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}
TINY = {"bf16": 0.0, "fp16": 2.0 ** -25}
EPS = 2.0 ** -16


def _visible(rows, cols, sq, sk, causal):
    if not causal:
        return np.ones((len(rows), len(cols)), bool)
    return np.asarray(cols)[None, :] <= (np.asarray(rows)[:, None] + (sk - sq))


def bounds(q, k, v, do, o, lse, dq_ref, dk_ref, dv_ref, causal, scale, dtype, rows=None, cols=None):
    """Per-element bounds for one head.  q, do, o: [sq, d]; k, v: [sk, d];
    lse: [sq] (oracle, natural log); dq_ref [len(rows), d], dk_ref / dv_ref
    [len(cols), d] are the oracle's gradients at those rows / keys.
    Returns (bound_dq, bound_dk, bound_dv)."""
    sq, sk = q.shape[0], k.shape[0]
    rows = np.arange(sq) if rows is None else np.asarray(rows)
    cols = np.arange(sk) if cols is None else np.asarray(cols)
    u, tiny = U[dtype], TINY[dtype]
    a = np.sum(np.abs(do) * np.abs(o), axis=1)   # [sq]
    D = np.sum(do * o, axis=1)                   # [sq]

    def block(ri, cj):
        vis = _visible(ri, cj, sq, sk, causal)
        with np.errstate(invalid="ignore", over="ignore"):
            P = np.where(vis & np.isfinite(lse[ri])[:, None],
                         np.exp(scale * (q[ri] @ k[cj].T) - lse[ri][:, None]), 0.0)
        dP = do[ri] @ v[cj].T
        dS = P * (dP - D[ri][:, None])
        B = np.abs(do[ri]) @ np.abs(v[cj]).T
        E = (scale * P * (u * a[ri][:, None] + EPS * (B + np.abs(dP - D[ri][:, None])))
             + (2 * u + EPS) * scale * np.abs(dS) + tiny)
        return P, dS, E

    # dQ at the sampled rows: all keys
    P, dS, E = block(rows, np.arange(sk))
    bdq = E @ np.abs(k) + EPS * scale * (np.abs(dS) @ np.abs(k)) + u * np.abs(dq_ref) + tiny
    # dK, dV at the sampled keys: all rows
    P, dS, E = block(np.arange(sq), cols)
    bdk = E.T @ np.abs(q) + EPS * scale * (np.abs(dS).T @ np.abs(q)) + u * np.abs(dk_ref) + tiny
    bdv = (u + EPS) * (P.T @ np.abs(do)) + u * np.abs(dv_ref) + tiny * np.sum(np.abs(do), axis=0)[None, :] + tiny
    return 1.125 * bdq, 1.125 * bdk, 1.125 * bdv


def check(name, got, ref, bound):
    """Element bound and the L2 criterion; returns (worst err/bound, rel-L2)."""
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values ({np.isnan(got).sum()} NaN)"
    err = np.abs(got - ref)
    zero = bound == 0.0  # exact zeros (e.g. scale 0): the result must be exact too
    assert (err[zero] == 0.0).all(), f"{name}: nonzero error where the gradient is exactly zero"
    ratio = float((err[~zero] / bound[~zero]).max()) if (~zero).any() else 0.0
    assert ratio <= 1.0, f"{name}: error above its bound (worst err/bound {ratio:.3f}, max err {err.max():.3e})"
    l2 = float(np.linalg.norm(err))
    l2_bound = float(np.linalg.norm(bound)) / math.sqrt(3.0)
    assert l2 <= l2_bound, f"{name}: ||err|| {l2:.3e} > ||bound||/sqrt(3) {l2_bound:.3e}"
    den = float(np.linalg.norm(ref))
    return ratio, (l2 / den if den > 0 else l2)
