"""fp64 CPU oracle for the fused attention forward and its gradients -- TEST
INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
this package.  It shares no code with the CUDA library and imports nothing
from the product package.

What it computes (attention formula of "flash-attn 实现 prefill 阶段",
problem analysis; scale after the dot product and natural-exp softmax of
flash-attention-minimal ``forward_kernel``) is documented in
``attn_oracle.c``.  ``build()`` compiles that file with the host C compiler
into ``liboracle.so`` next to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, -O2, OpenMP) if missing or stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_attn_fwd_f64.restype = ctypes.c_int
    lib.oracle_attn_fwd_f64.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                        ctypes.c_int, ctypes.c_double]
    lib.oracle_attn_online_f64.restype = ctypes.c_int
    lib.oracle_attn_online_f64.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                           ctypes.c_int, ctypes.c_double, i64]
    lib.oracle_attn_head_rows_f64.restype = ctypes.c_int
    lib.oracle_attn_head_rows_f64.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_int,
                                              ctypes.c_double,
                                              ctypes.POINTER(ctypes.c_int64), i64, dp, dp]
    lib.oracle_attn_probs_f64.restype = ctypes.c_int
    lib.oracle_attn_probs_f64.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, ctypes.c_int,
                                          ctypes.c_double]
    lib.oracle_attn_bwd_f64.restype = ctypes.c_int
    lib.oracle_attn_bwd_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                        ctypes.c_int, ctypes.c_double]
    lib.oracle_attn_bwd_dq_rows_f64.restype = ctypes.c_int
    lib.oracle_attn_bwd_dq_rows_f64.argtypes = [dp, dp, dp, dp, i64, i64, i64, ctypes.c_int,
                                                ctypes.c_double, ctypes.POINTER(ctypes.c_int64),
                                                i64, dp]
    lib.oracle_attn_bwd_dkv_cols_f64.restype = ctypes.c_int
    lib.oracle_attn_bwd_dkv_cols_f64.argtypes = [dp, dp, dp, dp, i64, i64, i64, ctypes.c_int,
                                                 ctypes.c_double, ctypes.POINTER(ctypes.c_int64),
                                                 i64, dp, dp]
    lib.oracle_attn_fwd_kvcache_f64.restype = ctypes.c_int
    lib.oracle_attn_fwd_kvcache_f64.argtypes = [dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64), dp, dp,
                                                i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def load_library(path: str):
    """Bind the oracle API of another build of attn_oracle.c (the tests use
    this to check that the pins reject deliberately broken copies)."""
    return _bind(ctypes.CDLL(path))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def num_threads(lib=None) -> int:
    return int((lib or _load()).oracle_num_threads())


def attn_fwd(q, k, v, causal: bool, scale: float, lib=None):
    """Definition: O = softmax(scale * Q K^T [+ causal mask]) V and LSE.

    q: [b, h, sq, d], k/v: [b, h, sk, d] (any float dtype; used as fp64).
    Returns (o [b, h, sq, d] fp64, lse [b, h, sq] fp64).
    """
    lib = lib or _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, sq, d = q.shape
    sk = k.shape[2]
    assert k.shape == (b, h, sk, d) and v.shape == (b, h, sk, d)
    o = np.zeros((b, h, sq, d), np.float64)
    lse = np.zeros((b, h, sq), np.float64)
    rc = lib.oracle_attn_fwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 b, h, sq, sk, d, int(bool(causal)), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_f64 failed: {rc}")
    return o, lse


def attn_fwd_online(q, k, v, causal: bool, scale: float, bc: int, lib=None):
    """The flash-attention-minimal tile recurrence (tile of ``bc`` keys)."""
    lib = lib or _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, sq, d = q.shape
    sk = k.shape[2]
    o = np.zeros((b, h, sq, d), np.float64)
    lse = np.zeros((b, h, sq), np.float64)
    rc = lib.oracle_attn_online_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                    b, h, sq, sk, d, int(bool(causal)), float(scale),
                                    int(bc))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_online_f64 failed: {rc}")
    return o, lse


def attn_head_rows(q_head, k_head, v_head, rows, causal: bool, scale: float, lib=None):
    """Selected query rows of one head: q_head [sq, d], k/v_head [sk, d]."""
    lib = lib or _load()
    q_head, k_head, v_head = _f64(q_head), _f64(k_head), _f64(v_head)
    sq, d = q_head.shape
    sk = k_head.shape[0]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((rows.size, d), np.float64)
    lse = np.zeros((rows.size,), np.float64)
    rc = lib.oracle_attn_head_rows_f64(
        _ptr(q_head), _ptr(k_head), _ptr(v_head), sq, sk, d, int(bool(causal)),
        float(scale), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.size,
        _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_head_rows_f64 failed: {rc}")
    return o, lse


def attn_probs(q, k, causal: bool, scale: float, lib=None):
    """P = softmax(scale * Q K^T [+ causal]) as [b, h, sq, sk] fp64."""
    lib = lib or _load()
    q, k = _f64(q), _f64(k)
    b, h, sq, d = q.shape
    sk = k.shape[2]
    p = np.zeros((b, h, sq, sk), np.float64)
    rc = lib.oracle_attn_probs_f64(_ptr(q), _ptr(k), _ptr(p), b, h, sq, sk, d,
                                   int(bool(causal)), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_probs_f64 failed: {rc}")
    return p


def attn_bwd(q, k, v, dout, causal: bool, scale: float, lib=None):
    """Gradients (dq, dk, dv) of the forward for the output gradient
    ``dout`` [b, h, sq, d], by the chain rule through the definition."""
    lib = lib or _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    b, h, sq, d = q.shape
    sk = k.shape[2]
    assert k.shape == (b, h, sk, d) and v.shape == (b, h, sk, d) and dout.shape == q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = lib.oracle_attn_bwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), b, h, sq, sk, d, int(bool(causal)), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_f64 failed: {rc}")
    return dq, dk, dv


def attn_bwd_dq_rows(q_head, k_head, v_head, do_head, rows, causal: bool, scale: float, lib=None):
    """dQ of selected query rows of one head ([sq, d] / [sk, d] inputs)."""
    lib = lib or _load()
    q_head, k_head, v_head, do_head = _f64(q_head), _f64(k_head), _f64(v_head), _f64(do_head)
    sq, d = q_head.shape
    sk = k_head.shape[0]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.zeros((rows.size, d), np.float64)
    rc = lib.oracle_attn_bwd_dq_rows_f64(
        _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(do_head), sq, sk, d, int(bool(causal)),
        float(scale), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.size, _ptr(dq))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_dq_rows_f64 failed: {rc}")
    return dq


def attn_bwd_dkv_cols(q_head, k_head, v_head, do_head, cols, causal: bool, scale: float, lib=None):
    """dK and dV of selected keys of one head ([sq, d] / [sk, d] inputs)."""
    lib = lib or _load()
    q_head, k_head, v_head, do_head = _f64(q_head), _f64(k_head), _f64(v_head), _f64(do_head)
    sq, d = q_head.shape
    sk = k_head.shape[0]
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    dk = np.zeros((cols.size, d), np.float64)
    dv = np.zeros((cols.size, d), np.float64)
    rc = lib.oracle_attn_bwd_dkv_cols_f64(
        _ptr(q_head), _ptr(k_head), _ptr(v_head), _ptr(do_head), sq, sk, d, int(bool(causal)),
        float(scale), cols.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), cols.size, _ptr(dk),
        _ptr(dv))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_dkv_cols_f64 failed: {rc}")
    return dk, dv


def attn_fwd_kvcache(q, k_cache, v_cache, cache_len, k_new=None, v_new=None, causal: bool = False,
                     scale: float = 1.0, lib=None):
    """KV-cache forward: the new rows written into (copies of) the caches at
    each batch element's length, then attention over the valid keys.

    q: [b, h, sq, d]; k_cache/v_cache: [b, h, s_cache, d]; cache_len: [b]
    ints; k_new/v_new: [b, h, s_new, d] or None.  Returns (o, lse, k_cache
    after the write, v_cache after the write), all fp64.
    """
    lib = lib or _load()
    q = _f64(q)
    kc = np.array(k_cache, dtype=np.float64, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.float64, copy=True, order="C")
    b, h, sq, d = q.shape
    s_cache = kc.shape[2]
    assert kc.shape == (b, h, s_cache, d) and vc.shape == kc.shape
    lens = np.ascontiguousarray(np.asarray(cache_len, dtype=np.int64))
    assert lens.shape == (b,)
    if k_new is None:
        kn = vn = None
        s_new = 0
    else:
        kn, vn = _f64(k_new), _f64(v_new)
        s_new = kn.shape[2]
        assert kn.shape == (b, h, s_new, d) and vn.shape == kn.shape
    o = np.zeros((b, h, sq, d), np.float64)
    lse = np.zeros((b, h, sq), np.float64)
    null = ctypes.POINTER(ctypes.c_double)()
    rc = lib.oracle_attn_fwd_kvcache_f64(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(kn) if kn is not None else null,
        _ptr(vn) if vn is not None else null, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _ptr(o), _ptr(lse), b, h, sq, s_cache, s_new, d, int(bool(causal)), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_kvcache_f64 failed: {rc}")
    return o, lse, kc, vc


def attn_fwd_kvcache_paged(q, k_pool, v_pool, block_table, cache_len, k_new=None, v_new=None, causal: bool = False,
                           scale: float = 1.0, lib=None):
    """The KV-cache forward over a paged cache.  A paged cache is a
    re-indexing of a dense one: batch element e's logical cache is the
    concatenation of the pool pages block_table[e, 0..P) ([num_pages,
    page_size, h, d], token-major within a page).  The logical caches are
    gathered, ``attn_fwd_kvcache`` runs on them, and the written rows go
    back to their pages.  Pages of different elements must be distinct.
    Returns (o, lse, k_pool after the write, v_pool after the write)."""
    kp = np.array(k_pool, dtype=np.float64, copy=True)
    vp = np.array(v_pool, dtype=np.float64, copy=True)
    table = np.asarray(block_table, dtype=np.int64)
    b, h, sq, d = np.shape(q)
    num_pages, page_size = kp.shape[0], kp.shape[1]
    pages = table.shape[1]
    assert kp.shape == (num_pages, page_size, h, d) and vp.shape == kp.shape and table.shape == (b, pages)

    def logical(pool):  # [b, P, page_size, h, d] -> [b, h, P * page_size, d]
        return pool[table].reshape(b, pages * page_size, h, d).transpose(0, 2, 1, 3)

    o, lse, kc, vc = attn_fwd_kvcache(q, logical(kp), logical(vp), cache_len, k_new, v_new, causal, scale, lib=lib)
    kp[table] = kc.transpose(0, 2, 1, 3).reshape(b, pages, page_size, h, d)
    vp[table] = vc.transpose(0, 2, 1, 3).reshape(b, pages, page_size, h, d)
    return o, lse, kp, vp
