"""ctypes binding of libattn_fwd.so (the C ABI in include/attn_fwd.h).

Argument marshalling only: every step of the forward and backward runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  If the library is
missing or cannot be loaded, every call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libattn_fwd.so")
CHECKED_LIB_PATH = os.path.join(HERE, "libattn_fwd_checked.so")  # every computed index bounds-checked
_lib = None
_lock = threading.Lock()

FP16, BF16 = 0, 1
ERRORS = {
    0: "ATTN_OK", -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_SHAPE", -3: "ATTN_ERR_HEADDIM", -4: "ATTN_ERR_DTYPE",
    -5: "ATTN_ERR_SCALE", -6: "ATTN_ERR_ALIGN", -7: "ATTN_ERR_ARCH", -8: "ATTN_ERR_CUDA", -9: "ATTN_ERR_WATCHDOG",
    -10: "ATTN_ERR_BUILD",
}
# Every function include/attn_fwd.h declares.
EXPORTS = ["attn_fwd", "attn_fwd_host", "attn_fwd_varlen", "attn_fwd_fp8", "attn_fwd_splitkv", "attn_fwd_splitkv_workspace_bytes",
           "attn_fwd_splitkv_default_splits", "attn_fwd_splitkv_noalloc", "attn_last_error", "attn_fwd_status", "attn_fwd_status_clear",
           "attn_fwd_debug_status", "attn_fwd_sched_pin_slot", "attn_fwd_bounds_selftest", "attn_bwd_bounds_selftest",
           "attn_fwd_watchdog_selftest", "attn_bwd_watchdog_selftest", "attn_version", "attn_bwd", "attn_bwd_workspace_bytes", "attn_bwd_varlen",
           "attn_bwd_varlen_workspace_bytes", "attn_fwd_kvcache", "attn_fwd_kvcache_paged"]


class AttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


def lib_path() -> str:
    return _LIB_PATH


def _bind(lib):
    i64, vp, c_int, c_float = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.restype = c_int
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float, c_int, vp]
    lib.attn_fwd_host.restype = c_int
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                  i64, i64, i64, i64, i64, c_int, c_float, c_int, vp]
    lib.attn_fwd_fp8.restype = c_int
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float, c_float, c_float,
                                 c_float, vp]
    lib.attn_fwd_varlen.restype = c_int
    lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, c_int, c_float,
                                    c_int, vp]
    lib.attn_fwd_splitkv.restype = c_int
    lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float, c_int, c_int,
                                     vp, i64, vp]
    lib.attn_fwd_splitkv_workspace_bytes.restype = i64
    lib.attn_fwd_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, c_int]
    lib.attn_fwd_splitkv_default_splits.restype = c_int
    lib.attn_fwd_splitkv_default_splits.argtypes = [i64, i64, i64, i64, i64, c_int]
    lib.attn_fwd_splitkv_noalloc.restype = c_int
    lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float, c_int,
                                             c_int, vp]
    lib.attn_fwd_kvcache.restype = c_int
    lib.attn_fwd_kvcache.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_float,
                                     c_int, c_int, vp, i64, vp]
    lib.attn_fwd_kvcache_paged.restype = c_int
    lib.attn_fwd_kvcache_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                           i64, c_int, c_float, c_int, c_int, vp, i64, vp]
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_last_error.argtypes = []
    lib.attn_fwd_status.restype = c_int
    lib.attn_fwd_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.attn_fwd_status_clear.restype = c_int
    lib.attn_fwd_status_clear.argtypes = []
    lib.attn_fwd_debug_status.restype = c_int
    lib.attn_fwd_debug_status.argtypes = []
    lib.attn_fwd_sched_pin_slot.restype = c_int
    lib.attn_fwd_sched_pin_slot.argtypes = [c_int]
    lib.attn_fwd_bounds_selftest.restype = c_int
    lib.attn_fwd_bounds_selftest.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_float, c_int, vp]
    lib.attn_bwd_watchdog_selftest.restype = c_int
    lib.attn_bwd_watchdog_selftest.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int,
                                               c_float, c_int, vp, i64, c_int, c_int, vp]
    lib.attn_bwd_bounds_selftest.restype = c_int
    lib.attn_bwd_bounds_selftest.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_float,
                                             c_int, vp, i64, vp]
    lib.attn_fwd_watchdog_selftest.restype = c_int
    lib.attn_fwd_watchdog_selftest.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float,
                                               c_int, c_int, c_int, vp]
    lib.attn_version.restype = ctypes.c_char_p
    lib.attn_version.argtypes = []
    lib.attn_bwd.restype = c_int
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_float, c_int,
                             vp, i64, vp]
    lib.attn_bwd_workspace_bytes.restype = i64
    lib.attn_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64]
    lib.attn_bwd_varlen.restype = c_int
    lib.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                    c_int, c_float, c_int, vp, i64, vp]
    lib.attn_bwd_varlen_workspace_bytes.restype = i64
    lib.attn_bwd_varlen_workspace_bytes.argtypes = [i64, i64, i64, i64, i64]
    return lib


def load(path: str | None = None):
    """Load (once) and bind the C ABI.  Raises if the library is absent."""
    global _lib
    if path is None and _lib is not None:  # the common case: no lock
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise AttnError(-8, f"{p} not built; run python -m attention_forward_14_gb300.build")
        lib = _bind(ctypes.CDLL(p))
        if path is None:
            _lib = lib
        return lib


def _check(rc: int, lib) -> int:
    if rc < 0:
        raise AttnError(rc, lib.attn_last_error().decode(errors="replace"))
    return rc


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FP16
    if t.dtype == torch.bfloat16:
        return BF16
    raise AttnError(-4, f"unsupported dtype {t.dtype}")


def _stream_handle(stream, device):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


class _OnDevice:
    """Make `device` current for the call (the library works on the current
    device); does nothing when it already is."""
    __slots__ = ("ctx",)

    def __init__(self, device):
        import torch
        idx = device.index if device.index is not None else torch.cuda.current_device()
        self.ctx = None if idx == torch.cuda.current_device() else torch.cuda.device(idx)

    def __enter__(self):
        if self.ctx is not None:
            self.ctx.__enter__()

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
             return_lse: bool = True, stream=None):
    """O = softmax(scale * Q K^T [+ causal]) V on the GPU.

    q: [b, h, sq, d], k/v: [b, h, sk, d] contiguous CUDA tensors (fp16 or
    bf16, same dtype and device).  ``scale`` defaults to 1/sqrt(d).  ``o``
    and ``lse`` may be given (preallocated outputs); otherwise they are
    allocated with torch.  Returns (o, lse) -- lse is None when
    ``return_lse`` is False and no ``lse`` was given.
    """
    import torch
    lib = load()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise AttnError(-2, "q, k, v must be 4-D [b, h, s, d]")
    b, h, sq, d = q.shape
    sk = k.shape[2]
    if tuple(k.shape) != (b, h, sk, d) or tuple(v.shape) != (b, h, sk, d):
        raise AttnError(-2, f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise AttnError(-4, "q, k, v dtypes differ")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((b, h, sq), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous():
        raise AttnError(-2, "o must be a contiguous tensor shaped and typed like q")
    if lse is not None and (tuple(lse.shape) != (b, h, sq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise AttnError(-2, "lse must be contiguous fp32 [b, h, sq]")
    with _OnDevice(q.device):
        rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr() if lse is not None else None,
                          b, h, sq, sk, d, int(bool(causal)), float(scale), _dtype_code(q),
                          _stream_handle(stream, q.device))
    _check(rc, lib)
    return o, lse


def attn_fwd_fp8(q, k, v, causal: bool = False, scale: float | None = None, descale_q: float = 1.0,
                 descale_k: float = 1.0, descale_v: float = 1.0, o=None, lse=None, stream=None):
    """e4m3 inputs [b, h, s, d], d = 64 or 128 (torch.float8_e4m3fn CUDA tensors) with
    per-tensor descales; returns (o bf16 [b, h, sq, d], lse fp32)."""
    import torch
    lib = load()
    b, h, sq, d = q.shape
    sk = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float8_e4m3fn:
            raise AttnError(-4, f"{name} must be a contiguous CUDA float8_e4m3fn tensor")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if o is None:
        o = torch.empty((b, h, sq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((b, h, sq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), b, h, sq, sk,
                              d, int(bool(causal)), float(scale), float(descale_q), float(descale_k),
                              float(descale_v), _stream_handle(stream, q.device))
    _check(rc, lib)
    return o, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                    causal: bool = False, scale: float | None = None, o=None, lse=None, stream=None):
    """Packed variable-length forward.  q: [total_q, h, d], k/v: [total_k,
    h, d] CUDA tensors; cu_seqlens_*: int32 CUDA tensors [batch + 1].
    Returns (o [total_q, h, d], lse [h, total_q])."""
    import torch
    lib = load()
    total_q, h, d = q.shape
    total_k = k.shape[0]
    batch = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != batch + 1:
        raise AttnError(-2, "cu_seqlens_q and cu_seqlens_k sizes differ")
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise AttnError(-4, "cu_seqlens must be int32")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((h, total_q), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), batch, h, total_q, total_k,
                                 int(max_seqlen_q), int(max_seqlen_k), d, int(bool(causal)), float(scale),
                                 _dtype_code(q), _stream_handle(stream, q.device))
    _check(rc, lib)
    return o, lse


def splitkv_workspace_bytes(b, h, sq, d, num_splits) -> int:
    lib = load()
    return _check(int(lib.attn_fwd_splitkv_workspace_bytes(b, h, sq, d, num_splits)), lib)


def splitkv_default_splits(b, h, sq, sk, d, causal=False) -> int:
    lib = load()
    return _check(int(lib.attn_fwd_splitkv_default_splits(b, h, sq, sk, d, int(bool(causal)))), lib)


def attn_fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int | None = None,
                     o=None, lse=None, workspace=None, stream=None):
    """Split-KV forward (same result as attn_fwd).  ``num_splits`` defaults
    to the library's choice for the device; ``workspace`` (a CUDA uint8
    tensor) is allocated with torch when not given.  Returns (o, lse)."""
    import torch
    lib = load()
    b, h, sq, d = q.shape
    sk = k.shape[2]
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if num_splits is None:
        with torch.cuda.device(q.device):
            num_splits = splitkv_default_splits(b, h, sq, sk, d, causal)
    need = splitkv_workspace_bytes(b, h, sq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, h, sq), dtype=torch.float32, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  b, h, sq, sk, d, int(bool(causal)), float(scale), _dtype_code(q), int(num_splits),
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream, q.device))
    _check(rc, lib)
    return o, lse


def attn_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, k_new=None, v_new=None, causal: bool = False,
                     scale: float | None = None, num_splits: int | None = None, o=None, lse=None, workspace=None,
                     stream=None):
    """Attention of q [b, h, sq, d] against a KV cache [b, h, s_cache, d]
    whose batch element i holds cache_seqlens[i] valid tokens (int32 CUDA
    tensor [b]).  With k_new / v_new [b, h, s_new, d] the new rows are
    first written into the cache at each element's length (the caches are
    updated in place; cache_seqlens is not) and attended to as well.
    ``num_splits`` defaults to the library's split-KV choice for s_cache.
    Returns (o, lse)."""
    import torch
    lib = load()
    b, h, sq, d = q.shape
    s_cache = k_cache.shape[2]
    if tuple(k_cache.shape) != (b, h, s_cache, d) or tuple(v_cache.shape) != (b, h, s_cache, d):
        raise AttnError(-2, f"cache shapes {tuple(k_cache.shape)} / {tuple(v_cache.shape)} do not match q")
    if (k_new is None) != (v_new is None):
        raise AttnError(-1, "k_new and v_new must both be given or both be None")
    s_new = 0 if k_new is None else k_new.shape[2]
    if k_new is not None and (tuple(k_new.shape) != (b, h, s_new, d) or tuple(v_new.shape) != (b, h, s_new, d)):
        raise AttnError(-2, "k_new / v_new must be [b, h, s_new, d]")
    if cache_seqlens.dtype != torch.int32 or cache_seqlens.numel() != b:
        raise AttnError(-4, "cache_seqlens must be an int32 tensor of b elements")
    tensors = [("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("cache_seqlens", cache_seqlens)]
    if k_new is not None:
        tensors += [("k_new", k_new), ("v_new", v_new)]
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
        if name != "cache_seqlens" and t.dtype != q.dtype:
            raise AttnError(-4, f"{name} dtype differs from q")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if num_splits is None:
        with torch.cuda.device(q.device):
            num_splits = splitkv_default_splits(b, h, sq, max(s_cache, 1), d, causal)
        num_splits = max(1, min(num_splits, (s_cache + 127) // 128))
    need = splitkv_workspace_bytes(b, h, sq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, h, sq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_kvcache(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                  k_new.data_ptr() if k_new is not None else None,
                                  v_new.data_ptr() if v_new is not None else None,
                                  cache_seqlens.data_ptr(), o.data_ptr(), lse.data_ptr(), b, h, sq, s_cache, s_new,
                                  d, int(bool(causal)), float(scale), _dtype_code(q), int(num_splits),
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream, q.device))
    _check(rc, lib)
    return o, lse


def attn_fwd_kvcache_paged(q, k_pool, v_pool, cache_seqlens, block_table, k_new=None, v_new=None,
                           causal: bool = False, scale: float | None = None, num_splits: int | None = None, o=None,
                           lse=None, workspace=None, stream=None):
    """attn_fwd_kvcache over a paged cache: k_pool / v_pool [num_pages,
    page_size, h, d], block_table int32 [b, pages_per_seq] (CUDA tensors).
    Returns (o, lse)."""
    import torch
    lib = load()
    b, h, sq, d = q.shape
    num_pages, page_size = k_pool.shape[0], k_pool.shape[1]
    if tuple(k_pool.shape) != (num_pages, page_size, h, d) or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise AttnError(-2, f"pool shapes {tuple(k_pool.shape)} / {tuple(v_pool.shape)} do not match q")
    if block_table.dim() != 2 or block_table.shape[0] != b or block_table.dtype != torch.int32:
        raise AttnError(-2, "block_table must be int32 [b, pages_per_seq]")
    pages_per_seq = block_table.shape[1]
    if (k_new is None) != (v_new is None):
        raise AttnError(-1, "k_new and v_new must both be given or both be None")
    s_new = 0 if k_new is None else k_new.shape[2]
    if k_new is not None and (tuple(k_new.shape) != (b, h, s_new, d) or tuple(v_new.shape) != (b, h, s_new, d)):
        raise AttnError(-2, "k_new / v_new must be [b, h, s_new, d]")
    if cache_seqlens.dtype != torch.int32 or cache_seqlens.numel() != b:
        raise AttnError(-4, "cache_seqlens must be an int32 tensor of b elements")
    tensors = [("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("cache_seqlens", cache_seqlens),
               ("block_table", block_table)]
    if k_new is not None:
        tensors += [("k_new", k_new), ("v_new", v_new)]
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
        if name not in ("cache_seqlens", "block_table") and t.dtype != q.dtype:
            raise AttnError(-4, f"{name} dtype differs from q")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    cap = pages_per_seq * page_size
    if num_splits is None:
        with torch.cuda.device(q.device):
            num_splits = splitkv_default_splits(b, h, sq, max(cap, 1), d, causal)
        num_splits = max(1, min(num_splits, (cap + 127) // 128))
    need = splitkv_workspace_bytes(b, h, sq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, h, sq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_kvcache_paged(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                        k_new.data_ptr() if k_new is not None else None,
                                        v_new.data_ptr() if v_new is not None else None,
                                        cache_seqlens.data_ptr(), block_table.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        b, h, sq, num_pages, page_size, pages_per_seq, s_new, d, int(bool(causal)),
                                        float(scale), _dtype_code(q), int(num_splits), workspace.data_ptr(),
                                        workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    _check(rc, lib)
    return o, lse


def attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev,
                  causal: bool = False, scale: float | None = None, stream=None):
    """End-to-end call on host (ideally pinned) tensors through the C ABI:
    host->device copies, the forward, device->host copies, all enqueued on
    ``stream``.  The caller synchronises the stream before reading o_host."""
    import torch
    lib = load()
    b, h, sq, d = q_host.shape
    sk = k_host.shape[2]
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    with torch.cuda.device(q_dev.device):
        rc = lib.attn_fwd_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
                               lse_host.data_ptr() if lse_host is not None else None,
                               q_dev.data_ptr(), k_dev.data_ptr(), v_dev.data_ptr(), o_dev.data_ptr(),
                               lse_dev.data_ptr() if lse_dev is not None else None,
                               b, h, sq, sk, d, int(bool(causal)), float(scale), _dtype_code(q_host),
                               _stream_handle(stream, q_dev.device))
    _check(rc, lib)


def status():
    """(code, block, warp, site) of the device watchdog (synchronises)."""
    lib = load()
    out = (ctypes.c_uint32 * 4)()
    _check(lib.attn_fwd_status(out), lib)
    return tuple(int(x) for x in out)


def status_clear():
    lib = load()
    _check(lib.attn_fwd_status_clear(), lib)


def watchdog_selftest(q, k, v, o, lse, causal, scale, withheld_load: int, timeout_ms: int):
    """Run the forward with one K/V load withheld; returns the recorded code."""
    import torch
    lib = load()
    b, h, sq, d = q.shape
    sk = k.shape[2]
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_watchdog_selftest(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                            lse.data_ptr() if lse is not None else None,
                                            b, h, sq, sk, d, int(bool(causal)), float(scale), _dtype_code(q),
                                            int(withheld_load), int(timeout_ms),
                                            _stream_handle(None, q.device))
    return _check(rc, lib)


def bwd_watchdog_selftest(q, k, v, o, dout, lse, causal, scale, withheld_load: int, timeout_ms: int):
    """Run the backward with one query-tile load withheld in every CTA;
    returns the recorded code.  The gradients are not meaningful."""
    import torch
    lib = load()
    b, h, sq, d = q.shape
    sk = k.shape[2]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = bwd_workspace_bytes(b, h, sq, d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.attn_bwd_watchdog_selftest(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                            b, h, sq, sk, d, int(bool(causal)), float(scale), _dtype_code(q),
                                            ws.data_ptr(), nbytes, int(withheld_load), int(timeout_ms),
                                            _stream_handle(None, q.device))
    return _check(rc, lib)


def bwd_workspace_bytes(b: int, h: int, sq: int, d: int) -> int:
    lib = load()
    return _check(int(lib.attn_bwd_workspace_bytes(b, h, sq, d)), lib)


def attn_bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for the output gradient ``dout``.

    q, o, dout: [b, h, sq, 128]; k, v: [b, h, sk, 128] contiguous CUDA
    tensors of one dtype (fp16 or bf16); lse: fp32 [b, h, sq] from the
    forward.  Outputs and the workspace (a CUDA uint8 tensor of at least
    bwd_workspace_bytes bytes) are allocated with torch when not given."""
    import torch
    lib = load()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise AttnError(-2, "q, k, v must be 4-D [b, h, s, d]")
    b, h, sq, d = q.shape
    sk = k.shape[2]
    if tuple(k.shape) != (b, h, sk, d) or tuple(v.shape) != (b, h, sk, d) or o.shape != q.shape or \
            dout.shape != q.shape or tuple(lse.shape) != (b, h, sq):
        raise AttnError(-2, "shape mismatch among q, k, v, o, dout, lse")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype) or lse.dtype != torch.float32:
        raise AttnError(-4, "q, k, v, o, dout must share a dtype; lse must be fp32")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if workspace is None:
        with torch.cuda.device(q.device):
            need = bwd_workspace_bytes(b, h, sq, d)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("lse", lse), ("dq", dq), ("dk", dk),
                    ("dv", dv), ("workspace", workspace)):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
    with torch.cuda.device(q.device):
        rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), b, h, sq, sk, d, int(bool(causal)),
                          float(scale), _dtype_code(q), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    _check(rc, lib)
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, o, dout, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                    causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None, workspace=None,
                    stream=None):
    """Gradients (dq, dk, dv) of attn_fwd_varlen.  q, o, dout: [total_q, h, d];
    k, v: [total_k, h, d] of one dtype; lse: fp32 [h, total_q];
    cu_seqlens_q / _k: int32 CUDA tensors [batch + 1]."""
    import torch
    lib = load()
    total_q, h, d = q.shape
    total_k = k.shape[0]
    batch = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != batch + 1 or tuple(k.shape) != (total_k, h, d) or tuple(v.shape) != (total_k, h, d) \
            or o.shape != q.shape or dout.shape != q.shape or tuple(lse.shape) != (h, total_q):
        raise AttnError(-2, "shape mismatch among q, k, v, o, dout, lse, cu_seqlens")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        need = _check(int(lib.attn_bwd_varlen_workspace_bytes(batch, h, total_q, max_seqlen_q, d)), lib)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("lse", lse), ("dq", dq), ("dk", dk),
                    ("dv", dv), ("workspace", workspace), ("cu_seqlens_q", cu_seqlens_q),
                    ("cu_seqlens_k", cu_seqlens_k)):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError(-2, f"{name} must be a contiguous CUDA tensor")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise AttnError(-4, "cu_seqlens must be int32")
    with torch.cuda.device(q.device):
        rc = lib.attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                 lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens_q.data_ptr(),
                                 cu_seqlens_k.data_ptr(), batch, h, total_q, total_k, int(max_seqlen_q),
                                 int(max_seqlen_k), d, int(bool(causal)), float(scale), _dtype_code(q),
                                 workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                 _stream_handle(stream, q.device))
    _check(rc, lib)
    return dq, dk, dv
