"""Seeded synthetic inputs for the attention forward.

This module is shared by the tests, the benchmark and the smoke check; it
holds no attention arithmetic, only shapes, seeds and random draws, so that the
CUDA path and the fp64 oracle always see the same inputs.  It imports nothing
from the rest of the package.

Recipe: a CPU ``torch.Generator`` seeded per workload draws Q, K, V in that
order with ``randn`` in fp32 (Q and K multiplied by ``qk_std``), then each is
rounded to the workload dtype.  The oracle consumes the rounded values, so
input quantisation is not counted as kernel error.  The shapes follow the
[b, h, s, d] layout of "flash-attn 实现 prefill 阶段" (问题分析); the scale is
1/sqrt(d) as in flash-attention-minimal ``forward()``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    h: int
    sq: int
    sk: int
    d: int
    dtype: str
    causal: bool
    qk_std: float
    seed: int
    splitkv: bool = False  # run through the split-KV entry point (decode shapes)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def flops(self) -> float:
        """Counted work: 4*b*h*sq*sk*d, half of it when causal."""
        f = 4.0 * self.b * self.h * self.sq * self.sk * self.d
        return f * 0.5 if self.causal else f

    def bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O written once, fp32 LSE."""
        if self.dtype == "e4m3":  # 1-byte Q, K, V; bf16 O
            return (self.b * self.h * (self.sq * self.d + 2 * self.sk * self.d) + 2 * self.b * self.h * self.sq * self.d
                    + 4 * self.b * self.h * self.sq)
        e = 2
        return (e * self.b * self.h * (2 * self.sq * self.d + 2 * self.sk * self.d)
                + 4 * self.b * self.h * self.sq)


# The five workloads the project is measured on, named by what they are.
WORKLOADS = {
    w.name: w for w in [
        Workload("noncausal_b1_h2_s256_d128_fp16", 1, 2, 256, 256, 128, "fp16", False, 1.0, 20260000),
        Workload("noncausal_b4_h16_s1024_d128_fp16", 4, 16, 1024, 1024, 128, "fp16", False, 1.0, 20260001),
        Workload("noncausal_b8_h16_s1000_d64_bf16", 8, 16, 1000, 1000, 64, "bf16", False, 1.0, 20260002),
        Workload("causal_b2_h32_s4096_d128_bf16", 2, 32, 4096, 4096, 128, "bf16", True, 1.0, 20260003),
        Workload("causal_b1_h32_s16384_d128_bf16_qk3", 1, 32, 16384, 16384, 128, "bf16", True, 3.0, 20260004),
        # the long causal problem with 8-bit (e4m3) inputs
        Workload("causal_b1_h32_s16384_d128_e4m3", 1, 32, 16384, 16384, 128, "e4m3", True, 1.0, 20260007),
        # the ragged head-dim-64 problem with 8-bit (e4m3) inputs
        Workload("noncausal_b8_h16_s1000_d64_e4m3", 8, 16, 1000, 1000, 64, "e4m3", False, 1.0, 20260013),
        # decode step: one query row per (batch, head) against a 16k-key cache
        Workload("decode_b8_h32_q1_s16384_d128_bf16", 8, 32, 1, 16384, 128, "bf16", False, 1.0, 20260005,
                 splitkv=True),
    ]
}
ORDER = [n for n in WORKLOADS if not WORKLOADS[n].splitkv and WORKLOADS[n].dtype != "e4m3"]
FP8 = [n for n in WORKLOADS if WORKLOADS[n].dtype == "e4m3"]
DECODE = [n for n in WORKLOADS if WORKLOADS[n].splitkv]
HEADLINE = "causal_b1_h32_s16384_d128_bf16_qk3"


def draw(b, h, sq, sk, d, dtype, seed, qk_std=1.0, v_std=1.0):
    """Seeded Q [b,h,sq,d], K/V [b,h,sk,d] as CPU tensors of ``dtype``."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((b, h, sq, d), generator=g, dtype=torch.float32)
    k = torch.randn((b, h, sk, d), generator=g, dtype=torch.float32)
    v = torch.randn((b, h, sk, d), generator=g, dtype=torch.float32)
    if qk_std != 1.0:
        q.mul_(qk_std)
        k.mul_(qk_std)
    if v_std != 1.0:
        v.mul_(v_std)
    return q.to(tdt), k.to(tdt), v.to(tdt)


def randn_device(shape, dtype, seed, device, std=1.0, chunk=1 << 26):
    """Seeded N(0, std^2) values of ``shape``, drawn on ``device`` in fp32
    ``chunk`` elements at a time (so a tensor of several GiB needs no
    full-size fp32 copy) and rounded to ``dtype``.  The values depend on the
    seed, the shape and the device type only.  For problems too large to draw
    on the host; the tests copy the parts they check back to the host."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(shape, dtype=tdt, device=device)
    flat = out.view(-1)
    for a in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - a)
        t = torch.randn(n, generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            t.mul_(std)
        flat[a:a + n].copy_(t)
    return out


def draw_grad(b, h, sq, d, dtype, seed):
    """Seeded output gradient dO [b, h, sq, d] ~ N(0, 1) as a CPU tensor."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn((b, h, sq, d), generator=g, dtype=torch.float32).to(tdt)


def inputs(w: Workload):
    """CPU tensors (q, k, v) of the workload."""
    return draw(w.b, w.h, w.sq, w.sk, w.d, w.dtype, w.seed, w.qk_std)


def sample_heads(w: Workload, n: int = 4, seed: int = 7):
    """Seeded sample of (batch, head) pairs, always including the first and
    the last pair."""
    pairs = [(0, 0)]
    if (w.b - 1, w.h - 1) != (0, 0):
        pairs.append((w.b - 1, w.h - 1))
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    while len(pairs) < min(n, w.b * w.h):
        bi = int(torch.randint(0, w.b, (1,), generator=g))
        hi = int(torch.randint(0, w.h, (1,), generator=g))
        if (bi, hi) not in pairs:
            pairs.append((bi, hi))
    return pairs


@dataclass(frozen=True)
class VarlenWorkload:
    """Packed batch of sequences with seeded lengths in [lo, hi] (self
    attention: query and key lengths equal per sequence)."""
    name: str
    n: int
    lo: int
    hi: int
    h: int
    d: int
    dtype: str
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def lengths(self):
        return varlen_lengths(self.n, self.lo, self.hi, self.seed)

    def flops(self) -> float:
        f = sum(4.0 * self.h * s * s * self.d for s in self.lengths())
        return f * 0.5 if self.causal else f

    def bytes(self) -> int:
        t = sum(self.lengths())
        return 2 * t * self.h * self.d * 4 + 4 * self.h * t


VARLEN = {
    w.name: w for w in [
        VarlenWorkload("varlen_16seq_512to8192_h32_d128_bf16_causal", 16, 512, 8192, 32, 128, "bf16", True,
                       20260006),
    ]
}


def varlen_inputs(w: VarlenWorkload):
    lens = w.lengths()
    return draw_varlen(lens, lens, w.h, w.d, w.dtype, w.seed)


def draw_varlen(lens_q, lens_k, h, d, dtype, seed, qk_std=1.0):
    """Packed variable-length inputs: sequence s draws its own dense
    [1, h, lens_q[s], d] / [1, h, lens_k[s], d] tensors (seed + s), which are
    laid out token-major and concatenated.  Returns (q, k, v) packed
    [total, h, d] CPU tensors, cu_seqlens_q, cu_seqlens_k (int32) and the
    per-sequence dense tensors [(q_s, k_s, v_s), ...]."""
    dense = [draw(1, h, int(a), int(b), d, dtype, seed + i, qk_std) for i, (a, b) in enumerate(zip(lens_q, lens_k))]

    def pack(idx):
        parts = [t[idx][0].transpose(0, 1).contiguous() for t in dense]  # [s, h, d]
        return torch.cat(parts, 0) if parts else torch.empty(0, h, d, dtype=DTYPES[dtype])

    cu_q = torch.zeros(len(lens_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(lens_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor([int(x) for x in lens_q], dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.tensor([int(x) for x in lens_k], dtype=torch.int64), 0).to(torch.int32)
    return pack(0), pack(1), pack(2), cu_q, cu_k, dense


def varlen_lengths(n, lo, hi, seed):
    """Seeded sequence lengths, uniform in [lo, hi]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


# Backward workloads: the forward's problem plus a seeded dO.  One step is
# one attn_bwd call; its work is the five products of the gradient (S, dP,
# dV, dK, dQ), 2.5x the forward's FLOPs.
@dataclass(frozen=True)
class BwdWorkload:
    fwd: str        # the forward workload whose q, k, v are used
    grad_seed: int

    @property
    def w(self) -> Workload:
        return WORKLOADS[self.fwd]

    @property
    def name(self) -> str:
        return "bwd_" + self.fwd

    def flops(self) -> float:
        return 2.5 * self.w.flops()

    def bytes(self) -> int:
        w = self.w
        e = 2  # 16-bit inputs and gradients
        # read q, k, v, o, dO, lse; write dq, dk, dv
        return (e * w.b * w.h * (3 * w.sq * w.d + 2 * w.sk * w.d) + 4 * w.b * w.h * w.sq
                + e * w.b * w.h * (w.sq * w.d + 2 * w.sk * w.d))


BWD = {bw.name: bw for bw in [
    BwdWorkload("causal_b1_h32_s16384_d128_bf16_qk3", 20260008),
    BwdWorkload("causal_b2_h32_s4096_d128_bf16", 20260009),
    BwdWorkload("noncausal_b8_h16_s1000_d64_bf16", 20260010),
]}


# KV-cache decoding: b sequences whose cached lengths are seeded, uniform in
# [lo, hi], in a cache of capacity `cap`; each step writes s_new new tokens
# per sequence and their s_new queries attend (causally) to everything
# cached.  The lengths do not advance between steps, so every step repeats
# the same work.
@dataclass(frozen=True)
class KvcacheWorkload:
    name: str
    b: int
    h: int
    cap: int
    lo: int
    hi: int
    s_new: int
    d: int
    dtype: str
    seed: int
    causal: bool = True
    page_size: int = 0  # > 0: a paged cache of pages of this many keys (capacity / page_size per sequence)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def sq(self) -> int:
        return self.s_new

    def lengths(self):
        """Cached tokens per sequence before the step."""
        return varlen_lengths(self.b, self.lo, self.hi, self.seed)

    def visible(self):
        """Keys seen by each query row, summed (causal: row i of a sequence
        with n = min(len + s_new, cap) keys sees min(n, n - s_new + i + 1))."""
        tot = 0
        for l0 in self.lengths():
            n = min(max(l0, 0) + self.s_new, self.cap)
            for i in range(self.sq):
                tot += max(0, min(n, n - self.sq + i + 1)) if self.causal else n
        return tot

    def flops(self) -> float:
        return 4.0 * self.h * self.d * self.visible()

    def bytes(self) -> int:
        """Algorithmic HBM bytes of one step: the valid K and V read once,
        Q and the new K/V rows read, the new rows written into the cache,
        O and the fp32 LSE written."""
        e = 2
        valid = sum(min(max(l0, 0) + self.s_new, self.cap) for l0 in self.lengths())
        rows = self.b * self.h
        return (e * self.h * self.d * 2 * valid + e * rows * self.sq * self.d + 2 * e * rows * self.s_new * self.d
                + 2 * e * rows * self.s_new * self.d + e * rows * self.sq * self.d + 4 * rows * self.sq)


KVCACHE = {kw.name: kw for kw in [
    KvcacheWorkload("kvcache_decode_b8_h32_cap16384_len1to16383_d128_bf16", 8, 32, 16384, 1, 16383, 1, 128, "bf16",
                    20260011),
    # the same decoding step over a paged cache: 256-key pages, shuffled in the pool
    KvcacheWorkload("kvcache_paged_decode_b8_h32_page256_len1to16383_d128_bf16", 8, 32, 16384, 1, 16383, 1, 128,
                    "bf16", 20260011, page_size=256),
]}


def kvcache_inputs(kw: KvcacheWorkload):
    """CPU tensors q [b,h,s_new,d], k_cache/v_cache [b,h,cap,d] (every slot
    drawn: the unused ones take no part), k_new/v_new [b,h,s_new,d] and the
    int32 lengths [b]."""
    q, kc, vc = draw(kw.b, kw.h, kw.sq, kw.cap, kw.d, kw.dtype, kw.seed)
    _, kn, vn = draw(kw.b, kw.h, 1, kw.s_new, kw.d, kw.dtype, kw.seed + 1)
    lens = torch.tensor(kw.lengths(), dtype=torch.int32)
    return q, kc, vc, kn, vn, lens


def kvcache_paged_inputs(kw: KvcacheWorkload):
    """The dense workload's caches cut into pages of kw.page_size keys,
    placed in the pool [b * pages, page_size, h, d] in a seeded random order;
    returns (q, k_pool, v_pool, k_new, v_new, lengths, block_table)."""
    q, kc, vc, kn, vn, lens = kvcache_inputs(kw)
    pages = kw.cap // kw.page_size
    g = torch.Generator(device="cpu")
    g.manual_seed(int(kw.seed) + 7)
    table = torch.randperm(kw.b * pages, generator=g).reshape(kw.b, pages).to(torch.int32)

    def pool(c):  # [b, h, cap, d] -> pages [b*pages, page_size, h, d] at their table slots
        out = torch.empty((kw.b * pages, kw.page_size, kw.h, kw.d), dtype=c.dtype)
        paged = c.reshape(kw.b, kw.h, pages, kw.page_size, kw.d).permute(0, 2, 3, 1, 4)
        out[table.reshape(-1).long()] = paged.reshape(kw.b * pages, kw.page_size, kw.h, kw.d)
        return out

    return q, pool(kc), pool(vc), kn, vn, lens, table


# Backward of the packed workload: its q, k, v plus a seeded output gradient
# dO ~ N(0, 1) [total, h, d]; one step is one attn_bwd_varlen call.
@dataclass(frozen=True)
class BwdVarlenWorkload:
    fwd: str
    grad_seed: int

    @property
    def w(self) -> VarlenWorkload:
        return VARLEN[self.fwd]

    @property
    def name(self) -> str:
        return "bwd_" + self.fwd

    def flops(self) -> float:
        return 2.5 * self.w.flops()

    def bytes(self) -> int:
        t = sum(self.w.lengths())
        e = 2
        # read q, k, v, o, dO and lse; write dq, dk, dv
        return 8 * e * t * self.w.h * self.w.d + 4 * self.w.h * t


BWD_VARLEN = {bw.name: bw for bw in [
    BwdVarlenWorkload("varlen_16seq_512to8192_h32_d128_bf16_causal", 20260012),
]}


def bwd_varlen_grad(bw: BwdVarlenWorkload):
    """The seeded dO [total, h, d] of the packed backward workload."""
    t = sum(bw.w.lengths())
    return draw_grad(1, t, bw.w.h, bw.w.d, bw.w.dtype, bw.grad_seed)[0]
