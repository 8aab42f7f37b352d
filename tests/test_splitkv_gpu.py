"""Split-KV forward (key range cut into splits, partial softmaxes merged by
the online-recurrence step) against the fp64 oracle on seeded inputs."""
import math
import zlib

import numpy as np
import pytest
import torch

import attention_forward_14_gb300 as af
from attention_forward_14_gb300 import binding
from attention_forward_14_gb300 import workloads as W
from parity import compare, dtype_name
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # b, h, sq, sk, d, dtype, causal, splits
    (1, 8, 1, 4096, 128, "bf16", False, 4),
    (1, 8, 1, 4096, 128, "bf16", True, 7),
    (2, 4, 7, 3000, 128, "fp16", False, 3),
    (2, 4, 7, 3000, 64, "bf16", True, 24),     # one tile per split, ragged last tile
    (1, 2, 64, 1000, 64, "fp16", False, 2),
    (1, 2, 300, 700, 128, "bf16", True, 5),    # several row blocks, diagonal tiles
    (1, 1, 513, 100, 128, "bf16", True, 1),    # rows with no visible key
    (1, 2, 600, 200, 64, "fp16", True, 2),     # rows with no visible key, split
    (1, 3, 256, 256, 128, "fp16", False, 2),
]


def _run(q, k, v, causal, scale, splits):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    af.attn_fwd_splitkv(qd, kd, vd, causal=causal, scale=scale, num_splits=splits, o=o, lse=lse)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
def test_splitkv_matches_oracle(case):
    b, h, sq, sk, d, dt, causal, splits = case
    q, k, v = W.draw(b, h, sq, sk, d, dt, seed=zlib.crc32(repr(case).encode()))
    scale = 1 / math.sqrt(d)
    o, lse = _run(q, k, v, causal, scale, splits)
    o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal, scale)
    compare(o, lse, o_ref, lse_ref, dt, f"splitkv {case}")


def test_splitkv_large_logits():
    """Q, K ~ N(0, 9): splits whose maxima differ by many units of log2."""
    q, k, v = W.draw(1, 4, 16, 8192, 128, "bf16", seed=77, qk_std=3.0)
    scale = 1 / math.sqrt(128)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal, scale, 16)
        o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal, scale)
        compare(o, lse, o_ref, lse_ref, "bf16", f"splitkv qk3 c{causal}")


def test_splitkv_default_splits_and_agreement():
    q, k, v = W.draw(1, 4, 1, 16384, 128, "bf16", seed=5)
    dev = torch.device("cuda", 0)
    s = binding.splitkv_default_splits(1, 4, 1, 16384, 128)
    assert 1 < s <= 64
    o1, l1 = af.attn_fwd_splitkv(q.to(dev), k.to(dev), v.to(dev))
    o2, l2 = af.attn_fwd(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), False, 1 / math.sqrt(128))
    compare(o1.float().cpu().double().numpy(), l1.cpu().double().numpy(), o_ref, lse_ref, "bf16", "default splits")
    compare(o2.float().cpu().double().numpy(), l2.cpu().double().numpy(), o_ref, lse_ref, "bf16", "no split")


def test_splitkv_workspace_reuse_across_calls():
    """The workspace's previous contents do not matter (two calls, one buffer)."""
    dev = torch.device("cuda", 0)
    ws = torch.full((binding.splitkv_workspace_bytes(2, 2, 5, 128, 4),), 0x7f, dtype=torch.uint8, device=dev)
    for seed in (1, 2):
        q, k, v = W.draw(2, 2, 5, 2048, 128, "fp16", seed=seed)
        o, lse = af.attn_fwd_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=True, num_splits=4, workspace=ws)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), True,
                                         1 / math.sqrt(128))
        compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, "fp16", f"reuse {seed}")


@pytest.mark.parametrize("name", W.DECODE)
def test_decode_workload_full(name):
    """The decode workload at full size, in the launch configuration the
    benchmark times (default split count), every row against the oracle."""
    w = W.WORKLOADS[name]
    q, k, v = W.inputs(w)
    splits = binding.splitkv_default_splits(w.b, w.h, w.sq, w.sk, w.d, w.causal)
    o, lse = _run(q, k, v, w.causal, w.scale, splits)
    o_ref, lse_ref = oracle.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), w.causal, w.scale)
    compare(o, lse, o_ref, lse_ref, w.dtype, name)


def test_default_split_counts():
    """The default fills whole waves of the SMs for short queries and does
    not split problems with many query rows that already fill the GPU."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # many query rows, at least one unit per SM: no split
    assert binding.splitkv_default_splits(1, 32, 2048, 16384, 128, True) == 1
    # decode, b*h = 256 units: the count with the best wave fill
    s = binding.splitkv_default_splits(8, 32, 1, 16384, 128)
    units = 256 * s
    fill = units / (sms * -(-units // sms))
    assert s > 1 and fill > 0.9, (s, fill)
    # one key tile: nothing to split
    assert binding.splitkv_default_splits(4, 4, 1, 100, 64) == 1
    # every split keeps at least two key tiles
    s = binding.splitkv_default_splits(1, 1, 1, 1024, 128)
    assert 1 <= s <= 4
