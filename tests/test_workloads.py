"""The seeded input generators (host logic, no GPU): shapes, types,
determinism and the distributions the workloads state."""
import torch

from attention_forward_14_gb300 import workloads as W


def test_draw_is_seeded_and_shaped():
    a = W.draw(2, 3, 5, 7, 64, "bf16", seed=11, qk_std=3.0)
    b = W.draw(2, 3, 5, 7, 64, "bf16", seed=11, qk_std=3.0)
    c = W.draw(2, 3, 5, 7, 64, "bf16", seed=12, qk_std=3.0)
    assert [tuple(t.shape) for t in a] == [(2, 3, 5, 64), (2, 3, 7, 64), (2, 3, 7, 64)]
    assert all(t.dtype == torch.bfloat16 for t in a)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[0], c[0])


def test_draw_scales_q_and_k_only():
    q1, k1, v1 = W.draw(1, 1, 4096, 4096, 64, "fp16", seed=5, qk_std=1.0)
    q3, k3, v3 = W.draw(1, 1, 4096, 4096, 64, "fp16", seed=5, qk_std=3.0)
    assert abs(q3.float().std().item() / q1.float().std().item() - 3.0) < 0.01
    assert abs(k3.float().std().item() / k1.float().std().item() - 3.0) < 0.01
    assert torch.equal(v1, v3)


def test_randn_device_is_seeded_and_chunk_consistent():
    shape = (3, 1000, 7)
    a = W.randn_device(shape, "bf16", 41001, torch.device("cpu"), chunk=4096)
    b = W.randn_device(shape, "bf16", 41001, torch.device("cpu"), chunk=4096)
    c = W.randn_device(shape, "bf16", 41002, torch.device("cpu"), chunk=4096)
    assert a.shape == shape and a.dtype == torch.bfloat16
    assert torch.equal(a, b) and not torch.equal(a, c)
    # the chunks draw one stream in order: a single chunk gives the same values
    whole = W.randn_device(shape, "bf16", 41001, torch.device("cpu"), chunk=1 << 26)
    assert torch.equal(a, whole)
    x = W.randn_device((1 << 20,), torch.float32, 7, torch.device("cpu"), std=2.0, chunk=1 << 16).double()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 2.0) < 0.02


def test_varlen_lengths_in_range_and_seeded():
    lens = W.varlen_lengths(500, 3, 40, 9)
    assert len(lens) == 500 and min(lens) >= 3 and max(lens) <= 40
    assert lens == W.varlen_lengths(500, 3, 40, 9)
    assert len(set(lens)) > 20


def test_sample_heads_keeps_first_and_last():
    w = W.WORKLOADS["noncausal_b8_h16_s1000_d64_bf16"]
    pairs = W.sample_heads(w, n=6)
    assert pairs[0] == (0, 0) and pairs[1] == (w.b - 1, w.h - 1)
    assert len(set(pairs)) == 6
    assert all(0 <= bi < w.b and 0 <= hi < w.h for bi, hi in pairs)


def test_draw_varlen_packs_the_dense_draws():
    q, k, v, cu_q, cu_k, dense = W.draw_varlen([3, 0, 5], [4, 2, 5], 2, 64, "bf16", seed=21)
    assert cu_q.tolist() == [0, 3, 3, 8] and cu_k.tolist() == [0, 4, 6, 11]
    assert tuple(q.shape) == (8, 2, 64) and tuple(k.shape) == (11, 2, 64)
    # token-major packing of sequence 2's dense [1, h, s, d] tensors
    assert torch.equal(q[3:8], dense[2][0][0].transpose(0, 1))
    assert torch.equal(v[6:11], dense[2][2][0].transpose(0, 1))
