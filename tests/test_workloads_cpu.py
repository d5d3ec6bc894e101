"""The seeded input generators and the work counts the benchmark divides by.

The generators hold none of the attention arithmetic; these checks pin their
layouts (what the oracle and the kernels both read) and the algorithmic
counts against brute-force enumeration.
"""
import torch

from gqa_attention_head_sink_gb300 import workloads


def test_generators_are_reproducible():
    a = workloads.make_decode([40, 17], num_q_heads=8, num_kv_heads=2, seed=7, q_len=3)
    b = workloads.make_decode([40, 17], num_q_heads=8, num_kv_heads=2, seed=7, q_len=3)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_pages, b.k_pages) and torch.equal(a.page_table, b.page_table)
    assert a.q.shape == (2, 3, 8, 64) and a.q_len == 3


def test_paged_prefill_layout():
    d = workloads.make_paged_prefill([100, 5, 300], [20, 5, 0], num_q_heads=8, num_kv_heads=2, seed=1)
    assert d.q.shape == (25, 8, 64)
    assert d.cu_seqlens_q.tolist() == [0, 20, 25, 25]
    # every sequence owns distinct pool pages, enough for its cached length
    owned = [set(d.page_table[b, :(L + 15) // 16].tolist()) for b, L in enumerate(d.seqlens)]
    assert sum(len(o) for o in owned) == len(set().union(*owned))


def test_prefill_flops_count_causal_pairs():
    for lens in ([1], [5, 0, 7], [128, 129]):
        pairs = sum(i + 1 for L in lens for i in range(L))
        assert workloads.prefill_flops(lens, 3) == 4 * 64 * 3 * pairs


def test_paged_prefill_flops_count_visible_pairs():
    for lens, new in (([16384], [8192]), ([5], [8]), ([100, 7], [1, 7]), ([33], [0])):
        pairs = sum(max(0, L - n + t + 1) for L, n in zip(lens, new) for t in range(n))
        assert workloads.paged_prefill_flops(lens, new, 2) == 4 * 64 * 2 * pairs
    # every token new: the causal prefill count
    assert workloads.paged_prefill_flops([8192], [8192], 64) == workloads.prefill_flops([8192], 64)


def test_decode_bytes_count_each_kv_byte_once():
    n = workloads.decode_bytes([8192] * 64, 64, 8, out_bytes=2, q_len=4)
    kv = 64 * 8192 * 8 * 64 * 2 * 2
    q = o = 64 * 4 * 64 * 64 * 2
    assert n == kv + q + o + 64 * 512 * 4 + 64 * 4


def test_qkv_rope_inputs_and_bytes():
    r = workloads.make_qkv_rope(10, num_q_heads=8, num_kv_heads=2)
    assert r.q.shape == (10, 8, 64) and r.k_bias.shape == (2, 64) and r.positions.tolist() == list(range(10))
    assert workloads.qkv_rope_bytes(10, 8, 2) == 2 * 10 * 12 * 64 * 2 + 40 + 12 * 64 * 2
