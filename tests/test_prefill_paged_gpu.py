"""GPU parity of chunked prefill against the paged cache (float64 oracle).

Runs of at least 128 new tokens (with the key length not split) take the
persistent prefill kernel's paged mode; the others the tensor-core decode
kernel; the cases below exercise both.

Sequence b has n_b new tokens, the last n_b of its L_b cached ones; new token
t sees keys 0 .. L_b - n_b + t.  Cases: prefixes of every length including
none (plain causal prefill) and sequences with no new token, more new tokens
than cached ones, groups 1 to 16, forced and automatic chunking of the key
length, ragged page tails with poisoned slots, and at full size 8192 new
tokens after an 8192-token prefix (the benchmark's workload), checked on
every element.  All calls go through the C ABI.
"""
import pytest
import torch

import gqa_attention_head_sink_gb300 as sa
import oracle
from gqa_attention_head_sink_gb300 import build, workloads
from tests.full_parity import check_paged_prefill_everywhere
from tests.parity import assert_parity, lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    sa.load()
    yield
    assert sa.sink_attn_get_device_error() == 0, "a bounded device wait timed out"


def run(inp, num_splits=None, out_dtype=torch.float32, with_lse=False):
    total_q, hq = inp.q.shape[0], inp.q.shape[1]
    lse = torch.empty((total_q, hq), dtype=torch.float32, device="cuda") if with_lse else None
    out = sa.sink_attn_prefill_paged(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.cu_seqlens_q,
                                     inp.seqlens_t, inp.sinks, inp.scale,
                                     num_splits=inp.num_splits if num_splits is None else num_splits,
                                     out_dtype=out_dtype, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def oracle_paged(inp):
    return oracle.paged_attention(inp.q.cpu(), inp.k_pages.cpu(), inp.v_pages.cpu(), inp.page_table.cpu(),
                                  inp.seqlens_t.cpu(), inp.cu_seqlens_q.cpu(), inp.sinks.cpu(), inp.scale,
                                  page_size=inp.page_size)


SMALL = [
    # cached lengths L_b, new tokens n_b, Hq, Hkv, sink mode, splits
    ([100, 5, 300], [20, 5, 0], 8, 2, "mixed", 0),
    ([1000, 2000, 17], [300, 1, 17], 64, 8, "normal2", 0),
    ([4096], [1024], 64, 8, "mixed", 3),
    ([700, 800], [900, 10], 16, 1, "normal1", 0),       # 200 new tokens before the cache start
    ([129, 130, 131], [129, 130, 131], 24, 3, "zero", 1),  # every token new: causal prefill
    ([500, 64], [333, 64], 4, 4, "normal2", 0),         # group 1
    ([2500, 1], [2500, 1], 64, 4, "neginf", 0),         # group 16
]


@pytest.mark.parametrize("lens,new,hq,hkv,sink,splits", SMALL)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_paged_small(lens, new, hq, hkv, sink, splits, out_dtype):
    inp = workloads.make_paged_prefill(lens, new, num_q_heads=hq, num_kv_heads=hkv, seed=sum(new) % 97 + hq,
                                       sink_mode=sink, num_splits=splits, spare_pages=3, poison=True,
                                       device="cuda")
    out, lse = run(inp, out_dtype=out_dtype, with_lse=True)
    want, want_lse = oracle_paged(inp)
    assert_parity(out, want, bf16_output=out_dtype == torch.bfloat16)
    lse_close(lse, want_lse)


def test_prefill_paged_all_new_matches_contiguous_prefill():
    # n_b = L_b: the same numbers as the contiguous causal prefill of the gathered cache
    lens = [333, 1000, 64]
    inp = workloads.make_paged_prefill(lens, lens, seed=51, sink_mode="mixed", num_splits=1, device="cuda")
    out, _ = run(inp)
    j = [torch.arange(L, device="cuda") for L in lens]
    k = torch.cat([inp.k_pages[inp.page_table[b, jj // 16].long(), :, jj % 16] for b, jj in enumerate(j)])
    v = torch.cat([inp.v_pages[inp.page_table[b, jj // 16].long(), :, jj % 16] for b, jj in enumerate(j)])
    ref = sa.sink_attn_prefill(inp.q, k.contiguous(), v.contiguous(), inp.sinks, inp.cu_seqlens_q, inp.scale,
                               max_seqlen=max(lens))
    torch.cuda.synchronize()
    assert_parity(out, ref.double().cpu().numpy())


def test_prefill_paged_long_runs_equal_contiguous_prefill_bit_for_bit():
    # runs of >= 128 new tokens go to the persistent prefill kernel's paged mode: with every
    # token new it must give exactly what the contiguous prefill gives on the gathered cache
    lens = [1000, 333, 4097]
    inp = workloads.make_paged_prefill(lens, lens, seed=54, sink_mode="mixed", num_splits=0, spare_pages=2,
                                       poison=True, device="cuda")
    out, lse = run(inp, with_lse=True)
    j = [torch.arange(L, device="cuda") for L in lens]
    k = torch.cat([inp.k_pages[inp.page_table[b, jj // 16].long(), :, jj % 16] for b, jj in enumerate(j)])
    v = torch.cat([inp.v_pages[inp.page_table[b, jj // 16].long(), :, jj % 16] for b, jj in enumerate(j)])
    lse_ref = torch.empty_like(lse)
    ref = sa.sink_attn_prefill(inp.q, k.contiguous(), v.contiguous(), inp.sinks, inp.cu_seqlens_q, inp.scale,
                               max_seqlen=max(lens), lse=lse_ref)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, lse_ref)


def test_prefill_paged_splits_agree():
    inp = workloads.make_paged_prefill([3000, 1200], [700, 1200], seed=52, sink_mode="normal2", device="cuda")
    want, _ = oracle_paged(inp)
    for splits in [1, 2, 5, 0]:
        out, _ = run(inp, num_splits=splits)
        assert_parity(out, want)


def test_prefill_paged_full_size():
    # 8192 new tokens after an 8192-token prefix (Hq 64, Hkv 8): the benchmark's launch (keys not
    # split, the prefill kernel's paged mode); every element of the bf16 output and the lse
    L, n = 16384, 8192
    inp = workloads.workload("chunked_prefill", device="cuda")
    assert inp.seqlens == [L] and inp.q_lens == [n]
    out, lse = run(inp, out_dtype=torch.bfloat16, with_lse=True)
    total = check_paged_prefill_everywhere(inp, out16=out, lse=lse)
    assert total["out16"]["n"] == n * inp.num_q_heads * 64


@pytest.mark.parametrize("n_new", [700, 90])  # the prefill kernel's paged mode, then the tensor-core decode kernel
def test_prefill_paged_running_max_moves_often(n_new):
    # keys whose norm grows along the cache raise the running maximum at nearly every key tile
    L = 1500
    inp = workloads.make_paged_prefill([L], [n_new], num_q_heads=16, num_kv_heads=2, seed=55, sink_mode="mixed",
                                       device="cuda")
    j = torch.arange(L, device="cuda")
    grow = (1.0 + j.float() / 80.0)[:, None]
    pages = inp.page_table[0, j // 16].long()
    inp.k_pages[pages, :, j % 16] = (inp.k_pages[pages, :, j % 16].float() * grow[:, None, :]).to(torch.bfloat16)
    out, lse = run(inp, with_lse=True)
    want, want_lse = oracle_paged(inp)
    assert_parity(out, want)
    lse_close(lse, want_lse)
