"""The whole-output comparison used for the full-size prefill workloads,
checked on the CPU: fed the oracle's own output it must pass, fed an output
with one element off by more than the tolerance, or a mean error over the
bound, it must fail.  No GPU is involved."""
import numpy as np
import pytest
import torch

import oracle
from gqa_attention_head_sink_gb300 import workloads
from tests.full_parity import check_paged_prefill_everywhere, check_prefill_everywhere


@pytest.fixture(scope="module")
def case():
    inp = workloads.make_prefill([200, 0, 77, 130], num_q_heads=8, num_kv_heads=2, seed=5, sink_mode="mixed")
    want, want_lse = oracle.prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale)
    return inp, torch.from_numpy(want).float(), torch.from_numpy(want_lse).float()


def test_passes_on_the_oracle_output(case):
    inp, out, lse = case
    total = check_prefill_everywhere(inp, out32=out, out16=out.to(torch.bfloat16), lse=lse, processes=2)
    assert total["out32"]["n"] == inp.total_tokens * inp.num_q_heads * 64
    assert total["out32"]["max"] < 1e-6 and total["out16"]["excess"] <= 0.0


def test_fails_on_one_bad_element(case):
    inp, out, lse = case
    bad = out.clone()
    bad[250, 5, 17] += 0.02
    with pytest.raises(AssertionError, match="per-element"):
        check_prefill_everywhere(inp, out32=bad, processes=2)


def test_fails_on_a_mean_error_over_the_bound(case):
    inp, out, lse = case
    with pytest.raises(AssertionError, match="mean"):
        check_prefill_everywhere(inp, out32=out + 0.005, processes=2)


def test_fails_on_a_non_finite_value(case):
    inp, out, lse = case
    bad = out.clone()
    bad[3, 0, 0] = float("nan")
    with pytest.raises(AssertionError, match="non-finite"):
        check_prefill_everywhere(inp, out32=bad, processes=2)


@pytest.fixture(scope="module")
def paged_case():
    # two sequences: 300 new tokens after 200 cached, and 40 new tokens with 10 before the cache start
    inp = workloads.make_paged_prefill([500, 30], [300, 40], num_q_heads=8, num_kv_heads=2, seed=6, sink_mode="mixed")
    want, want_lse = oracle.paged_attention(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t,
                                            inp.cu_seqlens_q, inp.sinks, inp.scale)
    return inp, torch.from_numpy(want).float(), torch.from_numpy(want_lse).float()


def test_paged_passes_on_the_oracle_output(paged_case):
    inp, out, lse = paged_case
    # blocks of 64 rows: the positions of each block's queries are kept
    total = check_paged_prefill_everywhere(inp, out16=out.to(torch.bfloat16), lse=lse, rows_per_task=64,
                                           processes=2)
    assert total["out16"]["excess"] <= 0.0 and total["lse"]["max"] < 1e-6
    assert total["out16"]["n"] == 340 * inp.num_q_heads * 64  # every row, those before the cache start too


def test_paged_fails_on_one_bad_element(paged_case):
    inp, out, lse = paged_case
    bad = out.clone()
    bad[123, 6, 40] += 0.05
    with pytest.raises(AssertionError, match="per-element"):
        check_paged_prefill_everywhere(inp, out16=bad.to(torch.bfloat16), rows_per_task=64, processes=2)
