"""GPU parity of causal varlen prefill against the float64 oracle.

All calls go through the C ABI.  Small and medium cases (several 128-row
tiles, ragged tails, empty and one-token sequences, odd GQA groups, every
sink edge case) are compared on every element, and so are the full-size
workloads (one 8192-token sequence with 64/8 heads, and 16 ragged sequences
of 256..32768 tokens), with the mean error taken over the whole workload; a
131072-token sequence is compared on sampled rows.
"""
import numpy as np
import pytest
import torch

import gqa_attention_head_sink_gb300 as sa
import oracle
from gqa_attention_head_sink_gb300 import build, workloads
from tests.full_parity import check_prefill_everywhere
from tests.parity import assert_parity, lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    sa.load()
    yield
    assert sa.sink_attn_get_device_error() == 0, "a bounded device wait timed out"


def run(inp, out_dtype=torch.float32, with_lse=False):
    lse = torch.empty((inp.total_tokens, inp.num_q_heads), dtype=torch.float32, device="cuda") if with_lse else None
    out = sa.sink_attn_prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale, out_dtype=out_dtype,
                               lse=lse, max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    return out, lse


def full_oracle(inp):
    return oracle.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.sinks.cpu(), inp.cu_seqlens.cpu(), inp.scale)


def sampled_rows(seqlens, extra=()):
    """Token indices at sequence starts/ends and 128-row tile boundaries."""
    toks, start = set(extra), 0
    for L in seqlens:
        for r in (0, 1, 126, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1):
            if 0 <= r < L:
                toks.add(start + r)
        start += L
    return sorted(toks)


def test_prefill_tiny_workload():
    inp = workloads.workload("tiny_prefill", device="cuda")
    want, want_lse = full_oracle(inp)
    out, lse = run(inp, with_lse=True)
    assert_parity(out, want)
    lse_close(lse, want_lse)
    out_bf, _ = run(inp, out_dtype=torch.bfloat16)
    assert_parity(out_bf, want, bf16_output=True)


CASES = [
    # lengths, Hq, Hkv, sink mode
    ([1, 127, 128, 129, 300, 0, 517], 8, 2, "mixed"),
    ([256, 255, 257], 16, 2, "normal2"),
    ([200, 65], 6, 2, "normal1"),        # odd group: the second head of a pair is absent
    ([333], 4, 4, "neginf"),              # plain MHA without sinks
    ([1000, 1], 64, 8, "mixed"),
    ([129] * 7, 4, 1, "zero"),
]


@pytest.mark.parametrize("lens,hq,hkv,sink", CASES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_small(lens, hq, hkv, sink, out_dtype):
    inp = workloads.make_prefill(lens, num_q_heads=hq, num_kv_heads=hkv, seed=sum(lens) % 97, sink_mode=sink,
                                 device="cuda")
    want, want_lse = full_oracle(inp)
    out, lse = run(inp, out_dtype=out_dtype, with_lse=True)
    assert_parity(out, want, bf16_output=out_dtype == torch.bfloat16)
    lse_close(lse, want_lse)


def test_prefill_many_short_sequences():
    g = torch.Generator().manual_seed(3)
    lens = [int(x) for x in torch.randint(0, 300, (200,), generator=g)]
    inp = workloads.make_prefill(lens, num_q_heads=16, num_kv_heads=2, seed=21, sink_mode="mixed", device="cuda")
    want, _ = full_oracle(inp)
    out, _ = run(inp)
    assert_parity(out, want)


def test_prefill_is_deterministic():
    inp = workloads.make_prefill([700, 1300], seed=8, device="cuda")
    a, _ = run(inp)
    b, _ = run(inp)
    assert torch.equal(a, b)


def test_prefill_sequences_do_not_leak_into_each_other():
    # changing one sequence's tokens must not change another sequence's output
    inp = workloads.make_prefill([300, 260], num_q_heads=8, num_kv_heads=1, seed=9, device="cuda")
    a, _ = run(inp)
    inp.k[300:] = 100.0
    inp.v[300:] = 1000.0
    b, _ = run(inp)
    assert torch.equal(a[:300], b[:300])


@pytest.mark.parametrize("poison", [float("nan"), float("inf"), -float("inf")])
def test_prefill_packed_neighbours_may_hold_non_finite_values(poison):
    # the first sequence (300 = 2 x 128 + 44 tokens) shares its last key tile with the
    # second one's first 84 tokens; whatever those hold, even NaN or Inf, the first
    # sequence's output must equal the clean run and the oracle
    lens = [300, 260, 129]
    inp = workloads.make_prefill(lens, num_q_heads=16, num_kv_heads=2, seed=15, sink_mode="mixed", device="cuda")
    want, want_lse = full_oracle(inp)
    clean, clean_lse = run(inp, with_lse=True)
    inp.k[300:560] = poison
    inp.v[300:560] = poison
    dirty, dirty_lse = run(inp, with_lse=True)
    for out, lse in ((clean, clean_lse), (dirty, dirty_lse)):
        assert_parity(out[:300], want[:300])
        lse_close(lse[:300], want_lse[:300])
        assert_parity(out[560:], want[560:])  # the third sequence reads none of the poisoned tokens
    assert torch.equal(clean[:300], dirty[:300]) and torch.equal(clean[560:], dirty[560:])


@pytest.mark.slow
def test_prefill_full_len8192_every_element():
    # the 8192-token gpt-oss prefill: every row and head, fp32 and bf16 output and the lse,
    # against the float64 oracle (about 0.55 TFLOP of float64 work, spread over the host cores)
    inp = workloads.workload("gptoss_prefill", device="cuda")
    out32, lse = run(inp, with_lse=True)
    out16, _ = run(inp, out_dtype=torch.bfloat16)
    total = check_prefill_everywhere(inp, out32=out32, out16=out16, lse=lse)
    assert total["out32"]["n"] == inp.total_tokens * inp.num_q_heads * 64


@pytest.mark.slow
def test_prefill_full_ragged16_every_element():
    # 16 ragged sequences (215586 tokens, sinks -inf / 0 / N(0,2) / +20 by head): every row and
    # head, fp32 and bf16 output and the lse (about 34 TFLOP of float64 work over the host cores)
    inp = workloads.workload("ragged_prefill", device="cuda")
    out32, lse = run(inp, with_lse=True)
    out16, _ = run(inp, out_dtype=torch.bfloat16)
    total = check_prefill_everywhere(inp, out32=out32, out16=out16, lse=lse)
    assert total["out32"]["n"] == inp.total_tokens * inp.num_q_heads * 64


@pytest.mark.slow
def test_prefill_131072_tokens_sampled():
    # the longest prompts the pages discuss (128000 tokens and beyond): one 131072-token
    # sequence, rows near tile edges and the end, a few heads of different kv groups
    L = 131072
    inp = workloads.make_prefill([L], seed=12, sink_mode="normal2", device="cuda")
    out, lse = run(inp, with_lse=True)
    assert torch.isfinite(out).all()
    toks = [0, 127, 128, 65535, 100000, L - 1]
    heads = [0, 9, 63]
    cpu = (inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.sinks.cpu(), inp.cu_seqlens.cpu())
    want, want_lse = oracle.prefill_rows(*cpu, inp.scale, toks, heads)
    assert_parity(out[toks][:, heads], want)
    lse_close(lse[toks][:, heads], want_lse)


@pytest.mark.parametrize("how", ["growing_keys", "scale_1"])
def test_prefill_running_max_moves_often(how):
    # the running maximum is raised only when a tile beats it by more than 8 (log2 units), and
    # O is rescaled then: keys whose norm grows along the sequence raise it at nearly every key
    # tile; a softmax scale of 1 (logits ~8x larger) raises it often and by a lot
    lens = [1000, 700]
    inp = workloads.make_prefill(lens, num_q_heads=16, num_kv_heads=2, seed=14, sink_mode="mixed", device="cuda")
    scale = inp.scale
    if how == "growing_keys":
        start = 0
        for L in lens:
            grow = (1.0 + torch.arange(L, device="cuda", dtype=torch.float32) / 60.0)[:, None, None]
            inp.k[start:start + L] = (inp.k[start:start + L].float() * grow).to(torch.bfloat16)
            start += L
    else:
        scale = 1.0
    lse = torch.empty((inp.total_tokens, inp.num_q_heads), dtype=torch.float32, device="cuda")
    out = sa.sink_attn_prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, scale, lse=lse,
                               max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    want, want_lse = oracle.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.sinks.cpu(), inp.cu_seqlens.cpu(),
                                    scale)
    assert_parity(out, want)
    lse_close(lse, want_lse)

@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_prefill_writes_only_its_output_rows(out_dtype):
    """The output may be a view into a larger buffer: whole 128-row bf16 blocks
    leave by bulk tensor store (bounded by the view's T rows), partial blocks and
    fp32 rows by direct stores; rows before and after the view stay as they were."""
    lens = [384, 200, 256]  # whole blocks, a partial last block, whole blocks again
    inp = workloads.make_prefill(lens, num_q_heads=16, num_kv_heads=2, seed=33, sink_mode="mixed", device="cuda")
    T, H = inp.total_tokens, inp.num_q_heads
    big = torch.full((T + 320, H, 64), float("nan"), dtype=out_dtype, device="cuda")
    out = big[64:64 + T]  # starts 64 rows into the allocation
    sa.sink_attn_prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale, out=out, max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    assert torch.isnan(big[:64].float()).all() and torch.isnan(big[64 + T:].float()).all()
    want, _ = full_oracle(inp)
    assert_parity(out, want, bf16_output=out_dtype == torch.bfloat16)

def test_prefill_concurrent_launches_on_several_streams():
    """Launches running at the same time on different streams each take their
    units from their own counter: every output equals the one of a lone launch,
    bit for bit (the work split between CTAs does not change any result)."""
    inp = workloads.make_prefill([640, 384, 1000, 257], num_q_heads=16, num_kv_heads=2, seed=41, sink_mode="mixed",
                                 device="cuda")
    ref, _ = run(inp, out_dtype=torch.bfloat16)
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = [torch.empty_like(ref) for _ in range(len(streams) * 4)]
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        with torch.cuda.stream(streams[i % len(streams)]):
            sa.sink_attn_prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale, out=out,
                                 max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    for out in outs:
        assert torch.equal(out, ref)
