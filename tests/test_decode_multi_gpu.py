"""GPU parity of multi-token decode against the float64 oracle.

q_len new tokens per sequence are the last q_len tokens of its paged cache:
token t sits at position L - q_len + t and sees keys 0..L - q_len + t.  Up
to 16 query rows per kv head (group x q_len) run on the warp-level-MMA split
kernel, more on the tensor-core kernel in tiles of 128 (new token, head)
rows.  The cases cover both kernels, one and several row tiles, groups of 1,
4, 8 and 16, sequences shorter than q_len (tokens before the cache start see
only the sink), sequences that are all new, long runs of new tokens against
a cached prefix, ragged tails with poisoned slots, and every chunking.  All
calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import gqa_attention_head_sink_gb300 as sa
import oracle
from gqa_attention_head_sink_gb300 import build, workloads
from tests.parity import assert_parity, lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    sa.load()
    yield
    assert sa.sink_attn_get_device_error() == 0, "a bounded device wait timed out"


def run(inp, num_splits=None, out_dtype=torch.float32, with_lse=False, workspace=None):
    lse = None
    if with_lse:
        lse = torch.empty((inp.batch, inp.q_len, inp.num_q_heads), dtype=torch.float32, device="cuda")
    out = sa.sink_attn_decode_multi(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                                    inp.scale, num_splits=inp.num_splits if num_splits is None else num_splits,
                                    out_dtype=out_dtype, lse=lse, max_seqlen=inp.max_seqlen, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def oracle_multi(inp, seqs=None):
    seqs = list(range(inp.batch)) if seqs is None else list(seqs)
    big = inp.k_pages.numel() >= (1 << 26)
    return oracle.decode_multi(inp.q[seqs].cpu(), inp.k_pages if big else inp.k_pages.cpu(),
                               inp.v_pages if big else inp.v_pages.cpu(), inp.page_table[seqs].cpu(),
                               inp.seqlens_t[seqs].cpu(), inp.sinks.cpu(), inp.scale, page_size=inp.page_size)


SMALL = [
    # lengths, q_len, Hq, Hkv, sink mode, splits      (rows per kv head = Hq/Hkv * q_len)
    ([1, 2, 15, 16, 17, 100, 333], 2, 64, 8, "normal2", 0),     # 16 rows: warp-level MMAs
    ([1, 2, 15, 16, 17, 100, 333], 2, 64, 8, "normal2", 3),
    ([300, 31], 5, 8, 8, "zero", 2),                            # group 1: 5 rows
    ([0, 1, 3, 5, 2048, 1999], 4, 64, 8, "mixed", 0),           # 32 rows: tensor cores; L < q_len
    ([0, 5, 2048, 1999], 8, 64, 8, "mixed", 7),                 # 64 rows
    ([4000, 17, 1], 3, 16, 1, "mixed", 0),                      # group 16: 48 rows
    ([777, 778, 779, 780], 4, 16, 1, "normal1", 5),             # group 16: 64 rows
    ([5000], 8, 64, 8, "normal2", 256),                         # one page per chunk
    ([129] * 9, 6, 24, 3, "normal2", 0),                        # 48 rows
    ([16, 32, 48], 16, 16, 4, "neginf", 1),                     # q_len 16 x group 4; first sequence all new
    ([1, 100, 4000], 16, 64, 8, "mixed", 0),                    # 128 rows: one full tile
    ([50, 700, 3000], 40, 64, 8, "normal2", 0),                 # three row tiles (16 + 16 + 8 tokens)
    ([300, 1000], 12, 32, 2, "normal2", 3),                     # group 16: two row tiles (8 + 4 tokens)
    ([129, 260], 33, 8, 8, "normal1", 2),                       # group 1: 33 rows
]


@pytest.mark.parametrize("lens,q_len,hq,hkv,sink,splits", SMALL)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_multi_small(lens, q_len, hq, hkv, sink, splits, out_dtype):
    inp = workloads.make_decode(lens, num_q_heads=hq, num_kv_heads=hkv, seed=len(lens) + hq + q_len,
                                sink_mode=sink, num_splits=splits, spare_pages=3, poison=True, q_len=q_len,
                                device="cuda")
    out, lse = run(inp, out_dtype=out_dtype, with_lse=True)
    want, want_lse = oracle_multi(inp)
    assert_parity(out, want, bf16_output=out_dtype == torch.bfloat16)
    lse_close(lse, want_lse)


def test_decode_multi_all_splits_agree():
    inp = workloads.make_decode([3000, 1, 16, 4097, 513], seed=31, sink_mode="mixed", q_len=4, device="cuda")
    want, _ = oracle_multi(inp)
    for splits in [1, 2, 3, 8, 64, 0]:
        out, _ = run(inp, num_splits=splits)
        assert_parity(out, want)


def test_decode_multi_one_token_is_decode():
    # q_len = 1 is plain decode: the same launch, bit for bit
    inp = workloads.make_decode([1, 17, 4000, 333], seed=32, sink_mode="mixed", q_len=1, num_splits=0,
                                device="cuda")
    out_m, _ = run(inp)
    out_d = sa.sink_attn_decode(inp.q[:, 0].contiguous(), inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t,
                                inp.sinks, inp.scale, num_splits=0, max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    assert torch.equal(out_m[:, 0], out_d)


def test_decode_multi_tokens_match_single_token_calls():
    # token t of a multi-token call = a one-token decode over the first L - q_len + t + 1 keys
    q_len = 4
    inp = workloads.make_decode([700, 64, 1025], seed=33, sink_mode="normal2", q_len=q_len, num_splits=0,
                                device="cuda")
    out, _ = run(inp)
    for t in range(q_len):
        lens = (inp.seqlens_t - (q_len - 1 - t)).contiguous()
        one = sa.sink_attn_decode(inp.q[:, t].contiguous(), inp.k_pages, inp.v_pages, inp.page_table, lens,
                                  inp.sinks, inp.scale, num_splits=0, max_seqlen=int(lens.max()))
        torch.cuda.synchronize()
        assert_parity(out[:, t], one.double().cpu().numpy())


def test_decode_multi_with_caller_workspace():
    inp = workloads.make_decode([2049, 4096], seed=34, sink_mode="normal2", q_len=8, num_splits=4, device="cuda")
    need = sa.sink_attn_decode_multi_workspace_bytes(inp.batch, 8, inp.max_seqlen, 64, 8, 64, 16, 4)
    ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")  # garbage: nothing may assume zeros
    out, _ = run(inp, workspace=ws)
    want, _ = oracle_multi(inp)
    assert_parity(out, want)


def test_decode_multi_new_tokens_against_cached_prefix():
    # 1000 new tokens per sequence after prefixes of 500 and 1100 cached ones:
    # 63 row tiles per sequence and kv head, causal skipping of key tiles
    inp = workloads.make_decode([1500, 2100], seed=36, sink_mode="mixed", q_len=1000, num_splits=0,
                                spare_pages=2, poison=True, device="cuda")
    out, lse = run(inp, with_lse=True)
    want, want_lse = oracle_multi(inp)
    assert_parity(out, want)
    lse_close(lse, want_lse)


def test_decode_multi_rejects_too_many_tokens():
    inp = workloads.make_decode([4097], seed=35, q_len=4097, num_q_heads=8, num_kv_heads=8, device="cuda")
    with pytest.raises(sa.SinkAttnError) as e:
        run(inp)
    assert e.value.status == 2


@pytest.mark.parametrize("q_len,splits", [(2, 8), (4, 0), (8, 0), (16, 0), (16, 8)])
def test_decode_multi_full_size(q_len, splits):
    # batch 64 x 8192 cached tokens: with chunks chosen per length (0) exactly the launch the
    # benchmark times, and with 8 chunks merged; every sequence, head and element compared
    if splits == 0:
        inp = workloads.workload("mtp_decode", device="cuda", q_len=q_len)
    else:
        inp = workloads.make_decode([8192] * 64, seed=2, sink_mode="normal2", num_splits=splits, q_len=q_len,
                                    device="cuda")
    out, lse = run(inp, out_dtype=torch.bfloat16, with_lse=True)
    want, want_lse = oracle_multi(inp)
    assert_parity(out, want, bf16_output=True)
    lse_close(lse, want_lse)


@pytest.mark.parametrize("q_len", [2, 8])  # the split kernel, then the tensor-core kernel
def test_decode_multi_large_logits(q_len):
    # softmax scale 1: logits ~8x larger, the running maximum moves often and far
    inp = workloads.make_decode([3000, 129, 7], seed=37, sink_mode="mixed", q_len=q_len, num_splits=0,
                                scale=1.0, device="cuda")
    out, lse = run(inp, with_lse=True)
    want, want_lse = oracle_multi(inp)
    assert_parity(out, want)
    lse_close(lse, want_lse)
