"""GPU parity of split-KV paged decode against the float64 oracle.

All calls go through the C ABI (ctypes binding).  Small cases are compared on
every element; so are the full-size workloads (batch 64 x 8192 tokens with 8
chunks, the launch the benchmark times, and batch 128 x 16K-32K tokens with
chunks chosen per length): every sequence, head and dimension, the mean error
taken over the whole output.
"""
import ctypes

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
    lse = torch.empty((inp.batch, inp.num_q_heads), dtype=torch.float32, device="cuda") if with_lse else None
    out = sa.sink_attn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                              inp.scale, num_splits=inp.num_splits if num_splits is None else num_splits,
                              out_dtype=out_dtype, lse=lse, max_seqlen=inp.max_seqlen, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(inp, seqs=None):
    seqs = list(range(inp.batch)) if seqs is None else list(seqs)
    cpu = lambda t: t.cpu()  # noqa: E731
    return oracle.decode(cpu(inp.q[seqs]), inp.k_pages.cpu() if inp.k_pages.numel() < (1 << 26) else inp.k_pages,
                         inp.v_pages.cpu() if inp.v_pages.numel() < (1 << 26) else inp.v_pages,
                         cpu(inp.page_table[seqs]), cpu(inp.seqlens_t[seqs]), cpu(inp.sinks), inp.scale,
                         page_size=inp.page_size)


SMALL = [
    # lengths, Hq, Hkv, sink mode, splits
    ([1, 15, 16, 17, 100, 333], 64, 8, "normal2", 0),
    ([1, 15, 16, 17, 100, 333], 64, 8, "normal2", 1),
    ([1, 15, 16, 17, 100, 333], 64, 8, "normal2", 3),
    ([0, 5, 2048, 1999], 16, 2, "neginf", 2),
    ([0, 5, 2048, 1999], 16, 2, "mixed", 7),
    ([4000, 17, 1], 4, 1, "mixed", 0),
    ([777, 778, 779, 780], 16, 1, "normal1", 5),
    ([300, 31], 8, 8, "zero", 2),
    ([5000], 64, 8, "normal2", 256),
    ([129] * 9, 24, 3, "normal2", 0),
]


@pytest.mark.parametrize("lens,hq,hkv,sink,splits", SMALL)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_small(lens, hq, hkv, sink, splits, out_dtype):
    inp = workloads.make_decode(lens, num_q_heads=hq, num_kv_heads=hkv, seed=len(lens) + hq, sink_mode=sink,
                                num_splits=splits, spare_pages=3, poison=True, device="cuda")
    out, lse = run(inp, out_dtype=out_dtype, with_lse=True)
    want, want_lse = oracle_decode(inp)
    assert_parity(out, want, bf16_output=out_dtype == torch.bfloat16)
    lse_close(lse, want_lse)


def test_decode_all_splits_agree():
    inp = workloads.make_decode([3000, 1, 16, 4097, 513], seed=11, sink_mode="mixed", device="cuda")
    want, _ = oracle_decode(inp)
    outs = []
    for splits in [1, 2, 3, 8, 16, 64, 0]:
        out, _ = run(inp, num_splits=splits)
        assert_parity(out, want)
        outs.append(out)
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 1e-3


def test_decode_is_deterministic_and_ignores_page_placement():
    inp = workloads.make_decode([1000, 2500, 77], seed=12, num_splits=4, device="cuda")
    a, _ = run(inp)
    b, _ = run(inp)
    assert torch.equal(a, b)
    # move every page to another pool slot and rewrite the table: bitwise equal
    n = inp.k_pages.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n, device="cuda")
    table2 = torch.where(inp.page_table >= 0, inv[inp.page_table.long().clamp(min=0)].int(), inp.page_table)
    inp2 = workloads.DecodeInputs(q=inp.q, k_pages=inp.k_pages[perm].contiguous(),
                                  v_pages=inp.v_pages[perm].contiguous(), page_table=table2.contiguous(),
                                  seqlens_t=inp.seqlens_t, seqlens=inp.seqlens, sinks=inp.sinks, scale=inp.scale,
                                  num_splits=inp.num_splits)
    c, _ = run(inp2)
    assert torch.equal(a, c)


def test_decode_caller_workspace_matches_library_workspace():
    # caller workspace, the binding's default (PyTorch's caching allocator) and the C ABI's own
    # stream-ordered allocation (null workspace) give the same bits
    inp = workloads.make_decode([2000, 3000], seed=13, num_splits=6, device="cuda")
    need = sa.sink_attn_decode_workspace_bytes(inp.batch, inp.max_seqlen, 64, 8, 64, 16, 6)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a, _ = run(inp, workspace=ws)
    b, _ = run(inp)
    c = torch.empty_like(a)
    st = sa.load().sink_attn_decode(inp.q.data_ptr(), inp.k_pages.data_ptr(), inp.v_pages.data_ptr(),
                                    inp.page_table.data_ptr(), inp.page_table.shape[1], inp.seqlens_t.data_ptr(),
                                    inp.batch, inp.max_seqlen, inp.k_pages.shape[0], inp.sinks.data_ptr(), 64, 8,
                                    64, 16, inp.scale, 6, c.data_ptr(), 1, None, None, 0,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_decode_default_workspace_on_another_stream():
    # the binding's default workspace is tied to the stream the call runs on: allocations made on
    # the current stream right after the call must not reuse it while that stream still works
    inp = workloads.make_decode([3000, 5000, 4000], seed=14, num_splits=5, device="cuda")
    want, _ = run(inp)
    need = sa.sink_attn_decode_workspace_bytes(inp.batch, inp.max_seqlen, 64, 8, 64, 16, 5)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out = torch.empty_like(want)
    for _ in range(3):
        sa.sink_attn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks, inp.scale,
                            num_splits=5, out=out, max_seqlen=inp.max_seqlen, stream=side)
        junk = [torch.full((need // 4 + 1,), float("nan"), device="cuda") for _ in range(8)]
        del junk
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_decode_rejects_bad_shapes():
    inp = workloads.make_decode([20], seed=1, device="cuda")
    with pytest.raises(sa.SinkAttnError) as e:
        sa.sink_attn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                            scale=-1.0)
    assert e.value.status == 1


@pytest.mark.slow
def test_decode_full_batch64_len8192_splits8():
    inp = workloads.workload("decode", device="cuda")
    out, lse = run(inp, with_lse=True)
    want, want_lse = oracle_decode(inp)  # all 64 sequences
    assert_parity(out, want)
    lse_close(lse, want_lse)
    out_bf, _ = run(inp, out_dtype=torch.bfloat16)
    assert_parity(out_bf, want, bf16_output=True)


@pytest.mark.slow
def test_decode_full_batch128_long_auto_splits():
    inp = workloads.workload("long_decode", device="cuda")
    out, lse = run(inp, with_lse=True)
    want, want_lse = oracle_decode(inp)  # all 128 sequences
    assert_parity(out, want)
    lse_close(lse, want_lse)


@pytest.mark.slow
def test_decode_131072_tokens():
    # one query against 131072 cached tokens (8192 pages), chunks chosen per length
    inp = workloads.make_decode([131072, 5], seed=13, sink_mode="normal2", num_splits=0, device="cuda")
    out, lse = run(inp, with_lse=True)
    want, want_lse = oracle_decode(inp)
    assert_parity(out, want)
    lse_close(lse, want_lse)
