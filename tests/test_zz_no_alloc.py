"""The allocation-free decode entry point.

sink_attn_decode_noalloc serves callers that are not allowed to allocate
device memory when they run decode (a fixed memory budget planned ahead, or a
host framework that forbids allocation on its decode path): it keeps the
per-chunk partial states in the library's own 16 MiB device array instead of
a workspace.  Its results must match sink_attn_decode's, call after call,
although the array keeps whatever the previous call left in it.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import gqa_attention_head_sink_gb300 as sa
import oracle
from gqa_attention_head_sink_gb300 import build, workloads
from tests.parity import MAX_ABS, MEAN_ABS, assert_parity


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sa.load()


def _close(a, b):
    err = (a.double() - b.double()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (err.max().item(), err.mean().item())


@pytest.mark.gpu
def test_noalloc_matches_decode_on_consecutive_calls(lib):
    # first call: 8 chunks per sequence; second: a different batch with chunks
    # chosen by length, so stale partials of the first call would show.
    first = workloads.make_decode([3000, 16, 1, 2049, 777, 4096], seed=31, sink_mode="mixed", num_splits=8,
                                  device="cuda")
    second = workloads.make_decode([5000, 33, 1200], num_q_heads=16, num_kv_heads=2, seed=32, sink_mode="normal2",
                                   num_splits=0, device="cuda")
    for inp in (first, second):
        need = sa.sink_attn_decode_workspace_bytes(inp.batch, inp.max_seqlen, inp.num_q_heads, inp.num_kv_heads, 64,
                                                   16, inp.num_splits)
        assert 0 < need <= sa.binding.NOALLOC_SCRATCH_BYTES  # the scratch array is really used
        out = torch.empty((inp.batch, inp.num_q_heads, 64), dtype=torch.float32, device="cuda")
        got = sa.sink_attn_decode_noalloc(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                                          inp.scale, num_splits=inp.num_splits, out=out, max_seqlen=inp.max_seqlen)
        ref = sa.sink_attn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                                  inp.scale, num_splits=inp.num_splits, max_seqlen=inp.max_seqlen)
        torch.cuda.synchronize()
        _close(got, ref)
        want, _ = oracle.decode(inp.q.cpu(), inp.k_pages.cpu(), inp.v_pages.cpu(), inp.page_table.cpu(),
                                inp.seqlens_t.cpu(), inp.sinks.cpu(), inp.scale)
        assert_parity(got, want)
    assert sa.sink_attn_get_device_error() == 0


def test_noalloc_rejects_partials_beyond_the_scratch_size(lib):
    # 128 sequences x 32768 tokens, 64/8 heads, 16 chunks: 33 MiB of partial
    # states, more than the 16 MiB array; refused on the host, nothing enqueued.
    assert sa.sink_attn_decode_workspace_bytes(128, 32768, 64, 8, 64, 16, 16) > 16 << 20
    fake = lambda x: ctypes.c_void_p(x)  # noqa: E731  (never dereferenced)
    st = lib.sink_attn_decode_noalloc(fake(256), fake(512), fake(768), fake(1024), 2048, fake(1280), 128, 32768,
                                      1 << 18, fake(1536), 64, 8, 64, 16, 0.125, 16, fake(1792), 1, None, None)
    assert st == 2  # SINK_ATTN_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_single_chunk_and_wide_groups(lib):
    # one chunk per sequence: the chunks write the output directly and no partial
    # state reaches the scratch array; still the same results as sink_attn_decode
    inp = workloads.make_decode([700, 5, 4096], num_q_heads=16, num_kv_heads=1, seed=33, sink_mode="mixed",
                                num_splits=1, device="cuda")
    assert sa.sink_attn_decode_workspace_bytes(inp.batch, inp.max_seqlen, 16, 1, 64, 16, 1) == 0
    got = sa.sink_attn_decode_noalloc(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                                      inp.scale, num_splits=1, max_seqlen=inp.max_seqlen)
    ref = sa.sink_attn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks, inp.scale,
                              num_splits=1, max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    _close(got, ref)
    want, _ = oracle.decode(inp.q.cpu(), inp.k_pages.cpu(), inp.v_pages.cpu(), inp.page_table.cpu(),
                            inp.seqlens_t.cpu(), inp.sinks.cpu(), inp.scale)
    assert_parity(got, want)
    # a group of 32 query heads per kv head is outside what one-token decode supports,
    # with or without the scratch array: refused on the host with the same status
    wide = workloads.make_decode([64, 32], num_q_heads=64, num_kv_heads=2, seed=34, device="cuda")
    for fn in (sa.sink_attn_decode_noalloc, sa.sink_attn_decode):
        with pytest.raises(sa.SinkAttnError) as e:
            fn(wide.q, wide.k_pages, wide.v_pages, wide.page_table, wide.seqlens_t, wide.sinks, wide.scale,
               num_splits=2, max_seqlen=wide.max_seqlen)
        assert e.value.status == 2
    assert sa.sink_attn_get_device_error() == 0
