"""Decode and prefill captured in a CUDA graph and replayed on new inputs.

A serving loop replays one captured decode step per token.  The decode plans
its chunks on the device from the lengths in `seqlens`; the host only passes
an upper bound (max_seqlen) that fixes the grid.  So a graph captured once
(with a caller-owned workspace, outputs preallocated, bound fixed) must give,
after the inputs are overwritten in place, exactly what a direct call on the
new inputs gives -- including new lengths up to the bound.  The first call on
a device does one-time set-up and must happen before capture.
"""
import pytest
import torch

import gqa_attention_head_sink_gb300 as sa
from gqa_attention_head_sink_gb300 import build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    sa.load()


def test_decode_graph_replay_follows_new_lengths_and_data():
    bound = 4096
    d = workloads.make_decode([bound, bound, bound], seed=41, sink_mode="mixed", num_splits=0, device="cuda")
    need = sa.sink_attn_decode_workspace_bytes(d.batch, bound, 64, 8, 64, 16, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty((d.batch, 64, 64), dtype=torch.float32, device="cuda")

    def step():
        sa.sink_attn_decode(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale, num_splits=0,
                            out=out, max_seqlen=bound, workspace=ws)

    step()  # one-time set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    # overwrite the inputs in place: other lengths (within the bound), new query and cache contents
    g = torch.Generator(device="cuda").manual_seed(7)
    d.seqlens_t.copy_(torch.tensor([17, 4096, 2049], dtype=torch.int32, device="cuda"))
    d.q.copy_(torch.randn(d.q.shape, generator=g, device="cuda").to(torch.bfloat16))
    d.k_pages.copy_(torch.randn(d.k_pages.shape, generator=g, device="cuda").to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    want = sa.sink_attn_decode(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale, num_splits=0,
                               max_seqlen=bound, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    assert sa.sink_attn_get_device_error() == 0


def test_prefill_graph_replay_follows_new_data():
    p = workloads.make_prefill([700, 129, 1000], num_q_heads=16, num_kv_heads=2, seed=42, device="cuda")
    out = torch.empty(p.q.shape, dtype=torch.bfloat16, device="cuda")

    def step():
        sa.sink_attn_prefill(p.q, p.k, p.v, p.sinks, p.cu_seqlens, p.scale, out=out, max_seqlen=p.max_seqlen)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    g = torch.Generator(device="cuda").manual_seed(8)
    p.q.copy_(torch.randn(p.q.shape, generator=g, device="cuda").to(torch.bfloat16))
    p.v.copy_(torch.randn(p.v.shape, generator=g, device="cuda").to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    want = sa.sink_attn_prefill(p.q, p.k, p.v, p.sinks, p.cu_seqlens, p.scale, out_dtype=torch.bfloat16,
                                max_seqlen=p.max_seqlen)
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_capture_with_default_bounds_needs_no_device_read():
    # without max_seqlen the bindings use bounds known on the host (page-table width, token
    # count): nothing reads the device, so capture works and replays follow new inputs
    d = workloads.make_decode([700, 1500], seed=43, sink_mode="normal2", num_splits=0, q_len=4, device="cuda")
    bound = d.page_table.shape[1] * 16
    need = sa.sink_attn_decode_multi_workspace_bytes(d.batch, 4, bound, 64, 8, 64, 16, 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty(d.q.shape, dtype=torch.float32, device="cuda")
    c = workloads.make_paged_prefill([900, 300], [300, 300], seed=44, sink_mode="mixed", device="cuda")
    out_c = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")

    def step():
        sa.sink_attn_decode_multi(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale,
                                  out=out, workspace=ws)
        sa.sink_attn_prefill_paged(c.q, c.k_pages, c.v_pages, c.page_table, c.cu_seqlens_q, c.seqlens_t, c.sinks,
                                   c.scale, out=out_c)

    step()  # one-time set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    g = torch.Generator(device="cuda").manual_seed(9)
    d.q.copy_(torch.randn(d.q.shape, generator=g, device="cuda").to(torch.bfloat16))
    c.q.copy_(torch.randn(c.q.shape, generator=g, device="cuda").to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    want = sa.sink_attn_decode_multi(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale,
                                     workspace=ws)
    want_c = sa.sink_attn_prefill_paged(c.q, c.k_pages, c.v_pages, c.page_table, c.cu_seqlens_q, c.seqlens_t,
                                        c.sinks, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, want) and torch.equal(out_c, want_c)


def test_capture_with_default_workspaces():
    # neither a caller workspace from the binding (PyTorch's graph pool serves it) nor one
    # through the C ABI (a null pointer: the library records a graph allocation node)
    import ctypes

    bound = 2048
    d = workloads.make_decode([bound, 700], seed=44, sink_mode="normal2", num_splits=4, device="cuda")
    out_a = torch.empty((d.batch, 64, 64), dtype=torch.float32, device="cuda")
    out_b = torch.empty_like(out_a)
    lib = sa.load()

    def step():
        sa.sink_attn_decode(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale, num_splits=4,
                            out=out_a, max_seqlen=bound)
        st = lib.sink_attn_decode(d.q.data_ptr(), d.k_pages.data_ptr(), d.v_pages.data_ptr(), d.page_table.data_ptr(),
                                  d.page_table.shape[1], d.seqlens_t.data_ptr(), d.batch, bound, d.k_pages.shape[0],
                                  d.sinks.data_ptr(), 64, 8, 64, 16, d.scale, 4, out_b.data_ptr(), 1, None, None, 0,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, st

    step()  # one-time set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    g = torch.Generator(device="cuda").manual_seed(9)
    d.q.copy_(torch.randn(d.q.shape, generator=g, device="cuda").to(torch.bfloat16))
    d.seqlens_t.copy_(torch.tensor([1500, 2048], dtype=torch.int32, device="cuda"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    want = sa.sink_attn_decode(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale, num_splits=4,
                               max_seqlen=bound)
    torch.cuda.synchronize()
    assert torch.equal(out_a, want) and torch.equal(out_b, want)
    assert sa.sink_attn_get_device_error() == 0
