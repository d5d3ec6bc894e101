"""Host-side checks of the C-ABI library that need no GPU.

The library must build, load on a machine without a GPU, export every entry
point include/sink_attn.h declares, and reject bad arguments on the host
before touching the device.
"""
import ctypes
import os
import re

import pytest

import gqa_attention_head_sink_gb300 as sa
from gqa_attention_head_sink_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sink_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sink_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["sink_attn_prefill", "sink_attn_decode", "sink_attn_decode_workspace_bytes",
                 "sink_attn_status_string", "sink_attn_get_device_error"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sink_attn.h but not exported"
        assert name in binding.EXPORTS, f"{name} has no Python binding"


def test_library_has_no_gpu_runtime_dependency():
    # static CUDA runtime, driver reached at run time: loads on CPU-only hosts
    out = os.popen(f"readelf -d {build.LIB}").read()
    needed = re.findall(r"Shared library: \[(.*?)\]", out)
    assert not any(n.startswith("libcudart") or n.startswith("libcuda.") for n in needed), needed


def test_status_strings(lib):
    assert sa.sink_attn_status_string(0) == "ok"
    assert sa.sink_attn_status_string(4) == "device-side wait timed out"
    assert sa.sink_attn_status_string(99) == "unknown status"
    assert sa.sink_attn_version() >= 100


def _decode_call(lib, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, table=8 * 64, stride=4, seqlens=8 * 80, batch=2, max_seqlen=64,
                num_pages=8, sinks=8 * 96, hq=8, hkv=2, d=64, page=16, scale=0.125, splits=0, out=8 * 112,
                out_dtype=1, lse=None, ws=None, ws_bytes=0)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731  (fake, never dereferenced)
    return lib.sink_attn_decode(P(args["q"]), P(args["k"]), P(args["v"]), P(args["table"]), args["stride"],
                                P(args["seqlens"]), args["batch"], args["max_seqlen"], args["num_pages"],
                                P(args["sinks"]), args["hq"], args["hkv"], args["d"], args["page"],
                                args["scale"], args["splits"], P(args["out"]), args["out_dtype"], P(args["lse"]),
                                P(args["ws"]), args["ws_bytes"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=128), 2),                 # head_dim 64 only
    (dict(page=32), 2),               # page size 16 only
    (dict(hq=7), 1),                  # Hq % Hkv != 0
    (dict(hq=64, hkv=2), 2),          # group of 32 query heads: more than one MMA row block
    (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(splits=-1), 1),
    (dict(splits=257), 1),
    (dict(out_dtype=7), 1),
    (dict(q=None), 1),
    (dict(q=8 * 16 + 4), 1),          # misaligned
    (dict(stride=3), 1),              # page table too narrow for max_seqlen
    (dict(num_pages=0), 1),
    (dict(batch=-1), 1),
    (dict(ws=8 * 128 + 64, ws_bytes=1 << 20), 1),  # workspace not 256-byte aligned
    (dict(ws=256 * 4096, ws_bytes=16, splits=2), 1),  # workspace too small
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode_call(lib, **kw) == status


def test_decode_empty_batch_is_noop(lib):
    assert _decode_call(lib, batch=0, q=None, out=None) == 0


def _prefill_call(lib, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, sinks=8 * 64, cu=8 * 80, batch=2, total=300, max_seqlen=200,
                hq=8, hkv=2, d=64, scale=0.125, out=8 * 96, out_dtype=1, lse=None)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.sink_attn_prefill(P(args["q"]), P(args["k"]), P(args["v"]), P(args["sinks"]), P(args["cu"]),
                                 args["batch"], args["total"], args["max_seqlen"], args["hq"], args["hkv"],
                                 args["d"], args["scale"], P(args["out"]), args["out_dtype"], P(args["lse"]), None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), 2),
    (dict(hq=6, hkv=4), 1),
    (dict(scale=-1.0), 1),
    (dict(max_seqlen=301), 1),        # longer than the packed batch
    (dict(batch=5000), 2),            # schedule table holds 1024 sequences
    (dict(cu=None), 1),
    (dict(out=8 * 96 + 2), 1),
    (dict(out_dtype=3), 1),
])
def test_prefill_rejects_bad_arguments_on_host(lib, kw, status):
    assert _prefill_call(lib, **kw) == status


def test_prefill_empty_is_noop(lib):
    assert _prefill_call(lib, batch=0) == 0
    assert _prefill_call(lib, total=0, max_seqlen=0) == 0


def _prefill_rope_call(lib, inv_freq=8 * 200, q_bias=None, attn_factor=1.0, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, sinks=8 * 64, cu=8 * 80, batch=2, total=300, max_seqlen=200,
                hq=8, hkv=2, d=64, scale=0.125, out=8 * 96, out_dtype=1, lse=None)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731  (fake, never dereferenced)
    return lib.sink_attn_prefill_rope(P(args["q"]), P(args["k"]), P(args["v"]), P(args["sinks"]), P(args["cu"]),
                                      args["batch"], args["total"], args["max_seqlen"], args["hq"], args["hkv"],
                                      args["d"], args["scale"], P(q_bias), P(inv_freq), attn_factor, P(args["out"]),
                                      args["out_dtype"], P(args["lse"]), None)


def _decode_rope_call(lib, inv_freq=8 * 200, q_bias=None, attn_factor=1.0, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, table=8 * 64, stride=4, seqlens=8 * 80, batch=2, max_seqlen=64,
                num_pages=8, sinks=8 * 96, hq=8, hkv=2, d=64, page=16, scale=0.125, splits=0, out=8 * 112,
                out_dtype=1, lse=None)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.sink_attn_decode_rope(P(args["q"]), P(args["k"]), P(args["v"]), P(args["table"]), args["stride"],
                                     P(args["seqlens"]), args["batch"], args["max_seqlen"], args["num_pages"],
                                     P(args["sinks"]), args["hq"], args["hkv"], args["d"], args["page"],
                                     args["scale"], args["splits"], P(q_bias), P(inv_freq), attn_factor,
                                     P(args["out"]), args["out_dtype"], P(args["lse"]), None, 0, None)


@pytest.mark.parametrize("call", [_prefill_rope_call, _decode_rope_call])
@pytest.mark.parametrize("kw", [
    dict(inv_freq=None),                  # the frequency table is required
    dict(inv_freq=8 * 200 + 8),           # misaligned table
    dict(q_bias=8 * 300 + 2),             # misaligned bias
    dict(attn_factor=float("inf")),
    dict(attn_factor=float("nan")),
    dict(scale=-1.0),
])
def test_fused_rotary_calls_reject_bad_arguments_on_host(lib, call, kw):
    assert call(lib, **kw) == 1  # SINK_ATTN_ERR_INVALID_ARG, nothing enqueued


def test_fused_rotary_calls_empty_is_noop(lib):
    assert _prefill_rope_call(lib, batch=0) == 0
    assert _decode_rope_call(lib, batch=0) == 0


def test_decode_planning(lib):
    # fixed splits: at most one chunk per page
    assert sa.sink_attn_decode_max_splits(64, 8192, 8, 16, 8) == 8
    assert sa.sink_attn_decode_max_splits(4, 20, 8, 16, 8) == 2
    # chosen per length: enough chunks to fill the GPU, 16..128 pages each
    assert sa.sink_attn_decode_max_splits(128, 32768, 8, 16, 0) == 16
    assert sa.sink_attn_decode_max_splits(1, 8192, 8, 16, 0) == 32
    assert sa.sink_attn_decode_max_splits(1, 16, 8, 16, 0) == 1
    # a single chunk writes the output directly: no workspace
    assert sa.sink_attn_decode_workspace_bytes(4, 16, 64, 8, 64, 16, 0) == 0
    n = sa.sink_attn_decode_workspace_bytes(64, 8192, 64, 8, 64, 16, 8)
    slots = 64 * 64 * 8
    assert n == slots * 64 * 4 + slots * 2 * 4
    with pytest.raises(sa.SinkAttnError):
        sa.sink_attn_decode_workspace_bytes(1, 16, 64, 8, 128, 16, 0)


def _decode_multi_call(lib, q_len, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, table=8 * 64, stride=4, seqlens=8 * 80, batch=2, max_seqlen=64,
                num_pages=8, sinks=8 * 96, hq=64, hkv=8, d=64, page=16, scale=0.125, splits=0, out=8 * 112,
                out_dtype=1)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731  (fake, never dereferenced)
    return lib.sink_attn_decode_multi(P(args["q"]), P(args["k"]), P(args["v"]), P(args["table"]), args["stride"],
                                      P(args["seqlens"]), args["batch"], q_len, args["max_seqlen"],
                                      args["num_pages"], P(args["sinks"]), args["hq"], args["hkv"], args["d"],
                                      args["page"], args["scale"], args["splits"], P(args["out"]),
                                      args["out_dtype"], None, None, 0, None)


@pytest.mark.parametrize("q_len,kw,status", [
    (0, {}, 1),                       # at least one new token
    (-3, {}, 1),
    (4097, {}, 2),                    # at most 4096 new tokens per call
    (2048, dict(batch=600), 2),       # 600 sequences x 128 row tiles: beyond the grid
    (4, dict(hq=64, hkv=2), 2),       # group of 32: beyond one row block per head group
    (2, dict(d=128), 2),
    (2, dict(q=8 * 16 + 8), 1),       # misaligned
])
def test_decode_multi_rejects_bad_arguments_on_host(lib, q_len, kw, status):
    assert _decode_multi_call(lib, q_len, **kw) == status


def test_decode_multi_empty_batch_is_noop(lib):
    assert _decode_multi_call(lib, 8, batch=0, q=None, out=None) == 0


def test_decode_multi_workspace(lib):
    # q_len rows per (sequence, head): q_len times the single-token workspace
    one = sa.sink_attn_decode_workspace_bytes(64, 8192, 64, 8, 64, 16, 8)
    assert sa.sink_attn_decode_multi_workspace_bytes(64, 1, 8192, 64, 8, 64, 16, 8) == one
    slots = 64 * 4 * 64 * 8
    assert sa.sink_attn_decode_multi_workspace_bytes(64, 4, 8192, 64, 8, 64, 16, 8) == slots * 64 * 4 + slots * 8
    with pytest.raises(sa.SinkAttnError):
        sa.sink_attn_decode_multi_workspace_bytes(64, 0, 8192, 64, 8, 64, 16, 8)


def _prefill_paged_call(lib, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, table=8 * 64, stride=8, cu=8 * 72, seqlens=8 * 80, batch=2,
                total_q=100, max_q=60, max_k=120, num_pages=16, sinks=8 * 96, hq=64, hkv=8, d=64, page=16,
                scale=0.125, splits=0, out=8 * 112, out_dtype=1)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731  (fake, never dereferenced)
    return lib.sink_attn_prefill_paged(P(args["q"]), P(args["k"]), P(args["v"]), P(args["table"]), args["stride"],
                                       P(args["cu"]), P(args["seqlens"]), args["batch"], args["total_q"],
                                       args["max_q"], args["max_k"], args["num_pages"], P(args["sinks"]), args["hq"],
                                       args["hkv"], args["d"], args["page"], args["scale"], args["splits"],
                                       P(args["out"]), args["out_dtype"], None, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(max_q=101), 1),             # more new tokens in one sequence than in the batch
    (dict(total_q=-1), 1),
    (dict(cu=None), 1),
    (dict(cu=8 * 72 + 4), 1),         # misaligned offsets
    (dict(stride=7), 1),              # page table too narrow for max_seqlen_k
    (dict(hq=64, hkv=2), 2),          # group of 32
    (dict(d=128), 2),
    (dict(batch=40000, total_q=4000000, max_q=2048), 2),  # 40000 x 128 row tiles: beyond the grid
])
def test_prefill_paged_rejects_bad_arguments_on_host(lib, kw, status):
    assert _prefill_paged_call(lib, **kw) == status


def test_prefill_paged_empty_is_noop(lib):
    assert _prefill_paged_call(lib, batch=0) == 0
    assert _prefill_paged_call(lib, total_q=0, max_q=0, q=None, out=None) == 0


def test_prefill_paged_workspace(lib):
    # new tokens filling the GPU: the key length is not split, no workspace
    assert sa.sink_attn_prefill_paged_workspace_bytes(1, 8192, 8192, 16384, 64, 8) == 0
    # a few new tokens over long caches: split, partial state per (row, head, chunk)
    n = sa.sink_attn_prefill_paged_workspace_bytes(4, 64, 16, 8192, 64, 8, 64, 16, 4)
    slots = 64 * 64 * 4
    assert n == slots * 64 * 4 + slots * 8


def test_yarn_inv_freq_matches_the_oracle(lib):
    import numpy as np
    import torch

    import oracle
    for args in [(64, 150000.0, 32.0, 4096, 32.0, 1.0), (64, 10000.0, 1.0, 4096, 32.0, 1.0),
                 (128, 500000.0, 8.0, 8192, 16.0, 2.0)]:
        f, af = sa.sink_attn_yarn_inv_freq(*args)
        want, want_af = oracle.yarn_inv_freq(*args)
        assert f.dtype == torch.float64
        np.testing.assert_allclose(f.numpy(), want, rtol=2.0 ** -50, atol=0)
        assert abs(af - want_af) <= 2.0 ** -23 * want_af


@pytest.mark.parametrize("args", [(63, 1e4, 2.0, 4096, 32.0, 1.0), (64, 1.0, 2.0, 4096, 32.0, 1.0),
                                  (64, 1e4, 0.0, 4096, 32.0, 1.0), (64, 1e4, 2.0, 0, 32.0, 1.0),
                                  (64, 1e4, 2.0, 4096, 1.0, 32.0)])
def test_yarn_inv_freq_rejects_bad_arguments(lib, args):
    with pytest.raises(sa.SinkAttnError):
        sa.sink_attn_yarn_inv_freq(*args)


def _rope_call(lib, **kw):
    args = dict(q=8 * 16, k=8 * 32, v=8 * 48, qb=None, kb=None, vb=None, pos=8 * 64, freq=8 * 80, af=1.0, T=10,
                hq=8, hkv=2, d=64, slots=None, kp=None, vp=None, npages=0, page=16)
    args.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731  (fake, never dereferenced)
    return lib.sink_attn_qkv_rope(P(args["q"]), P(args["k"]), P(args["v"]), P(args["qb"]), P(args["kb"]),
                                  P(args["vb"]), P(args["pos"]), P(args["freq"]), args["af"], args["T"], args["hq"],
                                  args["hkv"], args["d"], P(args["slots"]), P(args["kp"]), P(args["vp"]),
                                  args["npages"], args["page"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=128), 2),
    (dict(hq=6, hkv=4), 1),
    (dict(pos=None), 1),
    (dict(freq=8 * 80 + 4), 1),        # misaligned
    (dict(qb=8 * 96 + 8), 1),
    (dict(af=float("inf")), 1),
    (dict(slots=8 * 112), 1),          # cache write without pages
    (dict(slots=8 * 112, kp=8 * 128, vp=8 * 144, npages=4, page=32), 2),
    (dict(T=-1), 1),
])
def test_qkv_rope_rejects_bad_arguments_on_host(lib, kw, status):
    assert _rope_call(lib, **kw) == status


def test_qkv_rope_empty_is_noop(lib):
    assert _rope_call(lib, T=0, q=None) == 0


def _declared_arities():
    """Parameter count of every function the header declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(sink_attn_\w+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_binding_signatures_match_the_header():
    # a ctypes signature with a missing or extra argument would silently shift every later one
    arities = _declared_arities()
    assert set(arities) == set(binding.EXPORTS), set(arities) ^ set(binding.EXPORTS)
    for name, (_, args) in binding.EXPORTS.items():
        assert len(args) == arities[name], f"{name}: binding has {len(args)} arguments, header {arities[name]}"


def test_paged_shape_checks_reject_mismatches_before_any_launch():
    # the C ABI takes the pool size from k_pages and the batch from q, so a short v_pool,
    # page table, length vector or sink vector would be read past its end on the device:
    # the binding refuses them first (shapes only; no device is touched)
    import torch
    q = torch.empty(4, 16, 64)
    kp = torch.empty(10, 2, 16, 64)
    table, lens, sinks = torch.empty(4, 3), torch.empty(4), torch.empty(16)
    binding._check_paged(q, kp, kp, table, lens, sinks, 4, 16, 64)  # consistent: passes
    bad = [
        dict(v_pages=torch.empty(9, 2, 16, 64)),
        dict(page_table=torch.empty(3, 3)),
        dict(seqlens=torch.empty(3)),
        dict(sinks=torch.empty(8)),
    ]
    for kw in bad:
        args = dict(q=q, k_pages=kp, v_pages=kp, page_table=table, seqlens=lens, sinks=sinks)
        args.update(kw)
        with pytest.raises(ValueError):
            binding._check_paged(args["q"], args["k_pages"], args["v_pages"], args["page_table"], args["seqlens"],
                                 args["sinks"], 4, 16, 64)


@pytest.mark.parametrize("out_shape,lse_shape", [((4, 16, 63), None), ((3, 16, 64), None), ((4, 16, 64), (4, 15)),
                                                 ((4, 16, 64), (4, 16, 1))])
def test_output_shape_checks_reject_short_buffers(out_shape, lse_shape):
    import torch
    out = torch.empty(*out_shape)
    lse = None if lse_shape is None else torch.empty(*lse_shape)
    with pytest.raises(ValueError, match="shape"):
        binding._check_outputs(out, lse, (4, 16, 64), (4, 16))
