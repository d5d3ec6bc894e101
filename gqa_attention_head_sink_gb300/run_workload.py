"""Run one named synthetic workload through the library a few times.

    python -m gqa_attention_head_sink_gb300.run_workload <workload> [--calls N] [--q-len N]

Meant for profiling one kernel on one workload (e.g. under ncu with -k and
-c), so that the profiled process holds only that workload's tensors on the
device, not the whole benchmark.  Workloads are those of workloads.py:
tiny_prefill, gptoss_prefill, ragged_prefill, decode, long_decode,
mtp_decode (--q-len new tokens per sequence), chunked_prefill, qkv_rope, and
rope_prefill (the 8192 raw projections of qkv_rope through the rotary-mode
prefill, k and v rotated once beforehand).
Outputs are bf16.  Prints the mean device time per call (CUDA events; not a
benchmark figure: no L2 flush, few calls).
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

from . import binding as sa
from . import build, workloads


def _call(name: str, dev, q_len: int):
    if name in ("tiny_prefill", "gptoss_prefill", "ragged_prefill"):
        w = workloads.workload(name, device=dev)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device=dev)
        return lambda: sa.sink_attn_prefill(w.q, w.k, w.v, w.sinks, w.cu_seqlens, w.scale, out=out,
                                            max_seqlen=w.max_seqlen)
    if name in ("decode", "long_decode"):
        w = workloads.workload(name, device=dev)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(256, sa.sink_attn_decode_workspace_bytes(w.batch, w.max_seqlen, w.num_q_heads,
                                                                      w.num_kv_heads, 64, 16, w.num_splits)),
                         dtype=torch.uint8, device=dev)
        return lambda: sa.sink_attn_decode(w.q, w.k_pages, w.v_pages, w.page_table, w.seqlens_t, w.sinks, w.scale,
                                           num_splits=w.num_splits, out=out, max_seqlen=w.max_seqlen, workspace=ws)
    if name == "mtp_decode":
        w = workloads.workload(name, device=dev, q_len=q_len)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device=dev)
        return lambda: sa.sink_attn_decode_multi(w.q, w.k_pages, w.v_pages, w.page_table, w.seqlens_t, w.sinks,
                                                 w.scale, num_splits=w.num_splits, out=out, max_seqlen=w.max_seqlen)
    if name == "chunked_prefill":
        w = workloads.workload(name, device=dev)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device=dev)
        return lambda: sa.sink_attn_prefill_paged(w.q, w.k_pages, w.v_pages, w.page_table, w.cu_seqlens_q,
                                                  w.seqlens_t, w.sinks, w.scale, num_splits=w.num_splits, out=out,
                                                  max_seqlen_q=max(w.q_lens), max_seqlen_k=w.max_seqlen)
    if name == "qkv_rope":
        w = workloads.make_qkv_rope(8192, device=dev)
        f, af = sa.sink_attn_yarn_inv_freq(64, **workloads.YARN_SETTINGS)
        f = f.to(dev)
        return lambda: sa.sink_attn_qkv_rope(w.q, w.k, w.v, w.positions, f, af, w.q_bias, w.k_bias, w.v_bias)
    if name == "rope_prefill":
        w = workloads.make_qkv_rope(8192, device=dev)
        f, af = sa.sink_attn_yarn_inv_freq(64, **workloads.YARN_SETTINGS)
        f = f.to(dev)
        sa.sink_attn_qkv_rope(None, w.k, w.v, w.positions, f, af, None, w.k_bias, w.v_bias)
        sinks = (2.0 * torch.randn(64, generator=torch.Generator(device=dev).manual_seed(1), device=dev)).float()
        cu = torch.tensor([0, 8192], dtype=torch.int32, device=dev)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device=dev)
        return lambda: sa.sink_attn_prefill_rope(w.q, w.k, w.v, sinks, cu, 0.125, f, af, q_bias=w.q_bias, out=out,
                                                 max_seqlen=8192)
    raise SystemExit(f"unknown workload {name!r}")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("workload")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--q-len", type=int, default=4)
    a = ap.parse_args(argv)
    build.build()
    sa.load()
    dev = torch.device("cuda", 0)
    call = _call(a.workload, dev, a.q_len)
    call()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(a.calls):
        call()
    end.record()
    torch.cuda.synchronize()
    status = sa.sink_attn_get_device_error()
    print(f"{a.workload}: {a.calls} calls, {start.elapsed_time(end) / max(1, a.calls):.4f} ms per call, "
          f"device status {status}")
    sys.exit(0 if status == 0 else 1)


if __name__ == "__main__":
    main()
