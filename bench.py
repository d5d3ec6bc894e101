"""Benchmark of the sink-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill: causal, one sequence of 8192 tokens, Hq=64, Hkv=8, D=64, bf16
    q/k/v ~ N(0,1), sinks ~ N(0,2), scale 1/8 (the gpt-oss-shaped prefill);
  * decode: 64 sequences x 8192 cached tokens, one query each, paged bf16 KV
    (16-token pages, randomly permuted page table), 8 chunks per sequence,
    merged.
After the timed steps, the two largest workloads are timed per call, each
with its own roofline line: `long_decode` (128 sequences of 16384..32768
cached tokens) and `ragged_prefill` (16 packed sequences of 256..32768
tokens); then the rows built beyond the hot path (`next_rows`).
Inputs are resident in HBM before timing starts.  Between timed steps a
256 MiB buffer is written to flush L2 (the prefill's 80 MiB of inputs would
otherwise stay cached); the flush is outside the timed events.

Reported (rank 0, one JSON line): `value` = prefill TFLOP/s (algorithmic
flops: 4*D per unmasked query-key pair per query head) summed over ranks;
`decode` = HBM GB/s of algorithmic bytes (K/V of every cached token once,
queries, outputs, page-table entries); `roofline` for the prefill kernel
(tensor bound) and decode (HBM bound) against the measured peaks of this
GPU pool; `e2e` = the same through host buffers with the copies timed;
`cpu_baseline` = the float64 oracle timed on a bounded sample on this host.

`--sweep` instead prints one JSON line per shape: the prefill over single
sequences of 1K..128K tokens and packed batches, the decode over batch sizes
and cache lengths (default splits), each timed per call with L2 flushed.

`--impl reference` times the float64 CPU oracle (the only implementation the
method's source provides a definition for) on bounded samples of the same
workload and prints the same line with "impl": "reference".

Several GPUs (torchrun): every rank runs its own replica of the workload
(weak scaling, no collective on the data path); the timed region is
bracketed by a barrier and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gqa_attention_head_sink_gb300 import workloads  # noqa: E402

METRIC = "sink-attn prefill TFLOP/s and decode HBM GB/s, % of GB300 roofline"
PREFILL = "gptoss_prefill"
DECODE = "decode"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return None, 0, 1
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend)
    return dist, dist.get_rank(), ws


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _kernel_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gqa_attention_head_sink_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ["prefill.cu", "prefill.h", "tcgen05.cuh", "common.cuh"]
DECODE_SOURCES = ["decode.cu", "decode.h", "common.cuh"]
DECODE_TC_SOURCES = ["decode_tc.cu", "decode.h", "tcgen05.cuh", "common.cuh"]
ROPE_SOURCES = ["rope.cu", "rope.h", "common.cuh"]


def _traffic(kernel: str, files):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel
    source is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = _kernel_hash(files)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel and parts[1] == want:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def reduce_max(dist, values, device):
    """Element-wise maximum of `values` over all ranks (the slowest rank's
    time is the job's time); identity without a process group."""
    if dist is None:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _events():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def run_ours(args, dist, rank, world):
    import gqa_attention_head_sink_gb300 as sa
    from gqa_attention_head_sink_gb300 import build

    if rank == 0 or dist is None:
        build.build()
    if dist is not None:
        dist.barrier()
    sa.load()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    pre = workloads.workload(PREFILL, device=dev)
    dec = workloads.workload(DECODE, device=dev)
    out_p = torch.empty(pre.q.shape, dtype=torch.bfloat16, device=dev)
    out_d = torch.empty(dec.q.shape, dtype=torch.bfloat16, device=dev)
    ws_bytes = sa.sink_attn_decode_workspace_bytes(dec.batch, dec.max_seqlen, dec.num_q_heads, dec.num_kv_heads,
                                                   64, 16, dec.num_splits)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def prefill():
        sa.sink_attn_prefill(pre.q, pre.k, pre.v, pre.sinks, pre.cu_seqlens, pre.scale, out=out_p,
                             max_seqlen=pre.max_seqlen)

    def decode():
        sa.sink_attn_decode(dec.q, dec.k_pages, dec.v_pages, dec.page_table, dec.seqlens_t, dec.sinks, dec.scale,
                            num_splits=dec.num_splits, out=out_d, max_seqlen=dec.max_seqlen, workspace=ws)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        prefill()
        decode()
    torch.cuda.synchronize()

    ev = [(_events(), _events()) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # first samples land before the timed region
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        (pa, pb), (da, db) = ev[i]
        pa.record(stream)
        prefill()
        pb.record(stream)
        da.record(stream)
        decode()
        db.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    t_pre = [a.elapsed_time(b) for (a, b), _ in ev]
    t_dec = [a.elapsed_time(b) for _, (a, b) in ev]
    ms_pre = sum(t_pre) / len(t_pre)
    ms_dec = sum(t_dec) / len(t_dec)
    total_ms = sum(t_pre) + sum(t_dec)
    total_ms, ms_pre, ms_dec = reduce_max(dist, [total_ms, ms_pre, ms_dec], dev)

    flops = workloads.prefill_flops(pre.seqlens, pre.num_q_heads)
    dbytes = workloads.decode_bytes(dec.seqlens, dec.num_q_heads, dec.num_kv_heads, out_bytes=2)
    pre_tflops = flops / (ms_pre * 1e-3) / 1e12
    dec_gbs = dbytes / (ms_dec * 1e-3) / 1e9

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    if rank == 0:
        e2e = _e2e(sa, pre, dec, dev, stream, args)
    peaks, peak_src = _peaks()
    large = _large_configs(sa, dev, stream, flush, peaks, peak_src) if rank == 0 else None
    next_rows = _next_rows(sa, dev, stream, flush, peaks, peak_src) if rank == 0 else None

    if rank != 0:
        return None
    cpu = _cpu_baseline()
    line = {
        "metric": METRIC,
        "value": round(pre_tflops * world, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": _config(world),
        "prefill": {"value": round(pre_tflops * world, 3), "unit": "TFLOP/s", "ms": round(ms_pre, 4),
                    "flops_per_launch": flops},
        "decode": {"value": round(dec_gbs * world, 2), "unit": "GB/s", "ms": round(ms_dec, 4),
                   "bytes_per_launch": dbytes,
                   "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": round(dec_gbs / peaks["hbm_gbs"], 4),
                                "traffic": _traffic("decode_split_kernel", DECODE_SOURCES),
                                "peak_source": f"{peak_src} (STREAM-style copy)"}},
        "roofline": {"bound": "tensor", "achieved": round(pre_tflops, 3), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(pre_tflops / peaks["bf16_tflops"], 4),
                     "traffic": _traffic("prefill_kernel", PREFILL_SOURCES),
                     "kernel": "prefill_kernel",
                     "peak_source": f"{peak_src} (cuBLAS bf16 burst)"},
        "e2e": e2e,
        "long_decode": large["long_decode"],
        "ragged_prefill": large["ragged_prefill"],
        "next_rows": next_rows,
        "cpu_baseline": cpu,
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
    }
    return line


def _config(world):
    """The workload both arms report (the reference arm times a bounded sample
    of it, described in its cpu_baseline)."""
    return {
        "workload": "prefill: batch 1, causal, seq 8192, Hq 64, Hkv 8, head_dim 64, sinks N(0,2), scale 1/8; "
                    "decode: batch 64 x 8192 cached tokens, paged KV (page 16, permuted), num_splits 8",
        "prefill_out": "bf16", "decode_out": "bf16",
        "l2": "256 MiB buffer written between timed steps (outside the events)",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def _time_calls(fn, stream, flush=None, steps=20, warmup=3, prepare=None):
    """Mean device time (ms) of `fn` over `steps` calls, each bracketed by
    CUDA events on `stream`; `prepare` (if given) runs and `flush` (if given)
    is rewritten before each call, both outside the events."""
    for _ in range(warmup):
        if prepare is not None:
            prepare()
        fn()
    torch.cuda.synchronize()
    ev = [_events() for _ in range(steps)]
    for i, (a, b) in enumerate(ev):
        if prepare is not None:
            prepare()
        if flush is not None:
            flush.fill_(float(i))
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def _large_configs(sa, dev, stream, flush, peaks, peak_src):
    """The two largest workloads, timed per call after the hot-path region:
    the long decode (128 sequences of 16384..32768 cached tokens, chunks
    chosen per length: chunk kernel + merge) against HBM, and the ragged
    16-sequence prefill (215586 packed tokens) against the bf16 tensor peak."""
    res = {}
    ld = workloads.workload("long_decode", device=dev)
    out = torch.empty(ld.q.shape, dtype=torch.bfloat16, device=dev)
    need = sa.sink_attn_decode_workspace_bytes(ld.batch, ld.max_seqlen, ld.num_q_heads, ld.num_kv_heads, 64, 16,
                                               ld.num_splits)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def call_ld():
        sa.sink_attn_decode(ld.q, ld.k_pages, ld.v_pages, ld.page_table, ld.seqlens_t, ld.sinks, ld.scale,
                            num_splits=ld.num_splits, out=out, max_seqlen=ld.max_seqlen, workspace=ws)

    ms = _time_calls(call_ld, stream)  # 6.4 GB of K/V: far larger than L2, no flush needed
    nb = workloads.decode_bytes(ld.seqlens, ld.num_q_heads, ld.num_kv_heads, out_bytes=2)
    gbs = nb / (ms * 1e-3) / 1e9
    res["long_decode"] = {
        "workload": workloads.WORKLOADS["long_decode"], "value": round(gbs, 2), "unit": "GB/s", "ms": round(ms, 4),
        "bytes_per_launch": nb, "kernels": "decode_split_kernel + decode_merge_kernel",
        "chunks": sa.sink_attn_decode_max_splits(ld.batch, ld.max_seqlen, ld.num_kv_heads, 16, ld.num_splits),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "traffic": _traffic("decode_split_kernel/long_decode", DECODE_SOURCES),
                     "peak_source": f"{peak_src} (STREAM-style copy)"}}
    del ld, out, ws
    torch.cuda.empty_cache()
    rp = workloads.workload("ragged_prefill", device=dev)
    out = torch.empty(rp.q.shape, dtype=torch.bfloat16, device=dev)

    def call_rp():
        sa.sink_attn_prefill(rp.q, rp.k, rp.v, rp.sinks, rp.cu_seqlens, rp.scale, out=out, max_seqlen=rp.max_seqlen)

    ms = _time_calls(call_rp, stream, steps=10, flush=flush)
    fl = workloads.prefill_flops(rp.seqlens, rp.num_q_heads)
    tf = fl / (ms * 1e-3) / 1e12
    res["ragged_prefill"] = {
        "workload": workloads.WORKLOADS["ragged_prefill"], "value": round(tf, 3), "unit": "TFLOP/s",
        "ms": round(ms, 4), "flops_per_launch": fl, "kernels": "prefill_kernel",
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tf / peaks["bf16_tflops"], 4),
                     "traffic": _traffic("prefill_kernel/ragged_prefill", PREFILL_SOURCES),
                     "peak_source": f"{peak_src} (cuBLAS bf16 burst)"}}
    del rp, out
    torch.cuda.empty_cache()
    return res


def _next_rows(sa, dev, stream, flush, peaks, peak_src):
    """The rows built beyond the hot path, each on its own synthetic workload:
    multi-token decode (HBM bound), chunked prefill against the paged cache
    (tensor bound) and the QKV bias + YaRN rotary pass (HBM bound).  Timed
    per call (chunk kernel + merge kernel where there is one)."""
    res = {}
    for q_len in (4, 8, 16):
        mtp = workloads.workload("mtp_decode", device=dev, q_len=q_len)
        out = torch.empty(mtp.q.shape, dtype=torch.bfloat16, device=dev)
        need = sa.sink_attn_decode_multi_workspace_bytes(mtp.batch, mtp.q_len, mtp.max_seqlen, mtp.num_q_heads,
                                                         mtp.num_kv_heads, 64, 16, mtp.num_splits)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

        def call_mtp():
            sa.sink_attn_decode_multi(mtp.q, mtp.k_pages, mtp.v_pages, mtp.page_table, mtp.seqlens_t, mtp.sinks,
                                      mtp.scale, num_splits=mtp.num_splits, out=out, max_seqlen=mtp.max_seqlen,
                                      workspace=ws)

        ms = _time_calls(call_mtp, stream)  # 1 GiB of K/V: larger than L2, no flush needed
        nb = workloads.decode_bytes(mtp.seqlens, mtp.num_q_heads, mtp.num_kv_heads, out_bytes=2, q_len=mtp.q_len)
        gbs = nb / (ms * 1e-3) / 1e9
        key = "multi_token_decode" if q_len == 4 else f"multi_token_decode_q{q_len}"
        res[key] = {
            "workload": workloads.WORKLOADS["mtp_decode"].replace("the last 4 of them new (4 queries",
                                                                  f"the last {q_len} of them new ({q_len} queries"),
            "value": round(gbs, 2), "unit": "GB/s", "ms": round(ms, 4), "bytes_per_launch": nb,
            "kernels": ("decode_tc_kernel + decode_merge_kernel" if need > 0
                        else "decode_tc_kernel (one chunk per sequence, written directly: no merge)"),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": _traffic(f"decode_tc_kernel/mtp_decode_q{q_len}", DECODE_TC_SOURCES),
                         "peak_source": f"{peak_src} (STREAM-style copy)"}}
    del mtp, out, ws
    cp = workloads.workload("chunked_prefill", device=dev)
    out = torch.empty(cp.q.shape, dtype=torch.bfloat16, device=dev)

    def call_cp():
        sa.sink_attn_prefill_paged(cp.q, cp.k_pages, cp.v_pages, cp.page_table, cp.cu_seqlens_q, cp.seqlens_t,
                                   cp.sinks, cp.scale, num_splits=cp.num_splits, out=out,
                                   max_seqlen_q=max(cp.q_lens), max_seqlen_k=cp.max_seqlen)

    ms = _time_calls(call_cp, stream, flush=flush)  # 96 MiB of inputs would stay in L2
    fl = workloads.paged_prefill_flops(cp.seqlens, cp.q_lens, cp.num_q_heads)
    tf = fl / (ms * 1e-3) / 1e12
    res["chunked_prefill"] = {
        "workload": workloads.WORKLOADS["chunked_prefill"], "value": round(tf, 3), "unit": "TFLOP/s",
        "ms": round(ms, 4), "flops_per_launch": fl,
        "kernels": "prefill_kernel, paged mode (runs of >= 128 new tokens, keys not split: no merge)",
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tf / peaks["bf16_tflops"], 4),
                     "traffic": _traffic("prefill_kernel/chunked_prefill", PREFILL_SOURCES),
                     "peak_source": f"{peak_src} (cuBLAS bf16 burst)"}}
    del cp, out
    # QKV bias + YaRN rotary pass over the prefill's 8192 tokens (in place: the
    # inputs are restored from a pristine copy before each call, then L2 flushed)
    ro = workloads.make_qkv_rope(8192, device=dev)
    pristine = (ro.q.clone(), ro.k.clone(), ro.v.clone())
    f, af = sa.sink_attn_yarn_inv_freq(64, **workloads.YARN_SETTINGS)
    f = f.to(dev)

    def restore():
        ro.q.copy_(pristine[0])
        ro.k.copy_(pristine[1])
        ro.v.copy_(pristine[2])

    def call_rope():
        sa.sink_attn_qkv_rope(ro.q, ro.k, ro.v, ro.positions, f, af, ro.q_bias, ro.k_bias, ro.v_bias)

    ms = _time_calls(call_rope, stream, flush=flush, prepare=restore)
    nb = workloads.qkv_rope_bytes(8192, 64, 8)
    gbs = nb / (ms * 1e-3) / 1e9
    res["qkv_rope"] = {
        "workload": workloads.WORKLOADS["qkv_rope"], "value": round(gbs, 2), "unit": "GB/s", "ms": round(ms, 4),
        "bytes_per_launch": nb, "kernels": "qkv_rope_kernel",
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": _traffic("qkv_rope_kernel", ROPE_SOURCES),
                     "peak_source": f"{peak_src} (STREAM-style copy)"}}
    # The same 8192 raw projections through attention, two ways: the query's
    # bias and rotation inside the prefill kernel (the pass then handles k and
    # v only), against the full pass followed by the plain prefill.
    sinks = (2.0 * torch.randn(64, generator=torch.Generator(device=dev).manual_seed(1), device=dev)).float()
    cu = torch.tensor([0, 8192], dtype=torch.int32, device=dev)
    out = torch.empty(ro.q.shape, dtype=torch.bfloat16, device=dev)

    def call_fused():
        sa.sink_attn_qkv_rope(None, ro.k, ro.v, ro.positions, f, af, None, ro.k_bias, ro.v_bias)
        sa.sink_attn_prefill_rope(ro.q, ro.k, ro.v, sinks, cu, 0.125, f, af, q_bias=ro.q_bias, out=out,
                                  max_seqlen=8192)

    def call_separate():
        sa.sink_attn_qkv_rope(ro.q, ro.k, ro.v, ro.positions, f, af, ro.q_bias, ro.k_bias, ro.v_bias)
        sa.sink_attn_prefill(ro.q, ro.k, ro.v, sinks, cu, 0.125, out=out, max_seqlen=8192)

    ms_fused = _time_calls(call_fused, stream, flush=flush, prepare=restore)
    ms_sep = _time_calls(call_separate, stream, flush=flush, prepare=restore)
    fl = workloads.prefill_flops([8192], 64)
    tf = fl / (ms_fused * 1e-3) / 1e12
    res["rope_prefill"] = {
        "workload": "the 8192-token rotary workload's raw q/k/v (positions 0..8191, YaRN and biases as qkv_rope) "
                    "through the gpt-oss prefill (one sequence, causal, Hq=64, Hkv=8, D=64, sinks 2*N(0,1), "
                    "scale 1/8)",
        "value": round(tf, 3), "unit": "TFLOP/s", "ms": round(ms_fused, 4), "flops_per_launch": fl,
        "kernels": "qkv_rope_kernel (k and v) + prefill_kernel, rotary mode (query rotated in shared memory)",
        "separate": {"value": round(fl / (ms_sep * 1e-3) / 1e12, 3), "ms": round(ms_sep, 4),
                     "kernels": "qkv_rope_kernel (q, k and v) + prefill_kernel"},
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tf / peaks["bf16_tflops"], 4),
                     "traffic": _traffic("prefill_kernel/rope_prefill", PREFILL_SOURCES),
                     "kernel": "prefill_kernel (rotary mode)", "peak_source": f"{peak_src} (cuBLAS bf16 burst)"}}
    del ro, pristine, out
    torch.cuda.empty_cache()
    return res


def _e2e(sa, pre, dec, dev, stream, args):
    """Prefill and decode through the public API from pinned host buffers:
    every step copies its inputs host->device, runs, and reads its output
    back.  Serial: one stream, each step's copies and call back to back.
    Pipelined (the reported value): a double-buffered serving loop, step i's
    input copy on a copy-in stream overlapping step i-1's call and step i-2's
    read-back on a copy-out stream; events order each buffer's reuse."""
    steps = max(4, min(args.steps, 20))
    h = {n: getattr(pre, n).cpu().pin_memory() for n in ("q", "k", "v", "sinks", "cu_seqlens")}
    hd = {n: getattr(dec, n).cpu().pin_memory() for n in ("q", "k_pages", "v_pages", "page_table", "seqlens_t",
                                                           "sinks")}
    d = [{n: torch.empty_like(t, device=dev) for n, t in h.items()} for _ in range(2)]
    dd = [{n: torch.empty_like(t, device=dev) for n, t in hd.items()} for _ in range(2)]
    out_p = [torch.empty(pre.q.shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    out_d = [torch.empty(dec.q.shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    host_p = [torch.empty(out_p[0].shape, dtype=out_p[0].dtype).pin_memory() for _ in range(2)]
    host_d = [torch.empty(out_d[0].shape, dtype=out_d[0].dtype).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def call_prefill(b):
        sa.sink_attn_prefill(d[b]["q"], d[b]["k"], d[b]["v"], d[b]["sinks"], d[b]["cu_seqlens"], pre.scale,
                             out=out_p[b], max_seqlen=pre.max_seqlen)

    def call_decode(b):
        x = dd[b]
        sa.sink_attn_decode(x["q"], x["k_pages"], x["v_pages"], x["page_table"], x["seqlens_t"], x["sinks"],
                            dec.scale, num_splits=dec.num_splits, out=out_d[b], max_seqlen=dec.max_seqlen)

    def serial(src, dst, call, out, host):
        def step(i):
            for n in src:
                dst[0][n].copy_(src[n], non_blocking=True)
            call(0)
            host[0].copy_(out[0], non_blocking=True)
        return step

    def timed_serial(step):
        with torch.cuda.stream(stream):
            step(0)
            torch.cuda.synchronize()
            a, b = _events()
            a.record(stream)
            for i in range(steps):
                step(i)
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    def timed_pipelined(src, dst, call, out, host):
        in_done = [torch.cuda.Event() for _ in range(2)]
        run_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def run(n_steps, first, last):
            for i in range(n_steps):
                b = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(run_done[b])  # the call of step i-2 has read buffer b
                    if i == 0 and first is not None:
                        first.record(s_in)
                    for n in src:
                        dst[b][n].copy_(src[n], non_blocking=True)
                    in_done[b].record(s_in)
                with torch.cuda.stream(stream):
                    stream.wait_event(in_done[b])
                    if i >= 2:
                        stream.wait_event(out_done[b])  # step i-2's output has been read back
                    call(b)
                    run_done[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(run_done[b])
                    host[b].copy_(out[b], non_blocking=True)
                    out_done[b].record(s_out)
                    if i == n_steps - 1 and last is not None:
                        last.record(s_out)

        run(2, None, None)
        torch.cuda.synchronize()
        a, b = _events()
        run(steps, a, b)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    res = {}
    res["prefill_serial"] = timed_serial(serial(h, d, call_prefill, out_p, host_p))
    res["prefill"] = timed_pipelined(h, d, call_prefill, out_p, host_p)
    res["decode_serial"] = timed_serial(serial(hd, dd, call_decode, out_d, host_d))
    res["decode"] = timed_pipelined(hd, dd, call_decode, out_d, host_d)
    flops = workloads.prefill_flops(pre.seqlens, pre.num_q_heads)
    dbytes = workloads.decode_bytes(dec.seqlens, dec.num_q_heads, dec.num_kv_heads, out_bytes=2)
    h2d_p = sum(t.numel() * t.element_size() for t in h.values())
    h2d_d = sum(t.numel() * t.element_size() for t in hd.values())
    return {"value": round(flops / (res["prefill"] * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d_p, "d2h_bytes_per_step": host_p[0].numel() * 2,
            "ms_per_step": round(res["prefill"], 4),
            "loop": "pipelined: double-buffered, input copy / call / read-back on three streams",
            "serial": {"value": round(flops / (res["prefill_serial"] * 1e-3) / 1e12, 3),
                       "ms_per_step": round(res["prefill_serial"], 4)},
            "decode": {"value": round(dbytes / (res["decode"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "h2d_bytes_per_step": h2d_d, "d2h_bytes_per_step": host_d[0].numel() * 2,
                       "ms_per_step": round(res["decode"], 4),
                       "serial": {"value": round(dbytes / (res["decode_serial"] * 1e-3) / 1e9, 2),
                                  "ms_per_step": round(res["decode_serial"], 4)}},
            "steps": steps}


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


PREFILL_SAMPLE_HEADS = 16  # two kv groups of the 8192-token sequence
REFERENCE_BUDGET_S = 150.0  # the reference arm's whole timed run (warm-up + steps), about


def _oracle_prefill_sample(pre, nh=PREFILL_SAMPLE_HEADS):
    """Time the oracle on the first `nh` query heads (a power of two: their kv
    heads) of the full 8192-token sequence; returns (seconds, flops)."""
    import oracle
    group = pre.num_q_heads // pre.num_kv_heads
    nkv = max(1, nh // group)
    q, k, v = pre.q[:, :nh].cpu(), pre.k[:, :nkv].cpu(), pre.v[:, :nkv].cpu()
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, pre.sinks[:nh].cpu(), pre.cu_seqlens.cpu(), pre.scale)
    return time.perf_counter() - t0, workloads.prefill_flops(pre.seqlens, nh)


def _oracle_decode_sample(dec, seqs=8):
    import oracle
    sel = list(range(seqs))
    t0 = time.perf_counter()
    oracle.decode(dec.q[sel], dec.k_pages, dec.v_pages, dec.page_table[sel], dec.seqlens_t[sel], dec.sinks,
                  dec.scale)
    dt = time.perf_counter() - t0
    return dt, workloads.decode_bytes([dec.seqlens[i] for i in sel], dec.num_q_heads, dec.num_kv_heads,
                                      out_bytes=2)


def _oracle_large_samples():
    """The oracle on samples of the two largest workloads: 4 sequences of the
    long decode (their own lengths), and kv head 0 (8 query heads) of one
    3314-token sequence of the ragged prefill."""
    import oracle
    lens = workloads.workload_seqlens("long_decode")[:4]
    ld = workloads.make_decode(lens, seed=3, sink_mode="normal2", scale=0.125)
    t0 = time.perf_counter()
    oracle.decode(ld.q, ld.k_pages, ld.v_pages, ld.page_table, ld.seqlens_t, ld.sinks, ld.scale)
    dt = time.perf_counter() - t0
    nb = workloads.decode_bytes(lens, 64, 8, out_bytes=2)
    L = 3314
    rp = workloads.make_prefill([L], num_q_heads=8, num_kv_heads=1, seed=4, sink_mode="mixed", scale=0.125)
    t0 = time.perf_counter()
    oracle.prefill(rp.q, rp.k, rp.v, rp.sinks, rp.cu_seqlens, rp.scale)
    pt = time.perf_counter() - t0
    fl = workloads.prefill_flops([L], 8)
    return ({"value": round(nb / dt / 1e9, 4), "unit": "GB/s",
             "sample": f"4 of the 128 sequences ({sum(lens)} tokens, {nb} algorithmic bytes, {dt:.2f} s)"},
            {"value": round(fl / pt / 1e12, 6), "unit": "TFLOP/s",
             "sample": f"one kv head (8 query heads) of a {L}-token sequence ({fl:.3e} flop, {pt:.2f} s)"})


def _cpu_baseline():
    """The float64 oracle, as it stands, on a bounded sample of the workload."""
    pre = workloads.workload(PREFILL, device="cpu")
    dt, flops = _oracle_prefill_sample(pre)
    dec = workloads.make_decode([8192] * 8, seed=2, sink_mode="normal2", scale=0.125, num_splits=8)
    ddt, dbytes = _oracle_decode_sample(dec)
    ld, rp = _oracle_large_samples()
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
            "sample": f"prefill of the 8192-token sequence restricted to {PREFILL_SAMPLE_HEADS} of 64 query heads "
                      f"({flops:.3e} algorithmic flop, {dt:.2f} s)",
            "decode": {"value": round(dbytes / ddt / 1e9, 4), "unit": "GB/s",
                       "sample": f"8 sequences x 8192 tokens of the decode batch ({dbytes} algorithmic bytes, "
                                 f"{ddt:.2f} s)"},
            "long_decode": ld, "ragged_prefill": rp}


def run_reference(args, dist, rank, world):
    """The float64 CPU oracle as the reference arm, timed on the host cores."""
    if rank != 0:
        return None
    pre = workloads.workload(PREFILL, device="cpu")
    dec = workloads.make_decode([8192] * 16, seed=2, sink_mode="normal2", scale=0.125, num_splits=8)
    # Exactly the requested steps and warm-up; each step is a sample of the workload sized
    # so the whole run stays within a few minutes: the first nh query heads of the prefill
    # (a power of two) and the first ns (<= 16) of its 8192-token decode sequences, from one
    # timed head and sequence.
    steps, warm = max(1, args.steps), max(0, args.warmup)
    per_step = min(4.0, REFERENCE_BUDGET_S / (steps + warm))
    t_head, _ = _oracle_prefill_sample(pre, 1)
    t_seq, _ = _oracle_decode_sample(dec, 1)
    nh = 1
    while nh < pre.num_q_heads and 2 * nh * t_head <= 0.85 * per_step:
        nh *= 2
    ns = max(1, min(dec.batch, int(0.15 * per_step / max(t_seq, 1e-9))))
    for _ in range(warm):
        _oracle_prefill_sample(pre, nh)
        _oracle_decode_sample(dec, ns)
    tp, td, flops, dbytes = 0.0, 0.0, 0, 0
    for _ in range(steps):
        dt, flops = _oracle_prefill_sample(pre, nh)
        tp += dt
        ddt, dbytes = _oracle_decode_sample(dec, ns)
        td += ddt
    val = flops * steps / tp / 1e12
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(val, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": round((tp + td) / steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": _config(world),
        "decode": {"value": round(dbytes * steps / td / 1e9, 4), "unit": "GB/s"},
        "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                         "sample": f"{nh}/64 query heads of the 8192-token prefill and {ns} of the 64 decode "
                                   "sequences (8192 tokens each) per step"},
        "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_sweep(args):
    """Prefill TFLOP/s and decode GB/s across shapes (gpt-oss heads: 64 query,
    8 kv, head_dim 64), each shape timed per call (median of `args.steps`
    calls after `args.warmup`), L2 flushed between calls outside the events."""
    import statistics
    import torch
    import gqa_attention_head_sink_gb300 as sa
    from gqa_attention_head_sink_gb300 import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sa.load()
    peaks, _ = _peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    steps, warm = max(5, min(args.steps, 50)), max(3, args.warmup)

    def timed(call):
        for _ in range(warm):
            call()
        ts = []
        for i in range(steps):
            flush.fill_(float(i))
            a, b = _events()
            a.record()
            call()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    prefill_shapes = [[n] for n in (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)]
    prefill_shapes += [[4096] * 8, [1024] * 32, [512] * 64]
    for lens in prefill_shapes:
        inp = workloads.make_prefill(lens, seed=11, device=dev)
        out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: sa.sink_attn_prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale, out=out,
                                                max_seqlen=inp.max_seqlen))
        tf = workloads.prefill_flops(lens, inp.num_q_heads) / (ms * 1e-3) / 1e12
        print(json.dumps({"sweep": "prefill", "seqlens": f"{len(lens)} x {lens[0]}", "ms": round(ms, 4),
                          "TFLOP/s": round(tf, 1), "frac": round(tf / peaks["bf16_tflops"], 4)}), flush=True)
        del inp, out
    for batch, L in [(1, 8192), (8, 8192), (64, 1024), (64, 8192), (256, 8192), (16, 32768), (128, 32768)]:
        dec = workloads.make_decode([L] * batch, seed=12, device=dev)
        out = torch.empty(dec.q.shape, dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: sa.sink_attn_decode(dec.q, dec.k_pages, dec.v_pages, dec.page_table, dec.seqlens_t,
                                               dec.sinks, dec.scale, out=out, max_seqlen=dec.max_seqlen))
        gbs = workloads.decode_bytes(dec.seqlens, dec.num_q_heads, dec.num_kv_heads, out_bytes=2) / (ms * 1e-3) / 1e9
        print(json.dumps({"sweep": "decode", "batch": batch, "cached": L, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                          "frac": round(gbs / peaks["hbm_gbs"], 4)}), flush=True)
        del dec, out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true", help="one line per prefill / decode shape instead")
    args = ap.parse_args(argv)
    if args.sweep:
        run_sweep(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        # rank 0 alone times the CPU oracle; other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, None, rank, int(os.environ.get("WORLD_SIZE", "1")))
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    dist, rank, world = _dist()
    line = run_ours(args, dist, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
