"""Whole-output parity of full-size prefill workloads against the float64 oracle.

The oracle's prefill evaluates each (sequence, kv head) block on its own: the
query heads of one GQA group over one sequence, every (token, head) row an
independent softmax.  The blocks of a workload are spread over a pool of
worker processes, one per host core, started with "spawn" (a process forked
after the first CUDA call can hang).  Each worker evaluates its block with the
oracle and compares it at once with the GPU's outputs for the same rows; only
error statistics come back, which are combined into the workload-wide
maximum and mean.

Inputs and GPU outputs travel as raw bf16 bits (uint16) or fp32, so nothing
is rounded on the way.  This module computes none of the attention itself.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from tests.parity import LSE_ATOL, MAX_ABS, MEAN_ABS, bf16_spacing


def _bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the exact fp32 values."""
    return (u16.astype(np.uint32) << 16).view(np.float32)


def _bf16_bits(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _stats(got: np.ndarray, want: np.ndarray, bf16: bool):
    finite = np.isfinite(want)
    bad = int(np.count_nonzero(finite & ~np.isfinite(got)))
    # where the oracle value is not finite (the lse of an empty row) the GPU must agree exactly
    mismatch = int(np.count_nonzero(~finite & (got != want)))
    err = np.abs(got[finite].astype(np.float64) - want[finite])
    allowed = np.full_like(err, MAX_ABS)
    if bf16:
        allowed = np.maximum(allowed, bf16_spacing(want[finite]))
    excess = float(np.max(err - allowed)) if err.size else -1.0
    return {"max": float(err.max()) if err.size else 0.0, "sum": float(err.sum()), "n": int(err.size),
            "excess": excess, "nonfinite": bad + mismatch}


def _block(task):
    """Oracle prefill of one (sequence, kv head) block and its error statistics."""
    import oracle
    q = _bits_to_f32(task["q"])              # [L, G, D]
    k = _bits_to_f32(task["k"])[:, None, :]  # [L, 1, D]
    v = _bits_to_f32(task["v"])[:, None, :]
    L = q.shape[0]
    want, want_lse = oracle.prefill(q, k, v, task["sinks"], np.array([0, L]), task["scale"])
    res = {"key": task["key"]}
    if task.get("out32") is not None:
        res["out32"] = _stats(task["out32"], want, bf16=False)
    if task.get("out16") is not None:
        res["out16"] = _stats(_bits_to_f32(task["out16"]), want, bf16=True)
    if task.get("lse") is not None:
        res["lse"] = _stats(task["lse"], want_lse, bf16=False)
    return res


def _tasks(inp, out32, out16, lse):
    """One task per (sequence, kv head), longest sequences first."""
    q, k, v = _bf16_bits(inp.q), _bf16_bits(inp.k), _bf16_bits(inp.v)
    sinks = inp.sinks.detach().cpu().numpy().astype(np.float32)
    o32 = None if out32 is None else out32.detach().cpu().numpy()
    o16 = None if out16 is None else _bf16_bits(out16)
    l32 = None if lse is None else lse.detach().cpu().numpy()
    G = inp.num_q_heads // inp.num_kv_heads
    cu = inp.cu_seqlens.detach().cpu().numpy().astype(np.int64)
    order = sorted(range(len(cu) - 1), key=lambda b: -(cu[b + 1] - cu[b]))
    for b in order:
        t0, t1 = int(cu[b]), int(cu[b + 1])
        if t1 == t0:
            continue
        for g in range(inp.num_kv_heads):
            hs = slice(g * G, (g + 1) * G)
            yield {"key": (b, g), "q": q[t0:t1, hs], "k": k[t0:t1, g], "v": v[t0:t1, g], "sinks": sinks[hs],
                   "scale": float(inp.scale),
                   "out32": None if o32 is None else o32[t0:t1, hs],
                   "out16": None if o16 is None else o16[t0:t1, hs],
                   "lse": None if l32 is None else l32[t0:t1, hs]}


def check_prefill_everywhere(inp, out32=None, out16=None, lse=None, processes=None):
    """Compare every element of the GPU outputs (fp32 out, bf16 out, lse; any
    may be None) with the float64 oracle and assert the tolerances: each
    element within 1e-2 (bf16: or one bf16 spacing of the oracle value), the
    mean over the whole workload within 1e-3; lse within LSE_ATOL.  Returns the
    workload-wide statistics."""
    n_proc = processes or len(os.sched_getaffinity(0))
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"  # one BLAS thread per worker: the pool already uses every core
    try:
        with mp.get_context("spawn").Pool(n_proc) as pool:
            results = list(pool.imap_unordered(_block, _tasks(inp, out32, out16, lse)))
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
    total = {}
    for name in ("out32", "out16", "lse"):
        parts = [r[name] for r in results if name in r]
        if not parts:
            continue
        n = sum(p["n"] for p in parts)
        total[name] = {"max": max(p["max"] for p in parts), "mean": sum(p["sum"] for p in parts) / max(1, n),
                       "excess": max(p["excess"] for p in parts), "nonfinite": sum(p["nonfinite"] for p in parts),
                       "n": n, "blocks": len(parts)}
    for name in ("out32", "out16"):
        if name in total:
            t = total[name]
            assert t["nonfinite"] == 0, f"{name}: {t['nonfinite']} non-finite values"
            assert t["excess"] <= 0.0, f"{name}: max abs err {t['max']:.3e} over the per-element bound"
            assert t["mean"] <= MEAN_ABS, f"{name}: mean abs err {t['mean']:.3e} over the workload"
    if "lse" in total:
        t = total["lse"]
        assert t["nonfinite"] == 0, f"lse: {t['nonfinite']} values differ from a non-finite oracle value"
        assert t["max"] <= LSE_ATOL, f"lse max abs err {t['max']:.3e}"
    return total


def _paged_block(task):
    """Oracle of one (sequence, kv head, block of query rows) of a chunked
    prefill against a paged cache, and its error statistics.  The block's keys
    arrive gathered in position order and are laid out as consecutive pages of
    one kv head; its queries keep their positions (the cache is cut after the
    block's last query, so query i of the block sits at L_blk - n_blk + i)."""
    import oracle
    q = _bits_to_f32(task["q"])                      # [n_blk, G, D]
    keys = _bits_to_f32(task["k"])                   # [L_blk, D]
    vals = _bits_to_f32(task["v"])
    L, d = keys.shape
    ps = 16
    pages = (L + ps - 1) // ps
    kp = np.zeros((pages * ps, d), np.float32)
    vp = np.zeros((pages * ps, d), np.float32)
    kp[:L], vp[:L] = keys, vals
    kp = kp.reshape(pages, 1, ps, d)
    vp = vp.reshape(pages, 1, ps, d)
    n = q.shape[0]
    want, want_lse = oracle.paged_attention(q, kp, vp, np.arange(pages)[None, :], np.array([L]),
                                            np.array([0, n]), task["sinks"], task["scale"], page_size=ps)
    res = {"key": task["key"]}
    if task.get("out16") is not None:
        res["out16"] = _stats(_bits_to_f32(task["out16"]), want, bf16=True)
    if task.get("lse") is not None:
        res["lse"] = _stats(task["lse"], want_lse, bf16=False)
    return res


def _paged_tasks(inp, out16, lse, rows_per_task):
    q = _bf16_bits(inp.q)
    sinks = inp.sinks.detach().cpu().numpy().astype(np.float32)
    o16 = None if out16 is None else _bf16_bits(out16)
    l32 = None if lse is None else lse.detach().cpu().numpy()
    G = inp.num_q_heads // inp.num_kv_heads
    cu = inp.cu_seqlens_q.detach().cpu().numpy().astype(np.int64)
    lens = inp.seqlens_t.detach().cpu().numpy().astype(np.int64)
    ps = inp.k_pages.shape[2]
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        n, L = t1 - t0, int(lens[b])
        if n == 0 or L == 0:
            continue
        pages = inp.page_table[b, :(L + ps - 1) // ps].long()
        for g in range(inp.num_kv_heads):
            # keys of kv head g in position order (plain indexing of the pool)
            ks = _bf16_bits(inp.k_pages[pages, g].reshape(-1, inp.k_pages.shape[3])[:L])
            vs = _bf16_bits(inp.v_pages[pages, g].reshape(-1, inp.v_pages.shape[3])[:L])
            hs = slice(g * G, (g + 1) * G)
            for a in range(0, n, rows_per_task):
                e = min(n, a + rows_per_task)
                L_blk = L - n + e  # keys up to the block's last query
                if L_blk <= 0:
                    continue  # these rows see no key: checked by the small cases
                yield {"key": (b, g, a), "q": q[t0 + a:t0 + e, hs], "k": ks[:L_blk], "v": vs[:L_blk],
                       "sinks": sinks[hs], "scale": float(inp.scale),
                       "out16": None if o16 is None else o16[t0 + a:t0 + e, hs],
                       "lse": None if l32 is None else l32[t0 + a:t0 + e, hs]}


def check_paged_prefill_everywhere(inp, out16=None, lse=None, rows_per_task=2048, processes=None):
    """Every element of a chunked prefill's bf16 output (and lse) against the
    float64 oracle, with the same bounds as check_prefill_everywhere."""
    n_proc = processes or len(os.sched_getaffinity(0))
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(n_proc) as pool:
            results = list(pool.imap_unordered(_paged_block, _paged_tasks(inp, out16, lse, rows_per_task)))
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
    total = {}
    for name in ("out16", "lse"):
        parts = [r[name] for r in results if name in r]
        if not parts:
            continue
        n = sum(p["n"] for p in parts)
        total[name] = {"max": max(p["max"] for p in parts), "mean": sum(p["sum"] for p in parts) / max(1, n),
                       "excess": max(p["excess"] for p in parts), "nonfinite": sum(p["nonfinite"] for p in parts),
                       "n": n, "blocks": len(parts)}
    if "out16" in total:
        t = total["out16"]
        assert t["nonfinite"] == 0, f"out16: {t['nonfinite']} non-finite values"
        assert t["excess"] <= 0.0, f"out16: max abs err {t['max']:.3e} over the per-element bound"
        assert t["mean"] <= MEAN_ABS, f"out16: mean abs err {t['mean']:.3e} over the workload"
    if "lse" in total:
        t = total["lse"]
        assert t["nonfinite"] == 0, f"lse: {t['nonfinite']} values differ from a non-finite oracle value"
        assert t["max"] <= LSE_ATOL, f"lse max abs err {t['max']:.3e}"
    return total
