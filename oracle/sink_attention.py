"""Float64 CPU oracle for grouped-query attention with a per-head sink logit.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
table or helper with the CUDA library.

Source: Perplexity, "GPT-OSS on day 0" (2025-08-08).
  * Model overview, attention bullet: the attention is grouped-query attention
    (several query heads read one key/value head) and every attention head
    owns one trained sink parameter that takes part in the softmax.
  * Section "Sink Attention" (under "Kernels for GPT-OSS"):
      - first formula: the attention weights are a softmax of the scaled
        query-key products together with the head's sink, and the result is
        multiplied by V;
      - second formula: softmax written with the row maximum subtracted;
      - closing paragraph: the online form keeps a running maximum m and a
        running scale d; starting m at the head's sink (with d = 1) folds the
        sink into the normaliser once, and when the key/value length is split
        into chunks only the first chunk may be seeded with it.

Readings taken where the pages leave a step open (each also listed in the
design notes of this repository):
  * The sink is one extra logit per query head in the softmax normaliser; it
    has no value vector, so its column is dropped before multiplying by V.
    (Adding the sink to every logit would cancel inside the softmax and could
    not be what "initialise m to the sink, d to 1" implements.)
  * The sink is not multiplied by the softmax scale; it is already a logit.
  * Query head h reads key/value head h // (Hq / Hkv).
  * Prefill is causal with query length equal to key length: query i of a
    sequence sees keys 0..i of the same sequence.
  * Decode: the single query of sequence b sees all seqlens[b] cached keys.
  * Several new queries per sequence against a paged cache (multi-token
    decode for speculative / multi-token-prediction drafts, and chunked
    prefill): the n queries are the last n tokens of the cache, so query t
    (0-based) sits at position seqlens[b] - n + t and sees keys 0..that
    position.  The causal mask is aligned to the end of the key range.
  * Degenerate rows: with no key and sink = -inf the output is defined as 0;
    sink = +inf is taken as its limit (output 0).

Precision: every quantity is float64; bf16 inputs are upcast exactly.

Parity pins (tests/test_oracle_pins.py): every public function here is pinned
against something other than itself -- brute force at 50 digits, a library
attention routine, closed forms, hand-derived golden values, and invariants
(normalisation, split invariance, GQA = repeated-KV MHA, page permutation
invariance).  No function here is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "sink_softmax_rows",
    "attend_rows",
    "prefill",
    "prefill_rows",
    "decode",
    "gather_paged_kv",
    "online_split_merge",
    "paged_attention",
    "decode_multi",
]

# Rows of the score matrix computed at once, only to bound memory (the result
# does not depend on it: each row is an independent softmax).
_ROW_BLOCK = 512


def _as_f64(x) -> np.ndarray:
    """Upcast a numpy array or a (CPU) torch tensor exactly to float64."""
    if hasattr(x, "detach"):  # torch tensor; bf16 -> f32 -> f64 is exact
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _as_int(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.asarray(x, dtype=np.int64)


def _sink_exp_rows(s: np.ndarray, sink):
    """Exponentials of a block of rows relative to each row's maximum, the
    sink included (the second formula of "Sink Attention").

    s    : [r, n] float64 logits (masked entries are -inf)
    sink : the head's sink logit, one scalar for every row or one per row [r]
    Returns (e [r, n], e_sink [r], z [r], m [r], empty [r], inf_sink [r]):
    e = exp(s - m), e_sink = exp(sink - m), z = sum(e) + e_sink, with m the
    row maximum over the logits and the sink; rows with no finite logit and
    sink = -inf are flagged ``empty``, rows with sink = +inf ``inf_sink``
    (their e, e_sink and z are not used).
    """
    s = np.asarray(s, dtype=np.float64)
    r, n = s.shape
    sink = np.broadcast_to(np.asarray(sink, dtype=np.float64), (r,))
    row_max = s.max(axis=1) if n > 0 else np.full(r, -math.inf)
    m = np.maximum(row_max, sink)  # the subtracted maximum includes the sink
    empty = m == -math.inf
    inf_sink = sink == math.inf
    m_safe = np.where(empty | inf_sink, 0.0, m)
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(s - m_safe[:, None])
        e_sink = np.exp(sink - m_safe)
        z = e.sum(axis=1) + e_sink
    return e, e_sink, z, m, empty, inf_sink


def sink_softmax_rows(s: np.ndarray, sink):
    """Softmax of each row of ``s`` extended by one extra logit ``sink``.

    GPT-OSS on day 0, "Sink Attention": softmax of the scaled products with the
    head's sink, evaluated with the maximum subtracted (second formula).

    s    : [r, n] float64 logits (masked entries are -inf)
    sink : logit of the head (may be +-inf); a scalar, or one per row [r]
    Returns (p [r, n], p_sink [r]) with p.sum(1) + p_sink == 1 for every row
    that has at least one finite logit.  A row with no finite logit and
    sink = -inf has no defined softmax: it returns all zeros (output 0).
    sink = +inf gives p = 0, p_sink = 1 (the limit).
    """
    e, e_sink, z, _, empty, inf_sink = _sink_exp_rows(s, sink)
    z_safe = np.where(empty | inf_sink, 1.0, z)
    p = e / z_safe[:, None]
    p_sink = e_sink / z_safe
    p[empty | inf_sink] = 0.0
    p_sink = np.where(empty, 0.0, np.where(inf_sink, 1.0, p_sink))
    return p, p_sink


def attend_rows(s: np.ndarray, sink, v: np.ndarray):
    """Sink attention for a block of query rows sharing one key/value set.

    s : [r, n] scaled logits (masked = -inf), v : [n, D]; sink a scalar or one
    per row [r].
    Returns (out [r, D], lse [r]) where out = sum_j e^(s_j - m) v_j / z (the
    softmax weights times V; the sink column is dropped: it has no value
    vector) and lse = log(sum_j e^s_j + e^sink), the natural-log normaliser
    including the sink (-inf for an empty row, +inf for sink = +inf).
    """
    e, e_sink, z, m, empty, inf_sink = _sink_exp_rows(s, sink)
    skip = empty | inf_sink
    z_safe = np.where(skip, 1.0, z)
    out = (e @ np.asarray(v, dtype=np.float64)) / z_safe[:, None]
    out[skip] = 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(skip, m, m + np.log(z_safe))
    return out, lse


def prefill(q, k, v, sinks, cu_seqlens, scale: float):
    """Causal variable-length prefill (definition, float64).

    q : [T, Hq, D], k, v : [T, Hkv, D] packed over sequences,
    sinks : [Hq], cu_seqlens : [B+1] (cu[0] = 0, non-decreasing, cu[B] = T).
    For sequence b, local query i and head h (kv head g = h // (Hq/Hkv)):
        s_j = scale * <q[i,h], k[j,g]>   for j = 0..i
        out[i,h] = softmax([s_0..s_i, sinks[h]]) restricted to j, times v[j,g].
    Returns (out [T, Hq, D], lse [T, Hq]).

    Every (token, head) row is an independent softmax; the rows of the query
    heads that share one kv head are evaluated together, token-major, in
    blocks of about _ROW_BLOCK rows (to bound memory only).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    sinks = _as_f64(sinks)
    cu = _as_int(cu_seqlens)
    T, hq, d = q.shape
    hkv = k.shape[1]
    assert hq % hkv == 0, "query heads must be a multiple of kv heads"
    group = hq // hkv
    tokens_per_block = max(1, _ROW_BLOCK // group)
    out = np.zeros((T, hq, d))
    lse = np.full((T, hq), -math.inf)
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        L = t1 - t0
        if L == 0:
            continue
        for g in range(hkv):
            heads = slice(g * group, (g + 1) * group)
            kk = k[t0:t1, g, :]
            vv = v[t0:t1, g, :]
            for r0 in range(0, L, tokens_per_block):
                r1 = min(L, r0 + tokens_per_block)
                # rows (token i, head h), token-major; keys beyond r1-1 are masked for every row
                s = scale * (q[t0 + r0:t0 + r1, heads, :].reshape(-1, d) @ kk[:r1].T)
                tok = np.repeat(np.arange(r0, r1), group)[:, None]
                cols = np.arange(r0, r1)[None, :]  # only these keys lie past some row's own position
                s[:, r0:r1] = np.where(cols <= tok, s[:, r0:r1], -math.inf)
                o, l = attend_rows(s, np.tile(sinks[heads], r1 - r0), vv[:r1])
                out[t0 + r0:t0 + r1, heads, :] = o.reshape(r1 - r0, group, d)
                lse[t0 + r0:t0 + r1, heads] = l.reshape(r1 - r0, group)
    return out, lse


def prefill_rows(q, k, v, sinks, cu_seqlens, scale: float, tokens, heads):
    """The prefill definition evaluated only at selected (token, head) pairs.

    Same arithmetic as ``prefill`` (row i of a sequence sees keys 0..i of that
    sequence), for the cross product of ``tokens`` (packed token indices) and
    ``heads``; only the keys each row needs are upcast.  Inputs may be CPU
    torch tensors or numpy arrays.  Returns (out [len(tokens), len(heads), D],
    lse [len(tokens), len(heads)]).
    """
    cu = _as_int(cu_seqlens)
    sinks = _as_f64(sinks)
    hq = q.shape[1]
    hkv = k.shape[1]
    group = hq // hkv
    tokens = [int(t) for t in tokens]
    heads = [int(h) for h in heads]
    d = q.shape[2]
    out = np.zeros((len(tokens), len(heads), d))
    lse = np.zeros((len(tokens), len(heads)))
    for ti, t in enumerate(tokens):
        b = int(np.searchsorted(cu, t, side="right")) - 1
        t0 = int(cu[b])
        keys = slice(t0, t + 1)  # causal: keys of the same sequence up to t
        for hi, h in enumerate(heads):
            g = h // group
            kk = _as_f64(k[keys, g, :])
            vv = _as_f64(v[keys, g, :])
            s = scale * (_as_f64(q[t, h, :])[None, :] @ kk.T)
            o, l = attend_rows(s, float(sinks[h]), vv)
            out[ti, hi] = o[0]
            lse[ti, hi] = l[0]
    return out, lse


def gather_paged_kv(pages, page_table_row, length: int, page_size: int):
    """Contiguous [length, Hkv, D] view of one sequence's paged cache.

    pages : [num_pages, Hkv, page_size, D]; token j of the sequence lives at
    pages[page_table_row[j // page_size], :, j % page_size, :].  Only the
    pages the sequence owns are read (and upcast).
    """
    row = _as_int(page_table_row)
    n_pages = (length + page_size - 1) // page_size
    hkv, d = pages.shape[1], pages.shape[3]
    out = np.zeros((n_pages * page_size, hkv, d))
    for p in range(n_pages):
        out[p * page_size:(p + 1) * page_size] = _as_f64(pages[int(row[p])]).transpose(1, 0, 2)
    return out[:length]


def decode(q, k_pages, v_pages, page_table, seqlens, sinks, scale: float,
           page_size: int = 16):
    """One query per sequence against a paged KV cache (definition, float64).

    q : [B, Hq, D]; k_pages, v_pages : [num_pages, Hkv, page_size, D];
    page_table : [B, stride]; seqlens : [B].  The query of sequence b attends
    to all seqlens[b] cached keys (no mask).  Returns (out [B,Hq,D], lse [B,Hq]).
    """
    q = _as_f64(q)
    sinks = _as_f64(sinks)
    table = _as_int(page_table)
    lens = _as_int(seqlens)
    B, hq, d = q.shape
    kp, vp = k_pages, v_pages  # gathered (and upcast) per sequence below
    hkv = kp.shape[1]
    group = hq // hkv
    out = np.zeros((B, hq, d))
    lse = np.full((B, hq), -math.inf)
    for b in range(B):
        L = int(lens[b])
        kk = gather_paged_kv(kp, table[b], L, page_size)
        vv = gather_paged_kv(vp, table[b], L, page_size)
        for h in range(hq):
            g = h // group
            s = scale * (q[b, h][None, :] @ kk[:, g, :].T)
            o, l = attend_rows(s, float(sinks[h]), vv[:, g, :])
            out[b, h] = o[0]
            lse[b, h] = l[0]
    return out, lse


def online_split_merge(s_row, sink: float, v, cuts):
    """The pages' online algorithm for one query row, split along key length.

    GPT-OSS on day 0, "Sink Attention", closing paragraph: each chunk keeps a
    running maximum m and scale d (plus the weighted value sum).  The first
    chunk starts from m = sink, d = 1, which counts the sink once; every other
    chunk starts from the plain state m = -inf, d = 1.  Partial states are then
    combined by rescaling to the common maximum (the pages only imply this
    step; it is the standard combination of softmax partial sums).

    s_row : [n] logits, v : [n, D], cuts : sorted chunk boundaries inside
    (0, n).  Pure Python loops: small inputs only.  Returns out [D].
    """
    s_row = [float(x) for x in s_row]
    v = _as_f64(v)
    n, d = v.shape
    bounds = [0] + [int(c) for c in cuts] + [n]
    states = []
    for c in range(len(bounds) - 1):
        m, dd = (sink, 1.0) if c == 0 else (-math.inf, 1.0)
        acc = np.zeros(d)
        for j in range(bounds[c], bounds[c + 1]):
            x = s_row[j]
            if x == -math.inf:
                continue  # e^-inf = 0 adds nothing
            m_new = max(m, x)
            alpha = math.exp(m - m_new) if m != -math.inf else 0.0
            w = math.exp(x - m_new)
            dd = dd * alpha + w
            acc = acc * alpha + w * v[j]
            m = m_new
        if m == -math.inf:
            dd = 0.0  # a chunk that saw nothing holds no mass
        states.append((m, dd, acc))
    big_m = max(st[0] for st in states)
    if big_m == -math.inf:
        return np.zeros(d)
    if big_m == math.inf:
        return np.zeros(d)
    total_d = 0.0
    total = np.zeros(d)
    for m, dd, acc in states:
        if m == -math.inf:
            continue
        w = math.exp(m - big_m)
        total_d += dd * w
        total += acc * w
    return total / total_d


def paged_attention(q, k_pages, v_pages, page_table, seqlens, cu_seqlens_q, sinks, scale: float,
                    page_size: int = 16):
    """Queries that are the last tokens of their sequences, against a paged
    KV cache (definition, float64).

    q : [Tq, Hq, D] packed over sequences by cu_seqlens_q [B+1];
    k_pages, v_pages : [num_pages, Hkv, page_size, D]; page_table : [B, stride];
    seqlens : [B] cached tokens per sequence, the new ones included.
    Sequence b has n_b = cu_q[b+1] - cu_q[b] queries; query t of it sits at
    position seqlens[b] - n_b + t and sees keys 0..that position (causal, the
    mask aligned to the end of the cache; a query whose position is negative
    sees no key).  n_b = 1 is plain decode; n_b = seqlens[b] is causal prefill
    of the whole sequence.  Returns (out [Tq, Hq, D], lse [Tq, Hq]).
    """
    q = _as_f64(q)
    sinks = _as_f64(sinks)
    table = _as_int(page_table)
    lens = _as_int(seqlens)
    cu = _as_int(cu_seqlens_q)
    Tq, hq, d = q.shape
    hkv = k_pages.shape[1]
    group = hq // hkv
    out = np.zeros((Tq, hq, d))
    lse = np.full((Tq, hq), -math.inf)
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        n, L = t1 - t0, int(lens[b])
        if n == 0:
            continue
        kk = gather_paged_kv(k_pages, table[b], L, page_size)
        vv = gather_paged_kv(v_pages, table[b], L, page_size)
        pos = L - n + np.arange(n)  # absolute position of each query
        mask = np.arange(L)[None, :] <= pos[:, None]
        for h in range(hq):
            g = h // group
            for r0 in range(0, n, _ROW_BLOCK):
                r1 = min(n, r0 + _ROW_BLOCK)
                s = scale * (q[t0 + r0:t0 + r1, h, :] @ kk[:, g, :].T)
                s = np.where(mask[r0:r1], s, -math.inf)
                o, l = attend_rows(s, float(sinks[h]), vv[:, g, :])
                out[t0 + r0:t0 + r1, h] = o
                lse[t0 + r0:t0 + r1, h] = l
    return out, lse


def decode_multi(q, k_pages, v_pages, page_table, seqlens, sinks, scale: float, page_size: int = 16):
    """Multi-token decode: the same number of new queries for every sequence.

    q : [B, n, Hq, D], the last n tokens of each sequence's cache (query t at
    position seqlens[b] - n + t, causal among the new tokens).  Returns
    (out [B, n, Hq, D], lse [B, n, Hq]); ``paged_attention`` with n queries
    per sequence.
    """
    B, n, hq, d = q.shape
    cu = np.arange(B + 1, dtype=np.int64) * n
    qp = q.reshape(B * n, hq, d)
    out, lse = paged_attention(qp, k_pages, v_pages, page_table, seqlens, cu, sinks, scale, page_size)
    return out.reshape(B, n, hq, d), lse.reshape(B, n, hq)
