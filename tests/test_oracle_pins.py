"""Pins of the float64 oracle against things other than itself.

Each pin is chosen so that a plausible mistake in the oracle (a dropped sink
term, the sink scaled by the softmax scale, an off-by-one causal mask, a wrong
GQA head mapping, a transposed operand, a wrong page gather) fails at least
one test:

  * golden fixtures derived by hand from the definition (tests/golden/);
  * brute force in 50-digit arithmetic (mpmath) on tiny inputs;
  * sink = -inf reduces to textbook attention: torch's
    scaled_dot_product_attention in float64 on the CPU (a library routine);
  * closed forms for the sink's effect: out = out_nosink / (1 + e^(sink - lse_nosink))
    and lse = logaddexp(lse_nosink, sink); causal row 0 = v_0 * sigmoid(s_0 - sink);
  * invariants: probabilities plus the sink probability sum to 1; a large
    sink drives the output to 0 monotonically; the pages' online algorithm
    split at any cut points (sink only in the first chunk) gives the direct
    result; GQA equals MHA with each kv head repeated for its group; decode
    equals the last causal prefill row; page permutations do not matter;
  * several new queries per sequence against the paged cache: 50-digit brute
    force reading keys straight from the pages, torch SDPA with an explicit
    mask aligned to the end of the cache, one query = decode, every token new
    = causal prefill, and queries placed before the cache start see only the
    sink.

Source of the definition: Perplexity, "GPT-OSS on day 0", section
"Sink Attention" and the model overview's attention bullet.
"""
import glob
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_head_sink_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f(x):
    return -math.inf if x == "-inf" else (math.inf if x == "inf" else float(x))


# --------------------------------------------------------------------------
# golden fixtures
# --------------------------------------------------------------------------
@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "*.json"))))
def test_golden_fixture(path):
    g = json.load(open(path))
    tol = g["tol"]
    sinks = np.array([_f(x) for x in g["sinks"]])
    if g["kind"] == "prefill":
        out, lse = oracle.prefill(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]), sinks,
                                  np.array(g["cu_seqlens"]), g["scale"])
    else:
        out, lse = oracle.decode(np.array(g["q"]), np.array(g["k_pages"]), np.array(g["v_pages"]),
                                 np.array(g["page_table"]), np.array(g["seqlens"]), sinks,
                                 g["scale"], page_size=g["page_size"])
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=tol)
    if "expected_lse" in g:
        np.testing.assert_allclose(lse, np.array(g["expected_lse"]), rtol=0, atol=tol)


# --------------------------------------------------------------------------
# brute force, 50 digits
# --------------------------------------------------------------------------
def _brute_prefill(q, k, v, sinks, cu, scale):
    import mpmath
    mpmath.mp.dps = 50
    T, hq, d = q.shape
    hkv = k.shape[1]
    out = np.zeros((T, hq, d))
    lse = np.zeros((T, hq))
    for b in range(len(cu) - 1):
        t0, t1 = cu[b], cu[b + 1]
        for i in range(t0, t1):
            for h in range(hq):
                g = h * hkv // hq  # contiguous groups, written independently
                logits = []
                for j in range(t0, i + 1):
                    dot = mpmath.mpf(0)
                    for e in range(d):
                        dot += mpmath.mpf(float(q[i, h, e])) * mpmath.mpf(float(k[j, g, e]))
                    logits.append(mpmath.mpf(scale) * dot)
                terms = [mpmath.e ** x for x in logits]
                z = sum(terms) + (mpmath.e ** mpmath.mpf(float(sinks[h])) if sinks[h] != -math.inf else 0)
                for e in range(d):
                    acc = mpmath.mpf(0)
                    for jj, j in enumerate(range(t0, i + 1)):
                        acc += terms[jj] * mpmath.mpf(float(v[j, g, e]))
                    out[i, h, e] = float(acc / z)
                lse[i, h] = float(mpmath.log(z))
    return out, lse


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefill_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    lens = [1, 3, 0, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 3
    q = rng.normal(size=(T, hq, d))
    k = rng.normal(size=(T, hkv, d))
    v = rng.normal(size=(T, hkv, d))
    sinks = np.array([0.3, -1.7, 2.5, -math.inf])
    scale = 0.7
    out, lse = oracle.prefill(q, k, v, sinks, cu, scale)
    bo, bl = _brute_prefill(q, k, v, sinks, cu, scale)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# reduction to textbook attention (library routine)
# --------------------------------------------------------------------------
def _sdpa_causal(q, k, v, scale):
    """torch SDPA in float64 on the CPU, one sequence, kv repeated per group."""
    T, hq, d = q.shape
    hkv = k.shape[1]
    rep = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(np.repeat(k, rep, axis=1)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(np.repeat(v, rep, axis=1)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_no_sink_is_textbook_attention():
    rng = np.random.default_rng(7)
    T, hq, hkv, d = 300, 8, 2, 16
    q, k, v = rng.normal(size=(T, hq, d)), rng.normal(size=(T, hkv, d)), rng.normal(size=(T, hkv, d))
    out, _ = oracle.prefill(q, k, v, np.full(hq, -math.inf), np.array([0, T]), 0.25)
    np.testing.assert_allclose(out, _sdpa_causal(q, k, v, 0.25), rtol=0, atol=1e-12)


def test_row_block_boundary_textbook():
    # more rows than the oracle's internal row block, to cover its seams
    rng = np.random.default_rng(8)
    T, hq, hkv, d = 1100, 2, 1, 8
    q, k, v = rng.normal(size=(T, hq, d)), rng.normal(size=(T, hkv, d)), rng.normal(size=(T, hkv, d))
    out, _ = oracle.prefill(q, k, v, np.full(hq, -math.inf), np.array([0, T]), 0.3)
    np.testing.assert_allclose(out, _sdpa_causal(q, k, v, 0.3), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# closed forms for the sink term
# --------------------------------------------------------------------------
def test_sink_closed_form():
    rng = np.random.default_rng(11)
    T, hq, hkv, d = 200, 4, 1, 8
    q, k, v = rng.normal(size=(T, hq, d)), rng.normal(size=(T, hkv, d)), rng.normal(size=(T, hkv, d))
    sinks = np.array([-3.0, 0.0, 1.5, 6.0])
    cu = np.array([0, 77, T])
    out, lse = oracle.prefill(q, k, v, sinks, cu, 0.5)
    out0, lse0 = oracle.prefill(q, k, v, np.full(hq, -math.inf), cu, 0.5)
    frac = 1.0 / (1.0 + np.exp(sinks[None, :] - lse0))  # share of mass left to the keys
    np.testing.assert_allclose(out, out0 * frac[:, :, None], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.logaddexp(lse0, sinks[None, :]), rtol=0, atol=1e-12)


def test_causal_row_zero_is_sigmoid():
    rng = np.random.default_rng(12)
    T, hq, d = 5, 3, 4
    q, k, v = rng.normal(size=(T, hq, d)), rng.normal(size=(T, 1, d)), rng.normal(size=(T, 1, d))
    sinks = np.array([0.4, -2.0, 3.0])
    out, _ = oracle.prefill(q, k, v, sinks, np.array([0, T]), 0.9)
    for h in range(hq):
        s0 = 0.9 * float(q[0, h] @ k[0, 0])
        sig = 1.0 / (1.0 + math.exp(sinks[h] - s0))
        np.testing.assert_allclose(out[0, h], v[0, 0] * sig, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_probabilities_sum_to_one():
    rng = np.random.default_rng(13)
    s = rng.normal(size=(50, 37)) * 4
    s[3, :] = -math.inf
    s[4, 10:] = -math.inf
    for sink in [-math.inf, -5.0, 0.0, 2.0, 40.0]:
        p, ps = oracle.sink_softmax_rows(s, sink)
        tot = p.sum(axis=1) + ps
        ok = np.ones(50, dtype=bool)
        if sink == -math.inf:
            ok[3] = False  # no key and no sink: defined as all-zero
            assert np.all(p[3] == 0) and ps[3] == 0
        np.testing.assert_allclose(tot[ok], 1.0, rtol=0, atol=1e-15)
        assert np.all(p >= 0) and np.all(ps >= 0)
    # sink = +inf takes all the mass
    p, ps = oracle.sink_softmax_rows(s, math.inf)
    assert np.all(p == 0) and np.all(ps == 1)


def test_large_sink_drives_output_to_zero():
    rng = np.random.default_rng(14)
    L, d = 2048, 16
    q, k, v = rng.normal(size=(L, 1, d)), rng.normal(size=(L, 1, d)), rng.normal(size=(L, 1, d))
    norms = []
    for sink in [-1.0, 2.0, 5.0, 10.0, 20.0, 40.0]:
        out, _ = oracle.prefill(q, k, v, np.array([sink]), np.array([0, L]), 0.25)
        norms.append(np.abs(out).max(axis=(1, 2)))
    norms = np.array(norms)
    assert np.all(np.diff(norms, axis=0) <= 1e-15)  # every row shrinks as the sink grows
    assert norms[-2].max() < 1e-4  # sink = +20
    assert norms[-1].max() < 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_online_split_merge_matches_direct(seed):
    rng = np.random.default_rng(100 + seed)
    n, d = 61, 5
    s = rng.normal(size=n) * 3
    s[rng.integers(0, n, 5)] = -math.inf  # masked keys inside chunks
    v = rng.normal(size=(n, d))
    for sink in [-math.inf, -2.0, 0.7, 9.0]:
        ref, _ = oracle.attend_rows(s[None, :], sink, v)
        cut_sets = [[], [30], [1, 2, 3], list(range(1, n)), sorted(rng.choice(np.arange(1, n), 7, replace=False))]
        for cuts in cut_sets:
            got = oracle.online_split_merge(s, sink, v, cuts)
            np.testing.assert_allclose(got, ref[0], rtol=0, atol=1e-12)


def test_online_split_seeds_sink_only_once():
    # If every chunk were seeded with the sink, the sink would be counted
    # once per chunk; the result must equal the single-count definition.
    s = np.array([0.0, 0.0, 0.0, 0.0])
    v = np.array([[1.0], [1.0], [1.0], [1.0]])
    got = oracle.online_split_merge(s, 0.0, v, [1, 2, 3])
    np.testing.assert_allclose(got, [4.0 / 5.0], rtol=0, atol=1e-15)


def test_gqa_equals_repeated_mha():
    rng = np.random.default_rng(15)
    T, hq, hkv, d = 40, 8, 2, 4
    q, k, v = rng.normal(size=(T, hq, d)), rng.normal(size=(T, hkv, d)), rng.normal(size=(T, hkv, d))
    sinks = rng.normal(size=hq)
    cu = np.array([0, 13, 40])
    out, lse = oracle.prefill(q, k, v, sinks, cu, 0.5)
    out_m, lse_m = oracle.prefill(q, np.repeat(k, hq // hkv, axis=1), np.repeat(v, hq // hkv, axis=1),
                                  sinks, cu, 0.5)
    np.testing.assert_allclose(out, out_m, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_m, rtol=0, atol=1e-14)
    # and the kv heads are really different: head 0 and head hq-1 disagree
    assert np.abs(out[:, 0] - out[:, -1]).max() > 1e-3


def test_packed_sequences_are_independent():
    rng = np.random.default_rng(16)
    lens = [5, 0, 9, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, hq, hkv, d = int(cu[-1]), 2, 1, 3
    q, k, v = rng.normal(size=(T, hq, d)), rng.normal(size=(T, hkv, d)), rng.normal(size=(T, hkv, d))
    sinks = np.array([0.5, -0.5])
    out, _ = oracle.prefill(q, k, v, sinks, cu, 1.0)
    for b in range(len(lens)):
        a, e = cu[b], cu[b + 1]
        o1, _ = oracle.prefill(q[a:e], k[a:e], v[a:e], sinks, np.array([0, e - a]), 1.0)
        np.testing.assert_allclose(out[a:e], o1, rtol=0, atol=1e-15)


def test_decode_equals_last_prefill_row_and_ignores_page_order():
    inp = workloads.make_decode([37, 16, 1, 0, 50], num_q_heads=4, num_kv_heads=2, head_dim=8, seed=5,
                                sink_mode="normal2", page_size=16, spare_pages=3, poison=True)
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                             inp.scale, page_size=16)
    assert np.all(np.isfinite(out))  # poisoned slots were never read
    for b, L in enumerate(inp.seqlens):
        if L == 0:
            sink_only = np.isfinite(inp.sinks.numpy())
            np.testing.assert_allclose(out[b], 0.0)
            np.testing.assert_allclose(lse[b][sink_only], inp.sinks.numpy()[sink_only], atol=1e-7)
            continue
        kk = oracle.gather_paged_kv(inp.k_pages, inp.page_table[b], L, 16)
        vv = oracle.gather_paged_kv(inp.v_pages, inp.page_table[b], L, 16)
        qq = np.zeros((L, 4, 8))
        qq[L - 1] = inp.q[b].float().numpy()
        o2, l2 = oracle.prefill(qq, kk, vv, inp.sinks, np.array([0, L]), inp.scale)
        np.testing.assert_allclose(out[b], o2[L - 1], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], l2[L - 1], rtol=0, atol=1e-13)
    # move every used page to a different pool slot: the result is unchanged
    perm = torch.randperm(inp.k_pages.shape[0], generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    k2, v2 = inp.k_pages[perm], inp.v_pages[perm]  # new slot i holds old page perm[i]
    table2 = torch.where(inp.page_table >= 0, inv[inp.page_table.long().clamp(min=0)].to(torch.int32),
                         inp.page_table)
    out2, _ = oracle.decode(inp.q, k2, v2, table2, inp.seqlens_t, inp.sinks, inp.scale, page_size=16)
    np.testing.assert_array_equal(out, out2)


def test_gather_paged_kv_layout():
    # token j of a sequence is pages[table[j // P], :, j % P, :]
    P, hkv, d = 4, 2, 3
    pages = np.arange(5 * hkv * P * d, dtype=np.float64).reshape(5, hkv, P, d)
    table = np.array([3, 0, 4])
    got = oracle.gather_paged_kv(pages, table, 10, P)
    for j in range(10):
        np.testing.assert_array_equal(got[j], pages[table[j // P], :, j % P, :])


def test_oracle_takes_bf16_values_exactly():
    inp = workloads.workload("tiny_prefill")
    out_t, _ = oracle.prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale)
    out_n, _ = oracle.prefill(inp.q.float().numpy().astype(np.float64), inp.k.float().numpy(),
                              inp.v.float().numpy(), inp.sinks.numpy(), inp.cu_seqlens.numpy(), inp.scale)
    np.testing.assert_array_equal(out_t, out_n)


def test_prefill_rows_agrees_with_full_definition():
    inp = workloads.make_prefill([5, 130, 1, 64], num_q_heads=6, num_kv_heads=2, head_dim=16, seed=3,
                                 sink_mode="mixed")
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale)
    toks = [0, 4, 5, 6, 134, 135, 136, 199]
    heads = [0, 3, 5]
    o2, l2 = oracle.prefill_rows(inp.q, inp.k, inp.v, inp.sinks, inp.cu_seqlens, inp.scale, toks, heads)
    np.testing.assert_allclose(o2, out[toks][:, heads], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l2, lse[toks][:, heads], rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# several new queries per sequence against the paged cache
# --------------------------------------------------------------------------
def _brute_paged(q, k_pages, v_pages, table, lens, cu_q, sinks, scale, P):
    """50-digit brute force; keys fetched straight from the pages, query t of
    sequence b at absolute position lens[b] - n_b + t sees keys 0..position."""
    import mpmath
    mpmath.mp.dps = 50
    Tq, hq, d = q.shape
    hkv = k_pages.shape[1]
    out = np.zeros((Tq, hq, d))
    lse = np.zeros((Tq, hq))
    for b in range(len(lens)):
        n = cu_q[b + 1] - cu_q[b]
        for t in range(n):
            pos = lens[b] - n + t
            for h in range(hq):
                g = h * hkv // hq
                terms, vals = [], []
                for j in range(0, pos + 1):
                    page = table[b][j // P]
                    dot = mpmath.mpf(0)
                    for e in range(d):
                        dot += mpmath.mpf(float(q[cu_q[b] + t, h, e])) * mpmath.mpf(float(k_pages[page, g, j % P, e]))
                    terms.append(mpmath.e ** (mpmath.mpf(scale) * dot))
                    vals.append([mpmath.mpf(float(v_pages[page, g, j % P, e])) for e in range(d)])
                z = sum(terms) + (mpmath.e ** mpmath.mpf(float(sinks[h])) if sinks[h] != -math.inf else 0)
                for e in range(d):
                    out[cu_q[b] + t, h, e] = float(sum(w * vv[e] for w, vv in zip(terms, vals)) / z) if z else 0.0
                lse[cu_q[b] + t, h] = float(mpmath.log(z)) if z else -math.inf
    return out, lse


@pytest.mark.parametrize("seed", [0, 1])
def test_paged_attention_matches_brute_force(seed):
    rng = np.random.default_rng(200 + seed)
    P, hq, hkv, d = 2, 4, 2, 3
    lens = [3, 0, 5, 2, 4]
    n_q = [2, 1, 3, 4, 4]  # the fourth sequence has more queries than cached tokens
    cu_q = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int64)
    pages = 16
    k_pages, v_pages = rng.normal(size=(pages, hkv, P, d)), rng.normal(size=(pages, hkv, P, d))
    table = rng.permutation(pages)[:15].reshape(5, 3)
    q = rng.normal(size=(int(cu_q[-1]), hq, d))
    sinks = np.array([0.3, -math.inf, 2.5, -1.1])
    out, lse = oracle.paged_attention(q, k_pages, v_pages, table, np.array(lens), cu_q, sinks, 0.8, page_size=P)
    bo, bl = _brute_paged(q, k_pages, v_pages, table, lens, cu_q, sinks, 0.8, P)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-13)


def _gather_torch(pages, row, L, P):
    """[L, Hkv, D] keys of one sequence by index arithmetic on the pool."""
    j = torch.arange(L)
    return pages[torch.as_tensor(row).long()[j // P], :, j % P, :]


def test_decode_multi_no_sink_is_sdpa_with_bottom_right_mask():
    inp = workloads.make_decode([40, 17, 64, 5], num_q_heads=8, num_kv_heads=2, head_dim=16, seed=21,
                                sink_mode="neginf", q_len=5, spare_pages=2, poison=True)
    out, _ = oracle.decode_multi(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.seqlens_t, inp.sinks,
                                 inp.scale)
    assert np.all(np.isfinite(out))
    for b, L in enumerate(inp.seqlens):
        n = 5
        kk = _gather_torch(inp.k_pages, inp.page_table[b], L, 16).double()
        vv = _gather_torch(inp.v_pages, inp.page_table[b], L, 16).double()
        kk, vv = kk.repeat_interleave(4, dim=1), vv.repeat_interleave(4, dim=1)
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            inp.q[b].double().permute(1, 0, 2), kk.permute(1, 0, 2), vv.permute(1, 0, 2), attn_mask=mask,
            scale=inp.scale)
        np.testing.assert_allclose(out[b], o.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_decode_multi_one_token_is_decode_and_last_token_sees_all():
    d1 = workloads.make_decode([37, 16, 1, 0, 50], num_q_heads=4, num_kv_heads=2, head_dim=8, seed=22,
                               sink_mode="normal2", q_len=1)
    out, lse = oracle.decode_multi(d1.q, d1.k_pages, d1.v_pages, d1.page_table, d1.seqlens_t, d1.sinks, d1.scale)
    o1, l1 = oracle.decode(d1.q[:, 0], d1.k_pages, d1.v_pages, d1.page_table, d1.seqlens_t, d1.sinks, d1.scale)
    np.testing.assert_allclose(out[:, 0], o1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, 0], l1, rtol=0, atol=1e-14)
    d4 = workloads.make_decode([37, 16, 50], num_q_heads=4, num_kv_heads=2, head_dim=8, seed=23,
                               sink_mode="normal2", q_len=4)
    out, lse = oracle.decode_multi(d4.q, d4.k_pages, d4.v_pages, d4.page_table, d4.seqlens_t, d4.sinks, d4.scale)
    o1, l1 = oracle.decode(d4.q[:, 3], d4.k_pages, d4.v_pages, d4.page_table, d4.seqlens_t, d4.sinks, d4.scale)
    np.testing.assert_allclose(out[:, 3], o1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, 3], l1, rtol=0, atol=1e-14)


def test_paged_attention_whole_sequence_is_causal_prefill():
    # every token new (n = L): the mask aligned to the end is the prefill mask
    lens = [33, 1, 20]
    d = workloads.make_decode(lens, num_q_heads=6, num_kv_heads=3, head_dim=8, seed=24, sink_mode="mixed")
    rng = np.random.default_rng(25)
    q = rng.normal(size=(sum(lens), 6, 8))
    cu = np.concatenate([[0], np.cumsum(lens)])
    out, lse = oracle.paged_attention(q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, cu, d.sinks, 0.3)
    kk = np.concatenate([oracle.gather_paged_kv(d.k_pages, d.page_table[b], L, 16) for b, L in enumerate(lens)])
    vv = np.concatenate([oracle.gather_paged_kv(d.v_pages, d.page_table[b], L, 16) for b, L in enumerate(lens)])
    o2, l2 = oracle.prefill(q, kk, vv, d.sinks, cu, 0.3)
    np.testing.assert_allclose(out, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, l2, rtol=0, atol=1e-13)


def test_queries_before_the_cache_start_see_only_the_sink():
    d = workloads.make_decode([2], num_q_heads=4, num_kv_heads=1, head_dim=8, seed=26, sink_mode="mixed", q_len=5)
    out, lse = oracle.decode_multi(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale)
    sinks = d.sinks.numpy().astype(np.float64)
    # queries 0..2 sit at positions -3..-1: no key, so out = 0 and lse = sink
    np.testing.assert_array_equal(out[0, :3], 0.0)
    np.testing.assert_array_equal(lse[0, :3], np.broadcast_to(sinks, (3, 4)))
    assert np.abs(out[0, 3:]).max() > 0
