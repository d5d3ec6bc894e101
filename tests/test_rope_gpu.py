"""GPU parity of the QKV bias + YaRN rotary pass against the float64 oracle.

The pass rotates q and k in place (planes (i, i + D/2), angle position x
frequency, times YaRN's temperature) after adding their biases, biases v,
and optionally appends the new k and v to the paged cache.  Outputs are
bf16: each element may differ from the float64 value by one bf16 spacing
(the single rounding of the result, which a last-bit difference of the fp32
arithmetic can push to the other neighbour).  The expected values use the
oracle's float64 YaRN table, the kernel the library's fp64 table: the angle the
kernel forms must keep that precision at every int32 position, up to 2^31 - 1.
The end-to-end test runs the
pass and then prefill, against the oracle's float64 pass, rounded once to
bf16 (the pass's output type, which attention consumes), followed by its
prefill.  All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import gqa_attention_head_sink_gb300 as sa
import oracle
from gqa_attention_head_sink_gb300 import build, workloads
from tests.parity import assert_parity, bf16_spacing, lse_close, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    sa.load()


def _inputs(T, hq, hkv, seed, with_bias=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    q, k, v = r(T, hq, 64), r(T, hkv, 64), r(T, hkv, 64)
    biases = (r(hq, 64), r(hkv, 64), r(hkv, 64)) if with_bias else (None, None, None)
    return q, k, v, biases


def _close_bf16(got, want):
    g, w = to_f64(got), np.asarray(want, dtype=np.float64)
    err = np.abs(g - w)
    allowed = bf16_spacing(w) + 1e-6
    assert np.all(err <= allowed), f"max excess {np.max(err - allowed):.3e}"


@pytest.mark.parametrize("T,hq,hkv,yarn,with_bias,max_pos", [
    (1, 64, 8, (150000.0, 32.0, 4096, 32.0, 1.0), True, 131072),
    (300, 64, 8, (150000.0, 32.0, 4096, 32.0, 1.0), True, 1 << 20),
    (77, 8, 8, (10000.0, 1.0, 4096, 32.0, 1.0), False, 4096),
    (129, 16, 1, (500000.0, 8.0, 8192, 16.0, 2.0), True, 70000),
    (256, 64, 8, (150000.0, 32.0, 4096, 32.0, 1.0), True, 1 << 24),
    (200, 16, 2, (150000.0, 32.0, 4096, 32.0, 1.0), True, (1 << 31) - 1),
    (100, 16, 2, (10000.0, 1.0, 4096, 32.0, 1.0), True, (1 << 31) - 1),
])
def test_qkv_rope_matches_oracle(T, hq, hkv, yarn, with_bias, max_pos):
    q, k, v, (bq, bk, bv) = _inputs(T, hq, hkv, seed=T + hq)
    pos = torch.randint(0, max_pos, (T,), generator=torch.Generator().manual_seed(T), dtype=torch.int32)
    pos[0] = max_pos - 1  # the largest position of the range is always there
    f, af = sa.sink_attn_yarn_inv_freq(64, *yarn)  # the library's fp64 table goes to the kernel
    f64, af64 = oracle.yarn_inv_freq(64, *yarn)     # the expected values use the oracle's own table
    want_q, want_k, want_v = oracle.qkv_bias_rope(q, k, v, bq, bk, bv, pos, f64, af64)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    cu = lambda t: None if t is None else t.cuda()  # noqa: E731
    sa.sink_attn_qkv_rope(dq, dk, dv, pos.cuda(), f.cuda(), af, cu(bq), cu(bk), cu(bv))
    torch.cuda.synchronize()
    _close_bf16(dq, want_q)
    _close_bf16(dk, want_k)
    _close_bf16(dv, want_v)


def test_qkv_rope_appends_to_the_paged_cache():
    T, hq, hkv, num_pages = 40, 64, 8, 12
    q, k, v, (bq, bk, bv) = _inputs(T, hq, hkv, seed=5)
    g = torch.Generator(device="cpu").manual_seed(6)
    slots = torch.randperm(num_pages * 16, generator=g)[:T].to(torch.int32)
    slots[::7] = -1  # these tokens are not cached
    pos = torch.arange(T, dtype=torch.int32) + 1000
    f, af = sa.sink_attn_yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    kp = torch.full((num_pages, hkv, 16, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    vp = kp.clone()
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    sa.sink_attn_qkv_rope(dq, dk, dv, pos.cuda(), f.cuda(), af, bq.cuda(), bk.cuda(), bv.cuda(),
                          slot_mapping=slots.cuda(), k_pages=kp, v_pages=vp)
    torch.cuda.synchronize()
    touched = torch.zeros(num_pages, 16, dtype=torch.bool)
    for t in range(T):
        s = int(slots[t])
        if s < 0:
            continue
        touched[s // 16, s % 16] = True
        assert torch.equal(kp[s // 16, :, s % 16], dk[t]) and torch.equal(vp[s // 16, :, s % 16], dv[t])
    untouched = ~touched.cuda()
    assert bool((kp.permute(0, 2, 1, 3)[untouched] == 7.0).all()) and bool((vp.permute(0, 2, 1, 3)[untouched] == 7.0).all())


def test_qkv_rope_rejects_buffers_it_would_overrun():
    # a bias with fewer heads, a slot mapping shorter than the tokens, or cache pools with
    # fewer kv heads would be read or written past their ends: refused before any launch
    T, hq, hkv = 16, 8, 2
    q, k, v, (bq, bk, bv) = _inputs(T, hq, hkv, seed=9)
    q, k, v, bq, bk, bv = (t.cuda() for t in (q, k, v, bq, bk, bv))
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    f, af = sa.sink_attn_yarn_inv_freq(64)
    f = f.cuda()
    kp = torch.zeros((4, hkv, 16, 64), dtype=torch.bfloat16, device="cuda")
    slots = torch.arange(T, dtype=torch.int32, device="cuda")
    bad = [
        dict(q_bias=bq[:4]),
        dict(k_bias=bk[:1]),
        dict(v_bias=bv[:, :32].contiguous()),
        dict(slot_mapping=slots[:8], k_pages=kp, v_pages=kp.clone()),
        dict(slot_mapping=slots, k_pages=kp[:, :1].contiguous(), v_pages=kp[:, :1].contiguous()),
        dict(slot_mapping=slots, k_pages=kp, v_pages=kp[:2].contiguous()),
    ]
    before = (q.clone(), k.clone(), v.clone())
    for kw in bad:
        with pytest.raises(ValueError):
            sa.sink_attn_qkv_rope(q, k, v, pos, f, af, **kw)
    torch.cuda.synchronize()
    assert torch.equal(q, before[0]) and torch.equal(k, before[1]) and torch.equal(v, before[2])


def test_bias_rope_then_prefill_matches_oracle():
    lens = [300, 129]
    inp = workloads.make_prefill(lens, seed=7, sink_mode="normal2")
    T = sum(lens)
    g = torch.Generator(device="cpu").manual_seed(8)
    bq = (0.5 * torch.randn(64, 64, generator=g)).to(torch.bfloat16)
    bk = (0.5 * torch.randn(8, 64, generator=g)).to(torch.bfloat16)
    bv = (0.5 * torch.randn(8, 64, generator=g)).to(torch.bfloat16)
    pos = torch.cat([torch.arange(L, dtype=torch.int32) for L in lens])
    f, af = sa.sink_attn_yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    f64, af64 = oracle.yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    q2, k2, v2 = oracle.qkv_bias_rope(inp.q, inp.k, inp.v, bq, bk, bv, pos, f64, af64)
    # the pass hands bf16 q, k, v to attention: round the float64 results once
    # (nearest even), as the pass's contract says, then take the attention
    r = lambda x: torch.from_numpy(x).to(torch.bfloat16)  # noqa: E731
    want, _ = oracle.prefill(r(q2), r(k2), r(v2), inp.sinks, inp.cu_seqlens, inp.scale)
    d = inp.to("cuda")
    sa.sink_attn_qkv_rope(d.q, d.k, d.v, pos.cuda(), f.cuda(), af, bq.cuda(), bk.cuda(), bv.cuda())
    out = sa.sink_attn_prefill(d.q, d.k, d.v, d.sinks, d.cu_seqlens, d.scale, max_seqlen=max(lens))
    torch.cuda.synchronize()
    assert_parity(out, want)


@pytest.mark.parametrize("lens,hq,hkv,splits,yarn,with_bias", [
    ([500, 77, 1, 4096], 64, 8, 8, (150000.0, 32.0, 4096, 32.0, 1.0), True),
    ([300, 16, 2000], 16, 2, 0, (10000.0, 1.0, 4096, 32.0, 1.0), False),
    ([8192] * 4, 64, 8, 0, (150000.0, 32.0, 4096, 32.0, 1.0), True),
])
def test_decode_rope_fuses_the_query_rotation(lens, hq, hkv, splits, yarn, with_bias):
    # the query of each sequence is rotated inside the decode kernel by position
    # seqlens[b] - 1: the same bits as the rotary pass followed by plain decode, and
    # within tolerance of the oracle's float64 rotation (rounded to bf16) + decode
    d = workloads.make_decode(lens, num_q_heads=hq, num_kv_heads=hkv, seed=len(lens) + hq, sink_mode="mixed",
                              num_splits=splits, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(41)
    bq = (0.5 * torch.randn(hq, 64, generator=g)).to(torch.bfloat16).cuda() if with_bias else None
    f, af = sa.sink_attn_yarn_inv_freq(64, *yarn)
    f = f.cuda()
    pos = (d.seqlens_t - 1).clamp(min=0)
    fused = sa.sink_attn_decode_rope(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale, f, af,
                                     q_bias=bq, num_splits=splits, max_seqlen=d.max_seqlen)
    q2 = d.q.clone()
    dummy = torch.zeros((d.batch, hkv, 64), dtype=torch.bfloat16, device="cuda")
    sa.sink_attn_qkv_rope(q2, dummy, dummy.clone(), pos, f, af, q_bias=bq)
    separate = sa.sink_attn_decode(q2, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale,
                                   num_splits=splits, max_seqlen=d.max_seqlen)
    torch.cuda.synchronize()
    assert torch.equal(fused, separate)
    f64, af64 = oracle.yarn_inv_freq(64, *yarn)
    qr, _, _ = oracle.qkv_bias_rope(d.q.cpu(), dummy.cpu(), dummy.cpu(), None if bq is None else bq.cpu(), None,
                                    None, pos.cpu(), f64, af64)
    want, _ = oracle.decode(torch.from_numpy(qr).to(torch.bfloat16), d.k_pages.cpu(), d.v_pages.cpu(),
                            d.page_table.cpu(), d.seqlens_t.cpu(), d.sinks.cpu(), d.scale)
    assert_parity(fused, want)


@pytest.mark.parametrize("lens,hq,hkv,yarn,with_bias", [
    ([300, 129, 1, 0, 517], 64, 8, (150000.0, 32.0, 4096, 32.0, 1.0), True),
    ([1000, 128, 256], 16, 2, (10000.0, 1.0, 4096, 32.0, 1.0), False),
    ([777], 6, 2, (500000.0, 8.0, 8192, 16.0, 2.0), True),  # odd group: a pair's second head is absent
])
def test_prefill_rope_fuses_the_query_rotation(lens, hq, hkv, yarn, with_bias):
    # q is rotated inside the prefill kernel (token i of a sequence at position i): the
    # same bits as the rotary pass on q followed by plain prefill, and within tolerance
    # of the oracle's float64 pass (rounded to bf16) + prefill
    inp = workloads.make_prefill(lens, num_q_heads=hq, num_kv_heads=hkv, seed=sum(lens) % 89, sink_mode="mixed",
                                 device="cuda")
    g = torch.Generator(device="cpu").manual_seed(42)
    r = lambda *shape: (0.5 * torch.randn(*shape, generator=g)).to(torch.bfloat16)  # noqa: E731
    bq, bk, bv = (r(hq, 64), r(hkv, 64), r(hkv, 64)) if with_bias else (None, None, None)
    cu = lambda t: None if t is None else t.cuda()  # noqa: E731
    pos = torch.cat([torch.arange(L, dtype=torch.int32) for L in lens])
    f, af = sa.sink_attn_yarn_inv_freq(64, *yarn)
    f = f.cuda()
    q_raw, k, v = inp.q.clone(), inp.k.clone(), inp.v.clone()
    sa.sink_attn_qkv_rope(None, k, v, pos.cuda(), f, af, q_bias=cu(bq), k_bias=cu(bk), v_bias=cu(bv))
    lse = torch.empty((inp.total_tokens, hq), dtype=torch.float32, device="cuda")
    fused = sa.sink_attn_prefill_rope(q_raw, k, v, inp.sinks, inp.cu_seqlens, inp.scale, f, af, q_bias=cu(bq),
                                      lse=lse, max_seqlen=inp.max_seqlen)
    q_rot = q_raw.clone()
    sa.sink_attn_qkv_rope(q_rot, torch.zeros_like(k), torch.zeros_like(v), pos.cuda(), f, af, q_bias=cu(bq))
    separate = sa.sink_attn_prefill(q_rot, k, v, inp.sinks, inp.cu_seqlens, inp.scale, max_seqlen=inp.max_seqlen)
    torch.cuda.synchronize()
    assert torch.equal(fused, separate)
    assert torch.equal(q_raw, inp.q)  # the caller's q is not modified
    f64, af64 = oracle.yarn_inv_freq(64, *yarn)
    q2, k2, v2 = oracle.qkv_bias_rope(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), bq, bk, bv, pos, f64, af64)
    rb = lambda x: torch.from_numpy(x).to(torch.bfloat16)  # noqa: E731
    want, want_lse = oracle.prefill(rb(q2), rb(k2), rb(v2), inp.sinks.cpu(), inp.cu_seqlens.cpu(), inp.scale)
    assert_parity(fused, want)
    lse_close(lse, want_lse)
