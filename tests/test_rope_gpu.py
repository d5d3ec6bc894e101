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
from tests.parity import assert_parity, bf16_spacing, to_f64

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
