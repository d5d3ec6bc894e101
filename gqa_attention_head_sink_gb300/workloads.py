"""Seeded synthetic inputs shaped like gpt-oss attention.

This module only draws random tensors and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the float64 oracle can be fed
from it.  Shapes follow the attention of gpt-oss: head_dim 64, 64 query heads,
8 key/value heads (GQA group 8), bf16 q/k/v, fp32 sinks, softmax scale
1/sqrt(64) = 1/8.

Draw order for one workload (all from one generator seeded with ``seed`` on
``device``): sinks, q, k, v, then (decode only) the page permutation.  Lengths
that are random are drawn first from a separate CPU generator with the same
seed, so they are identical whatever the device.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

HEAD_DIM = 64
PAGE_SIZE = 16

# Sink initialisations.
#   "normal1": N(0, 1);  "normal2": 2 * N(0, 1) (standard deviation 2);
#   "mixed":   by head index mod 4 -> -inf, 0, 2*N(0,1), +20;
#   "neginf":  all -inf (no sink: plain attention);  "zero": all 0.
SINK_MODES = ("normal1", "normal2", "mixed", "neginf", "zero")


@dataclasses.dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, Hq, D] bf16
    k: torch.Tensor            # [T, Hkv, D] bf16
    v: torch.Tensor            # [T, Hkv, D] bf16
    sinks: torch.Tensor        # [Hq] fp32
    cu_seqlens: torch.Tensor   # [B+1] int32
    seqlens: List[int]         # host copy of the lengths
    scale: float

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens)) if self.seqlens else 0

    @property
    def batch(self) -> int:
        return len(self.seqlens)

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k.shape[1]

    def to(self, device) -> "PrefillInputs":
        return dataclasses.replace(
            self, q=self.q.to(device), k=self.k.to(device), v=self.v.to(device),
            sinks=self.sinks.to(device), cu_seqlens=self.cu_seqlens.to(device))


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor            # [B, Hq, D] bf16, or [B, n, Hq, D] for n new tokens per sequence
    k_pages: torch.Tensor      # [num_pages, Hkv, page_size, D] bf16
    v_pages: torch.Tensor      # [num_pages, Hkv, page_size, D] bf16
    page_table: torch.Tensor   # [B, stride] int32, unused entries -1
    seqlens_t: torch.Tensor    # [B] int32
    seqlens: List[int]         # host copy
    sinks: torch.Tensor        # [Hq] fp32
    scale: float
    num_splits: int            # 0 = chosen per length by the library
    page_size: int = PAGE_SIZE
    # chunked prefill: q is [total_q, Hq, D], packed by these offsets [B+1]
    cu_seqlens_q: Optional[torch.Tensor] = None
    q_lens: Optional[List[int]] = None

    @property
    def batch(self) -> int:
        return len(self.seqlens)

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens)) if self.seqlens else 0

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[-2]

    @property
    def q_len(self) -> int:
        """New query tokens per sequence (1 for a [B, Hq, D] query)."""
        if self.q_lens is not None:
            raise ValueError("per-sequence new-token counts: see q_lens")
        return self.q.shape[1] if self.q.dim() == 4 else 1

    @property
    def num_kv_heads(self) -> int:
        return self.k_pages.shape[1]

    def to(self, device) -> "DecodeInputs":
        return dataclasses.replace(
            self, q=self.q.to(device), k_pages=self.k_pages.to(device),
            v_pages=self.v_pages.to(device), page_table=self.page_table.to(device),
            seqlens_t=self.seqlens_t.to(device), sinks=self.sinks.to(device),
            cu_seqlens_q=None if self.cu_seqlens_q is None else self.cu_seqlens_q.to(device))


def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_sinks(num_q_heads: int, mode: str, gen: torch.Generator, device) -> torch.Tensor:
    if mode not in SINK_MODES:
        raise ValueError(f"unknown sink mode {mode!r}")
    z = torch.randn(num_q_heads, generator=gen, device=device, dtype=torch.float32)
    if mode == "normal1":
        return z
    if mode == "normal2":
        return 2.0 * z
    if mode == "neginf":
        return torch.full_like(z, -math.inf)
    if mode == "zero":
        return torch.zeros_like(z)
    # mixed: one of four edge cases per head
    idx = torch.arange(num_q_heads, device=device) % 4
    out = 2.0 * z
    out = torch.where(idx == 0, torch.full_like(z, -math.inf), out)
    out = torch.where(idx == 1, torch.zeros_like(z), out)
    out = torch.where(idx == 3, torch.full_like(z, 20.0), out)
    return out


def _randn_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_prefill(seqlens, num_q_heads=64, num_kv_heads=8, head_dim=HEAD_DIM, seed=0,
                 sink_mode="normal2", scale: Optional[float] = None, device="cpu") -> PrefillInputs:
    """Packed causal prefill inputs: q/k/v ~ N(0,1) rounded once to bf16."""
    seqlens = [int(x) for x in seqlens]
    T = sum(seqlens)
    gen = _generator(device, seed)
    sinks = draw_sinks(num_q_heads, sink_mode, gen, device)
    q = _randn_bf16((T, num_q_heads, head_dim), gen, device)
    k = _randn_bf16((T, num_kv_heads, head_dim), gen, device)
    v = _randn_bf16((T, num_kv_heads, head_dim), gen, device)
    cu = torch.zeros(len(seqlens) + 1, dtype=torch.int32)
    if seqlens:
        cu[1:] = torch.cumsum(torch.tensor(seqlens, dtype=torch.int64), 0).to(torch.int32)
    return PrefillInputs(q=q, k=k, v=v, sinks=sinks, cu_seqlens=cu.to(device), seqlens=seqlens,
                         scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale))


def make_decode(seqlens, num_q_heads=64, num_kv_heads=8, head_dim=HEAD_DIM, seed=0,
                sink_mode="normal2", scale: Optional[float] = None, num_splits=0,
                page_size=PAGE_SIZE, spare_pages=0, poison=False, q_len: Optional[int] = None,
                q_lens: Optional[List[int]] = None, device="cpu") -> DecodeInputs:
    """Paged decode inputs: one bf16 query per sequence (q [B, Hq, D]), or
    ``q_len`` new query tokens per sequence (q [B, q_len, Hq, D]: the last
    q_len tokens of each sequence's cache), KV pool in pages of
    ``page_size`` tokens laid out [num_pages, Hkv, page_size, D], and a page
    table that maps each sequence's logical pages to a random permutation of
    the pool.  ``spare_pages`` adds pool pages that no sequence owns.  With
    ``poison`` the slots past each sequence's length in its last page and the
    spare pages hold NaN, so any read beyond the valid tokens shows up.
    ``q_lens`` (chunked prefill): per-sequence new-token counts instead; q is
    then [sum(q_lens), Hq, D] packed by ``cu_seqlens_q``."""
    seqlens = [int(x) for x in seqlens]
    B = len(seqlens)
    pages_per_seq = [(L + page_size - 1) // page_size for L in seqlens]
    used = sum(pages_per_seq)
    num_pages = max(1, used + int(spare_pages))
    gen = _generator(device, seed)
    sinks = draw_sinks(num_q_heads, sink_mode, gen, device)
    if q_lens is not None:
        q_lens = [int(x) for x in q_lens]
        q_shape = (sum(q_lens), num_q_heads, head_dim)
    elif q_len is None:
        q_shape = (B, num_q_heads, head_dim)
    else:
        q_shape = (B, int(q_len), num_q_heads, head_dim)
    q = _randn_bf16(q_shape, gen, device)
    k_pages = _randn_bf16((num_pages, num_kv_heads, page_size, head_dim), gen, device)
    v_pages = _randn_bf16((num_pages, num_kv_heads, page_size, head_dim), gen, device)
    perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    stride = max(1, max(pages_per_seq) if pages_per_seq else 1)
    table = torch.full((B, stride), -1, dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(pages_per_seq):
        if n:
            table[b, :n] = perm[off:off + n]
        off += n
    if poison:
        nan = float("nan")
        for b, L in enumerate(seqlens):
            n = pages_per_seq[b]
            tail = L - (n - 1) * page_size if n else page_size
            if n and tail < page_size:
                last = int(table[b, n - 1])
                k_pages[last, :, tail:, :] = nan
                v_pages[last, :, tail:, :] = nan
        if spare_pages:
            spare = perm[used:]
            k_pages[spare.long()] = nan
            v_pages[spare.long()] = nan
    lens_t = torch.tensor(seqlens, dtype=torch.int32, device=device)
    cu_q = None
    if q_lens is not None:
        cu_q = torch.zeros(B + 1, dtype=torch.int32)
        if B:
            cu_q[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
        cu_q = cu_q.to(device)
    return DecodeInputs(q=q, k_pages=k_pages, v_pages=v_pages, page_table=table, seqlens_t=lens_t,
                        seqlens=seqlens, sinks=sinks, num_splits=int(num_splits), page_size=page_size,
                        scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
                        cu_seqlens_q=cu_q, q_lens=q_lens)


def make_paged_prefill(seqlens_k, new_lens, **kw) -> DecodeInputs:
    """Chunked prefill inputs: sequence b holds seqlens_k[b] cached tokens in
    its pages, the last new_lens[b] of which are new and have a query each."""
    return make_decode(seqlens_k, q_lens=list(new_lens), **kw)


def _uniform_lengths(n, lo, hi, seed) -> List[int]:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


# The five named workloads.  Seeds: 0 for the tiny case, 1..4 for the others.
WORKLOADS = {
    "tiny_prefill": "batch 1, causal, seq 128, Hq=4, Hkv=1, D=64, sinks N(0,1), scale 1/8, seed 0",
    "gptoss_prefill": "batch 1, causal, seq 8192, Hq=64, Hkv=8, D=64, sinks N(0,2), scale 1/8, seed 1",
    "decode": "batch 64, 1 query each, Hq=64, Hkv=8, D=64, paged KV (page 16, permuted), "
              "all lengths 8192, sinks N(0,2), num_splits 8, seed 2",
    "long_decode": "batch 128, 1 query each, Hq=64, Hkv=8, D=64, paged KV (page 16), "
                   "lengths U[16384, 32768], sinks N(0,2), splits per length, seed 3",
    "ragged_prefill": "16 sequences, lengths U[256, 32768] packed by cu_seqlens, causal, Hq=64, "
                      "Hkv=8, D=64, sinks by head mod 4: -inf, 0, N(0,2), +20, seed 4",
    "mtp_decode": "batch 64 x 8192 cached tokens, the last 4 of them new (4 queries each, causal among "
                  "them), Hq=64, Hkv=8, D=64, paged KV (page 16), splits per length, sinks N(0,2), seed 5",
    "chunked_prefill": "1 sequence, 8192 new tokens after an 8192-token cached prefix (16384 paged), causal, "
                       "Hq=64, Hkv=8, D=64, splits per length, sinks N(0,2), seed 6",
    "qkv_rope": "8192 tokens (positions 0..8191), Hq=64, Hkv=8, D=64, q/k/v N(0,1), biases 0.5*N(0,1), all bf16; "
                "YaRN base 150000, factor 32, original context 4096, beta_fast 32, beta_slow 1, seed 7",
}

# YaRN settings of the rotary workload: those of the public gpt-oss model
# configuration (the pages name YaRN but give no parameters).
YARN_SETTINGS = dict(base=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)


@dataclasses.dataclass
class RopeInputs:
    q: torch.Tensor          # [T, Hq, D] bf16
    k: torch.Tensor          # [T, Hkv, D] bf16
    v: torch.Tensor          # [T, Hkv, D] bf16
    q_bias: torch.Tensor     # [Hq, D] bf16
    k_bias: torch.Tensor     # [Hkv, D] bf16
    v_bias: torch.Tensor     # [Hkv, D] bf16
    positions: torch.Tensor  # [T] int32


def make_qkv_rope(num_tokens, num_q_heads=64, num_kv_heads=8, head_dim=HEAD_DIM, seed=7, positions=None,
                  device="cpu") -> RopeInputs:
    """Inputs of the QKV bias + rotary pass: q/k/v ~ N(0,1) and biases
    0.5 * N(0,1), rounded once to bf16; positions 0..T-1 unless given."""
    gen = _generator(device, seed)
    q = _randn_bf16((num_tokens, num_q_heads, head_dim), gen, device)
    k = _randn_bf16((num_tokens, num_kv_heads, head_dim), gen, device)
    v = _randn_bf16((num_tokens, num_kv_heads, head_dim), gen, device)
    half = lambda *shape: (0.5 * torch.randn(*shape, generator=gen, device=device)).to(torch.bfloat16)  # noqa: E731
    bq, bk, bv = half(num_q_heads, head_dim), half(num_kv_heads, head_dim), half(num_kv_heads, head_dim)
    if positions is None:
        positions = torch.arange(num_tokens, dtype=torch.int32, device=device)
    return RopeInputs(q=q, k=k, v=v, q_bias=bq, k_bias=bk, v_bias=bv,
                      positions=torch.as_tensor(positions, dtype=torch.int32, device=device))


def qkv_rope_bytes(num_tokens, num_q_heads, num_kv_heads, head_dim=HEAD_DIM) -> int:
    """Bytes the rotary pass must move: q, k, v read and written once (bf16),
    the positions, and the biases."""
    qkv = num_tokens * (num_q_heads + 2 * num_kv_heads) * head_dim * 2
    return 2 * qkv + num_tokens * 4 + (num_q_heads + 2 * num_kv_heads) * head_dim * 2


def workload_seqlens(name: str) -> List[int]:
    if name == "tiny_prefill":
        return [128]
    if name == "gptoss_prefill":
        return [8192]
    if name == "decode":
        return [8192] * 64
    if name == "long_decode":
        return _uniform_lengths(128, 16384, 32768, 3)
    if name == "ragged_prefill":
        return _uniform_lengths(16, 256, 32768, 4)
    if name == "mtp_decode":
        return [8192] * 64
    if name == "chunked_prefill":
        return [16384]
    raise KeyError(name)


def workload(name: str, device="cpu", **overrides):
    """Inputs of one named workload on ``device``."""
    lens = workload_seqlens(name)
    if name == "tiny_prefill":
        kw = dict(num_q_heads=4, num_kv_heads=1, seed=0, sink_mode="normal1", scale=0.125)
        kw.update(overrides)
        return make_prefill(lens, device=device, **kw)
    if name == "gptoss_prefill":
        kw = dict(seed=1, sink_mode="normal2", scale=0.125)
        kw.update(overrides)
        return make_prefill(lens, device=device, **kw)
    if name == "decode":
        kw = dict(seed=2, sink_mode="normal2", scale=0.125, num_splits=8)
        kw.update(overrides)
        return make_decode(lens, device=device, **kw)
    if name == "long_decode":
        kw = dict(seed=3, sink_mode="normal2", scale=0.125, num_splits=0)
        kw.update(overrides)
        return make_decode(lens, device=device, **kw)
    if name == "ragged_prefill":
        kw = dict(seed=4, sink_mode="mixed", scale=0.125)
        kw.update(overrides)
        return make_prefill(lens, device=device, **kw)
    if name == "mtp_decode":
        kw = dict(seed=5, sink_mode="normal2", scale=0.125, num_splits=0, q_len=4)
        kw.update(overrides)
        return make_decode(lens, device=device, **kw)
    if name == "chunked_prefill":
        kw = dict(seed=6, sink_mode="normal2", scale=0.125, num_splits=0)
        kw.update(overrides)
        return make_paged_prefill(lens, [8192], device=device, **kw)
    raise KeyError(name)


# Algorithmic work per unit, used by the benchmark (counted, not measured).
def prefill_flops(seqlens, num_q_heads, head_dim=HEAD_DIM) -> int:
    """4*D flop (QK^T and PV multiply-adds) per unmasked (query, key) pair per
    query head; causal: L(L+1)/2 pairs per sequence."""
    pairs = sum(L * (L + 1) // 2 for L in seqlens)
    return 4 * head_dim * num_q_heads * pairs


def paged_prefill_flops(seqlens_k, new_lens, num_q_heads, head_dim=HEAD_DIM) -> int:
    """4*D flop per visible (query, key) pair per query head: new token t of
    a sequence with L keys and n new tokens sees L - n + t + 1 keys."""
    pairs = 0
    for L, n in zip(seqlens_k, new_lens):
        n_vis = min(n, L)  # tokens placed before the cache start see no key
        last = L  # keys seen by the last new token
        pairs += n_vis * last - n_vis * (n_vis - 1) // 2
    return 4 * head_dim * num_q_heads * pairs


def decode_bytes(seqlens, num_q_heads, num_kv_heads, head_dim=HEAD_DIM, out_bytes=2,
                 page_size=PAGE_SIZE, q_len=1) -> int:
    """Bytes a decode step must move at least once: K and V of every valid
    token (once per kv head), the queries (q_len per sequence), the outputs,
    the used page-table entries and the lengths."""
    kv = sum(seqlens) * num_kv_heads * head_dim * 2 * 2
    q = len(seqlens) * q_len * num_q_heads * head_dim * 2
    o = len(seqlens) * q_len * num_q_heads * head_dim * out_bytes
    table = sum((L + page_size - 1) // page_size for L in seqlens) * 4
    return kv + q + o + table + 4 * len(seqlens)
