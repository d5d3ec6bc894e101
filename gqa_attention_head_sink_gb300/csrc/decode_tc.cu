// Split-KV paged decode on the tensor cores, for many query rows per kv head
// (multi-token decode), with a per-head sink logit (sm_103a).
//
// Method: Perplexity, "GPT-OSS on day 0", section "Sink Attention": an online
// softmax whose running maximum m and scale d start at (sink, 1) in the first
// chunk of the key length only; chunks are combined afterwards by the merge
// kernel of the split decode (decode.cu).
//
// Work decomposition: one CTA per (chunk, kv head, sequence x row tile).  A
// row tile holds up to 128 query rows that read the same kv head: the G query
// heads of the group for tokens_per_tile consecutive new tokens, row
// rho = t_local * G + (h mod G).  That is exactly how a 3-D TMA box of
// (64 dims, G heads, tokens_per_tile tokens) lands in shared memory, so Q is
// one copy.  A sequence with L cached tokens has n new ones (the last n of
// the cache: q_len each, or from the offsets cu_q for a paged prefill); new
// token t sees keys 0 .. L - n + t.
//
// Per key tile of 128 tokens (8 pages):
//   * warp 0 (producer): one 2 KiB TMA copy per page for K and for V (the
//     (page, kv head) slab is contiguous), into a ring of five 16 KiB slots
//     (K_0, V_0, K_1, V_1, ...), 128-byte swizzle, byte-counting mbarriers;
//   * warp 1 (MMA): S = Q K^T (M=128, N=128, K=64) into TMEM; once the
//     softmax has written P, O += P V (M=128, N=64, K=128; P from TMEM, V from
//     shared memory).  The next tile's S is issued as soon as the softmax has
//     read the current one.  Before the last PV it zeroes the V rows past the
//     chunk's last key: stale or poisoned slots must not meet a zero weight
//     inside the MMA (0 x NaN = NaN);
//   * warps 2..5 (softmax, one thread per row; warp w reads TMEM lanes
//     32*(w%4) .. +31): mask keys past the row's limit, update (m, d) with the
//     rescale deferred until the maximum grows by more than 8 (log2 units),
//     write P (bf16) to TMEM, rescale O when needed.  Warps whose rows are all
//     padding sit out.  At the end: O / d (and lse) for a single chunk,
//     otherwise the partial (m, d, O) for the merge kernel.
// TMEM: S [0,128), P [128,192), O [192,256): 256 columns.  Shared memory
// (97 KiB) limits the SM to two of these CTAs, so two allocations always fit
// the 512 columns; no other kernel of this library that allocates TMEM fits
// beside them (the prefill kernel takes 181 KiB).
//
// The work is HBM-bound (at most 128 flop per byte of K/V, against ~300 for
// the tensor pipe's ridge point), so one MMA warp and a single S buffer
// suffice; what matters is copies in flight: 2 CTAs x up to five 16 KiB
// slots per SM.
#include "common.cuh"
#include "decode.h"
#include "tcgen05.cuh"

namespace sa {

namespace {

constexpr int kD = 64;
constexpr int kPage = 16;
constexpr int kKeyTile = 128;                    // keys per tile = 8 pages
constexpr int kPagesPerTile = kKeyTile / kPage;  // 8
constexpr int kSlabBytes = kPage * kD * 2;       // 2 KiB: one page of one kv head
constexpr int kSlotBytes = kKeyTile * kD * 2;    // 16 KiB
constexpr int kSlots = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, false, true);
constexpr float kRescaleThreshold = 8.f;

constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kDecodeTcRows * kD * 2;
constexpr int kOffBar = kOffRing + kSlots * kSlotBytes;
constexpr int kNumBars = 1 + 2 * kSlots + 5;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const DecodeParams& p,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, p.err, kErrDecodeFull, p.wait_limit_ns)) return true;
  *abort_flag = 1;
  return false;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  // the merge kernel may be scheduled once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int s = blockIdx.x, g = blockIdx.y;
  // blockIdx.z = r * batch + b with tile = row_tiles - 1 - r: the last tiles of
  // every sequence (which see the most keys) are launched first
  const int b = blockIdx.z % p.batch, tile = p.row_tiles - 1 - (int)(blockIdx.z / p.batch);
  int q0 = b * p.q_len, nq = p.q_len;  // first row of q and number of new tokens of the sequence
  if (p.cu_q) {                        // offsets are device data: clamp them to the rows of q
    q0 = min(max(0, p.cu_q[b]), p.total_q);
    nq = max(0, min(p.cu_q[b + 1], p.total_q) - q0);
  }
  const int G = p.group, tpt = p.tokens_per_tile;
  const int t0 = tile * tpt;  // first new token of the tile
  if (t0 >= nq) return;
  const int L = min(max(0, p.seqlens[b]), p.stride * kPage);
  const int npages = (L + kPage - 1) / kPage;
  const int n_chunks = decode_num_chunks(npages, p.num_splits, p.split_pages, p.max_splits);
  if (s >= n_chunks) return;
  const int chunk = npages > 0 ? (npages + n_chunks - 1) / n_chunks : 0;
  const int pg0 = s * chunk;
  const int pg1 = min(npages, pg0 + chunk);
  const int t_last = min(nq, t0 + tpt) - 1;  // last new token of the tile
  const int box_rows = G * tpt;              // rows the Q copy fills
  // keys [pg0*16, kend) of this chunk can be visible to some row of the tile
  const int kend = min(min(L, pg1 * kPage), L - nq + t_last + 1);
  const int nkeys = max(0, kend - pg0 * kPage);
  const int ntiles = (nkeys + kKeyTile - 1) / kKeyTile;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_tile = smem + kOffQ;
  uint8_t* ring = smem + kOffRing;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* slot_full = q_full + 1;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* s_full = slot_empty + kSlots;
  uint64_t* s_free = s_full + 1;
  uint64_t* p_full = s_free + 1;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int live_quads = (box_rows + 31) / 32;  // softmax warps with at least one real row
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(slot_full + i, 1);
      mbar_init(slot_empty + i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 32 * live_quads);
    mbar_init(p_full, 32 * live_quads);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ================================================================ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const uint64_t pol_stream = l2_policy_evict_first();
    if (ntiles > 0 && !p.withhold_copies && elect_one()) {  // no copy may outlive the CTA: Q only if used
      mbar_arrive_expect_tx(q_full, box_rows * kD * 2);
      tma_load_3d(q_tile, &qmap, q_full, 0, g * G, q0 + t0);
    }
    const int32_t* row = p.page_table + (size_t)b * p.stride;
    uint32_t ring_i = 0;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int first = pg0 + j * kPagesPerTile;
      const int np = min(kPagesPerTile, (kend - first * kPage + kPage - 1) / kPage);
      const int page = lane < np ? __ldg(row + first + lane) : 0;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const uint32_t slot = ring_i % kSlots;
        if (ring_i >= kSlots &&
            !(ok = __all_sync(0xffffffffu,
                              wait_or_abort(slot_empty + slot, ((ring_i / kSlots) - 1) & 1, p, abort_flag))))
          break;
        if (!p.withhold_copies) {
          if (elect_one()) mbar_arrive_expect_tx(slot_full + slot, np * kSlabBytes);
          __syncwarp();
          if (lane < np) {
            uint8_t* dst = ring + slot * kSlotBytes + lane * kSlabBytes;
            const int y = (page * p.hkv + g) * kPage;
            if (p.row_tiles == 1)  // read by this CTA only
              tma_load_2d_hint(dst, kv ? &vmap : &kmap, slot_full + slot, 0, y, pol_stream);
            else  // the sequence's other row tiles read it too
              tma_load_2d(dst, kv ? &vmap : &kmap, slot_full + slot, 0, y);
          }
        }
        ++ring_i;
      }
    }
    if (__any_sync(0xffffffffu, *abort_flag) && elect_one()) {
      // let copies already in flight land before the CTA can exit
      if (ntiles > 0) mbar_wait(q_full, 0, p.err, kErrDecodeFull, 10000000ull);
      for (uint32_t i = ring_i > kSlots ? ring_i - kSlots : 0; i < ring_i; ++i)
        mbar_wait(slot_full + (i % kSlots), (i / kSlots) & 1, p.err, kErrDecodeFull, 10000000ull);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    const uint64_t dq = smem_desc_sw128(smem_addr(q_tile));
    const uint64_t dring = smem_desc_sw128(smem_addr(ring));
    auto slot_desc = [&](uint32_t i) { return dring + (uint64_t)((i % kSlots) * (kSlotBytes >> 4)); };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p, abort_flag));
    };
    const uint32_t d_s = tmem + kColS, a_p = tmem + kColP, d_o = tmem + kColO;
    bool ok = ntiles > 0 && wait_all(q_full, 0);
    if (ok) ok = wait_all(slot_full + 0, 0);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_ss(d_s, dq + 2 * kk, slot_desc(0) + 2 * kk, kIdescQK, kk > 0);
        umma_commit(s_full);
        umma_commit(slot_empty + 0);
      }
    }
    for (int j = 0; j < ntiles && ok; ++j) {
      const uint32_t vi = 2 * j + 1, ki = 2 * j + 2;
      if (j + 1 < ntiles) {  // scores of tile j+1 once the softmax has read tile j's
        if (!(ok = wait_all(slot_full + ki % kSlots, (ki / kSlots) & 1))) break;
        if (!(ok = wait_all(s_free, j & 1))) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_ss(d_s, dq + 2 * kk, slot_desc(ki) + 2 * kk, kIdescQK, kk > 0);
          umma_commit(s_full);
          umma_commit(slot_empty + ki % kSlots);
        }
      }
      if (!(ok = wait_all(slot_full + vi % kSlots, (vi / kSlots) & 1))) break;
      if (!(ok = wait_all(p_full, j & 1))) break;
      tc_fence_after();
      const int valid = nkeys - j * kKeyTile;  // keys of this tile inside the chunk (>= 1)
      if (valid < kKeyTile) {
        // zero V rows [valid, 128): pages not copied or slots past the sequence end
        uint4* v = reinterpret_cast<uint4*>(ring + (vi % kSlots) * kSlotBytes);
        for (int i = valid * 8 + lane; i < kKeyTile * 8; i += 32) v[i] = make_uint4(0, 0, 0, 0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      if (elect_one()) {
        const uint64_t dv = slot_desc(vi);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) umma_ts(d_o, a_p + 8 * kk, dv + 128 * kk, kIdescPV, (j > 0 || kk > 0) ? 1 : 0);
        umma_commit(o_done);
        umma_commit(slot_empty + vi % kSlots);
      }
    }
    // every MMA issued here must finish before TMEM is released
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.err, kErrDecodeFull, p.wait_limit_ns);
  } else {
    // ================================================================ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row of the tile
    if (quad < live_quads) {
      const int t_loc = r / G;
      const int t = t0 + t_loc;                        // new token of the row
      const int h = g * G + (r - t_loc * G);           // query head of the row
      const bool row_ok = r < box_rows && t < nq;
      // keys visible to this row, relative to the chunk start
      const int lim = (row_ok ? min(kend, L - nq + t + 1) : kend) - pg0 * kPage;
      const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
      const uint32_t s_addr = tmem + lane_off + kColS;
      const uint32_t p_addr = tmem + lane_off + kColP;
      const uint32_t o_addr = tmem + lane_off + kColO;
      const float sl2 = p.scale_log2;
      const float2 sl2x2 = make_float2(sl2, sl2);
      float m = -INFINITY, d = 0.f;
      if (s == 0 && row_ok) {  // the first chunk starts from the sink
        m = __ldg(p.sinks + h) * kLog2e;
        d = 1.f;
      }
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        ok = __all_sync(0xffffffffu, wait_or_abort(s_full, j & 1, p, abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128(s_addr, sr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(s_free);  // the next tile's QK may overwrite S now
        const int vis = lim - j * kKeyTile;  // keys c < vis are visible
        float x[128];  // raw scores, -inf where masked
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
        if (__any_sync(0xffffffffu, vis < kKeyTile)) {  // only tiles that cross a row's last key
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= vis) x[c] = -INFINITY;
        }
        float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
        for (int c = 4; c < 124; c += 8) {
          mx0 = fmax3(mx0, x[c], x[c + 1]);
          mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
          mx2 = fmax3(mx2, x[c + 4], x[c + 5]);
          mx3 = fmax3(mx3, x[c + 6], x[c + 7]);
        }
        mx0 = fmax3(mx0, x[124], x[125]);
        mx1 = fmax3(mx1, x[126], x[127]);
        const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;  // log2 units
        const bool need = m_tile > m + kRescaleThreshold;  // also true the first time a -inf row sees a key
        const bool any_need = __any_sync(0xffffffffu, need);
        const float m_new = need ? m_tile : m;
        // -inf only while the row has seen neither sink nor key: subtract 0 then
        const float ms = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m - ms);
        const float2 neg_m2 = make_float2(-ms, -ms);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float2 e = ffma2(make_float2(x[2 * i], x[2 * i + 1]), sl2x2, neg_m2);
          pk[i] = pack_bf16x2(fast_exp2(e.x), fast_exp2(e.y));
          acc[i & 3] = add_bf16x2_f32x2(acc[i & 3], pk[i]);  // the normaliser sums the rounded weights
        }
        if (j > 0) {  // PV(j-1) reads P and accumulates into O until it is done
          ok = __all_sync(0xffffffffu, wait_or_abort(o_done, (j - 1) & 1, p, abort_flag));
          if (!ok) break;
          tc_fence_after();
          if (any_need) {
            uint32_t ob[64];
            tmem_ld64(o_addr, ob);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 64; ++e) ob[e] = __float_as_uint(__uint_as_float(ob[e]) * alpha);
            tmem_st64(o_addr, ob);
          }
        }
        tmem_st64(p_addr, pk);
        tmem_st_wait();
        const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
        d = d * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
        m = m_new;
        tc_fence_before();
        mbar_arrive(p_full);
      }
      // ---- epilogue
      uint32_t ob[64];
      if (ok && ntiles > 0) {
        ok = __all_sync(0xffffffffu, wait_or_abort(o_done, (ntiles - 1) & 1, p, abort_flag));
        if (ok) {
          tc_fence_after();
          tmem_ld64(o_addr, ob);
          tmem_ld_wait();
        }
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) ob[e] = 0u;  // no key in this chunk: O = 0
      }
      if (ok && row_ok) {
        const size_t qrow = ((size_t)q0 + t) * p.hq + h;  // (row of q, head)
        if (p.direct) {
          const float inv = d > 0.f ? 1.f / d : 0.f;
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + qrow * kD);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              dst[i] = make_float4(__uint_as_float(ob[4 * i]) * inv, __uint_as_float(ob[4 * i + 1]) * inv,
                                   __uint_as_float(ob[4 * i + 2]) * inv, __uint_as_float(ob[4 * i + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + qrow * kD);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(ob[8 * i + 0]) * inv, __uint_as_float(ob[8 * i + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(ob[8 * i + 2]) * inv, __uint_as_float(ob[8 * i + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(ob[8 * i + 4]) * inv, __uint_as_float(ob[8 * i + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(ob[8 * i + 6]) * inv, __uint_as_float(ob[8 * i + 7]) * inv);
              dst[i] = v;
            }
          }
          if (p.lse) p.lse[qrow] = d > 0.f ? (m + __log2f(d)) * kLn2 : -INFINITY;
        } else {
          const size_t slot = qrow * p.max_splits + s;
          float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * kD);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            dst[i] = make_float4(__uint_as_float(ob[4 * i]), __uint_as_float(ob[4 * i + 1]),
                                 __uint_as_float(ob[4 * i + 2]), __uint_as_float(ob[4 * i + 3]));
          p.ws_md[slot * 2] = m;
          p.ws_md[slot * 2 + 1] = d;
        }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t decode_tc_configure() {
  return cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_decode_tc(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.max_splits, p.hkv, p.batch * p.row_tiles);
  decode_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.direct) return e;
  return launch_decode_merge(p, stream);
}

}  // namespace sa
