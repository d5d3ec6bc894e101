// Causal variable-length prefill with a per-head sink logit (sm_103a).
//
// Method: Perplexity, "GPT-OSS on day 0", section "Sink Attention": the
// softmax of every query row is taken over its (causal) key logits plus the
// head's sink logit, evaluated online over key tiles with a running maximum m
// and running scale d; the state starts at m = sink, d = 1, which counts the
// sink once in the normaliser.  The sink has no value vector.
//
// Design (persistent, warp-specialised, one CTA per SM):
//   * work unit = (sequence, 128-row query block, pair of query heads of one
//     GQA group).  The two heads share every K/V tile, so a tile is staged once
//     for two 128x128 score tiles.  Units are ordered by sequence (longest
//     first) and within a sequence by query block (most key tiles first), the
//     heads of one group adjacent, so that concurrently running CTAs read the
//     same K/V from L2.  A CTA takes its next unit from a launch-wide counter
//     (a unit of schedule order at a time), so CTAs on slower SMs take fewer:
//     with a fixed serpentine deal the last CTA ended ~22 us after the first
//     on the 8192-token workload (some SMs run ~2 % slower throughout).
//     Launches captured into a graph keep the serpentine deal.
//   * warp 2 (elected lane): TMA producer.  Takes the CTA's units and publishes
//     each, one unit ahead, in a shared-memory ring every role reads; loads the
//     two 128x64 Q tiles of a unit, then K_0, V_0, K_1, V_1, ... through an
//     8-slot ring of 16 KiB tiles (128-byte swizzle), each slot guarded by a
//     full/empty mbarrier.
//   * warps 1 and 3: MMA issuers for head 0 and head 1.  S_t = Q_t K_j^T
//     (M=128, N=128, K=64) into TMEM, and O_t += P_t V_j (M=128, N=64, K=128)
//     with P_t read from TMEM (A operand) and V_j from shared memory (MN-major
//     B operand).  Each warp runs its loop as a whole warp and issues from an
//     elect.sync lane: from a lone lane the same MMAs issued ~40% slower.
//   * warps 4..7 / 8..11: softmax of head 0 / head 1, one thread per query row.
//     Each reads its 128 scores from TMEM and at once hands the S columns back
//     (so the MMA for the next key tile overlaps this tile's softmax), applies
//     the causal mask on the diagonal tile, updates (m, d), and writes P (bf16)
//     to its own TMEM columns once the previous tile's PV has finished with
//     them; at the end it normalises O by d and stores the row.  A bf16 block
//     whose 128 rows all belong to the sequence goes out through a staging
//     tile per head (the Q tile's swizzled layout) and one bulk tensor store:
//     128 threads each storing a 128-byte row 8 KiB away from its neighbours'
//     held up every unit change by about 2,000 cycles.  Partial blocks and
//     fp32 output store their rows directly.
//   * warp 0 allocates / frees the 512 TMEM columns:
//       S_0 [0,128)  S_1 [128,256)  O_0 [256,320)  O_1 [320,384)  P_0 [384,448)  P_1 [448,512)
//     P has two bf16 per column.  Keeping P apart from S means a QK MMA never
//     waits for the PV MMA reading the previous P.
// Per head and key tile the only waits are: softmax(j) needs S(j), which the
// MMA issued when softmax(j-1) released S; it needs PV(j-1) done before it
// writes P(j) (by then long finished); the MMA needs S released and P written.
// The running maximum is only raised when a tile's maximum exceeds it by more
// than 8 (log2 units), so O is rescaled rarely; the final O / d is exact for
// any reference point, and P stays <= 2^8 which bf16 and fp32 hold easily.
// d accumulates the bf16-rounded P (the values the PV MMA multiplies), so the
// rounding of P perturbs the weights of a convex combination of V rows
// instead of scaling the output.
//
// Paged mode (template flag; chunked prefill against the paged KV cache): a
// sequence's query rows are the last n of its L cached tokens, so row i sits
// at position L - n + i and sees keys 0 .. L - n + i.  K/V tiles of 128 keys
// are gathered as 8 page slabs (2 KiB TMA copies, 8 per tile); a unit needs
// the key tiles up to its last row's position; the causal mask applies to
// every tile that crosses a row's last key; rows may see no key at all (more
// query rows than cached tokens), which the softmax guards.  In both modes V
// rows past the last needed key are zeroed before the last PV: stale or
// poisoned slots, or the next packed sequence's tokens, must not meet a zero
// weight inside the MMA (0 x NaN = NaN), so a sequence's output never depends
// on another sequence's values.
#include "common.cuh"
#include "prefill.h"
#include "rope.h"
#include "tcgen05.cuh"

#include <algorithm>
#include <atomic>

namespace sa {

// Unit counters for the dynamic deal: slot s holds {units handed out, CTAs
// finished}, and the last CTA of a launch zeroes it again.  Launches take the
// slots in turn, so two launches share one only if they run at the same time
// kSchedSlots launches apart.
constexpr int kSchedSlots = 1 << 16;
__device__ unsigned g_prefill_sched[kSchedSlots][2];

namespace {

constexpr int kTile = kPrefillTileRows;
constexpr int kD = 64;
constexpr int kTileBytes = kTile * kD * 2;  // 16 KiB
constexpr int kSlots = 8;
constexpr int kThreads = 384;
// Warp roles 0..3: the TMA producer sits on the scheduler (warp % 4) that has
// no MMA issuer, so its copy instructions do not queue behind an issuer's.
constexpr int kProducerWarp = 2, kTmemWarp = 0;
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }   // S_t
__host__ __device__ constexpr uint32_t col_o(int t) { return t ? 320u : 256u; }  // O_t
__host__ __device__ constexpr uint32_t col_p(int t) { return t ? 448u : 384u; }  // P_t
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, false, true);
constexpr float kRescaleThreshold = 8.f;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                                // 2 Q tiles
constexpr int kOffRing = kOffQ + 2 * kTileBytes;         // kSlots K/V tiles
constexpr int kOffBar = kOffRing + kSlots * kTileBytes;  // mbarriers
constexpr int kUnitRing = 16;  // units published by the producer, read by every role
constexpr int kNumBars = 2 + 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 2 + 2 + kUnitRing;
constexpr int kBarBytes = 384;
constexpr int kOffMisc = kOffBar + kBarBytes;
constexpr int kOffSeq = kOffMisc + 64 + 4 * kUnitRing;
constexpr int kSeqArrays = 6;
// bf16 output of a whole 128-row block leaves through a staging tile per head
// (the Q tile's layout: 128-byte swizzle) and one bulk tensor store
constexpr int kOffStage = (kOffSeq + kSeqArrays * kPrefillMaxBatch * 4 + 1023) / 1024 * 1024;
constexpr int kSmemBytes = kOffStage + 2 * kTileBytes + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
// Rotary mode adds a table of cos/sin(r * f_i) for the 128 rows of a query
// tile and the 32 planes ([plane][row] float2: conflict-free row reads), and
// the planes' fixed-point turn increments.
constexpr int kOffRopeLo = kOffSeq + kSeqArrays * kPrefillMaxBatch * 4;
constexpr int kOffRopeTurn = kOffRopeLo + 32 * kTile * 8;
constexpr int kSmemBytesRope = kOffRopeTurn + 32 * 8 + 1024;
static_assert(kSmemBytesRope <= 227 * 1024, "shared memory of the rotary mode");
constexpr int kPage = 16;
constexpr int kSlabBytes = kPage * kD * 2;  // one (page, kv head) slab: 2 KiB
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

struct Bars {
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* slot_full;
  uint64_t* slot_empty;
  uint64_t* s_full;  // [2] MMA -> softmax: scores of the next tile ready
  uint64_t* s_free;  // [2] softmax -> MMA: scores read, S columns free
  uint64_t* p_full;  // [2] softmax -> MMA: P written (and O rescaled)
  uint64_t* o_done;  // [2] MMA -> softmax: a PV (hence every earlier MMA) finished
  uint64_t* drain;
  uint64_t* q_ready;  // [2] rotary mode, softmax -> MMA: the unit's Q tile of the head is rotated
};

// Walks the list of query blocks in schedule order: sequences longest first,
// and within a sequence its query blocks from the last (most key tiles) to the
// first.  Consecutive blocks, which concurrently running CTAs take, then read
// the same sequence's keys and values, so those stay in L2 (level by level
// across all sequences, the keys of every long sequence were live at once and
// re-read from HBM).  Sequences are sorted by block count.
struct Cursor {
  const int* nqb;  // sorted, descending
  int batch;
  int seq, start;  // current sequence (sorted index) and its first block's index
  __device__ void init(const int* nqb_sorted, int b) {
    nqb = nqb_sorted;
    batch = b;
    seq = 0;
    start = 0;
  }
  // qbl must not decrease between calls.  Returns the sorted sequence index.
  __device__ int seek(int qbl, int& qb) {
    while (seq < batch - 1 && qbl >= start + nqb[seq]) {
      start += nqb[seq];
      ++seq;
    }
    qb = nqb[seq] - 1 - (qbl - start);
    return seq;
  }
};

struct Unit {
  int seq;  // sorted index
  int qb;   // query block within the sequence
  int g;    // kv head
  int pair; // pair of query heads within the group
};

// Unit index (schedule order) -> unit.  Indices must not decrease between calls.
__device__ __forceinline__ void decode_unit(int ui, int pairs_per_group, int hkv, Cursor& cur, Unit& u) {
  u.pair = ui % pairs_per_group;
  const int rest = ui / pairs_per_group;
  u.g = rest % hkv;
  u.seq = cur.seek(rest / hkv, u.qb);
}

// The k-th unit index of this CTA under the static deal (serpentine), or -1.
__device__ __forceinline__ int static_unit(int k, int total) {
  const int c = blockIdx.x, G = gridDim.x;
  const long long idx = (long long)k * G + ((k & 1) ? (G - 1 - c) : c);
  return idx < total ? (int)idx : -1;
}

// Paged mode: keys a unit needs, [0, kend): up to the position of its last
// query row (may be <= 0 when every row sits before the cache start).
__device__ __forceinline__ int paged_kend(int kv_len, int q_len, int qb) {
  return kv_len - q_len + min(q_len, (qb + 1) * kTile);
}

// Rotary encoding of query row r of a Q tile in shared memory (128-byte swizzle:
// 16-byte chunk c of row r at chunk c ^ (r % 8)), in place.  Row r is token
// qb * 128 + r of its sequence, at that position: cos/sin of the position's
// multiple of 128 come from lane `plane` of the warp (ch, sh), those of r from
// the table lo[plane * 128 + r]; the angles are added, the bias added and the
// plane rotated exactly as the rotary pass does it (rope.h), then rounded to bf16.
__device__ __forceinline__ void rope_q_row(uint8_t* tile, int r, const __nv_bfloat16* bias_row, float ch, float sh,
                                           const float2* lo, float af) {
  uint4* row = reinterpret_cast<uint4*>(tile + r * 128);
  const uint4* b4 = reinterpret_cast<const uint4*>(bias_row);
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // chunk c holds dims 8c..8c+7, chunk c + 4 their plane partners
    const uint4 v1 = row[c ^ (r & 7)], v2 = row[(c + 4) ^ (r & 7)];
    const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w}, w2[4] = {v2.x, v2.y, v2.z, v2.w};
    uint32_t b1[4] = {0, 0, 0, 0}, b2[4] = {0, 0, 0, 0};
    if (bias_row) {
      const uint4 u1 = __ldg(b4 + c), u2 = __ldg(b4 + c + 4);
      b1[0] = u1.x; b1[1] = u1.y; b1[2] = u1.z; b1[3] = u1.w;
      b2[0] = u2.x; b2[1] = u2.y; b2[2] = u2.z; b2[3] = u2.w;
    }
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float y1[2], y2[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int plane = 8 * c + 2 * e + k;
        float x1 = k ? bf16x2_hi(w1[e]) : bf16x2_lo(w1[e]);
        float x2 = k ? bf16x2_hi(w2[e]) : bf16x2_lo(w2[e]);
        if (bias_row) {
          x1 = __fadd_rn(x1, k ? bf16x2_hi(b1[e]) : bf16x2_lo(b1[e]));
          x2 = __fadd_rn(x2, k ? bf16x2_hi(b2[e]) : bf16x2_lo(b2[e]));
        }
        const float chp = __shfl_sync(0xffffffffu, ch, plane), shp = __shfl_sync(0xffffffffu, sh, plane);
        const float2 l = lo[plane * kTile + r];
        float cc, sn;
        rope_angle_add(chp, shp, l.x, l.y, cc, sn);
        const float cs = __fmul_rn(cc, af), ss = __fmul_rn(sn, af);
        y1[k] = rope_first(x1, x2, cs, ss);
        y2[k] = rope_second(x1, x2, cs, ss);
      }
      o1[e] = pack_bf16x2(y1[0], y1[1]);
      o2[e] = pack_bf16x2(y2[0], y2[1]);
    }
    row[c ^ (r & 7)] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    row[(c + 4) ^ (r & 7)] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  }
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const PrefillParams& p,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;  // fast path: already complete
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, p.err, kErrPrefill, p.wait_limit_ns)) return true;
  *abort_flag = 1;
  return false;
}

}  // namespace

template <bool kPaged, bool kRopeQ>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                   const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Bars bars;
  bars.q_full = bar_base;
  bars.q_empty = bar_base + 1;
  bars.slot_full = bar_base + 2;
  bars.slot_empty = bars.slot_full + kSlots;
  bars.s_full = bars.slot_empty + kSlots;
  bars.s_free = bars.s_full + 2;
  bars.p_full = bars.s_free + 2;
  bars.o_done = bars.p_full + 2;
  bars.drain = bars.o_done + 2;
  bars.q_ready = bars.drain + 1;
  uint64_t* stg_full = bars.q_ready + 2;  // [2] softmax rows of a block written to the staging tile
  uint64_t* unit_ready = stg_full + 2;    // [kUnitRing] producer -> all: unit k published in unit_ring[k % kUnitRing]
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + kOffMisc + 64);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* total_qblocks = reinterpret_cast<int*>(smem + kOffMisc + 8);
  // tail-V zeroings head 0's MMA warp has finished (head 1's waits on the count, which
  // cannot alias the way a phase bit could when head 0 runs a unit ahead)
  volatile int* zeroed_count = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  int* seq_start = reinterpret_cast<int*>(smem + kOffSeq);   // sorted
  int* seq_len = seq_start + kPrefillMaxBatch;                // sorted
  int* seq_nqb = seq_len + kPrefillMaxBatch;                  // sorted, descending
  int* tmp_nqb = seq_nqb + kPrefillMaxBatch;                  // by batch index
  int* seq_kv = tmp_nqb + kPrefillMaxBatch;                   // sorted; paged mode: cached tokens
  int* seq_id = seq_kv + kPrefillMaxBatch;                    // sorted; paged mode: batch index
  float2* rope_lo = reinterpret_cast<float2*>(smem + kOffRopeLo);                    // rotary mode
  unsigned long long* rope_turn = reinterpret_cast<unsigned long long*>(smem + kOffRopeTurn);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.batch;

  // ---- per-CTA schedule table: sequences sorted by query-block count
  for (int i = tid; i < B; i += kThreads) {
    const int len = max(0, __ldg(p.cu_seqlens + i + 1) - __ldg(p.cu_seqlens + i));
    tmp_nqb[i] = (len + kTile - 1) / kTile;
  }
  if (kRopeQ && tid < 32) rope_turn[tid] = rope_turn_increment(__ldg(p.inv_freq + tid));
  if (tid == 0) {
    mbar_init(bars.q_full, 1);
    mbar_init(bars.q_empty, 2);  // released by both MMA warps
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bars.slot_full + i, 1);
      mbar_init(bars.slot_empty + i, 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_full + t, 1);
      mbar_init(bars.s_free + t, 128);  // every softmax thread of the head arrives
      mbar_init(bars.p_full + t, 128);
      mbar_init(bars.o_done + t, 1);
    }
    mbar_init(bars.drain, 2);
    mbar_init(bars.q_ready, 128);
    mbar_init(bars.q_ready + 1, 128);
    mbar_init(stg_full, 128);
    mbar_init(stg_full + 1, 128);
    for (int i = 0; i < kUnitRing; ++i) mbar_init(unit_ready + i, 1);
    *abort_flag = 0;
    *zeroed_count = 0;
    fence_barrier_init();
  }
  if (warp == kTmemWarp) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (kRopeQ) {  // cos/sin of r * f for the 128 rows of a tile, every plane
    for (int e = tid; e < 32 * kTile; e += kThreads) {
      float c, sn;
      rope_phase_cos_sin(e % kTile, rope_turn[e / kTile], c, sn);
      rope_lo[e] = make_float2(c, sn);
    }
  }
  for (int i = tid; i < B; i += kThreads) {
    const int mine = tmp_nqb[i];
    int rank = 0, total = 0;
    for (int j = 0; j < B; ++j) {
      const int o = tmp_nqb[j];
      rank += (o > mine) || (o == mine && j < i);
      total += o;
    }
    const int st = __ldg(p.cu_seqlens + i);
    seq_start[rank] = st;
    seq_len[rank] = max(0, __ldg(p.cu_seqlens + i + 1) - st);
    seq_nqb[rank] = mine;
    if constexpr (kPaged) {
      seq_kv[rank] = min(max(0, __ldg(p.kv_len + i)), p.stride * kPage);  // never past the page-table row
      seq_id[rank] = i;
    }
    if (i == 0) *total_qblocks = total;
  }
  tc_fence_after();
  __syncthreads();
  const uint32_t tmem = *tmem_holder;
  const int pairs_per_group = (p.group + 1) / 2;
  const long long total_ll = (long long)(*total_qblocks) * p.hkv * pairs_per_group;
  const int total_units = (int)min(total_ll, (long long)0x7fffffff);
  Cursor cur;
  cur.init(seq_nqb, B);
  // Unit k of this CTA (every role reads it from the ring): 1 got one, 0 none left, -1 aborted.
  auto unit_at = [&](int k, Unit& v) -> int {
    if (!__all_sync(0xffffffffu, wait_or_abort(unit_ready + (k % kUnitRing), (k / kUnitRing) & 1, p, abort_flag)))
      return -1;
    const int idx = unit_ring[k % kUnitRing];
    if (idx < 0) return 0;
    decode_unit(idx, pairs_per_group, p.hkv, cur, v);
    return 1;
  };

  uint8_t* q_tile[2] = {smem + kOffQ, smem + kOffQ + kTileBytes};
  uint8_t* ring = smem + kOffRing;

  if (warp == kProducerWarp) {
    // ================================================================ TMA producer
    // The whole warp runs the loop and waits; one elected lane issues the copies.
    if (elect_one()) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const uint64_t pol_stream = l2_policy_evict_first();
    uint32_t ring_i = 0;
    Unit u;
    bool ok = true;
    // The CTA's k-th unit: the next one of the launch (dynamic deal) or the static one,
    // published to every role one unit ahead (so the MMA warps know the next unit while
    // they work on this one).
    auto publish = [&](int kk) -> int {
      int v = 0;
      if (lane == 0) {
        if (p.sched_slot >= 0) {
          v = (int)atomicAdd(&g_prefill_sched[p.sched_slot][0], 1u);
          if (v >= total_units) v = -1;
        } else {
          v = static_unit(kk, total_units);
        }
        unit_ring[kk % kUnitRing] = v;
        mbar_arrive(unit_ready + (kk % kUnitRing));  // release: the ring entry is visible to its waiters
      }
      return __shfl_sync(0xffffffffu, v, 0);
    };
    int idx_next = publish(0);
    for (int k = 0; ok; ++k) {
      const int idx = idx_next;
      if (idx < 0) break;
      idx_next = publish(k + 1);
      decode_unit(idx, pairs_per_group, p.hkv, cur, u);
      if (k > 0 && !(ok = __all_sync(0xffffffffu, wait_or_abort(bars.q_empty, (k - 1) & 1, p, abort_flag)))) break;
      const int t0 = seq_start[u.seq] + u.qb * kTile;
      const int hA = u.g * p.group + 2 * u.pair;
      const int hB = (2 * u.pair + 1 < p.group) ? hA + 1 : hA;
      if (!p.withhold_copies && elect_one()) {
        mbar_arrive_expect_tx(bars.q_full, 2 * kTileBytes);
        tma_load_3d_hint(q_tile[0], &qmap, bars.q_full, 0, hA, t0, pol_stream);
        tma_load_3d_hint(q_tile[1], &qmap, bars.q_full, 0, hB, t0, pol_stream);
      }
      const int kv0 = seq_start[u.seq];
      int n = u.qb + 1, kend = 0;
      const int32_t* table_row = nullptr;
      if constexpr (kPaged) {
        kend = paged_kend(seq_kv[u.seq], seq_len[u.seq], u.qb);
        n = max(1, (kend + kTile - 1) / kTile);  // at least one (possibly empty) tile: the unit still runs
        table_row = p.page_table + (size_t)seq_id[u.seq] * p.stride;
      }
      if constexpr (kPaged) {
        // Per tile: both slots first, then its K and V slabs from 16 lanes in one go (lanes
        // 0..7 K, 8..15 V).  Copies issued lane-parallel: from one lane the copy issue alone
        // paced the kernel.  Page ids are read one tile ahead (lanes 0..7).
        auto slabs = [&](int j) { return min(kTile / kPage, max(0, (kend - j * kTile + kPage - 1) / kPage)); };
        int next_page = lane < slabs(0) ? __ldg(table_row + lane) : 0;
        for (int j = 0; j < n && ok; ++j) {
          const int np = slabs(j), page = next_page;
          if (j + 1 < n && lane < slabs(j + 1)) next_page = __ldg(table_row + (j + 1) * (kTile / kPage) + lane);
          const uint32_t ks = ring_i % kSlots, vs = (ring_i + 1) % kSlots;
          if (ring_i >= kSlots &&
              !(ok = __all_sync(0xffffffffu,
                                wait_or_abort(bars.slot_empty + ks, ((ring_i / kSlots) - 1) & 1, p, abort_flag))))
            break;
          if (ring_i + 1 >= kSlots &&
              !(ok = __all_sync(0xffffffffu, wait_or_abort(bars.slot_empty + vs, (((ring_i + 1) / kSlots) - 1) & 1,
                                                           p, abort_flag))))
            break;
          if (!p.withhold_copies) {
            if (elect_one()) {
              mbar_arrive_expect_tx(bars.slot_full + ks, np * kSlabBytes);
              mbar_arrive_expect_tx(bars.slot_full + vs, np * kSlabBytes);
            }
            __syncwarp();
            const int sl = lane & 7;
            const bool is_v = lane >= 8;
            const int pg = __shfl_sync(0xffffffffu, page, sl);
            const uint32_t slot = is_v ? vs : ks;
            if (lane < 16 && sl < np)
              tma_load_2d(ring + slot * kTileBytes + sl * kSlabBytes, is_v ? &vmap : &kmap, bars.slot_full + slot, 0,
                          (pg * p.hkv + u.g) * kPage);
          }
          ring_i += 2;
        }
      } else {
        for (int j = 0; j < n && ok; ++j) {
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t slot = ring_i % kSlots;
            if (ring_i >= kSlots &&
                !(ok = __all_sync(0xffffffffu,
                                  wait_or_abort(bars.slot_empty + slot, ((ring_i / kSlots) - 1) & 1, p, abort_flag))))
              break;
            if (!p.withhold_copies && elect_one()) {
              mbar_arrive_expect_tx(bars.slot_full + slot, kTileBytes);
              tma_load_3d(ring + slot * kTileBytes, kv ? &vmap : &kmap, bars.slot_full + slot, 0, u.g,
                          kv0 + j * kTile);
            }
            ++ring_i;
          }
        }
      }
    }
    if (__any_sync(0xffffffffu, *abort_flag) && elect_one()) {
      // let copies already in flight land before the CTA can exit
      for (uint32_t i = ring_i > kSlots ? ring_i - kSlots : 0; i < ring_i; ++i)
        mbar_wait(bars.slot_full + (i % kSlots), (i / kSlots) & 1, p.err, kErrPrefill, 10000000ull);
    }
  } else if (warp == 1 || warp == 3) {
    // ================================================================ MMA issuers
    // Warp 1 issues head 0's MMAs, warp 3 head 1's: each head's S, P and O are
    // touched only by its own warp's MMAs, whose order tcgen05 keeps; the K/V
    // slots and the Q tiles are released by a commit from each warp.  The whole
    // warp runs the loop and waits; one elected lane issues (warp-uniform operands).
    const int t = warp == 1 ? 0 : 1;
    uint32_t ring_i = 0, pph = 0, fph = 0;
    bool first_qk = true;
    const uint64_t dq = smem_desc_sw128(smem_addr(q_tile[t]));
    const uint64_t dring = smem_desc_sw128(smem_addr(ring));
    // descriptor of ring slot i: the start-address field advances 16 KiB >> 4 per slot
    auto slot_desc = [&](uint32_t i) { return dring + (uint64_t)((i % kSlots) * (kTileBytes >> 4)); };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p, abort_flag));
    };
    const uint32_t d_s = tmem + col_s(t), d_o = tmem + col_o(t), a_p = tmem + col_p(t);
    int zeroings = 0;  // tail-V zeroings met so far
    Unit u, un;
    int got = unit_at(0, u), got_next = 0;
    bool ok = got >= 0;
    for (int k = 0; ok && got > 0; ++k, u = un, got = got_next) {
      int n = u.qb + 1, kend = 0;
      if constexpr (kPaged) {
        kend = paged_kend(seq_kv[u.seq], seq_len[u.seq], u.qb);
        n = max(1, (kend + kTile - 1) / kTile);
      }
      // rotary mode: the softmax warps rotate the landed tile first
      if (!(ok = wait_all(kRopeQ ? bars.q_ready + t : bars.q_full, k & 1))) break;
      // K_0 -> S (once the softmax has released S)
      if (!(ok = wait_all(bars.slot_full + ring_i % kSlots, (ring_i / kSlots) & 1))) break;
      if (!first_qk) {
        if (!(ok = wait_all(bars.s_free + t, fph))) break;
        fph ^= 1;
      }
      first_qk = false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dk0 = slot_desc(ring_i);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_ss(d_s, dq + 2 * kk, dk0 + 2 * kk, kIdescQK, kk > 0);
        umma_commit(bars.s_full + t);
        umma_commit(bars.slot_empty + ring_i % kSlots);
        if (n == 1) umma_commit(bars.q_empty);
      }
      // the next unit (published before this unit's Q tiles were loaded), read here, where
      // the warp has only waits ahead of it
      got_next = unit_at(k + 1, un);
      if (!(ok = got_next >= 0)) break;
      ++ring_i;
      // keys of the unit's last tile it needs (only the last tile can end early)
      const int valid_last = (kPaged ? kend : seq_len[u.seq]) - (n - 1) * kTile;
      for (int j = 0; j < n; ++j) {
        const uint32_t vi = ring_i, ki = ring_i + 1;
        const bool more = j + 1 < n;
        if (more) {  // scores of tile j+1 as soon as the softmax has read tile j's
          if (!(ok = wait_all(bars.slot_full + ki % kSlots, (ki / kSlots) & 1))) break;
          if (!(ok = wait_all(bars.s_free + t, fph))) break;
          fph ^= 1;
          tc_fence_after();
          if (elect_one()) {
            const uint64_t dk = slot_desc(ki);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_ss(d_s, dq + 2 * kk, dk + 2 * kk, kIdescQK, kk > 0);
            umma_commit(bars.s_full + t);
            umma_commit(bars.slot_empty + ki % kSlots);
            if (j + 2 == n) umma_commit(bars.q_empty);
          }
        }
        if (!(ok = wait_all(bars.slot_full + vi % kSlots, (vi / kSlots) & 1))) break;
        if (!(ok = wait_all(bars.p_full + t, pph))) break;
        pph ^= 1;
        tc_fence_after();
        {
          // keys of this tile the unit needs: paged mode, up to its last row's position;
          // contiguous mode, up to the sequence end (only the last query block's
          // diagonal tile can end early, when the length is not a multiple of 128)
          const int valid = valid_last;
          if (j == n - 1 && valid < kTile) {
            // rows past them (slabs not copied, slots past the sequence end, or the next
            // packed sequence's tokens) enter the product with weight 0, and 0 x NaN is NaN:
            // head 0's warp zeroes them (fence for the tensor core's reads); head 1's waits.
            ++zeroings;
            if (t == 0) {
              uint4* vrows = reinterpret_cast<uint4*>(ring + (vi % kSlots) * kTileBytes);
              for (int i = max(0, valid) * 8 + lane; i < kTile * 8; i += 32) vrows[i] = make_uint4(0, 0, 0, 0);
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              __syncwarp();
              __threadfence_block();
              if (lane == 0) *zeroed_count = zeroings;
            } else {
              bool seen = *zeroed_count >= zeroings;
              const uint64_t t0 = seen ? 0 : global_timer_ns();
              while (!seen && !*abort_flag) {
                __nanosleep(64);
                seen = *zeroed_count >= zeroings;
                if (!seen && global_timer_ns() - t0 > p.wait_limit_ns) {
                  atomicOr(p.err, kErrPrefill);
                  *abort_flag = 1;
                }
              }
              if (!(ok = __all_sync(0xffffffffu, seen))) break;
              __threadfence_block();
            }
          }
        }
        if (elect_one()) {
          const uint64_t dv = slot_desc(vi);
          if (j > 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_ts(d_o, a_p + 8 * kk, dv + 128 * kk, kIdescPV, 1);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_ts(d_o, a_p + 8 * kk, dv + 128 * kk, kIdescPV, kk > 0);
          }
          umma_commit(bars.o_done + t);
          umma_commit(bars.slot_empty + vi % kSlots);
        }
        ring_i += more ? 2 : 1;
      }
    }
    // every MMA issued by these warps must finish before TMEM is released
    if (elect_one()) umma_commit(bars.drain);
    __syncwarp();
    mbar_wait(bars.drain, 0, p.err, kErrPrefill, p.wait_limit_ns);
  } else if (warp >= 4) {
    // ================================================================ softmax
    const int t = (warp - 4) >> 2;         // which query tile (head of the pair)
    const int quad = warp & 3;             // TMEM lane quarter of this warp
    const int r = quad * 32 + lane;        // query row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const bool stg_issuer = quad == 0 && lane == 0;  // issues and waits for this head's bulk stores
    uint32_t stg_phase = 0;
    const uint32_t s_addr = tmem + lane_off + col_s(t);
    const uint32_t o_addr = tmem + lane_off + col_o(t);
    const uint32_t p_addr = tmem + lane_off + col_p(t);
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    uint32_t sph = 0, oph = 0;
    // Rotary mode: rotate this thread's row of the head's Q tile of unit kk once it
    // has landed, then hand the tile to the MMA warp.
    auto rotate_unit = [&](const Unit& un, int kk) -> bool {
      if (!__all_sync(0xffffffffu, wait_or_abort(bars.q_full, kk & 1, p, abort_flag))) return false;
      const int hA = un.g * p.group + 2 * un.pair;
      const int hT = (t && 2 * un.pair + 1 < p.group) ? hA + 1 : hA;  // the head the producer loaded
      float ch, sh;
      rope_phase_cos_sin(un.qb * kTile, rope_turn[lane], ch, sh);
      rope_q_row(q_tile[t], r, p.q_bias ? p.q_bias + (size_t)hT * kD : nullptr, ch, sh, rope_lo, p.attn_factor);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor core reads
      mbar_arrive(bars.q_ready + t);
      return true;
    };
    Unit u;
    bool ok = true;
    int got = 0;
    for (int k = 0; ok && (got = unit_at(k, u)) > 0; ++k) {
      if constexpr (kRopeQ) {
        if (k == 0 && !(ok = rotate_unit(u, 0))) break;
      }
      // the previous block has left this head's staging tile before the unit starts: every
      // warp of the head writes the tile again only after this unit's last PV, which waits
      // for this thread's arrivals
      if (stg_issuer) bulk_wait_read0();
      int n = u.qb + 1;
      int lim0 = 0;     // paged mode: keys visible to this row, counted from the unit's first key tile
      int j_mask = 0;   // paged mode: first key tile that crosses the last key of some row of this warp
      if constexpr (kPaged) {
        const int kend = paged_kend(seq_kv[u.seq], seq_len[u.seq], u.qb);
        n = max(1, (kend + kTile - 1) / kTile);
        lim0 = seq_kv[u.seq] - seq_len[u.seq] + u.qb * kTile + r + 1;
        j_mask = __reduce_min_sync(0xffffffffu, (unsigned)max(0, lim0) / kTile);
      }
      const int h = u.g * p.group + 2 * u.pair + t;
      const bool head_ok = 2 * u.pair + t < p.group;
      float m = head_ok ? __ldg(p.sinks + h) * kLog2e : -INFINITY;  // sink-seeded state
      float d = 1.f;
      for (int j = 0; j < n; ++j) {
        ok = wait_or_abort(bars.s_full + t, sph, p, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        sph ^= 1;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128(s_addr, sr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bars.s_free + t);  // the next tile's QK may overwrite S now
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        if constexpr (kPaged) {
          if (j >= j_mask) {  // warp-uniform: the tiles before it are fully visible to every row
            const int lim = lim0 - j * kTile;  // key c of this tile is visible iff c < lim
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim) s[c] = -INFINITY;
          }
        } else {
          if (j == n - 1) {  // diagonal tile: key c is visible to row r iff c <= r
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > r) s[c] = -INFINITY;
          }
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < 124; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        mx0 = fmax3(mx0, s[124], s[125]);
        mx1 = fmax3(mx1, s[126], s[127]);
        const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
        const bool need = m_tile > m + kRescaleThreshold;
        const bool any_need = __any_sync(0xffffffffu, need);
        const float m_new = need ? m_tile : m;
        // paged mode: a row may have seen neither sink nor key yet (-inf); subtract 0 then
        const float m_ref = (kPaged && m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = fast_exp2(m - m_ref);  // 1 unless this row's maximum moved
        const float2 neg_m2 = make_float2(-m_ref, -m_ref);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), sl2x2, neg_m2);
          pk[i] = pack_bf16x2(fast_exp2(x.x), fast_exp2(x.y));
          // the normaliser sums the same bf16-rounded weights the PV MMA uses
          acc[i & 3] = add_bf16x2_f32x2(acc[i & 3], pk[i]);
        }
        if (j > 0) {  // PV(j-1) still reads P and accumulates into O until it is done
          ok = wait_or_abort(bars.o_done + t, oph, p, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          oph ^= 1;
          tc_fence_after();
          if (any_need) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
              uint32_t ob[16];
              tmem_ld16(o_addr + c0, ob);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) ob[e] = __float_as_uint(__uint_as_float(ob[e]) * alpha);
              tmem_st16(o_addr + c0, ob);
            }
          }
        }
        tmem_st64(p_addr, pk);
        tmem_st_wait();
        const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
        d = d * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
        m = m_new;
        tc_fence_before();
        mbar_arrive(bars.p_full + t);
      }
      if (!ok) break;
      if constexpr (kRopeQ) {
        // rotate the next unit's tile (loaded once this unit's last QK was issued) while
        // this unit's last PV runs; kept out of the tile loop, whose every iteration ran
        // slower with it inside
        Unit un;
        const int got_next = unit_at(k + 1, un);
        if (!(ok = got_next >= 0) || (got_next > 0 && !(ok = rotate_unit(un, k + 1)))) break;
      }
      // ---- epilogue: wait for the last PV, normalise, store
      ok = wait_or_abort(bars.o_done + t, oph, p, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      oph ^= 1;
      tc_fence_after();
      uint32_t ob[64];
      tmem_ld64(o_addr, ob);
      tmem_ld_wait();
      const int row_tok = u.qb * kTile + r;
      const int tok = seq_start[u.seq] + row_tok;  // checked against T too: cu_seqlens is not trusted
      const int tok0 = seq_start[u.seq] + u.qb * kTile;
      // a whole block of a head (uniform over the head's 128 threads) leaves by one bulk store
      const bool bulk = !kRopeQ && !p.out_f32 && head_ok && (u.qb + 1) * kTile <= seq_len[u.seq] && tok0 >= 0 &&
                        tok0 + kTile <= p.total_tokens;
      if (bulk) {
        const float inv = (!kPaged || d > 0.f) ? 1.f / d : 0.f;  // paged: no key and no sink gives 0
        uint4* rowp = reinterpret_cast<uint4*>(smem + kOffStage + t * kTileBytes + r * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(ob[8 * i + 0]) * inv, __uint_as_float(ob[8 * i + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(ob[8 * i + 2]) * inv, __uint_as_float(ob[8 * i + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(ob[8 * i + 4]) * inv, __uint_as_float(ob[8 * i + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(ob[8 * i + 6]) * inv, __uint_as_float(ob[8 * i + 7]) * inv);
          rowp[i ^ (r & 7)] = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> bulk copy reads
        mbar_arrive(stg_full + t);
        if (p.lse) p.lse[(size_t)tok * p.hq + h] = (!kPaged || d > 0.f) ? (m + __log2f(d)) * kLn2 : -INFINITY;
        if (stg_issuer) {
          ok = wait_or_abort(stg_full + t, stg_phase, p, abort_flag);
          stg_phase ^= 1;
          if (ok) {
            tma_store_3d(&omap, smem + kOffStage + t * kTileBytes, 0, h, tok0);
            bulk_commit();
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      } else if (head_ok && row_tok < seq_len[u.seq] && tok >= 0 && tok < p.total_tokens) {
        const float inv = (!kPaged || d > 0.f) ? 1.f / d : 0.f;  // paged: no key and no sink gives 0
        const size_t row = (size_t)tok * p.hq + h;
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * kD);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            dst[i] = make_float4(__uint_as_float(ob[4 * i]) * inv, __uint_as_float(ob[4 * i + 1]) * inv,
                                 __uint_as_float(ob[4 * i + 2]) * inv, __uint_as_float(ob[4 * i + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row * kD);
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
        if (p.lse) p.lse[row] = (!kPaged || d > 0.f) ? (m + __log2f(d)) * kLn2 : -INFINITY;
      }
    }
  }

  // ---- teardown
  if (warp >= 4 && (warp & 3) == 0 && lane == 0) bulk_wait0();  // bulk stores complete before exit
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && p.sched_slot >= 0) {
    // the last CTA of the launch zeroes its counters for the next launch (every unit
    // fetch of every CTA precedes its count here)
    __threadfence();
    if (atomicAdd(&g_prefill_sched[p.sched_slot][1], 1u) == gridDim.x - 1) {
      g_prefill_sched[p.sched_slot][0] = 0;
      g_prefill_sched[p.sched_slot][1] = 0;
      __threadfence();
    }
  }
  if (warp == kTmemWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t prefill_configure() {
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytesRope);
}

// Counter slot of a launch, or -1 for the static deal: a launch captured into a
// graph keeps the static deal, since every replay of the graph (and every
// instance made from it) would share the one slot baked into it.
static int prefill_sched_slot(cudaStream_t stream) {
  static std::atomic<unsigned> next{0};
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return -1;
  return (int)(next.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
}

cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& omap, const PrefillParams& params, int num_sms, bool paged,
                           cudaStream_t stream) {
  PrefillParams p = params;
  p.sched_slot = prefill_sched_slot(stream);
  const long long ppg = (p.group + 1) / 2;
  const long long upper = ppg * p.hkv * ((long long)(p.total_tokens + kTile - 1) / kTile + p.batch);
  const int grid = (int)std::min<long long>(std::max(1, num_sms), std::max(1LL, upper));
  if (paged)
    prefill_kernel<true, false><<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, omap, p);
  else if (p.inv_freq)
    prefill_kernel<false, true><<<grid, kThreads, kSmemBytesRope, stream>>>(qmap, kmap, vmap, omap, p);
  else
    prefill_kernel<false, false><<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, omap, p);
  return cudaGetLastError();
}

}  // namespace sa
