// Split-KV paged decode with a per-head sink logit (sm_103a).
//
// Method: Perplexity, "GPT-OSS on day 0", section "Sink Attention".  The key
// length of each sequence is cut into chunks of whole pages; every chunk keeps
// the online-softmax state (running max m, running scale d, weighted value sum)
// and only the first chunk's state starts from the head's sink (m = sink,
// d = 1).  A second kernel combines the chunks' (m, d, acc) triples.
//
// Work decomposition: one CTA per (chunk, kv head, sequence).  The CTA holds
// every query row that reads the kv head -- the G = Hq/Hkv query heads of the
// group times the n new tokens of the sequence (n = 1 for plain decode; n > 1
// for multi-token decode, where new token t sits at position L - n + t and
// sees keys 0..L - n + t) -- so every page of K/V is read from HBM exactly
// once.  Row rho = t*G + (h mod G), at most 16 rows (one MMA row tile; more
// rows go to the tensor-core kernel of decode_tc.cu).  Four warps; warp w
// takes pages w, w+4, ... of the chunk and streams each (page, kv head) slab
// -- 16 tokens x 64 dims x bf16 = 2 KiB of K and 2 KiB of V, contiguous in the
// [page, kv_head, slot, dim] layout -- into its own two shared-memory stages
// with 16-byte asynchronous copies (cp.async), page k + 2 in flight while page
// k is computed.  For one page the warp computes S = Q K^T (16 rows, padded;
// 16 tokens) and O += P V with warp-level bf16 MMAs (m16n8k16, fp32
// accumulate) and the online softmax in registers.  No wait in this kernel
// depends on another warp: a warp only waits for its own copies.
// The four warps' states are merged in shared memory; with a single chunk
// the CTA writes the normalised output directly, otherwise its partial
// state.  At 16 rows the work is at most 16 flop per byte of K/V, well
// within what the warp-level MMAs sustain at full HBM bandwidth.
//
// Fragment layouts (m16n8k16): lane = 4*r + qd.  The head dimension is used in
// a permuted order that is the same for Q and K (a dot product does not care),
// chosen so that each lane reads 32 contiguous bytes of a K row; the output
// dimension is permuted so that each lane reads 16 contiguous bytes of a V row
// and ends up owning 16 contiguous output dimensions.  Slabs are stored with a
// 128-byte swizzle (16-byte chunk c of row t at chunk c ^ (t % 8)), so every
// shared load below is free of bank conflicts.
#include "common.cuh"
#include "decode.h"
#include "rope.h"

namespace sa {

namespace {

constexpr int kD = 64;
constexpr int kPage = 16;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kStagesPerWarp = 2;  // pages each warp has in flight
constexpr int kStages = kConsumerWarps * kStagesPerWarp;
constexpr int kSlabBytes = kPage * kD * 2;      // 2048
constexpr int kStageBytes = 2 * kSlabBytes;     // K + V
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kRows = 16;                       // MMA rows of one row tile
// merge scratch per warp: m[16], d[16], o[16][64]
constexpr int kScratchFloatsPerWarp = kRows * 2 + kRows * kD;
static_assert(kConsumerWarps * kScratchFloatsPerWarp * 4 <= kRingBytes, "merge scratch aliases the ring");

// 16-byte asynchronous copy global -> shared; src_bytes 0 writes zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void chunk_range(const DecodeParams& p, int L, int s, int& n, int& pg0, int& pg1) {
  const int npages = (L + kPage - 1) / kPage;
  n = decode_num_chunks(npages, p.num_splits, p.split_pages, p.max_splits);
  const int chunk = npages > 0 ? (npages + n - 1) / n : 0;
  pg0 = s * chunk;
  pg1 = min(npages, pg0 + chunk);
}

// Sixteen dims [16qd, 16qd+16) of the query row (new token t, head h) as packed
// bf16 pairs.  With the rotary encoding on, the row's bias is added and the
// dims rotated against their plane partners (dim i pairs with i +- 32, the
// other half of the row), with the same roundings as the rotary pass.
__device__ __forceinline__ void load_query16(const DecodeParams& p, int b, int t, int h, int qd,
                                             const float2 (&rope_cs)[16][kD / 2], uint32_t (&w)[8]) {
  const uint4* qr = reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.q_len + t) * p.hq + h) * kD);
  const uint4 lo = __ldg(qr + 2 * qd), hi = __ldg(qr + 2 * qd + 1);
  const uint32_t own[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  if (!p.inv_freq) {
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = own[e];
    return;
  }
  const int pq = qd ^ 2;  // the 16 partner dims: the same planes in the other half
  const uint4 plo = __ldg(qr + 2 * pq), phi = __ldg(qr + 2 * pq + 1);
  const uint32_t par[8] = {plo.x, plo.y, plo.z, plo.w, phi.x, phi.y, phi.z, phi.w};
  uint32_t bo[8] = {}, bp[8] = {};
  if (p.q_bias) {
    const uint4* br = reinterpret_cast<const uint4*>(p.q_bias + (size_t)h * kD);
    const uint4 b0 = __ldg(br + 2 * qd), b1 = __ldg(br + 2 * qd + 1);
    const uint4 c0 = __ldg(br + 2 * pq), c1 = __ldg(br + 2 * pq + 1);
    const uint32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const uint32_t cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bo[e] = bb[e];
      bp[e] = cc[e];
    }
  }
  const bool first_half = qd < 2;
  const int plane0 = (16 * qd) & (kD / 2 - 1);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float y[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float x = __fadd_rn(k ? bf16x2_hi(own[e]) : bf16x2_lo(own[e]), k ? bf16x2_hi(bo[e]) : bf16x2_lo(bo[e]));
      const float xp = __fadd_rn(k ? bf16x2_hi(par[e]) : bf16x2_lo(par[e]), k ? bf16x2_hi(bp[e]) : bf16x2_lo(bp[e]));
      const float2 cs = rope_cs[t][plane0 + 2 * e + k];
      y[k] = first_half ? rope_first(x, xp, cs.x, cs.y) : rope_second(xp, x, cs.x, cs.y);
    }
    w[e] = pack_bf16x2(y[0], y[1]);
  }
}

}  // namespace

// Four CTAs per SM (up to 128 registers a thread, so nothing spills), each
// warp with two 4 KiB pages in flight.  Streaming the slabs this way, from
// sixteen warps per SM, ran 8-16 % faster than one TMA-issuing producer warp
// per CTA feeding an eight-stage ring.
__global__ void __launch_bounds__(kThreads, 4) decode_split_kernel(const DecodeParams p) {
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  // a length beyond the page-table row is clamped: never read past the row
  const int L = min(max(0, p.seqlens[b]), p.stride * kPage);
  int n, pg0, pg1;
  chunk_range(p, L, s, n, pg0, pg1);
  // the merge kernel may be scheduled once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (s >= n) return;
  const int count = max(0, pg1 - pg0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int r = lane >> 2, qd = lane & 3;
  const int G = p.group, nrows = G * p.q_len;  // <= 16
  const int rho = r, rho8 = r + 8;
  const bool row_ok = rho < nrows, row8_ok = rho8 < nrows;
  // new token t and query head h of rows rho and rho + 8
  const int t_r = rho / G, t_r8 = rho8 / G;
  const int h_r = g * G + rho - t_r * G, h_r8 = g * G + rho8 - t_r8 * G;
  // keys visible to a row: positions < lim (causal among the new tokens);
  // padding rows take every valid key so that their (unused) state stays finite
  const int lim_r = row_ok ? L - p.q_len + t_r + 1 : L;
  const int lim_r8 = row8_ok ? L - p.q_len + t_r8 + 1 : L;

  // Rotary encoding of q (optional): cos and sin of every (new token, plane),
  // times the factor, computed once for the CTA (q_len <= 16 tokens here).
  __shared__ float2 rope_cs[16][kD / 2];
  if (p.inv_freq) {
    for (int e = threadIdx.x; e < p.q_len * (kD / 2); e += kThreads) {
      const int t = e / (kD / 2), i = e % (kD / 2);
      float c, sn;
      rope_cos_sin(L - p.q_len + t, rope_turn_increment(__ldg(p.inv_freq + i)), c, sn);
      rope_cs[t][i] = make_float2(__fmul_rn(c, p.attn_factor), __fmul_rn(sn, p.attn_factor));
    }
    __syncthreads();
  }

  // Query fragments: row r holds dims [16qd, 16qd+16) of its head.
  uint32_t qa[4][4];
  {
    uint32_t wr[8] = {}, wr8[8] = {};
    if (row_ok) load_query16(p, b, t_r, h_r, qd, rope_cs, wr);
    if (row8_ok) load_query16(p, b, t_r8, h_r8, qd, rope_cs, wr8);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      qa[kk][0] = wr[2 * kk];
      qa[kk][1] = wr8[2 * kk];
      qa[kk][2] = wr[2 * kk + 1];
      qa[kk][3] = wr8[2 * kk + 1];
    }
  }

  // Online-softmax state for rows r and r+8 (log2 domain).  Only the first
  // chunk's first warp starts from the sink: m = sink * log2(e), d = 1.
  float m_r = -INFINITY, m_r8 = -INFINITY, d_r = 0.f, d_r8 = 0.f;
  if (s == 0 && warp == 0) {
    m_r = row_ok ? __ldg(p.sinks + h_r) * kLog2e : -INFINITY;
    m_r8 = row8_ok ? __ldg(p.sinks + h_r8) * kLog2e : -INFINITY;
    if (qd == 0) {
      d_r = 1.f;
      d_r8 = 1.f;
    }
  }
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  const float sl2 = p.scale_log2;
  // Each warp streams its own pages (i = warp + 4k) into its own two stages with
  // 16-byte asynchronous copies, page k + 2 issued while page k is computed.  A
  // slab lands in the 128-byte swizzled layout the fragment loads below expect
  // (16-byte chunk c of key row t at chunk c ^ (t % 8)); a page id outside the
  // pool yields zeros.
  const int32_t* prow = p.page_table + (size_t)b * p.stride + pg0;
  const int nw = count > warp ? (count - warp + kConsumerWarps - 1) / kConsumerWarps : 0;
  auto issue = [&](int k) {
    if (k < nw) {
      const int page = __ldg(prow + warp + kConsumerWarps * k);
      const bool ok = page >= 0 && page < p.num_pages;
      const size_t slab = ok ? ((size_t)page * p.hkv + g) * (size_t)(kPage * kD) : 0;
      const __nv_bfloat16* ksrc = p.k_pages + slab;
      const __nv_bfloat16* vsrc = p.v_pages + slab;
      uint8_t* st = smem + (warp * kStagesPerWarp + k % kStagesPerWarp) * kStageBytes;
#pragma unroll
      for (int u = 0; u < kSlabBytes / 16 / 32; ++u) {
        const int q = lane + 32 * u, t = q >> 3, c = q & 7;
        const int off = t * 128 + ((c ^ (t & 7)) << 4);
        cp_async16(st + off, ksrc + q * 8, ok ? 16u : 0u);
        cp_async16(st + kSlabBytes + off, vsrc + q * 8, ok ? 16u : 0u);
      }
    }
    cp_async_commit();  // one group per page slot, empty past the warp's pages
  };
#pragma unroll
  for (int k = 0; k < kStagesPerWarp; ++k) issue(k);
  for (int k = 0; k < nw; ++k) {
    const int i = warp + kConsumerWarps * k;
    cp_async_wait<kStagesPerWarp - 1>();
    __syncwarp();
    const uint8_t* ks = smem + (warp * kStagesPerWarp + k % kStagesPerWarp) * kStageBytes;
    const uint8_t* vs = ks + kSlabBytes;
    // K rows t = nt*8 + r, 16-byte chunks 2qd and 2qd+1 (swizzled by t % 8 = r)
    uint4 k0a = lds128(ks + r * 128 + (((2 * qd) ^ r) << 4));
    uint4 k0b = lds128(ks + r * 128 + (((2 * qd + 1) ^ r) << 4));
    uint4 k1a = lds128(ks + (8 + r) * 128 + (((2 * qd) ^ r) << 4));
    uint4 k1b = lds128(ks + (8 + r) * 128 + (((2 * qd + 1) ^ r) << 4));
    // V rows 2qd, 2qd+1, 2qd+8, 2qd+9, chunk r (dims 8r..8r+7)
    const int t0 = 2 * qd, t1 = 2 * qd + 1;
    uint4 va = lds128(vs + t0 * 128 + ((r ^ t0) << 4));
    uint4 vb = lds128(vs + t1 * 128 + ((r ^ t1) << 4));
    uint4 vc = lds128(vs + (t0 + 8) * 128 + ((r ^ t0) << 4));
    uint4 vd = lds128(vs + (t1 + 8) * 128 + ((r ^ t1) << 4));
    __syncwarp();
    issue(k + kStagesPerWarp);  // refills the stage just read

    const int base = (pg0 + i) * kPage;
    const int valid = min(kPage, L - base);  // >= 1
    if (valid < kPage) {  // tail page: unused slots may hold anything (even NaN)
      const uint4 z = make_uint4(0, 0, 0, 0);
      if (t0 >= valid) va = z;
      if (t1 >= valid) vb = z;
      if (t0 + 8 >= valid) vc = z;
      if (t1 + 8 >= valid) vd = z;
    }

    // S = Q K^T: two n-tiles of 8 tokens
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const uint4 ka = nt ? k1a : k0a, kb = nt ? k1b : k0b;
      mma_16816_bf16(sc[nt], qa[0], ka.x, ka.y);
      mma_16816_bf16(sc[nt], qa[1], ka.z, ka.w);
      mma_16816_bf16(sc[nt], qa[2], kb.x, kb.y);
      mma_16816_bf16(sc[nt], qa[3], kb.z, kb.w);
    }
    // scale to log2 units, mask slots past each row's last visible key
    // (lim <= L, so slots past the sequence end are always masked)
    const int vis_r = lim_r - base, vis_r8 = lim_r8 - base;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = nt * 8 + 2 * qd + (e & 1);
        sc[nt][e] = tok < (e < 2 ? vis_r : vis_r8) ? sc[nt][e] * sl2 : -INFINITY;
      }
    }
    float mx_r = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    float mx_r8 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    mx_r = fmaxf(mx_r, __shfl_xor_sync(0xffffffffu, mx_r, 1));
    mx_r = fmaxf(mx_r, __shfl_xor_sync(0xffffffffu, mx_r, 2));
    mx_r8 = fmaxf(mx_r8, __shfl_xor_sync(0xffffffffu, mx_r8, 1));
    mx_r8 = fmaxf(mx_r8, __shfl_xor_sync(0xffffffffu, mx_r8, 2));
    const float mn_r = fmaxf(m_r, mx_r), mn_r8 = fmaxf(m_r8, mx_r8);
    // -inf only while a row has seen neither the sink nor a key: subtract 0
    // then, so that alpha and every weight come out 0 instead of NaN
    const float ms_r = mn_r == -INFINITY ? 0.f : mn_r, ms_r8 = mn_r8 == -INFINITY ? 0.f : mn_r8;
    const float al_r = fast_exp2(m_r - ms_r), al_r8 = fast_exp2(m_r8 - ms_r8);
    m_r = mn_r;
    m_r8 = mn_r8;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = fast_exp2(sc[nt][0] - ms_r);
      pr[nt][1] = fast_exp2(sc[nt][1] - ms_r);
      pr[nt][2] = fast_exp2(sc[nt][2] - ms_r8);
      pr[nt][3] = fast_exp2(sc[nt][3] - ms_r8);
    }
    uint32_t pa[4];
    pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
    pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
    pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
    pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
    // the normaliser sums the same bf16-rounded weights the PV MMA uses
    d_r = d_r * al_r + (bf16x2_lo(pa[0]) + bf16x2_hi(pa[0])) + (bf16x2_lo(pa[2]) + bf16x2_hi(pa[2]));
    d_r8 = d_r8 * al_r8 + (bf16x2_lo(pa[1]) + bf16x2_hi(pa[1])) + (bf16x2_lo(pa[3]) + bf16x2_hi(pa[3]));
    // O = alpha * O + P V over 8 n-tiles of output dims
    const uint32_t vaw[4] = {va.x, va.y, va.z, va.w}, vbw[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t vcw[4] = {vc.x, vc.y, vc.z, vc.w}, vdw[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= al_r;
      o[j][1] *= al_r;
      o[j][2] *= al_r8;
      o[j][3] *= al_r8;
      const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
      const uint32_t b0 = __byte_perm(vaw[j >> 1], vbw[j >> 1], sel);
      const uint32_t b1 = __byte_perm(vcw[j >> 1], vdw[j >> 1], sel);
      mma_16816_bf16(o[j], pa, b0, b1);
    }
  }

  cp_async_wait<0>();

  // ---------------------------------------------- merge the four warps' states
  d_r += __shfl_xor_sync(0xffffffffu, d_r, 1);
  d_r += __shfl_xor_sync(0xffffffffu, d_r, 2);
  d_r8 += __shfl_xor_sync(0xffffffffu, d_r8, 1);
  d_r8 += __shfl_xor_sync(0xffffffffu, d_r8, 2);
  named_barrier(1, kConsumerWarps * 32);  // every consumer is done with the ring
  float* scr = reinterpret_cast<float*>(smem) + warp * kScratchFloatsPerWarp;
  float* sm = scr;
  float* sd = scr + kRows;
  float* so = scr + 2 * kRows;
  if (qd == 0) {
    sm[r] = m_r;
    sd[r] = d_r;
    sm[r + 8] = m_r8;
    sd[r + 8] = d_r8;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    so[r * kD + 16 * qd + j] = o[j][0];
    so[r * kD + 16 * qd + 8 + j] = o[j][1];
    so[(r + 8) * kD + 16 * qd + j] = o[j][2];
    so[(r + 8) * kD + 16 * qd + 8 + j] = o[j][3];
  }
  named_barrier(1, kConsumerWarps * 32);

  const int tid = threadIdx.x;  // 0..127
  const int row = tid >> 3, c8 = (tid & 7) * 8;
  if (row >= nrows) return;
  const float* scratch = reinterpret_cast<const float*>(smem);
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, scratch[w * kScratchFloatsPerWarp + row]);
  float W = 0.f, acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* ws = scratch + w * kScratchFloatsPerWarp;
      const float mw = ws[row];
      if (mw == -INFINITY) continue;
      const float f = fast_exp2(mw - M);
      W += ws[kRows + row] * f;
      const float* ow = ws + 2 * kRows + row * kD + c8;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += ow[e] * f;
    }
  }
  const int t = row / G;
  const size_t qrow = ((size_t)b * p.q_len + t) * p.hq + g * G + (row - t * G);  // (sequence, token, head)
  if (p.direct) {
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const size_t o_off = qrow * kD + c8;
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o_off);
      dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
    } else {
      uint4 v;
      v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o_off) = v;
    }
    if (p.lse && c8 == 0) p.lse[qrow] = W > 0.f ? (M + __log2f(W)) * kLn2 : -INFINITY;
  } else {
    const size_t slot = qrow * p.max_splits + s;
    float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * kD + c8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (c8 == 0) {
      p.ws_md[slot * 2] = M;
      p.ws_md[slot * 2 + 1] = W;
    }
  }
}

// Combine the chunks' partial states: one warp per (row of q, query head).
// Lane l owns output dims 2l, 2l+1.  Chunk c contributes with weight
// 2^(m_c - M), M = max_c m_c; chunks that saw nothing have m_c = -inf (and
// d_c = 0, o_c = 0), hence weight 0.  Launched as a programmatic dependent of
// the chunk kernel: it waits for that grid's results before reading them.
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (wid >= p.total_q * p.hq) return;
  const int row = wid / p.hq;
  int b;
  if (p.cu_q) {  // the last sequence whose new tokens start at or before this row
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu_q[mid] <= row) lo = mid;
      else hi = mid;
    }
    b = lo;
  } else {
    b = row / p.q_len;
  }
  const size_t slot0 = (size_t)wid * p.max_splits;
  const float2* md = reinterpret_cast<const float2*>(p.ws_md) + slot0;  // (m_c, d_c)
  const float2* o = reinterpret_cast<const float2*>(p.ws_o + slot0 * kD) + lane;  // chunk c at o[c * 32]
  float W = 0.f, a0 = 0.f, a1 = 0.f, M = -INFINITY;
  if (p.max_splits <= 16) {
    // Up to 16 chunks: every load of the row at once, before the length that says how
    // many of them this sequence used (slots past that count hold another call's
    // values and are skipped, never multiplied by a zero weight): one round trip to
    // L2 instead of three (3.6 against 5.7 us for the batch-64 decode's merge).
    float2 oc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) oc[u] = u < p.max_splits ? o[(size_t)u * 32] : make_float2(0.f, 0.f);
    const float2 v = lane < p.max_splits ? md[lane] : make_float2(-INFINITY, 0.f);
    const int L = min(max(0, p.seqlens[b]), p.stride * kPage);
    int n, pg0, pg1;
    chunk_range(p, L, 0, n, pg0, pg1);
    M = lane < n ? v.x : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M != -INFINITY) {
      const float f = lane < n ? fast_exp2(v.x - M) : 0.f;  // 0 for a chunk that saw nothing
      W = lane < n ? v.y * f : 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float fu = __shfl_sync(0xffffffffu, f, u);
        if (u < n) {
          a0 += oc[u].x * fu;
          a1 += oc[u].y * fu;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    }
  } else {
    const int L = min(max(0, p.seqlens[b]), p.stride * kPage);
    int n, pg0, pg1;
    chunk_range(p, L, 0, n, pg0, pg1);
    for (int c = lane; c < n; c += 32) M = fmaxf(M, md[c].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M != -INFINITY) {
      for (int base = 0; base < n; base += 32) {
        // chunk base + lane's weight on this lane; the dims loop reads it by shuffle
        float f = 0.f;
        if (base + lane < n) {
          const float2 v = md[base + lane];
          f = fast_exp2(v.x - M);  // 0 for a chunk that saw nothing
          W += v.y * f;
        }
        const int cnt = min(32, n - base);
        for (int k = 0; k < cnt; k += 8) {  // eight chunks' loads in flight before their adds
          float2 oc[8];
          float fk[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            fk[u] = __shfl_sync(0xffffffffu, f, k + u);
            oc[u] = k + u < cnt ? o[(size_t)(base + k + u) * 32] : make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            a0 += oc[u].x * fk[u];
            a1 += oc[u].y * fk[u];
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const size_t o_off = (size_t)wid * kD + 2 * lane;
  if (p.out_f32) {
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.out) + o_off) = make_float2(a0 * inv, a1 * inv);
  } else {
    *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o_off) = pack_bf16x2(a0 * inv, a1 * inv);
  }
  if (p.lse && lane == 0) p.lse[wid] = W > 0.f ? (M + __log2f(W)) * kLn2 : -INFINITY;
}

cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t stream) {
  const long long warps = (long long)p.total_q * p.hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel, p);
}

size_t decode_smem_bytes() { return kRingBytes + 1024; }

cudaError_t decode_configure() {
  // Prefer shared memory over L1 so four CTAs' rings fit on an SM.
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)decode_smem_bytes());
}
int decode_threads() { return kThreads; }

}  // namespace sa

namespace sa {

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.max_splits, p.hkv, p.batch);
  decode_split_kernel<<<grid, kThreads, decode_smem_bytes(), stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.direct) return e;
  return launch_decode_merge(p, stream);
}

}  // namespace sa
