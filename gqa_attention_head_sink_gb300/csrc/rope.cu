// QKV bias + rotary position encoding (YaRN frequencies) applied to q, k and
// v before sink attention, with an optional append of k and v to the paged
// KV cache (sm_103a).
//
// Method: Perplexity, "GPT-OSS on day 0", model overview: YaRN positional
// encoding (as in DeepSeek-V3) and biased QKV projections (as in Qwen 2).
// The pages give no formula; this follows the published definitions:
// rotary planes (dim i, dim i + D/2) rotated by position * inv_freq[i], the
// rotation multiplied by attn_factor (YaRN's temperature, 1 for plain RoPE),
// the bias added before the rotation; v gets its bias only.  YaRN's
// frequencies themselves are a per-model table computed once on the host
// (sink_attn_yarn_inv_freq in api.cu).
//
// Why K is rotated here and not at the attention kernels' tile loads: each K
// tile is read by every query block of its sequence (64 times at 8192
// tokens), so rotating at load would repeat the work 64 times on the softmax
// warps that already bound the prefill.  q may be left out (q == NULL): the
// prefill and decode kernels can rotate each query tile once themselves
// (their rotary mode, bit for bit the same as this pass); on the 8192-token
// prefill this pass over q, k and v plus the plain prefill is the faster
// route.  For decode and chunked prefill the same pass writes the new
// tokens' rotated k and v into their cache slots, so the attention kernels
// read the cache unchanged.
//
// One CTA per 8 tokens: each thread first forms one (token, plane) entry of
// the cos/sin table (the angle position * inv_freq as a 64-bit fixed-point
// phase, exact modulo one turn for any int32 position, then sincospif; see
// rope_cos_sin), then the threads take (token, head, lane) items, a lane
// rotating 8 planes of one head row with 16-byte loads of both halves, and v
// rows get their bias in 16-byte pieces.
#include "common.cuh"
#include "rope.h"

namespace sa {

namespace {

constexpr int kD = 64;
constexpr int kHalf = kD / 2;
constexpr int kThreads = 256;
constexpr int kTokensPerBlock = 8;
constexpr int kLanesPerRow = 4;  // a lane rotates 8 planes: 16 bytes of each half
// the table phase gives each thread exactly one (token, plane) entry
static_assert(kThreads == kTokensPerBlock * kHalf, "one cos/sin entry per thread");

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = bf16x2_lo(w[e]);
    f[2 * e + 1] = bf16x2_hi(w[e]);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

}  // namespace

__global__ void __launch_bounds__(kThreads) qkv_rope_kernel(const RopeParams p) {
  __shared__ float cs[kTokensPerBlock][kHalf], sn[kTokensPerBlock][kHalf];
  __shared__ unsigned long long turn[kHalf];
  __shared__ long long cache_row[kTokensPerBlock];
  const int tid = threadIdx.x;
  const int t_base = blockIdx.x * kTokensPerBlock;
  if (tid < kHalf) turn[tid] = rope_turn_increment(__ldg(p.inv_freq + tid));
  __syncthreads();
  {
    // one (token, plane) angle per thread: 8 tokens x 32 planes = 256
    const int tb = tid / kHalf, i = tid % kHalf, t = t_base + tb;
    if (t < p.tokens) {
      float s, c;
      rope_cos_sin(__ldg(p.positions + t), turn[i], c, s);
      cs[tb][i] = __fmul_rn(c, p.attn_factor);
      sn[tb][i] = __fmul_rn(s, p.attn_factor);
    }
    if (i == 0) {
      // cache slot of this token's k and v: row of the [num_pages * Hkv * page_size, 64] view (kv head 0)
      long long row = -1;
      if (p.slot_mapping && t < p.tokens) {
        const int slot = __ldg(p.slot_mapping + t);
        const int page = slot >= 0 ? slot / p.page_size : -1;
        if (page >= 0 && page < p.num_pages) row = ((long long)page * p.hkv) * p.page_size + (slot - page * p.page_size);
      }
      cache_row[tb] = row;
    }
  }
  __syncthreads();

  // q and k rows: items (token, head, lane); heads 0..Hq-1 are q (none when q is
  // left alone), then k
  const int q_rows = p.q ? p.hq : 0;
  const int rows = q_rows + p.hkv;
  const int qk_items = kTokensPerBlock * rows * kLanesPerRow;
  for (int item = tid; item < qk_items; item += kThreads) {
    const int tb = item / (rows * kLanesPerRow), rest = item % (rows * kLanesPerRow);
    const int h = rest / kLanesPerRow, l = rest % kLanesPerRow;
    const int t = t_base + tb;
    if (t >= p.tokens) break;  // items are token-major: the rest are past the end too
    const bool is_q = h < q_rows;
    const int hh = is_q ? h : h - q_rows;
    __nv_bfloat16* row = is_q ? p.q + ((size_t)t * p.hq + hh) * kD : p.k + ((size_t)t * p.hkv + hh) * kD;
    const __nv_bfloat16* bias = is_q ? p.q_bias : p.k_bias;
    float x1[8], x2[8];
    unpack8(*reinterpret_cast<const uint4*>(row + 8 * l), x1);
    unpack8(*reinterpret_cast<const uint4*>(row + kHalf + 8 * l), x2);
    if (bias) {
      float b1[8], b2[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(bias + (size_t)hh * kD + 8 * l)), b1);
      unpack8(__ldg(reinterpret_cast<const uint4*>(bias + (size_t)hh * kD + kHalf + 8 * l)), b2);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x1[e] = __fadd_rn(x1[e], b1[e]);
        x2[e] = __fadd_rn(x2[e], b2[e]);
      }
    }
    float y1[8], y2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float c = cs[tb][8 * l + e], s = sn[tb][8 * l + e];
      y1[e] = rope_first(x1[e], x2[e], c, s);
      y2[e] = rope_second(x1[e], x2[e], c, s);
    }
    const uint4 o1 = pack8(y1), o2 = pack8(y2);
    *reinterpret_cast<uint4*>(row + 8 * l) = o1;
    *reinterpret_cast<uint4*>(row + kHalf + 8 * l) = o2;
    if (!is_q && cache_row[tb] >= 0) {
      __nv_bfloat16* dst = p.k_pages + (cache_row[tb] + (long long)hh * p.page_size) * kD;
      *reinterpret_cast<uint4*>(dst + 8 * l) = o1;
      *reinterpret_cast<uint4*>(dst + kHalf + 8 * l) = o2;
    }
  }

  // v rows: bias only, 8 dims per item
  const int v_items = kTokensPerBlock * p.hkv * 8;
  for (int item = tid; item < v_items; item += kThreads) {
    const int tb = item / (p.hkv * 8), rest = item % (p.hkv * 8);
    const int hh = rest / 8, l = rest % 8;
    const int t = t_base + tb;
    if (t >= p.tokens) break;
    __nv_bfloat16* row = p.v + ((size_t)t * p.hkv + hh) * kD + 8 * l;
    uint4 v = *reinterpret_cast<const uint4*>(row);
    if (p.v_bias) {
      float x[8], b[8];
      unpack8(v, x);
      unpack8(__ldg(reinterpret_cast<const uint4*>(p.v_bias + (size_t)hh * kD + 8 * l)), b);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] += b[e];
      v = pack8(x);
      *reinterpret_cast<uint4*>(row) = v;
    }
    if (cache_row[tb] >= 0)
      *reinterpret_cast<uint4*>(p.v_pages + (cache_row[tb] + (long long)hh * p.page_size) * kD + 8 * l) = v;
  }
}

cudaError_t launch_qkv_rope(const RopeParams& p, cudaStream_t stream) {
  const int blocks = (p.tokens + kTokensPerBlock - 1) / kTokensPerBlock;
  qkv_rope_kernel<<<blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sa
