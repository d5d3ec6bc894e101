// Internal interface of the QKV bias + rotary encoding pass (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

struct RopeParams {
  __nv_bfloat16* q;  // [tokens, hq, 64], rotated in place; null: q is left alone
  __nv_bfloat16* k;  // [tokens, hkv, 64], rotated in place
  __nv_bfloat16* v;  // [tokens, hkv, 64], biased in place
  const __nv_bfloat16* q_bias;  // [hq, 64] or null
  const __nv_bfloat16* k_bias;  // [hkv, 64] or null
  const __nv_bfloat16* v_bias;  // [hkv, 64] or null
  const int32_t* positions;     // [tokens]
  const double* inv_freq;       // [32] rotation frequency of each plane (radians per position)
  float attn_factor;            // multiplies the rotated q and k
  const int32_t* slot_mapping;  // [tokens] cache slot (page * page_size + offset) or null; < 0 skips
  __nv_bfloat16* k_pages;       // [num_pages, hkv, page_size, 64] when slot_mapping is set
  __nv_bfloat16* v_pages;
  int num_pages, page_size;
  int tokens, hq, hkv;
};

// Rotation angles without fp64 arithmetic per element.  A plane's frequency f
// (radians per position) is turned once into a 64-bit fixed-point fraction of
// a turn, F = frac(f / 2 pi) * 2^64; the phase of position p is then the
// integer product p * F taken modulo 2^64, which is p * f modulo one turn with
// no rounding beyond that of F (a relative 2^-53, the precision of the fp64
// frequency itself).  The top 32 bits, read as a signed fraction of a half
// turn, go to sincospif.
__device__ __forceinline__ unsigned long long rope_turn_increment(double f) {
  double t = f / 6.283185307179586476925286766559;
  t -= floor(t);  // [0, 1]: whole turns contribute nothing
  const double scaled = t * 18446744073709551616.0;  // 2^64
  return scaled >= 18446744073709551616.0 ? 0ull : __double2ull_rn(scaled);
}

// cos and sin of position * f for a position held exactly by the phase.
__device__ __forceinline__ void rope_phase_cos_sin(int position, unsigned long long F, float& c, float& s) {
  const unsigned long long phase = (unsigned long long)(long long)position * F;  // modulo 2^64 = one turn
  const float half_turns = (float)(int)(phase >> 32) * 0x1p-31f;                 // in [-1, 1)
  sincospif(half_turns, &s, &c);
}

// Angle addition with every rounding explicit, so that each kernel applying
// the rotation gets the same bits: (c, s) of a + b from those of a and b.
__device__ __forceinline__ void rope_angle_add(float ca, float sa, float cb, float sb, float& c, float& s) {
  c = __fmaf_rn(ca, cb, -__fmul_rn(sa, sb));
  s = __fmaf_rn(sa, cb, __fmul_rn(ca, sb));
}

// cos and sin of position * f, F = rope_turn_increment(f).  The position is
// split into its multiple of 128 and its remainder (both exact phases), the
// two angles added: a kernel whose 128 consecutive positions share the first
// part (a prefill query tile) can keep the second part's 128 values in a
// table and reproduce these bits.
__device__ __forceinline__ void rope_cos_sin(int position, unsigned long long F, float& c, float& s) {
  const int lo = position & 127, hi = position - lo;
  float ch, sh, cl, sl;
  rope_phase_cos_sin(hi, F, ch, sh);
  rope_phase_cos_sin(lo, F, cl, sl);
  rope_angle_add(ch, sh, cl, sl, c, s);
}

// The rotation of one plane (x1 = dim i, x2 = dim i + D/2) by cs = c * factor,
// sn = s * factor, with explicit roundings (identical wherever it is used).
__device__ __forceinline__ float rope_first(float x1, float x2, float cs, float sn) {
  return __fmaf_rn(x1, cs, -__fmul_rn(x2, sn));
}
__device__ __forceinline__ float rope_second(float x1, float x2, float cs, float sn) {
  return __fmaf_rn(x2, cs, __fmul_rn(x1, sn));
}

__global__ void qkv_rope_kernel(const RopeParams p);
cudaError_t launch_qkv_rope(const RopeParams& p, cudaStream_t stream);

}  // namespace sa
