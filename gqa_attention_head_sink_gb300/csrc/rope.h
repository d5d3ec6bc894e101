// Internal interface of the QKV bias + rotary encoding pass (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

struct RopeParams {
  __nv_bfloat16* q;  // [tokens, hq, 64], rotated in place
  __nv_bfloat16* k;  // [tokens, hkv, 64], rotated in place
  __nv_bfloat16* v;  // [tokens, hkv, 64], biased in place
  const __nv_bfloat16* q_bias;  // [hq, 64] or null
  const __nv_bfloat16* k_bias;  // [hkv, 64] or null
  const __nv_bfloat16* v_bias;  // [hkv, 64] or null
  const int32_t* positions;     // [tokens]
  const float* inv_freq;        // [32] rotation frequency of each plane
  float attn_factor;            // multiplies the rotated q and k
  const int32_t* slot_mapping;  // [tokens] cache slot (page * page_size + offset) or null; < 0 skips
  __nv_bfloat16* k_pages;       // [num_pages, hkv, page_size, 64] when slot_mapping is set
  __nv_bfloat16* v_pages;
  int num_pages, page_size;
  int tokens, hq, hkv;
};

__global__ void qkv_rope_kernel(const RopeParams p);
cudaError_t launch_qkv_rope(const RopeParams& p, cudaStream_t stream);

}  // namespace sa
