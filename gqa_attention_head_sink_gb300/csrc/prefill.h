// Internal interface of the causal varlen prefill kernel (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sa {

constexpr int kPrefillTileRows = 128;   // query rows per tile
constexpr int kPrefillKeyRows = 128;    // keys per K/V tile
constexpr int kPrefillMaxBatch = 1024;  // sequences per call (per-CTA schedule table)

struct PrefillParams {
  const int32_t* cu_seqlens;  // [B+1]
  const float* sinks;         // [Hq]
  void* out;                  // [T, Hq, 64] bf16 or fp32
  float* lse;                 // [T, Hq] or null
  unsigned* err;              // device error word
  int batch, total_tokens, hq, hkv, group;
  int max_qblocks;  // ceil(max_seqlen / 128)
  int out_f32;
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  int withhold_copies;  // failure-path test: the producer issues no copies, so the waits time out
};

// One-time per-device kernel attributes (dynamic shared memory size).
cudaError_t prefill_configure();

// Enqueue the persistent prefill kernel: `grid_ctas` <= number of SMs.
// qmap / kmap / vmap are 3-D maps over [T, heads, 64] with boxes of 128 (q) or
// 64 (k, v) tokens x 1 head x 64 dims.
cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const PrefillParams& p, int num_sms, cudaStream_t stream);

}  // namespace sa
