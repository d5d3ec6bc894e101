// Internal interface of the causal varlen prefill kernel (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sa {

constexpr int kPrefillTileRows = 128;   // query rows per tile
constexpr int kPrefillKeyRows = 128;    // keys per K/V tile
constexpr int kPrefillMaxBatch = 1024;  // sequences per call (per-CTA schedule table)

struct PrefillParams {
  const int32_t* cu_seqlens;  // [B+1]: query rows of each sequence (contiguous mode: its keys too)
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
  // Work distribution: the slot of the per-device unit counters this launch
  // takes its units from (one at a time, in schedule order: longest first), or
  // -1 for the static deal (captured launches).  Set by launch_prefill.
  int sched_slot;
  // Paged mode (chunked prefill against the paged KV cache): the keys of
  // sequence b are its kv_len[b] cached tokens, read page by page, and its
  // n_b query rows are the last n_b of them (row i at position
  // kv_len[b] - n_b + i, causal).
  const int32_t* kv_len;      // [B]
  const int32_t* page_table;  // [B, stride]
  int stride;
  // Rotary mode (contiguous prefill only; null inv_freq: off): q is the raw
  // projection, and row i of a sequence becomes rot(q + q_bias) * attn_factor
  // at position i, rotated in shared memory before its first QK.
  const __nv_bfloat16* q_bias;  // [Hq, 64] or null
  const double* inv_freq;       // [32]
  float attn_factor;
};

// One-time per-device kernel attributes (dynamic shared memory size).
cudaError_t prefill_configure();

// Enqueue the persistent prefill kernel: `grid_ctas` <= number of SMs.
// qmap is a 3-D map over [T, Hq, 64] with boxes of 128 tokens x 1 head x 64
// dims; omap the same over the output (bf16 output only: whole 128-row blocks
// are written by bulk tensor stores; with fp32 output it is not used).  Contiguous mode: kmap / vmap are the same over [T, Hkv, 64].  Paged
// mode: 2-D maps over the pools viewed as [num_pages * Hkv * 16, 64] with
// boxes of one (page, kv head) slab of 16 rows.
cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& omap, const PrefillParams& p, int num_sms, bool paged,
                           cudaStream_t stream);

}  // namespace sa
