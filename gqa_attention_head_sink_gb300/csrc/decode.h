// Internal interface of the split-KV decode kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sa {

struct DecodeParams {
  const __nv_bfloat16* q;     // [total_q, Hq, 64]: [B, q_len, Hq, 64] or packed by cu_q
  const int32_t* page_table;  // [B, stride]
  const __nv_bfloat16* k_pages;  // [num_pages, Hkv, 16, 64]: read by the chunk kernel's copies
  const __nv_bfloat16* v_pages;
  int num_pages;                  // page ids outside [0, num_pages) read as zeros
  const int32_t* seqlens;     // [B]
  const float* sinks;         // [Hq]
  void* out;                  // [total_q, Hq, 64] bf16 or fp32
  float* lse;                 // [total_q, Hq] or null
  float* ws_o;                // [total_q, Hq, max_splits, 64] partial weighted sums
  float* ws_md;               // [total_q, Hq, max_splits, 2] partial (m, d), m in log2 units
  unsigned* err;              // device error word
  int batch, hq, hkv, group, stride;
  int q_len;            // new query tokens per sequence (the last q_len of its cache), when cu_q is null
  const int32_t* cu_q;  // tensor-core kernel: [B + 1] offsets of each sequence's new tokens, or null
  int total_q;          // rows of q / out: B * q_len, or cu_q[B]
  int tokens_per_tile;  // tensor-core kernel: new tokens per 128-row tile (tile rows = group * tokens_per_tile)
  int row_tiles;        // tensor-core kernel: tiles per sequence, ceil(q_len / tokens_per_tile)
  int num_splits;   // > 0: requested chunks per sequence; 0: by length
  int split_pages;  // pages per chunk when num_splits == 0
  int max_splits;   // grid extent of the chunk dimension
  int direct;       // 1: one chunk per sequence, write the output directly
  int out_f32;
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  int withhold_copies;  // failure-path test: the tensor-core kernel's producer issues no copies, so its waits time out
  // Rotary encoding of q inside the split kernel (null inv_freq: q is used as given).
  // New token t of a sequence with L cached tokens sits at position L - q_len + t;
  // its query rows become rot(q + q_bias) * attn_factor, rounded to bf16.
  const __nv_bfloat16* q_bias;  // [Hq, 64] or null
  const double* inv_freq;       // [32] radians per position, or null
  float attn_factor;
};

// Number of chunks sequence with `npages` pages is cut into.  Every chunk is
// non-empty (a sequence with no page still gets one chunk: the sink alone).
__host__ __device__ inline int decode_num_chunks(int npages, int num_splits, int split_pages, int max_splits) {
  if (npages <= 0) return 1;
  int n = num_splits > 0 ? num_splits : (npages + split_pages - 1) / split_pages;
  if (n > npages) n = npages;
  if (n > max_splits) n = max_splits;
  if (n < 1) n = 1;
  const int chunk = (npages + n - 1) / n;
  return (npages + chunk - 1) / chunk;
}

__global__ void decode_split_kernel(const DecodeParams p);
__global__ void decode_merge_kernel(const DecodeParams p);

// Tensor-core variant for many query rows per kv head (multi-token decode):
// 128-row tiles of (new token, query head) pairs, S and O in TMEM.
__global__ void decode_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                                 const __grid_constant__ CUtensorMap vmap, const DecodeParams p);
constexpr int kDecodeTcRows = 128;  // query rows of one tensor-core tile

size_t decode_smem_bytes();

// One-time per-device kernel attributes (shared-memory carveout, size).
cudaError_t decode_configure();
int decode_threads();

// Enqueue the merge kernel as a programmatic dependent launch of the chunk
// kernel just enqueued on the same stream.
cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t stream);

// Enqueue the chunk kernel and, when chunks are merged, the merge kernel.
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
// Same with the tensor-core chunk kernel (qmap: q as [B * q_len, Hq, 64],
// boxes of group heads x tokens_per_tile tokens).
cudaError_t decode_tc_configure();
cudaError_t launch_decode_tc(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const DecodeParams& p, cudaStream_t stream);

}  // namespace sa
