/*
 * sink_attn.h -- C ABI of the GB300 (sm_103a) sink-attention library.
 *
 * Grouped-query attention in which every query head owns one trained "sink"
 * logit that joins the softmax normaliser but carries no value vector
 * (Perplexity, "GPT-OSS on day 0": model overview, attention bullet, and the
 * section "Sink Attention").  For query head h, kv head g = h / (Hq / Hkv),
 * and the keys j visible to a query:
 *
 *     s_j    = scale * <q_h, k_{j,g}>
 *     M      = max(max_j s_j, sink_h)
 *     Z      = sum_j exp(s_j - M) + exp(sink_h - M)
 *     out_h  = sum_j exp(s_j - M) / Z * v_{j,g}
 *     lse_h  = M + log(Z)              (natural log, includes the sink)
 *
 * The kernels evaluate this with an online softmax whose running maximum
 * starts at the head's sink and whose running scale starts at 1 (same
 * section, closing paragraph); when the key length is split into chunks,
 * only the first chunk is seeded with the sink.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference to them after the call returns.
 *   - bf16 means IEEE bfloat16 stored in 2 bytes; tensors are dense and
 *     row-major in the order of the dimensions listed (no strides).
 *   - Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously on it; the call returns before it finishes.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-zero status means nothing was enqueued and no output was written
 *     (SINK_ATTN_ERR_CUDA can also report a failed launch).
 *   - No C++ exception crosses this interface.
 *   - Supported: head_dim == 64, page_size == 16, scale > 0 and finite,
 *     Hq % Hkv == 0.  Sinks may be -inf (no sink).  +inf / NaN sinks are
 *     outside the contract.
 *   - Device-side waits are bounded; a wait that gives up records a timeout
 *     that sink_attn_get_device_error() reports.
 *   - The prefill kernels hand work units to their CTAs at run time from one
 *     of 65,536 per-device counter slots, taken in turn by successive launches
 *     (calls may run concurrently on different streams); a launch captured
 *     into a CUDA graph uses a fixed deal instead.  Results do not depend on
 *     the deal.
 */
#ifndef SINK_ATTN_H_
#define SINK_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SINK_ATTN_OK = 0,
  SINK_ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or count */
  SINK_ATTN_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement */
  SINK_ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  SINK_ATTN_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
  SINK_ATTN_ERR_NO_MEMORY = 5    /* workspace allocation failed */
} sink_attn_status;

typedef enum {
  SINK_ATTN_OUT_BF16 = 0, /* out is bf16 */
  SINK_ATTN_OUT_F32 = 1   /* out is fp32 */
} sink_attn_out_dtype;

/*
 * Causal variable-length prefill ("GPT-OSS on day 0", section Sink Attention,
 * applied to every query of a packed batch; query length = key length).
 *
 *   q           bf16 [total_tokens, num_q_heads, head_dim]
 *   k, v        bf16 [total_tokens, num_kv_heads, head_dim]
 *   sinks       fp32 [num_q_heads] (per query head, not multiplied by scale)
 *   cu_seqlens  int32 [batch + 1], DEVICE memory: cu[0] = 0, non-decreasing,
 *               cu[batch] = total_tokens.  Sequence b owns tokens
 *               [cu[b], cu[b+1]); token i of a sequence sees keys 0..i of the
 *               same sequence.  Zero-length sequences are allowed.
 *   batch, total_tokens, max_seqlen
 *               host copies used to size the grid without a device sync;
 *               max_seqlen must be >= every sequence length.
 *   scale       softmax scale applied to q.k (typically 1/sqrt(head_dim)).
 *               A sequence's output depends on its own q, k and v only: the
 *               next packed sequence's tokens, which share its last 128-key
 *               tile, are masked and their values zeroed before the product,
 *               so even NaN or Inf there does not reach it.
 *   out         [total_tokens, num_q_heads, head_dim], bf16 or fp32 per
 *               out_dtype, 16-byte aligned, not overlapping q, k or v.
 *               Written for every token of every sequence and nowhere else
 *               (bf16: a head's 128-row block lying wholly inside its
 *               sequence goes out as one bulk tensor store).
 *   lse         optional fp32 [total_tokens, num_q_heads] (natural-log
 *               normaliser including the sink); NULL to skip.
 * Limits: batch <= 1024; max_seqlen < 2^24; total_tokens * num_q_heads < 2^31.
 * batch == 0 or total_tokens == 0 is a no-op returning SINK_ATTN_OK.
 */
int sink_attn_prefill(const void* q, const void* k, const void* v, const float* sinks,
                      const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen,
                      int num_q_heads, int num_kv_heads, int head_dim, float scale,
                      void* out, int out_dtype, float* lse, void* stream);

/*
 * sink_attn_prefill with the query's bias and rotary position encoding applied
 * inside the prefill kernel ("GPT-OSS on day 0": model overview, YaRN
 * positional encoding and biased QKV projections; section Sink Attention for
 * the attention).  Each 128-row query tile is rotated in shared memory after
 * it lands and before its first score product, so the rotated query never
 * goes through HBM.
 *
 * q is the query projection before its bias and rotation; k and v are ready
 * (biased and rotated k, biased v: sink_attn_qkv_rope with q = NULL).  Token
 * i of a sequence (0-based within it) is at position i, so its query rows
 * become rot(q + q_bias) * attn_factor at position i, computed exactly as
 * sink_attn_qkv_rope computes them at that position (same bits) and rounded
 * to bf16 before the attention: the output equals that of sink_attn_qkv_rope
 * followed by sink_attn_prefill, bit for bit.
 *   q_bias      bf16 [num_q_heads, head_dim] DEVICE, or NULL for no bias
 *   inv_freq    fp64 [head_dim / 2] DEVICE, radians per position
 *   attn_factor YaRN's temperature, 1 for plain RoPE
 * Every other argument, limit and result is that of sink_attn_prefill.
 */
int sink_attn_prefill_rope(const void* q, const void* k, const void* v, const float* sinks,
                           const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen,
                           int num_q_heads, int num_kv_heads, int head_dim, float scale,
                           const void* q_bias, const double* inv_freq, float attn_factor,
                           void* out, int out_dtype, float* lse, void* stream);

/*
 * Split-KV decode: one query token per sequence against a paged KV cache
 * ("GPT-OSS on day 0", section Sink Attention: the key length is split into
 * chunks and only the first chunk's online state starts from the sink).
 *
 *   q           bf16 [batch, num_q_heads, head_dim]
 *   k_pages,    bf16 [num_pages, num_kv_heads, page_size, head_dim]: one
 *   v_pages     (page, kv head) slab is page_size*head_dim contiguous values.
 *   page_table  int32 [batch, page_table_stride], DEVICE: token j of
 *               sequence b lives in page page_table[b][j / page_size], slot
 *               j % page_size.  Only the first ceil(seqlens[b]/page_size)
 *               entries of a row are read; each must be in [0, num_pages).
 *   seqlens     int32 [batch], DEVICE: number of cached tokens of each
 *               sequence (the query sees all of them).  A length of 0 gives
 *               out = 0 (only the sink is in the softmax).
 *   batch, max_seqlen, num_pages
 *               host values: max_seqlen >= every seqlens[b] and
 *               max_seqlen <= page_table_stride * page_size.
 *   sinks       fp32 [num_q_heads]
 *   num_q_heads / num_kv_heads must be <= 16 (one MMA row block per group).
 *   num_splits  > 0: every sequence is split into that many chunks of pages
 *               (fewer if it has fewer pages); 0: chosen per sequence length
 *               by the library.  At most 256.
 *   out         [batch, num_q_heads, head_dim], bf16 or fp32 per out_dtype.
 *   lse         optional fp32 [batch, num_q_heads]; NULL to skip.
 *   workspace   device scratch for the per-chunk partial states, at least
 *               sink_attn_decode_workspace_bytes(...) bytes, 256-byte
 *               aligned.  NULL: the library allocates and frees it in stream
 *               order when it is needed: from a library-owned memory pool
 *               per device (cudaMallocFromPoolAsync / cudaFreeAsync), which
 *               keeps freed memory for later calls (up to the largest
 *               workspace used) until the process exits; during stream
 *               capture with cudaMallocAsync (a graph allocation node).
 * batch == 0 is a no-op returning SINK_ATTN_OK.
 */
int sink_attn_decode(const void* q, const void* k_pages, const void* v_pages,
                     const int32_t* page_table, int page_table_stride,
                     const int32_t* seqlens, int batch, int max_seqlen, int num_pages,
                     const float* sinks, int num_q_heads, int num_kv_heads, int head_dim,
                     int page_size, float scale, int num_splits,
                     void* out, int out_dtype, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * sink_attn_decode with the query's bias and rotary position encoding applied
 * inside the decode kernel, so the query of a decode step needs no separate
 * pass ("GPT-OSS on day 0": model overview, YaRN positional encoding and
 * biased QKV projections; section Sink Attention for the attention).
 *
 * q is the query projection before its bias and rotation.  The keys and
 * values in the cache are already biased and rotated (sink_attn_qkv_rope with
 * q = NULL appends the step's k and v that way).  The query of sequence b is
 * the last of its seqlens[b] cached tokens, so it is rotated by position
 * seqlens[b] - 1: every query row becomes rot(q + q_bias) * attn_factor,
 * computed exactly as sink_attn_qkv_rope computes it (same bits) and rounded
 * to bf16 before the attention.
 *   q_bias      bf16 [num_q_heads, head_dim] DEVICE, or NULL for no bias
 *   inv_freq    fp64 [head_dim / 2] DEVICE, radians per position
 *               (sink_attn_yarn_inv_freq)
 *   attn_factor YaRN's temperature, 1 for plain RoPE
 * Every other argument, limit and result is that of sink_attn_decode.
 */
int sink_attn_decode_rope(const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* page_table, int page_table_stride,
                          const int32_t* seqlens, int batch, int max_seqlen, int num_pages,
                          const float* sinks, int num_q_heads, int num_kv_heads, int head_dim,
                          int page_size, float scale, int num_splits,
                          const void* q_bias, const double* inv_freq, float attn_factor,
                          void* out, int out_dtype, float* lse,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace sink_attn_decode needs for these arguments (0 when no
 * sequence is split, i.e. the chunks write the output directly).  Returns
 * (size_t)-1 for arguments sink_attn_decode would reject.
 */
size_t sink_attn_decode_workspace_bytes(int batch, int max_seqlen, int num_q_heads,
                                        int num_kv_heads, int head_dim, int page_size,
                                        int num_splits);

/*
 * Multi-token decode: q_len new query tokens per sequence against the paged
 * KV cache, for speculative or multi-token-prediction drafts that verify
 * several tokens in one step ("GPT-OSS on day 0" mentions both; the
 * attention is the one of section Sink Attention, split along the key
 * length exactly as in sink_attn_decode, sink only in the first chunk).
 *
 * The q_len new tokens are the LAST q_len tokens already written to each
 * sequence's cache: with L = seqlens[b], new token t (0-based) sits at
 * position L - q_len + t and sees keys 0 .. L - q_len + t (causal among the
 * new tokens, every older token visible).  If L < q_len, the tokens placed
 * before the cache start see no key: out = 0 and lse = sink (or -inf).
 *
 *   q       bf16 [batch, q_len, num_q_heads, head_dim]
 *   out     [batch, q_len, num_q_heads, head_dim], bf16 or fp32 per out_dtype
 *   lse     optional fp32 [batch, q_len, num_q_heads]; NULL to skip
 *   q_len   1 .. 4096.  The query rows that share one kv head (group x
 *           q_len) are processed together, so every page is read once for
 *           all of them: up to 16 rows with warp-level MMAs, more on the
 *           tensor cores in tiles of 128 (new token, query head) rows, which
 *           also skip the key tiles no row of a tile can see.  Limits:
 *           num_q_heads / num_kv_heads <= 16 and batch x ceil(q_len /
 *           floor(128 / group)) <= 65535.
 *   workspace
 *           at least sink_attn_decode_multi_workspace_bytes(...) bytes,
 *           256-byte aligned, or NULL (allocated in stream order).
 * Every other argument, limit and error is that of sink_attn_decode, which
 * equals this call with q_len = 1.
 */
int sink_attn_decode_multi(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, int page_table_stride,
                           const int32_t* seqlens, int batch, int q_len, int max_seqlen,
                           int num_pages, const float* sinks, int num_q_heads, int num_kv_heads,
                           int head_dim, int page_size, float scale, int num_splits,
                           void* out, int out_dtype, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace sink_attn_decode_multi needs (0 when no sequence is
 * split); (size_t)-1 for arguments it would reject on size grounds.
 */
size_t sink_attn_decode_multi_workspace_bytes(int batch, int q_len, int max_seqlen, int num_q_heads,
                                              int num_kv_heads, int head_dim, int page_size,
                                              int num_splits);

/*
 * Chunked prefill against the paged KV cache: a run of new tokens per
 * sequence, already appended to its paged cache, attends causally to the
 * whole cache ("GPT-OSS on day 0", section Sink Attention; the same online
 * softmax, sink counted once, in the first chunk of the key length when the
 * keys are split).  This is how a long prompt is prefilled piece by piece, or
 * new tokens are appended to a sequence that already has a cache.
 *
 * Sequence b has n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens; they
 * are the LAST n_b of its L_b = seqlens_k[b] cached tokens, so new token t
 * (0-based) sits at position L_b - n_b + t and sees keys 0 .. L_b - n_b + t.
 * n_b = L_b is plain causal prefill; n_b = 1 is decode.  New tokens placed
 * before the cache start (n_b > L_b) see no key: out = 0, lse = sink.
 *
 *   q             bf16 [total_q, num_q_heads, head_dim], packed by cu_seqlens_q
 *   k_pages, v_pages, page_table, page_table_stride, num_pages, sinks,
 *   num_q_heads, num_kv_heads, head_dim, page_size, scale, num_splits
 *                 as in sink_attn_decode
 *   cu_seqlens_q  int32 [batch + 1], DEVICE: cu[0] = 0, non-decreasing,
 *                 cu[batch] = total_q
 *   seqlens_k     int32 [batch], DEVICE: cached tokens of each sequence, the
 *                 new ones included
 *   total_q, max_seqlen_q, max_seqlen_k
 *                 host values: max_seqlen_q >= every n_b, max_seqlen_k >=
 *                 every L_b and <= page_table_stride * page_size
 *   out           [total_q, num_q_heads, head_dim], bf16 or fp32 per out_dtype
 *   lse           optional fp32 [total_q, num_q_heads]; NULL to skip
 *   workspace     at least sink_attn_prefill_paged_workspace_bytes(...)
 *                 bytes (0 when no sequence's keys are split: with num_splits
 *                 = 0 that is the case once the new tokens alone fill the
 *                 GPU), 256-byte aligned, or NULL (allocated in stream order)
 * Runs on the tensor cores in tiles of 128 (new token, query head) rows of
 * one kv head; key tiles no row of a tile can see are skipped.
 * Limits: num_q_heads / num_kv_heads <= 16; batch x ceil(max_seqlen_q /
 * floor(128 / group)) <= 65535; total_q * num_q_heads < 2^31.
 * batch == 0 or total_q == 0 is a no-op returning SINK_ATTN_OK.
 */
int sink_attn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int32_t* page_table, int page_table_stride,
                            const int32_t* cu_seqlens_q, const int32_t* seqlens_k, int batch,
                            int total_q, int max_seqlen_q, int max_seqlen_k, int num_pages,
                            const float* sinks, int num_q_heads, int num_kv_heads, int head_dim,
                            int page_size, float scale, int num_splits,
                            void* out, int out_dtype, float* lse,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace sink_attn_prefill_paged needs; (size_t)-1 for arguments
 * it would reject on size grounds. */
size_t sink_attn_prefill_paged_workspace_bytes(int batch, int total_q, int max_seqlen_q,
                                               int max_seqlen_k, int num_q_heads,
                                               int num_kv_heads, int head_dim, int page_size,
                                               int num_splits);

/*
 * The largest number of chunks any sequence gets for these arguments
 * (the grid's chunk dimension); 0 for arguments sink_attn_decode would reject.
 */
int sink_attn_decode_max_splits(int batch, int max_seqlen, int num_kv_heads, int page_size,
                                int num_splits);

/*
 * sink_attn_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that are not allowed to call cudaMalloc or any other allocator when they
 * run decode -- code working inside a memory budget fixed in advance, or a
 * host framework whose decode step forbids allocation.  sink_attn_decode
 * would otherwise need a caller workspace or allocate one in stream order.
 *
 * Same arguments and results as sink_attn_decode, without the workspace:
 * the per-chunk partial states go to one scratch array owned by the library,
 * SINK_ATTN_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory that every GPU
 * loading the library holds until the process exits.  Nothing is allocated.
 *   - Calls whose partial states need more than that (see
 *     sink_attn_decode_workspace_bytes) return SINK_ATTN_ERR_UNSUPPORTED and
 *     enqueue nothing; e.g. batch 64 x 8192 tokens, 64/8 heads, 8 chunks
 *     needs 8.25 MiB and fits.
 *   - Every call shares the one array: calls whose kernels overlap on the GPU
 *     (different streams, or different threads) race and corrupt each other's
 *     results; serialise them.  The array keeps the last call's contents;
 *     nothing in it needs clearing between calls.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: resetting the device (cudaDeviceReset) after that first call is
 *     not supported.
 *   - If any call reported SINK_ATTN_ERR_TIMEOUT through
 *     sink_attn_get_device_error(), the outputs of the calls it covers are
 *     undefined.
 */
#define SINK_ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)

int sink_attn_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                             const int32_t* page_table, int page_table_stride,
                             const int32_t* seqlens, int batch, int max_seqlen, int num_pages,
                             const float* sinks, int num_q_heads, int num_kv_heads, int head_dim,
                             int page_size, float scale, int num_splits,
                             void* out, int out_dtype, float* lse, void* stream);

/*
 * QKV bias + rotary position encoding with YaRN frequencies, applied to the
 * projections before attention ("GPT-OSS on day 0", model overview: YaRN
 * positional encoding as in DeepSeek-V3, QKV projections with biases as in
 * Qwen 2; the pages give no formula, the published definitions are used).
 *
 * In place, for every token t and head:
 *   q[t,h] <- rot(q[t,h] + q_bias[h]),  k[t,g] <- rot(k[t,g] + k_bias[g]),
 *   v[t,g] <- v[t,g] + v_bias[g]
 * where rot rotates each plane (dim i, dim i + D/2) by the angle
 * positions[t] * inv_freq[i] and multiplies the result by attn_factor.  The
 * angle is formed modulo one turn as a 64-bit fixed-point product of the
 * position and the frequency (in turns per position, from the fp64 table),
 * so it keeps the precision of the fp64 frequency at every int32 position
 * (within ~1e-7 rad before sincospif); the sum and rotation run in fp32, the
 * result is rounded once to bf16.
 *
 *   q, k, v     bf16 [num_tokens, H, head_dim] (H = num_q_heads for q,
 *               num_kv_heads for k and v), DEVICE, modified in place.  q may
 *               be NULL: only k and v are processed, for attention calls
 *               that rotate q themselves (sink_attn_prefill_rope,
 *               sink_attn_decode_rope).
 *   q_bias, k_bias, v_bias
 *               bf16 [H, head_dim] DEVICE, or NULL for no bias
 *   positions   int32 [num_tokens] DEVICE: position of each token in its
 *               sequence (e.g. L - n + t for the n new tokens of a cache of L)
 *   inv_freq    fp64 [head_dim / 2] DEVICE, radians per position
 *               (sink_attn_yarn_inv_freq fills it)
 *   attn_factor YaRN's temperature (sink_attn_yarn_inv_freq), 1 for plain RoPE
 *   slot_mapping
 *               optional int32 [num_tokens] DEVICE: cache slot (page *
 *               page_size + offset) of each token; when given, the rotated k
 *               and the biased v are also written to k_pages / v_pages
 *               ([num_pages, num_kv_heads, page_size, head_dim] bf16) there.
 *               Slots < 0 or past the pool are skipped.  NULL: no cache write.
 * Limits: head_dim == 64, page_size == 16, num_tokens * num_q_heads < 2^31.
 * num_tokens == 0 is a no-op returning SINK_ATTN_OK.
 */
int sink_attn_qkv_rope(void* q, void* k, void* v, const void* q_bias, const void* k_bias,
                       const void* v_bias, const int32_t* positions, const double* inv_freq,
                       float attn_factor, int num_tokens, int num_q_heads, int num_kv_heads,
                       int head_dim, const int32_t* slot_mapping, void* k_pages, void* v_pages,
                       int num_pages, int page_size, void* stream);

/*
 * YaRN rotary frequencies (host computation, no GPU): for plane i the base
 * frequency theta_i = base^(-2i/head_dim); with factor s > 1 each plane's
 * number of turns over the original context, r = original_max_position *
 * theta_i / (2 pi), sets a ramp g = clamp((r - beta_slow) / (beta_fast -
 * beta_slow), 0, 1) and the frequency becomes (1 - g) theta_i / s + g theta_i
 * (YaRN's "NTK-by-parts" interpolation, linear in r as the YaRN paper writes
 * it); attn_factor = 0.1 ln(s) + 1.  s <= 1 gives plain RoPE and 1.
 *   inv_freq     HOST fp64 [head_dim / 2], written
 *   attn_factor  HOST fp32, written
 * Returns SINK_ATTN_ERR_INVALID_ARG for odd head_dim, base <= 1, factor <= 0,
 * or (factor > 1) original_max_position <= 0 or not 0 < beta_slow < beta_fast.
 */
int sink_attn_yarn_inv_freq(int head_dim, double base, double factor, int original_max_position,
                            double beta_fast, double beta_slow, double* inv_freq,
                            float* attn_factor);

/* Static, human-readable name of a status code (never NULL). */
const char* sink_attn_status_string(int status);

/*
 * Synchronises `stream`, then reports (and clears) any timeout recorded by a
 * bounded device-side wait on the current device since the last call:
 * SINK_ATTN_OK, SINK_ATTN_ERR_TIMEOUT, or SINK_ATTN_ERR_CUDA if the sync or
 * the read failed.
 */
int sink_attn_get_device_error(void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int sink_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SINK_ATTN_H_ */
