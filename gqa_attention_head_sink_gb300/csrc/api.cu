// C ABI of the sink-attention library: argument validation, planning, TMA
// tensor-map encoding, workspace handling and kernel launches.  The entry
// points are declared (and documented) in include/sink_attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "../../include/sink_attn.h"
#include "decode.h"
#include "prefill.h"
#include "rope.h"

namespace sa {

// Timeouts recorded by bounded device-side waits (see common.cuh).
__device__ unsigned g_error_word;

namespace {

constexpr int kHeadDim = 64;
constexpr int kPageSize = 16;
constexpr int kMaxSplits = 256;
constexpr int kMaxGroupDecode = 16;
// Query rows per kv head (group * new tokens) above which decode runs on the
// tensor cores (128-row tiles) instead of warp-level MMAs (16-row tiles).
constexpr int kTensorCoreMinRows = 17;
constexpr int kMaxDecodeTokens = 4096;  // new tokens per sequence in one decode call
constexpr int kMaxDevices = 64;
// Chunk sizing for num_splits == 0.  The split kernel (four small CTAs per
// SM) aims at about this many CTAs in the chunk grid (8 per SM of a 152-SM
// GB300) with 16..128 pages per chunk.
constexpr long long kDecodeTargetCtas = 152 * 8;
constexpr int kMinSplitPages = 16;
constexpr int kMaxSplitPages = 128;
// The tensor-core kernel (two large CTAs per SM, each paying a Q load and a
// first-tile latency of ~2.5 us before its first tile) aims at about 1.5
// waves of its CTAs, with chunks as long as that allows: at batch 64 x 8192
// one chunk per sequence (512 CTAs) ran at 85-90 % of the HBM copy figure for
// 4..16 new tokens, four chunks at 69-86 %.
constexpr long long kDecodeTcTargetCtas = 152 * 3;

std::mutex g_mutex;
unsigned* g_err_ptr[kMaxDevices] = {};
bool g_prefill_attr_set[kMaxDevices] = {};
bool g_decode_attr_set[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaMemPool_t g_ws_pool[kMaxDevices] = {};
bool g_ws_pool_failed[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace for a call that passes none, in stream order on `s`.  Outside
// stream capture it comes from a library-owned pool per device whose freed
// memory stays reserved for later calls (release threshold: unlimited), so a
// call after a synchronize does not go back to the driver; during capture (or
// if the pool cannot be made) from cudaMallocAsync, which capture records as a
// graph allocation node.
cudaError_t workspace_alloc(void** ws, size_t bytes, cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  int dev = -1;
  if (cap == cudaStreamCaptureStatusNone && cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
    cudaMemPool_t pool = nullptr;
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      if (!g_ws_pool[dev] && !g_ws_pool_failed[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        uint64_t keep = UINT64_MAX;
        if (cudaMemPoolCreate(&p, &props) == cudaSuccess &&
            cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep) == cudaSuccess) {
          g_ws_pool[dev] = p;
        } else {
          if (p) cudaMemPoolDestroy(p);
          cudaGetLastError();
          g_ws_pool_failed[dev] = true;
        }
      }
      pool = g_ws_pool[dev];
    }
    if (pool) return cudaMallocFromPoolAsync(ws, bytes, pool, s);
  }
  return cudaMallocAsync(ws, bytes, s);
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("SINK_ATTN_WAIT_LIMIT_MS");
    long long ms = s ? std::atoll(s) : 4000;
    if (ms <= 0) ms = 4000;
    return (uint64_t)ms * 1000000ull;
  }();
  return v;
}

// Failure-path testing only: SINK_ATTN_DEBUG_WITHHOLD_COPIES=1 makes the TMA
// producers issue nothing, so every bounded wait gives up and the call reports
// SINK_ATTN_ERR_TIMEOUT through sink_attn_get_device_error().  Read once.
int withhold_copies() {
  static int v = [] {
    const char* s = std::getenv("SINK_ATTN_DEBUG_WITHHOLD_COPIES");
    return (s && s[0] == '1') ? 1 : 0;
  }();
  return v;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return SINK_ATTN_ERR_UNSUPPORTED;
  return SINK_ATTN_OK;
}

int error_word(int dev, unsigned** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_ptr[dev];
  return SINK_ATTN_OK;
}

int get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return SINK_ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return SINK_ATTN_OK;
}

// 2-D bf16 tensor map over a row-major [rows, 64] view (128-byte rows) with
// boxes of `box_rows` x 64 and the 128-byte swizzle.
int encode_rows64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_stride_bytes, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int st = get_encoder(&enc);
  if (st) return st;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
  cuuint32_t box[2] = {(cuuint32_t)kHeadDim, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

// 3-D bf16 tensor map over a packed [tokens, heads, 64] tensor, boxes of
// box_tokens tokens x box_heads heads x 64 dims, 128-byte swizzle.  A box
// lands as box_tokens * box_heads rows of 128 bytes, token-major.
int encode_tokens_heads(CUtensorMap* map, const void* base, uint64_t tokens, uint64_t heads, uint32_t box_tokens,
                        uint32_t box_heads = 1) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int st = get_encoder(&enc);
  if (st) return st;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)heads * kHeadDim * 2};
  cuuint32_t box[3] = {(cuuint32_t)kHeadDim, box_heads, box_tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

struct DecodePlan {
  int max_splits;
  int split_pages;
  bool direct;
  size_t ws_bytes;
};

// Rows of one tensor-core decode tile are (new token, query head) pairs of one
// kv head: this many tokens per tile, and this many tiles per sequence
// (max_q = the most new tokens any sequence has).
int decode_tokens_per_tile(int group, int max_q) { return std::max(1, std::min(max_q, kDecodeTcRows / group)); }
int decode_row_tiles(int group, int max_q, bool tensor_cores) {
  if (!tensor_cores) return 1;
  const int tpt = decode_tokens_per_tile(group, max_q);
  return std::max(1, (max_q + tpt - 1) / tpt);
}
bool decode_uses_tensor_cores(int group, int q_len) { return group * q_len >= kTensorCoreMinRows; }

// Chunking of the key length.  num_splits > 0: that many chunks per sequence.
// 0: chunks of 16..128 pages aiming at kDecodeTargetCtas CTAs; when the row
// tiles alone give that many CTAs (long runs of new tokens), the chunks grow
// past 128 pages so that the key length is not split needlessly.
bool plan_decode(int batch, int max_q, long long total_q, int max_seqlen, int num_q_heads, int num_kv_heads,
                 int num_splits, bool tensor_cores, DecodePlan* pl) {
  if (batch < 0 || max_q < 0 || total_q < 0 || max_seqlen < 0 || num_kv_heads <= 0 || num_q_heads <= 0) return false;
  if (num_q_heads % num_kv_heads) return false;
  const int row_tiles = decode_row_tiles(num_q_heads / num_kv_heads, std::max(1, max_q), tensor_cores);
  if (num_splits < 0 || num_splits > kMaxSplits) return false;
  const long long max_pages = ((long long)max_seqlen + kPageSize - 1) / kPageSize;
  int split_pages = kMaxSplitPages;
  int max_splits;
  if (num_splits > 0) {
    max_splits = (int)std::max(1LL, std::min<long long>(num_splits, max_pages));
  } else {
    const long long target = tensor_cores ? kDecodeTcTargetCtas : kDecodeTargetCtas;
    long long sp = ((long long)batch * row_tiles * num_kv_heads * max_pages + target - 1) / target;
    sp = std::max<long long>(kMinSplitPages, sp);
    if (row_tiles == 1 && !tensor_cores) sp = std::min<long long>(kMaxSplitPages, sp);
    if ((max_pages + sp - 1) / sp > kMaxSplits) sp = (max_pages + kMaxSplits - 1) / kMaxSplits;
    split_pages = (int)sp;
    max_splits = (int)std::max(1LL, (max_pages + sp - 1) / sp);
  }
  pl->max_splits = max_splits;
  pl->split_pages = split_pages;
  pl->direct = max_splits == 1;
  if (pl->direct) {
    pl->ws_bytes = 0;
  } else {
    const size_t slots = (size_t)total_q * num_q_heads * max_splits;
    const size_t o_bytes = (slots * kHeadDim * 4 + 255) / 256 * 256;
    pl->ws_bytes = o_bytes + slots * 2 * 4;
  }
  return true;
}

// Which query rows a paged call has: q_len new tokens per sequence (cu_q
// null), or per-sequence counts from the device offsets cu_q [batch + 1].
struct QueryLayout {
  const int32_t* cu_q;
  int q_len;    // uniform count when cu_q is null
  int total_q;  // rows of q and out: batch * q_len, or cu_q[batch]
  int max_q;    // no sequence has more new tokens than this
};

// Chunked prefill on the persistent prefill kernel (paged mode).
int prefill_paged_impl(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                       int page_table_stride, const int32_t* cu_seqlens_q, const int32_t* seqlens_k, int batch,
                       int total_q, int max_seqlen_q, int max_seqlen_k, int num_pages, const float* sinks,
                       int num_q_heads, int num_kv_heads, int head_dim, int page_size, float scale, void* out,
                       int out_dtype, float* lse, void* stream);

// Rotary encoding of q applied inside the decode chunk kernel.
struct RopeQ {
  const void* q_bias;
  const double* inv_freq;
  float attn_factor;
};

// Shared body of sink_attn_decode (q_len = 1), sink_attn_decode_rope,
// sink_attn_decode_multi and sink_attn_prefill_paged.
int decode_impl(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                int page_table_stride, const int32_t* seqlens, int batch, const QueryLayout& ql, int max_seqlen,
                int num_pages, const float* sinks, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                float scale, int num_splits, void* out, int out_dtype, float* lse, void* workspace,
                size_t workspace_bytes, void* stream, const RopeQ* rope = nullptr);

}  // namespace
}  // namespace sa

using namespace sa;

extern "C" {

int sink_attn_version(void) { return 100; }

const char* sink_attn_status_string(int status) {
  switch (status) {
    case SINK_ATTN_OK: return "ok";
    case SINK_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case SINK_ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case SINK_ATTN_ERR_CUDA: return "CUDA error";
    case SINK_ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case SINK_ATTN_ERR_NO_MEMORY: return "out of device memory";
    default: return "unknown status";
  }
}

int sink_attn_get_device_error(void* stream) {
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  unsigned* w;
  if ((st = error_word(dev, &w))) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
    return SINK_ATTN_ERR_TIMEOUT;
  }
  return SINK_ATTN_OK;
}

int sink_attn_decode_max_splits(int batch, int max_seqlen, int num_kv_heads, int page_size, int num_splits) {
  if (page_size != kPageSize) return 0;
  DecodePlan pl;
  if (!plan_decode(batch, 1, batch, max_seqlen, num_kv_heads, num_kv_heads, num_splits, false, &pl)) return 0;
  return pl.max_splits;
}

size_t sink_attn_decode_workspace_bytes(int batch, int max_seqlen, int num_q_heads, int num_kv_heads,
                                        int head_dim, int page_size, int num_splits) {
  return sink_attn_decode_multi_workspace_bytes(batch, 1, max_seqlen, num_q_heads, num_kv_heads, head_dim,
                                                page_size, num_splits);
}

size_t sink_attn_decode_multi_workspace_bytes(int batch, int q_len, int max_seqlen, int num_q_heads,
                                              int num_kv_heads, int head_dim, int page_size, int num_splits) {
  if (head_dim != kHeadDim || page_size != kPageSize || q_len <= 0 || num_kv_heads <= 0) return (size_t)-1;
  DecodePlan pl;
  const bool tc = decode_uses_tensor_cores(num_q_heads / num_kv_heads, q_len);
  if (!plan_decode(batch, q_len, (long long)batch * q_len, max_seqlen, num_q_heads, num_kv_heads, num_splits, tc,
                   &pl))
    return (size_t)-1;
  return pl.ws_bytes;
}

size_t sink_attn_prefill_paged_workspace_bytes(int batch, int total_q, int max_seqlen_q, int max_seqlen_k,
                                               int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                                               int num_splits) {
  if (head_dim != kHeadDim || page_size != kPageSize) return (size_t)-1;
  DecodePlan pl;
  if (!plan_decode(batch, max_seqlen_q, total_q, max_seqlen_k, num_q_heads, num_kv_heads, num_splits, true, &pl))
    return (size_t)-1;
  // the same choice as sink_attn_prefill_paged: the persistent prefill kernel splits nothing
  if (num_splits == 0 && max_seqlen_q >= kPrefillTileRows && batch <= kPrefillMaxBatch) return 0;
  return pl.ws_bytes;
}

int sink_attn_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                     int page_table_stride, const int32_t* seqlens, int batch, int max_seqlen, int num_pages,
                     const float* sinks, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                     float scale, int num_splits, void* out, int out_dtype, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream) {
  const QueryLayout ql{nullptr, 1, batch, 1};
  return decode_impl(q, k_pages, v_pages, page_table, page_table_stride, seqlens, batch, ql, max_seqlen, num_pages,
                     sinks, num_q_heads, num_kv_heads, head_dim, page_size, scale, num_splits, out, out_dtype, lse,
                     workspace, workspace_bytes, stream);
}

int sink_attn_decode_rope(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                          int page_table_stride, const int32_t* seqlens, int batch, int max_seqlen, int num_pages,
                          const float* sinks, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                          float scale, int num_splits, const void* q_bias, const double* inv_freq,
                          float attn_factor, void* out, int out_dtype, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  const QueryLayout ql{nullptr, 1, batch, 1};
  const RopeQ rope{q_bias, inv_freq, attn_factor};
  return decode_impl(q, k_pages, v_pages, page_table, page_table_stride, seqlens, batch, ql, max_seqlen, num_pages,
                     sinks, num_q_heads, num_kv_heads, head_dim, page_size, scale, num_splits, out, out_dtype, lse,
                     workspace, workspace_bytes, stream, &rope);
}

int sink_attn_decode_multi(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                           int page_table_stride, const int32_t* seqlens, int batch, int q_len, int max_seqlen,
                           int num_pages, const float* sinks, int num_q_heads, int num_kv_heads, int head_dim,
                           int page_size, float scale, int num_splits, void* out, int out_dtype, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (q_len <= 0) return SINK_ATTN_ERR_INVALID_ARG;
  if ((long long)batch * q_len >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  const QueryLayout ql{nullptr, q_len, batch * q_len, q_len};
  return decode_impl(q, k_pages, v_pages, page_table, page_table_stride, seqlens, batch, ql, max_seqlen, num_pages,
                     sinks, num_q_heads, num_kv_heads, head_dim, page_size, scale, num_splits, out, out_dtype, lse,
                     workspace, workspace_bytes, stream);
}

int sink_attn_prefill_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                            int page_table_stride, const int32_t* cu_seqlens_q, const int32_t* seqlens_k, int batch,
                            int total_q, int max_seqlen_q, int max_seqlen_k, int num_pages, const float* sinks,
                            int num_q_heads, int num_kv_heads, int head_dim, int page_size, float scale,
                            int num_splits, void* out, int out_dtype, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_q > total_q) return SINK_ATTN_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0) return SINK_ATTN_OK;
  if (!cu_seqlens_q || !aligned16(cu_seqlens_q)) return SINK_ATTN_ERR_INVALID_ARG;
  // Runs of at least a query tile of new tokens: the persistent prefill kernel
  // in paged mode (two heads per CTA sharing each K/V tile).  Shorter runs, or
  // a requested split of the key length: the tensor-core decode kernel.
  if (num_splits == 0 && max_seqlen_q >= kPrefillTileRows && batch <= kPrefillMaxBatch)
    return prefill_paged_impl(q, k_pages, v_pages, page_table, page_table_stride, cu_seqlens_q, seqlens_k, batch,
                              total_q, max_seqlen_q, max_seqlen_k, num_pages, sinks, num_q_heads, num_kv_heads,
                              head_dim, page_size, scale, out, out_dtype, lse, stream);
  const QueryLayout ql{cu_seqlens_q, 0, total_q, max_seqlen_q};
  return decode_impl(q, k_pages, v_pages, page_table, page_table_stride, seqlens_k, batch, ql, max_seqlen_k,
                     num_pages, sinks, num_q_heads, num_kv_heads, head_dim, page_size, scale, num_splits, out,
                     out_dtype, lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace sa {
namespace {

int decode_impl(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                int page_table_stride, const int32_t* seqlens, int batch, const QueryLayout& ql, int max_seqlen,
                int num_pages, const float* sinks, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                float scale, int num_splits, void* out, int out_dtype, float* lse, void* workspace,
                size_t workspace_bytes, void* stream, const RopeQ* rope) {
  // ---- validation (nothing is enqueued on failure)
  if (batch < 0 || ql.max_q < 0 || ql.total_q < 0 || max_seqlen < 0 || num_q_heads <= 0 || num_kv_heads <= 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return SINK_ATTN_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return SINK_ATTN_ERR_INVALID_ARG;
  if (out_dtype != SINK_ATTN_OUT_BF16 && out_dtype != SINK_ATTN_OUT_F32) return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || page_size != kPageSize) return SINK_ATTN_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > kMaxGroupDecode) return SINK_ATTN_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  // per-sequence counts (paged prefill) always take the tensor-core kernel
  const bool tensor_cores = ql.cu_q != nullptr || decode_uses_tensor_cores(group, ql.q_len);
  if (!ql.cu_q && ql.q_len > kMaxDecodeTokens) return SINK_ATTN_ERR_UNSUPPORTED;
  const int row_tiles = decode_row_tiles(group, std::max(1, ql.max_q), tensor_cores);
  if (batch == 0) return SINK_ATTN_OK;
  if (!q || !k_pages || !v_pages || !page_table || !seqlens || !sinks || !out) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(page_table) ||
      !aligned16(seqlens) || !aligned16(sinks) || !aligned16(out) || (lse && !aligned16(lse)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || page_table_stride <= 0) return SINK_ATTN_ERR_INVALID_ARG;
  if ((long long)page_table_stride * kPageSize < max_seqlen) return SINK_ATTN_ERR_INVALID_ARG;
  if ((long long)batch * row_tiles > 65535 || num_kv_heads > 65535) return SINK_ATTN_ERR_UNSUPPORTED;
  if ((long long)ql.total_q * num_q_heads >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  if ((long long)num_pages * num_kv_heads * kPageSize >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  DecodePlan pl;
  if (!plan_decode(batch, std::max(1, ql.max_q), ql.total_q, max_seqlen, num_q_heads, num_kv_heads, num_splits,
                   tensor_cores, &pl))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SINK_ATTN_ERR_INVALID_ARG;
  if (workspace && workspace_bytes < pl.ws_bytes) return SINK_ATTN_ERR_INVALID_ARG;
  if (rope) {
    if (!rope->inv_freq || !aligned16(rope->inv_freq) || (rope->q_bias && !aligned16(rope->q_bias)))
      return SINK_ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(rope->attn_factor)) return SINK_ATTN_ERR_INVALID_ARG;
    if (tensor_cores) return SINK_ATTN_ERR_UNSUPPORTED;  // the rotation lives in the split kernel
  }

  int dev;
  int st = current_device(&dev);
  if (st) return st;
  unsigned* err;
  if ((st = error_word(dev, &err))) return st;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_decode_attr_set[dev]) {
      if (decode_configure() != cudaSuccess || decode_tc_configure() != cudaSuccess) return SINK_ATTN_ERR_CUDA;
      g_decode_attr_set[dev] = true;
    }
  }
  // tensor-core path: K/V as [pages * Hkv * 16, 64] (one 16-row slab per copy) and q as
  // [total_q tokens, Hq, 64] (one box = one row tile); the chunk kernel reads through pointers
  const int tokens_per_tile = decode_tokens_per_tile(group, std::max(1, ql.max_q));
  CUtensorMap kmap, vmap, qmap;
  if (tensor_cores) {
    const uint64_t rows = (uint64_t)num_pages * num_kv_heads * kPageSize;
    if ((st = encode_rows64(&kmap, k_pages, rows, kHeadDim * 2, kPageSize))) return st;
    if ((st = encode_rows64(&vmap, v_pages, rows, kHeadDim * 2, kPageSize))) return st;
    if ((st = encode_tokens_heads(&qmap, q, (uint64_t)ql.total_q, num_q_heads, tokens_per_tile, group))) return st;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  bool owned = false;
  if (pl.ws_bytes && !ws) {
    if (workspace_alloc(&ws, pl.ws_bytes, s) != cudaSuccess) {
      cudaGetLastError();
      return SINK_ATTN_ERR_NO_MEMORY;
    }
    owned = true;
  }
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.page_table = page_table;
  p.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
  p.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
  p.num_pages = num_pages;
  p.seqlens = seqlens;
  p.sinks = sinks;
  p.out = out;
  p.lse = lse;
  if (pl.ws_bytes) {
    const size_t slots = (size_t)ql.total_q * num_q_heads * pl.max_splits;
    p.ws_o = static_cast<float*>(ws);
    p.ws_md = reinterpret_cast<float*>(static_cast<char*>(ws) + (slots * kHeadDim * 4 + 255) / 256 * 256);
  }
  p.err = err;
  p.batch = batch;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.stride = page_table_stride;
  p.q_len = ql.q_len;
  p.cu_q = ql.cu_q;
  p.total_q = ql.total_q;
  p.tokens_per_tile = tokens_per_tile;
  p.row_tiles = row_tiles;
  p.num_splits = num_splits;
  p.split_pages = pl.split_pages;
  p.max_splits = pl.max_splits;
  p.direct = pl.direct ? 1 : 0;
  p.out_f32 = out_dtype == SINK_ATTN_OUT_F32;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.withhold_copies = withhold_copies();
  if (rope) {
    p.q_bias = static_cast<const __nv_bfloat16*>(rope->q_bias);
    p.inv_freq = rope->inv_freq;
    p.attn_factor = rope->attn_factor;
  }
  const cudaError_t e = tensor_cores ? launch_decode_tc(qmap, kmap, vmap, p, s) : launch_decode(p, s);
  if (owned) cudaFreeAsync(ws, s);
  return e == cudaSuccess ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace sa

extern "C" {

int sink_attn_yarn_inv_freq(int head_dim, double base, double factor, int original_max_position, double beta_fast,
                            double beta_slow, double* inv_freq, float* attn_factor) {
  if (!inv_freq || !attn_factor || head_dim <= 0 || head_dim % 2) return SINK_ATTN_ERR_INVALID_ARG;
  if (!(base > 1.0) || !std::isfinite(base) || !(factor > 0.0) || !std::isfinite(factor))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (factor > 1.0 && (original_max_position <= 0 || !(beta_fast > beta_slow) || !(beta_slow > 0.0)))
    return SINK_ATTN_ERR_INVALID_ARG;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < head_dim / 2; ++i) {
    const double theta = std::pow(base, -2.0 * i / head_dim);
    double f = theta;
    if (factor > 1.0) {
      // turns of this plane over the original context decide between keeping
      // the frequency (many turns) and dividing it by the factor (< 1 turn)
      const double turns = original_max_position * theta / two_pi;
      const double ramp = std::min(1.0, std::max(0.0, (turns - beta_slow) / (beta_fast - beta_slow)));
      f = (1.0 - ramp) * theta / factor + ramp * theta;
    }
    inv_freq[i] = f;
  }
  *attn_factor = factor > 1.0 ? (float)(0.1 * std::log(factor) + 1.0) : 1.0f;
  return SINK_ATTN_OK;
}

int sink_attn_qkv_rope(void* q, void* k, void* v, const void* q_bias, const void* k_bias, const void* v_bias,
                       const int32_t* positions, const double* inv_freq, float attn_factor, int num_tokens,
                       int num_q_heads, int num_kv_heads, int head_dim, const int32_t* slot_mapping,
                       void* k_pages, void* v_pages, int num_pages, int page_size, void* stream) {
  if (num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0) return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return SINK_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(attn_factor)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return SINK_ATTN_ERR_UNSUPPORTED;
  if (num_tokens == 0) return SINK_ATTN_OK;
  if (!k || !v || !positions || !inv_freq) return SINK_ATTN_ERR_INVALID_ARG;
  if ((q && !aligned16(q)) || !aligned16(k) || !aligned16(v) || !aligned16(positions) || !aligned16(inv_freq) ||
      (q_bias && !aligned16(q_bias)) || (k_bias && !aligned16(k_bias)) || (v_bias && !aligned16(v_bias)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (slot_mapping) {
    if (!aligned16(slot_mapping) || !k_pages || !v_pages || !aligned16(k_pages) || !aligned16(v_pages))
      return SINK_ATTN_ERR_INVALID_ARG;
    if (num_pages <= 0) return SINK_ATTN_ERR_INVALID_ARG;
    if (page_size != kPageSize) return SINK_ATTN_ERR_UNSUPPORTED;
  }
  if ((long long)num_tokens * num_q_heads >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  RopeParams p{};
  p.q = static_cast<__nv_bfloat16*>(q);
  p.k = static_cast<__nv_bfloat16*>(k);
  p.v = static_cast<__nv_bfloat16*>(v);
  p.q_bias = static_cast<const __nv_bfloat16*>(q_bias);
  p.k_bias = static_cast<const __nv_bfloat16*>(k_bias);
  p.v_bias = static_cast<const __nv_bfloat16*>(v_bias);
  p.positions = positions;
  p.inv_freq = inv_freq;
  p.attn_factor = attn_factor;
  p.slot_mapping = slot_mapping;
  p.k_pages = static_cast<__nv_bfloat16*>(k_pages);
  p.v_pages = static_cast<__nv_bfloat16*>(v_pages);
  p.num_pages = num_pages;
  p.page_size = kPageSize;
  p.tokens = num_tokens;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  return launch_qkv_rope(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

}  // extern "C"

namespace sa {
namespace {

int prefill_paged_impl(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                       int page_table_stride, const int32_t* cu_seqlens_q, const int32_t* seqlens_k, int batch,
                       int total_q, int max_seqlen_q, int max_seqlen_k, int num_pages, const float* sinks,
                       int num_q_heads, int num_kv_heads, int head_dim, int page_size, float scale, void* out,
                       int out_dtype, float* lse, void* stream) {
  // ---- validation (nothing is enqueued on failure); same rules as the decode paths
  if (num_q_heads <= 0 || num_kv_heads <= 0 || max_seqlen_k < 0) return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return SINK_ATTN_ERR_INVALID_ARG;
  if (out_dtype != SINK_ATTN_OUT_BF16 && out_dtype != SINK_ATTN_OUT_F32) return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || page_size != kPageSize) return SINK_ATTN_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > kMaxGroupDecode) return SINK_ATTN_ERR_UNSUPPORTED;
  if (!q || !k_pages || !v_pages || !page_table || !seqlens_k || !sinks || !out) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(page_table) ||
      !aligned16(seqlens_k) || !aligned16(sinks) || !aligned16(out) || (lse && !aligned16(lse)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || page_table_stride <= 0) return SINK_ATTN_ERR_INVALID_ARG;
  if ((long long)page_table_stride * kPageSize < max_seqlen_k) return SINK_ATTN_ERR_INVALID_ARG;
  if (max_seqlen_q >= (1 << 24) || num_kv_heads > 65535) return SINK_ATTN_ERR_UNSUPPORTED;
  if ((long long)total_q * num_q_heads >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  if ((long long)num_pages * num_kv_heads * kPageSize >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;

  int dev;
  int st = current_device(&dev);
  if (st) return st;
  unsigned* err;
  if ((st = error_word(dev, &err))) return st;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_prefill_attr_set[dev]) {
      if (prefill_configure() != cudaSuccess) return SINK_ATTN_ERR_CUDA;
      g_prefill_attr_set[dev] = true;
    }
  }
  const uint64_t rows = (uint64_t)num_pages * num_kv_heads * kPageSize;
  CUtensorMap qmap, kmap, vmap;
  if ((st = encode_tokens_heads(&qmap, q, total_q, num_q_heads, kPrefillTileRows))) return st;
  if ((st = encode_rows64(&kmap, k_pages, rows, kHeadDim * 2, kPageSize))) return st;
  if ((st = encode_rows64(&vmap, v_pages, rows, kHeadDim * 2, kPageSize))) return st;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SINK_ATTN_ERR_CUDA;

  PrefillParams p{};
  p.cu_seqlens = cu_seqlens_q;
  p.sinks = sinks;
  p.out = out;
  p.lse = lse;
  p.err = err;
  p.batch = batch;
  p.total_tokens = total_q;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.max_qblocks = (max_seqlen_q + kPrefillTileRows - 1) / kPrefillTileRows;
  p.out_f32 = out_dtype == SINK_ATTN_OUT_F32;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.withhold_copies = withhold_copies();
  p.kv_len = seqlens_k;
  p.page_table = page_table;
  p.stride = page_table_stride;
  CUtensorMap omap = qmap;
  if (!p.out_f32 && (st = encode_tokens_heads(&omap, out, total_q, num_q_heads, kPrefillTileRows))) return st;
  cudaError_t e = launch_prefill(qmap, kmap, vmap, omap, p, sms, true, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}


// Shared body of sink_attn_prefill and sink_attn_prefill_rope (rope: the
// query rotation inside the kernel, or null).
int prefill_impl(const void* q, const void* k, const void* v, const float* sinks, const int32_t* cu_seqlens,
                 int batch, int total_tokens, int max_seqlen, int num_q_heads, int num_kv_heads, int head_dim,
                 float scale, void* out, int out_dtype, float* lse, void* stream, const RopeQ* rope) {
  if (batch < 0 || total_tokens < 0 || max_seqlen < 0 || num_q_heads <= 0 || num_kv_heads <= 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return SINK_ATTN_ERR_INVALID_ARG;
  if (out_dtype != SINK_ATTN_OUT_BF16 && out_dtype != SINK_ATTN_OUT_F32) return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return SINK_ATTN_ERR_UNSUPPORTED;
  if (max_seqlen > total_tokens) return SINK_ATTN_ERR_INVALID_ARG;
  if (rope && (!rope->inv_freq || !aligned16(rope->inv_freq) || (rope->q_bias && !aligned16(rope->q_bias)) ||
               !std::isfinite(rope->attn_factor)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (batch == 0 || total_tokens == 0) return SINK_ATTN_OK;
  if (!q || !k || !v || !sinks || !cu_seqlens || !out) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(sinks) || !aligned16(cu_seqlens) ||
      !aligned16(out) || (lse && !aligned16(lse)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (batch > kPrefillMaxBatch || max_seqlen >= (1 << 24)) return SINK_ATTN_ERR_UNSUPPORTED;
  if ((long long)total_tokens * num_q_heads >= (1LL << 31)) return SINK_ATTN_ERR_UNSUPPORTED;

  int dev;
  int st = current_device(&dev);
  if (st) return st;
  unsigned* err;
  if ((st = error_word(dev, &err))) return st;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_prefill_attr_set[dev]) {
      if (prefill_configure() != cudaSuccess) return SINK_ATTN_ERR_CUDA;
      g_prefill_attr_set[dev] = true;
    }
  }
  CUtensorMap qmap, kmap, vmap;
  if ((st = encode_tokens_heads(&qmap, q, total_tokens, num_q_heads, kPrefillTileRows))) return st;
  if ((st = encode_tokens_heads(&kmap, k, total_tokens, num_kv_heads, kPrefillKeyRows))) return st;
  if ((st = encode_tokens_heads(&vmap, v, total_tokens, num_kv_heads, kPrefillKeyRows))) return st;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SINK_ATTN_ERR_CUDA;

  PrefillParams p{};
  p.cu_seqlens = cu_seqlens;
  p.sinks = sinks;
  p.out = out;
  p.lse = lse;
  p.err = err;
  p.batch = batch;
  p.total_tokens = total_tokens;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.max_qblocks = (max_seqlen + kPrefillTileRows - 1) / kPrefillTileRows;
  p.out_f32 = out_dtype == SINK_ATTN_OUT_F32;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.withhold_copies = withhold_copies();
  if (rope) {
    p.q_bias = static_cast<const __nv_bfloat16*>(rope->q_bias);
    p.inv_freq = rope->inv_freq;
    p.attn_factor = rope->attn_factor;
  }
  CUtensorMap omap = qmap;
  if (!p.out_f32 && (st = encode_tokens_heads(&omap, out, total_tokens, num_q_heads, kPrefillTileRows))) return st;
  cudaError_t e = launch_prefill(qmap, kmap, vmap, omap, p, sms, false, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace sa

extern "C" {

int sink_attn_prefill(const void* q, const void* k, const void* v, const float* sinks, const int32_t* cu_seqlens,
                      int batch, int total_tokens, int max_seqlen, int num_q_heads, int num_kv_heads,
                      int head_dim, float scale, void* out, int out_dtype, float* lse, void* stream) {
  return prefill_impl(q, k, v, sinks, cu_seqlens, batch, total_tokens, max_seqlen, num_q_heads, num_kv_heads,
                      head_dim, scale, out, out_dtype, lse, stream, nullptr);
}

int sink_attn_prefill_rope(const void* q, const void* k, const void* v, const float* sinks,
                           const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen, int num_q_heads,
                           int num_kv_heads, int head_dim, float scale, const void* q_bias, const double* inv_freq,
                           float attn_factor, void* out, int out_dtype, float* lse, void* stream) {
  const RopeQ rope{q_bias, inv_freq, attn_factor};
  return prefill_impl(q, k, v, sinks, cu_seqlens, batch, total_tokens, max_seqlen, num_q_heads, num_kv_heads,
                      head_dim, scale, out, out_dtype, lse, stream, &rope);
}

}  // extern "C"
