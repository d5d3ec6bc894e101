// Split-KV decode for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: code that runs inside a pre-planned memory budget, or a
// host framework that forbids allocation on its decode path.  For them,
// sink_attn_decode_noalloc keeps the per-chunk partial states in one
// library-owned device array, declared below at file scope.  Every GPU that
// loads this library holds that array (SINK_ATTN_NOALLOC_SCRATCH_BYTES) until
// the process exits.
//
// In host code the array's name is only a host-side stand-in for the symbol,
// never a device address: its device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and that address is
// what the kernels receive.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/sink_attn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SINK_ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SINK_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return SINK_ATTN_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SINK_ATTN_OK;
}

}  // namespace

extern "C" int sink_attn_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                        const int32_t* page_table, int page_table_stride, const int32_t* seqlens,
                                        int batch, int max_seqlen, int num_pages, const float* sinks,
                                        int num_q_heads, int num_kv_heads, int head_dim, int page_size, float scale,
                                        int num_splits, void* out, int out_dtype, float* lse, void* stream) {
  const size_t need = sink_attn_decode_workspace_bytes(batch, max_seqlen, num_q_heads, num_kv_heads, head_dim,
                                                       page_size, num_splits);
  // Arguments the decode rejects are passed through so it reports the exact
  // status; a valid call whose partial states do not fit is refused here.
  if (need != (size_t)-1 && need > (size_t)SINK_ATTN_NOALLOC_SCRATCH_BYTES) return SINK_ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != SINK_ATTN_OK) return st;
  // Every partial slot the merge kernel reads is written by this call's chunk
  // kernel first (one query token per sequence runs on the split kernel, which
  // has no bounded wait that could give up half way), so the contents left by
  // an earlier call never need clearing.
  return sink_attn_decode(q, k_pages, v_pages, page_table, page_table_stride, seqlens, batch, max_seqlen, num_pages,
                          sinks, num_q_heads, num_kv_heads, head_dim, page_size, scale, num_splits, out, out_dtype,
                          lse, scratch, (size_t)SINK_ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
