// pa_attention_varlen_noalloc: the attention call for callers that cannot
// allocate device memory.
//
// pa_attention_varlen needs a caller-provided workspace (the error word, the
// per-(request, kv head) counters of the persistent decode kernel and the
// partial results of key ranges cut between CTAs).  Some callers cannot
// obtain one: a real-time serving loop that must not touch the allocator
// between steps, a host framework whose device memory is all handed out to
// its own pool, or a plugin that is given only its input and output
// pointers.  This entry point serves them with a fixed scratch array that
// lives in the library's own device memory for as long as the library is
// loaded, on every GPU that loads it; it allocates nothing per call.
//
// The array is shared by every call on a device: calls on that device must
// not overlap on the GPU (they would race on the counters and partials);
// issue them on one stream or order them.  Each call first clears the part
// that must start at zero (error word and counters) on its stream.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "pa.h"

namespace {

constexpr size_t kNoAllocBytes = size_t(24) << 20;  // PA_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached.
pa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_attention_varlen_noalloc(
    const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks, const int32_t* block_tables,
    int32_t max_blocks_per_req, const int32_t* seq_lens, const int32_t* qo_indptr, const int32_t* seq_lens_host,
    const int32_t* qo_indptr_host, int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, float sm_scale, void* out, float* lse, int32_t* device_error,
    pa_stream_t stream) {
  // the same bound as pa_attention_varlen, checked before seq_lens_host is read
  if (!seq_lens_host || !qo_indptr_host || num_reqs < 0 || num_reqs > 65535)
    return pa::set_error(PA_ERR_INVALID_ARG, "noalloc: host metadata pointers and num_reqs in [0, 65535] are required");
  int32_t max_len = 1;
  for (int r = 0; r < num_reqs; ++r) max_len = seq_lens_host[r] > max_len ? seq_lens_host[r] : max_len;
  const size_t need = pa_attention_workspace_size(num_reqs, total_q, num_q_heads, head_dim, max_len);
  if (need == 0 || need > kNoAllocBytes)
    return pa::set_error(PA_ERR_UNSUPPORTED,
                         "noalloc: this batch needs %zu bytes of scratch, more than the fixed %zu bytes "
                         "(PA_NOALLOC_SCRATCH_BYTES); use pa_attention_varlen with a workspace",
                         need, kNoAllocBytes);
  void* ws = nullptr;
  pa_status s = scratch_address(&ws);
  if (s != PA_OK) return pa::set_error(s, "noalloc: cannot look up the scratch array on this device");
  // error word and counters must start at zero: everything below the first
  // partial-result byte, which is at or below 256 + 4 * num_reqs * Hkv
  // rounded up to 256 bytes
  const size_t clear = PA_ERROR_WORD_BYTES +
                       ((size_t(num_reqs > 0 ? num_reqs : 0) * size_t(num_kv_heads > 0 ? num_kv_heads : 1) * 4 +
                         255) & ~size_t(255));
  if (cudaMemsetAsync(ws, 0, clear < need ? clear : need, stream) != cudaSuccess)
    return pa::set_error(PA_ERR_CUDA, "noalloc: clearing the scratch counters failed");
  s = pa_attention_varlen(q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                          seq_lens_host, qo_indptr_host, num_reqs, total_q, num_q_heads, num_kv_heads, head_dim,
                          block_size, sm_scale, out, lse, ws, kNoAllocBytes, stream);
  if (s != PA_OK) return s;
  if (device_error &&
      cudaMemcpyAsync(device_error, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return pa::set_error(PA_ERR_CUDA, "noalloc: copying the error word failed");
  return PA_OK;
}
