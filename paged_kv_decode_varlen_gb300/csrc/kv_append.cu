// KV append: scatter this step's new K/V rows into their pool slots.
//
// "Inference optimisation" (AI-infra book ch. 8) §8.1.1: prefill stores the
// keys and values of each layer; §8.3.1: the sequence grows into a newly
// allocated block when the last one is full.  The slot of each new token is
// given by slot_mapping (block * 16 + offset); negative means padding.
//
// One (token, kv head) row is 256 B of K and 256 B of V.  Sixteen threads
// move one row with 16-byte loads and stores, so a warp moves two rows of K
// and two of V per instruction pair, fully coalesced on both sides.
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kLanesPerRow = kHeadDim * 2 / 16;  // 16 x 16 B = 256 B

__global__ void __launch_bounds__(kThreads) kv_append_kernel(const AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t rows = p.n_tokens * p.num_kv_heads;
  const int64_t stride = (int64_t)gridDim.x * (kThreads / kLanesPerRow);
  const int lane16 = threadIdx.x % kLanesPerRow;
  for (int64_t row = (int64_t)blockIdx.x * (kThreads / kLanesPerRow) + threadIdx.x / kLanesPerRow; row < rows;
       row += stride) {
    const int64_t tok = row / p.num_kv_heads;
    const int h = (int)(row % p.num_kv_heads);
    const int64_t slot = p.slot_mapping[tok];
    if (slot < 0) continue;
    const int64_t block = slot / kPage;
    const int off = (int)(slot % kPage);
    if (block >= p.num_blocks) {
      if (lane16 == 0) record_error(p.err, PA_ERR_DEVICE_INDEX);
      continue;
    }
    const int64_t src = row * kHeadDim;                                            // [tok, h, :]
    const int64_t dst = ((block * p.num_kv_heads + h) * kPage + off) * kHeadDim;   // [block, h, off, :]
    const uint4 kv = reinterpret_cast<const uint4*>(p.k_new + src)[lane16];
    const uint4 vv = reinterpret_cast<const uint4*>(p.v_new + src)[lane16];
    reinterpret_cast<uint4*>(p.k_cache + dst)[lane16] = kv;
    reinterpret_cast<uint4*>(p.v_cache + dst)[lane16] = vv;
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t rows = p.n_tokens * p.num_kv_heads;
  const int rows_per_cta = kThreads / kLanesPerRow;
  int64_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > 65535) grid = 65535;
  return launch_pdl(kv_append_kernel, dim3((unsigned)grid), dim3(kThreads), 0, stream, p);
}

}  // namespace pa
