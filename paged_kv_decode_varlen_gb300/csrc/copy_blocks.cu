// Block copy for copy-on-write: before a branch writes into a block it
// shares with another request it gets its own copy; the filled read-only
// blocks stay shared ("Inference optimisation", AI-infra book ch. 8, §8.3.2
// and Fig. 8-15).  Pair i copies the whole block src[i] -- every kv head and
// token slot, K and V (2 x 32 KiB for 8 kv heads) -- into block dst[i].
//
// HBM-bound: 16-byte loads and stores, consecutive threads on consecutive
// 16-byte words of one block, grid-stride over all pairs.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(const CopyParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t per_pair = 2 * p.block_vecs;  // K then V
  const int64_t total = p.n_pairs * per_pair;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total; i += (int64_t)gridDim.x * kThreads) {
    const int64_t pair = i / per_pair;
    const int64_t w = i - pair * per_pair;
    const int32_t s = p.src[pair], d = p.dst[pair];
    if (s < 0 || s >= p.num_blocks || d < 0 || d >= p.num_blocks) {
      if (w == 0) record_error(p.err, PA_ERR_DEVICE_INDEX);
      continue;
    }
    uint4* cache = reinterpret_cast<uint4*>(w < p.block_vecs ? p.k_cache : p.v_cache);
    const int64_t v = w < p.block_vecs ? w : w - p.block_vecs;
    cache[(int64_t)d * p.block_vecs + v] = cache[(int64_t)s * p.block_vecs + v];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream) {
  const int64_t total = p.n_pairs * 2 * p.block_vecs;
  const int64_t grid = std::min<int64_t>((total + kThreads - 1) / kThreads, 152 * 16);
  return launch_pdl(copy_blocks_kernel, dim3((unsigned)grid), dim3(kThreads), 0, stream, p);
}

}  // namespace pa
