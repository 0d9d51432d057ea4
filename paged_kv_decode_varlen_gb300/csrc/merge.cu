// LSE merge of two partial attentions over disjoint key sets.
//
//   M = max(lse_a, lse_b); w_x = exp(lse_x - M)
//   o = (w_a o_a + w_b o_b) / (w_a + w_b); lse = M + ln(w_a + w_b)
//
// A part with lse = -inf weighs 0 (its o is not read); two empty parts give
// o = 0, lse = -inf.  Element-wise and HBM-bound: one thread handles eight
// dims (one 16-byte load of each input), fp32 arithmetic, one RNE rounding.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int vecs_per_row = p.head_dim / 8;
  const int64_t n = p.rows * p.num_heads * vecs_per_row;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
    const int64_t rh = i / vecs_per_row;  // (row, head)
    const int vec = (int)(i % vecs_per_row);
    const float la = p.lse_a[rh], lb = p.lse_b[rh];
    const float M = fmaxf(la, lb);
    uint4 res = make_uint4(0, 0, 0, 0);
    float lse = -INFINITY;
    if (M != -INFINITY) {
      const float wa = (la == -INFINITY) ? 0.f : expf(la - M);
      const float wb = (lb == -INFINITY) ? 0.f : expf(lb - M);
      const float inv = 1.f / (wa + wb);
      float fa[8], fb[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) fa[j] = fb[j] = 0.f;
      if (wa > 0.f) {
        const uint4 a = reinterpret_cast<const uint4*>(p.o_a + rh * p.head_dim)[vec];
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          fa[2 * j] = wa * bf16lo(w[j]);
          fa[2 * j + 1] = wa * bf16hi(w[j]);
        }
      }
      if (wb > 0.f) {
        const uint4 b = reinterpret_cast<const uint4*>(p.o_b + rh * p.head_dim)[vec];
        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          fb[2 * j] = wb * bf16lo(w[j]);
          fb[2 * j + 1] = wb * bf16hi(w[j]);
        }
      }
      res.x = pack_bf16x2((fa[0] + fb[0]) * inv, (fa[1] + fb[1]) * inv);
      res.y = pack_bf16x2((fa[2] + fb[2]) * inv, (fa[3] + fb[3]) * inv);
      res.z = pack_bf16x2((fa[4] + fb[4]) * inv, (fa[5] + fb[5]) * inv);
      res.w = pack_bf16x2((fa[6] + fb[6]) * inv, (fa[7] + fb[7]) * inv);
      lse = M + logf(wa + wb);
    }
    // this thread read exactly the 16 bytes of o_a / o_b it overwrites, so
    // o_out may alias either input (lse_out may not: other threads of the
    // same row still read lse_a / lse_b)
    reinterpret_cast<uint4*>(p.o_out + rh * p.head_dim)[vec] = res;
    if (p.lse_out && vec == 0) p.lse_out[rh] = lse;
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int64_t n = p.rows * p.num_heads * (p.head_dim / 8);
  int64_t grid = (n + kThreads - 1) / kThreads;
  if (grid > 65535 * 4) grid = 65535 * 4;
  if (grid < 1) grid = 1;
  return launch_pdl(merge_kernel, dim3((unsigned)grid), dim3(kThreads), 0, stream, p);
}

}  // namespace pa
