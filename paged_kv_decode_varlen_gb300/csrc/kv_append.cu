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
#include <cuda_fp16.h>

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

// q8_0 pages ("Inference optimisation" §8.4.2 and Fig. 8-23: 32 values
// share one 2-byte scale next to their 8-bit codes).  A (block, kv head)
// slab is 16 x 128 codes, then 16 x 4 binary16 scales.  Per 32-value group:
// d = max|x| / 127 (binary32), stored as binary16 (round to nearest even);
// code = rint(x / d16) clamped to [-127, 127] with d16 the stored scale
// (all zero when d16 is 0).  The 16 lanes of a row hold 8 values each, so a
// group is 4 adjacent lanes.
constexpr int kQ8Slab = kPage * kHeadDim + kPage * (kHeadDim / 32) * 2;

__device__ __forceinline__ void quantize8_q8(const uint4& x, unsigned mask, uint2& codes, uint16_t& scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 2));
  const __half h = __float2half_rn(amax / 127.f);
  const float d16 = __half2float(h);
  uint32_t c[2] = {0u, 0u};
  if (d16 != 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float t = fminf(fmaxf(rintf(v[i] / d16), -127.f), 127.f);
      c[i >> 2] |= ((uint32_t)(int32_t)t & 0xffu) << (8 * (i & 3));
    }
  }
  codes = make_uint2(c[0], c[1]);
  scale = __half_as_ushort(h);
}

__global__ void __launch_bounds__(kThreads) kv_append_q8_kernel(const AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t rows = p.n_tokens * p.num_kv_heads;
  const int64_t stride = (int64_t)gridDim.x * (kThreads / kLanesPerRow);
  const int lane16 = threadIdx.x % kLanesPerRow;
  // the 16 lanes of this row (rows never split across a warp boundary)
  const unsigned mask = 0xffffu << (threadIdx.x & 16);
  uint8_t* kc = reinterpret_cast<uint8_t*>(p.k_cache);
  uint8_t* vc = reinterpret_cast<uint8_t*>(p.v_cache);
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
    const int64_t src = row * kHeadDim;
    const size_t slab = ((size_t)block * p.num_kv_heads + h) * kQ8Slab;
    const size_t code_at = slab + (size_t)off * kHeadDim + 8 * lane16;
    const size_t scale_at = slab + kPage * kHeadDim + 2 * ((size_t)off * (kHeadDim / 32) + lane16 / 4);
    uint2 codes;
    uint16_t scale;
    quantize8_q8(reinterpret_cast<const uint4*>(p.k_new + src)[lane16], mask, codes, scale);
    *reinterpret_cast<uint2*>(kc + code_at) = codes;
    if ((lane16 & 3) == 0) *reinterpret_cast<uint16_t*>(kc + scale_at) = scale;
    quantize8_q8(reinterpret_cast<const uint4*>(p.v_new + src)[lane16], mask, codes, scale);
    *reinterpret_cast<uint2*>(vc + code_at) = codes;
    if ((lane16 & 3) == 0) *reinterpret_cast<uint16_t*>(vc + scale_at) = scale;
  }
}

}  // namespace

cudaError_t launch_kv_append_q8(const AppendParams& p, cudaStream_t stream) {
  const int64_t rows = p.n_tokens * p.num_kv_heads;
  const int rows_per_cta = kThreads / kLanesPerRow;
  int64_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > 65535) grid = 65535;
  return launch_pdl(kv_append_q8_kernel, dim3((unsigned)grid), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t rows = p.n_tokens * p.num_kv_heads;
  const int rows_per_cta = kThreads / kLanesPerRow;
  int64_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > 65535) grid = 65535;
  return launch_pdl(kv_append_kernel, dim3((unsigned)grid), dim3(kThreads), 0, stream, p);
}

}  // namespace pa
