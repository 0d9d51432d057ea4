// Split-KV flash-decode over a paged KV cache (decode rows, qo_len = 1), and
// the log-sum-exp combine of the splits.
//
// What is computed: for a decode row, every q head attends to all seq_len
// keys of its kv head, read through the block table ("Inference
// optimisation", AI-infra book ch. 8, §8.3.1 / Fig. 8-10; "vLLM, SGLang and
// continuous batching", section "PagedAttention").  The softmax is computed
// online in fp32 (log2 domain), and partial results over disjoint key
// ranges are merged by the log-sum-exp identity.
//
// Design for GB300 (HBM-bound; ~1 FMA per byte per q head):
//   * grid = (split, kv head, request); one CTA streams the pages of one
//     (request, kv head) key range.  Each page's K slab and V slab (4 KiB
//     each, contiguous in the HND pool) are fetched by the TMA engine with
//     two 1-D bulk copies into an 8-deep shared-memory ring guarded by
//     mbarriers, so 64 KiB per CTA (3 CTAs per SM) are in flight.
//   * The 4 q heads of the GQA group share every K/V element read: each
//     K/V byte is read from HBM once per kv head.
//   * 128 threads = 16 token slots x 8 dim chunks.  Thread (t, c) owns dims
//     [8c, 8c+8) and [64+8c, 64+8c+8) of token t of each page, so every
//     shared-memory read is a conflict-free 16-byte load and a score needs
//     only a 3-step shuffle reduction over 8 lanes.
//   * Each token slot keeps its own running max / sum / accumulator (an
//     online softmax per slot); the 16 slots are merged once at the end.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 8;

struct __align__(128) DecodeSmem {
  uint8_t k[kStages][kSlabBytes];  // reused as the slot-merge buffer (32 KiB) after the loop
  uint8_t v[kStages][kSlabBytes];
  uint64_t full[kStages];
  int32_t ids[kDecodeMaxPagesPerCta];
  float red_m[kPage][kGroup];
  float red_l[kPage][kGroup];
  int abort_flag;
};
static_assert(kStages * kSlabBytes >= kPage * kGroup * kHeadDim * 4, "merge buffer must fit in the K ring");

__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
  f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
  f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

__device__ __forceinline__ float dot8(const float* q, const uint4& w) {
  float s = q[0] * bf16lo(w.x);
  s = fmaf(q[1], bf16hi(w.x), s);
  s = fmaf(q[2], bf16lo(w.y), s);
  s = fmaf(q[3], bf16hi(w.y), s);
  s = fmaf(q[4], bf16lo(w.z), s);
  s = fmaf(q[5], bf16hi(w.z), s);
  s = fmaf(q[6], bf16lo(w.w), s);
  s = fmaf(q[7], bf16hi(w.w), s);
  return s;
}

__device__ __forceinline__ void axpy8(float* acc, float p, const uint4& w) {
  acc[0] = fmaf(p, bf16lo(w.x), acc[0]);
  acc[1] = fmaf(p, bf16hi(w.x), acc[1]);
  acc[2] = fmaf(p, bf16lo(w.y), acc[2]);
  acc[3] = fmaf(p, bf16hi(w.y), acc[3]);
  acc[4] = fmaf(p, bf16lo(w.z), acc[4]);
  acc[5] = fmaf(p, bf16hi(w.z), acc[5]);
  acc[6] = fmaf(p, bf16lo(w.w), acc[6]);
  acc[7] = fmaf(p, bf16hi(w.w), acc[7]);
}

__global__ void __launch_bounds__(kThreads, 3) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int split = blockIdx.x, kvh = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x;
  const int tok = p.qo_indptr[r];
  if (p.qo_indptr[r + 1] - tok != 1) return;  // not a decode row
  const int L = p.seq_lens[r];
  const int n_pages = (L + kPage - 1) / kPage;
  const int per = (n_pages + p.num_splits - 1) / p.num_splits;
  const int pg0 = min(n_pages, split * per);
  const int npg = min(n_pages, pg0 + per) - pg0;

  const int ts = tid >> 3;  // token slot within a page
  const int c = tid & 7;    // dim chunk

  // Block ids of this split; an id outside the pool is recorded and its
  // page is masked (and fetched from block 0 so the copy stays in bounds).
  const int32_t* table = p.block_tables + (size_t)r * p.max_blocks_per_req;
  for (int i = tid; i < npg; i += kThreads) {
    int32_t b = table[pg0 + i];
    if (b < 0 || b >= p.num_blocks) {
      record_error(p.err, PA_ERR_DEVICE_INDEX);
      b = -1;
    }
    sm.ids[i] = b;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const size_t slab_elems = (size_t)kPage * kHeadDim;
  auto issue = [&](int i) {
    const int s = i % kStages;
    const int32_t b = max(sm.ids[i], 0);
    const size_t off = ((size_t)b * p.num_kv_heads + kvh) * slab_elems;
    mbar_arrive_expect_tx(&sm.full[s], 2 * kSlabBytes);
    bulk_g2s(sm.k[s], p.k_cache + off, kSlabBytes, &sm.full[s]);
    bulk_g2s(sm.v[s], p.v_cache + off, kSlabBytes, &sm.full[s]);
  };
  if (tid == 0) {
    const int n0 = min(npg, kStages);
    for (int i = 0; i < n0; ++i) issue(i);
  }

  // q of the 4 heads of this group, scaled into the log2 domain.
  float qf[kGroup][16];
  {
    const uint16_t* qrow = p.q + ((size_t)tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const uint4 a = *reinterpret_cast<const uint4*>(qrow + g * kHeadDim + 8 * c);
      const uint4 b = *reinterpret_cast<const uint4*>(qrow + g * kHeadDim + 64 + 8 * c);
      unpack8(a, qf[g]);
      unpack8(b, qf[g] + 8);
#pragma unroll
      for (int d = 0; d < 16; ++d) qf[g][d] *= p.scale_log2;
    }
  }

  float acc[kGroup][16];
  float m[kGroup], l[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int d = 0; d < 16; ++d) acc[g][d] = 0.f;
  }

  int stop_at = npg;
  for (int i = 0; i < npg; ++i) {
    const int s = i % kStages;
    if (!mbar_wait_bounded(&sm.full[s], (uint32_t)(i / kStages) & 1u)) {
      record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
      sm.abort_flag = 1;
    }
    const uint8_t* krow = sm.k[s] + ts * (kHeadDim * 2);
    const uint4 ka = *reinterpret_cast<const uint4*>(krow + 16 * c);
    const uint4 kb = *reinterpret_cast<const uint4*>(krow + 128 + 16 * c);
    float sc[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) sc[g] = dot8(qf[g], ka) + dot8(qf[g] + 8, kb);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], o);
    }
    const int t = (pg0 + i) * kPage + ts;
    const bool valid = (t < L) && (sm.ids[i] >= 0);
    const uint8_t* vrow = sm.v[s] + ts * (kHeadDim * 2);
    const uint4 va = *reinterpret_cast<const uint4*>(vrow + 16 * c);
    const uint4 vb = *reinterpret_cast<const uint4*>(vrow + 128 + 16 * c);
    if (valid) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        if (sc[g] > m[g]) {  // new running max for this slot: rescale
          const float corr = exp2f(m[g] - sc[g]);
          l[g] *= corr;
#pragma unroll
          for (int d = 0; d < 16; ++d) acc[g][d] *= corr;
          m[g] = sc[g];
        }
        const float pr = exp2f(sc[g] - m[g]);
        l[g] += pr;
        axpy8(acc[g], pr, va);
        axpy8(acc[g] + 8, pr, vb);
      }
    }
    __syncthreads();  // every thread is done with stage s
    if (sm.abort_flag) {
      stop_at = i;
      break;
    }
    if (tid == 0 && i + kStages < npg) issue(i + kStages);
  }

  if (stop_at < npg) {
    // A wait gave up: let the copies already issued land (bounded), then leave.
    if (tid == 0) {
      const int last = min(npg, stop_at + kStages);
      for (int j = stop_at; j < last; ++j)
        if (!mbar_wait_bounded(&sm.full[j % kStages], (uint32_t)(j / kStages) & 1u)) break;
    }
    return;
  }

  // Merge the 16 token slots: global max per head, then rescaled sums.
  if (c == 0) {
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      sm.red_m[ts][g] = m[g];
      sm.red_l[ts][g] = l[g];
    }
  }
  __syncthreads();
  float M[kGroup], Lsum[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPage; ++j) mx = fmaxf(mx, sm.red_m[j][g]);
    float sum = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int j = 0; j < kPage; ++j) {
        const float mj = sm.red_m[j][g];
        if (mj != -INFINITY) sum += sm.red_l[j][g] * exp2f(mj - mx);
      }
    }
    M[g] = mx;
    Lsum[g] = sum;
  }
  float* red = reinterpret_cast<float*>(&sm.k[0][0]);  // [16 slots][4 heads][128 dims]
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    const float f = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - M[g]);
    float* dst = red + (ts * kGroup + g) * kHeadDim;
#pragma unroll
    for (int d = 0; d < 8; d += 4) {
      *reinterpret_cast<float4*>(dst + 8 * c + d) =
          make_float4(acc[g][d] * f, acc[g][d + 1] * f, acc[g][d + 2] * f, acc[g][d + 3] * f);
      *reinterpret_cast<float4*>(dst + 64 + 8 * c + d) =
          make_float4(acc[g][8 + d] * f, acc[g][9 + d] * f, acc[g][10 + d] * f, acc[g][11 + d] * f);
    }
  }
  __syncthreads();
  const int g = tid >> 5;
  const int d0 = (tid & 31) * 4;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(red + (j * kGroup + g) * kHeadDim + d0);
    o.x += x.x;
    o.y += x.y;
    o.z += x.z;
    o.w += x.w;
  }
  const float inv = Lsum[g] > 0.f ? 1.f / Lsum[g] : 0.f;
  o.x *= inv;
  o.y *= inv;
  o.z *= inv;
  o.w *= inv;
  const int head = kvh * kGroup + g;
  const float lse2 = Lsum[g] > 0.f ? M[g] + log2f(Lsum[g]) : -INFINITY;
  if (p.num_splits == 1) {
    uint2 packed;
    packed.x = pack_bf16x2(o.x, o.y);
    packed.y = pack_bf16x2(o.z, o.w);
    *reinterpret_cast<uint2*>(p.out + ((size_t)tok * p.num_q_heads + head) * kHeadDim + d0) = packed;
    if (p.lse && (tid & 31) == 0) p.lse[(size_t)tok * p.num_q_heads + head] = lse2 * kLn2;
  } else {
    const size_t row = ((size_t)split * p.total_q + tok) * p.num_q_heads + head;
    *reinterpret_cast<float4*>(p.part_o + row * kHeadDim + d0) = o;
    if ((tid & 31) == 0) p.part_lse[row] = lse2;
  }
}

// One CTA per (kv head, request); warp w merges q head 4*kvh + w, each lane
// four dims.  Weights are 2^(lse_s - max); empty splits (lse = -inf) weigh 0.
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  const int kvh = blockIdx.x, r = blockIdx.y;
  const int tok = p.qo_indptr[r];
  if (p.qo_indptr[r + 1] - tok != 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = kvh * kGroup + warp;
  const size_t split_stride = (size_t)p.total_q * p.num_q_heads;
  const size_t row0 = (size_t)tok * p.num_q_heads + head;
  float M = -INFINITY;
  for (int s = 0; s < p.num_splits; ++s) M = fmaxf(M, p.part_lse[s * split_stride + row0]);
  float wsum = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int s = 0; s < p.num_splits; ++s) {
      const float ls = p.part_lse[s * split_stride + row0];
      if (ls == -INFINITY) continue;
      const float w = exp2f(ls - M);
      const float4 x = *reinterpret_cast<const float4*>(p.part_o + (s * split_stride + row0) * kHeadDim + lane * 4);
      wsum += w;
      o.x = fmaf(w, x.x, o.x);
      o.y = fmaf(w, x.y, o.y);
      o.z = fmaf(w, x.z, o.z);
      o.w = fmaf(w, x.w, o.w);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2 packed;
  packed.x = pack_bf16x2(o.x * inv, o.y * inv);
  packed.y = pack_bf16x2(o.z * inv, o.w * inv);
  *reinterpret_cast<uint2*>(p.out + row0 * kHeadDim + lane * 4) = packed;
  if (p.lse && lane == 0) p.lse[row0] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
}

bool g_decode_attr_set[64] = {};

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !g_decode_attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(DecodeSmem));
    if (e != cudaSuccess) return e;
    g_decode_attr_set[dev] = true;
  }
  dim3 grid(p.num_splits, p.num_kv_heads, p.num_reqs);
  decode_kernel<<<grid, kThreads, sizeof(DecodeSmem), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.num_kv_heads, p.num_reqs);
  combine_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
