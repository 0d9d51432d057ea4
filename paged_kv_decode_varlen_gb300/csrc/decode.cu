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
// Design for GB300 (HBM-bound; 2 FMA per byte of K/V for the 4-head group):
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
//   * Products and sums use packed fp32x2 FMA (two lanes per instruction).
//     The 8-lane score reduction is transposed (each shuffle step halves the
//     values a lane keeps), so each lane ends with one head's score, takes
//     one exp2, and broadcasts its weight.  The running max is only re-based
//     when it grows by more than 2^8, so the rescale branch is rarely taken.
//   * No CTA-wide barrier in the page loop: each warp releases a stage on an
//     "empty" mbarrier and thread 0 refills it one page later.  (An L2
//     prefetch of the pages beyond the ring is available at compile time,
//     PA_DECODE_L2_AHEAD; measured on GB300 it lowers throughput, so it is
//     off.)
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 8;      // pages in the shared-memory ring
#ifndef PA_DECODE_L2_AHEAD
#define PA_DECODE_L2_AHEAD 0
#endif
constexpr int kL2Ahead = PA_DECODE_L2_AHEAD;  // pages prefetched into L2 beyond the ring (0 = none)
// Rescale the running sums only when the running max grows by more than
// 2^kRescaleSlack; until then exp2(s - m) stays below 2^kRescaleSlack.
constexpr float kRescaleSlack = 8.f;

struct __align__(128) DecodeSmem {
  uint8_t k[kStages][kSlabBytes];  // reused as the slot-merge buffer (32 KiB) after the loop
  uint8_t v[kStages][kSlabBytes];
  uint64_t full[kStages];   // TMA landed
  uint64_t empty[kStages];  // all warps done reading
  int32_t ids[kDecodeMaxPagesPerCta];
  float red_m[kPage][kGroup];
  float red_l[kPage][kGroup];
  int abort_flag;
};
static_assert(kStages * kSlabBytes >= kPage * kGroup * kHeadDim * 4, "merge buffer must fit in the K ring");

// 8 packed bf16 pairs (two 16-byte loads) -> 8 float2
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float2* f) {
  f[0] = bf16x2_to_f2(a.x); f[1] = bf16x2_to_f2(a.y); f[2] = bf16x2_to_f2(a.z); f[3] = bf16x2_to_f2(a.w);
  f[4] = bf16x2_to_f2(b.x); f[5] = bf16x2_to_f2(b.y); f[6] = bf16x2_to_f2(b.z); f[7] = bf16x2_to_f2(b.w);
}

__global__ void __launch_bounds__(kThreads, 3) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int split = blockIdx.x, kvh = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tok = p.qo_indptr[r];
  if (p.qo_indptr[r + 1] - tok != 1) return;  // not a decode row
  const int L = p.seq_lens[r];
  const int n_pages = (L + kPage - 1) / kPage;
  const int per = (n_pages + p.num_splits - 1) / p.num_splits;
  const int pg0 = min(n_pages, split * per);
  const int npg = min(n_pages, pg0 + per) - pg0;

  const int ts = tid >> 3;  // token slot within a page
  const int c = tid & 7;    // dim chunk: dims [8c, 8c+8) and [64+8c, 64+8c+8)
  // After the transposed reduction below, lane c of a token slot holds the
  // score of head hd = 2 * bit2(c) + bit1(c); lane base + cg[g] holds head g.
  const int hd = ((c >> 2) & 1) * 2 + ((c >> 1) & 1);
  const int slot_base = lane & ~7;

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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kWarps);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const size_t slab_elems = (size_t)kPage * kHeadDim;
  auto slab_off = [&](int i) {
    return ((size_t)max(sm.ids[i], 0) * p.num_kv_heads + kvh) * slab_elems;
  };
  auto issue = [&](int i) {  // page i of this split -> stage i % kStages; page i + kL2Ahead -> L2
    const int s = i % kStages;
    const size_t off = slab_off(i);
    mbar_arrive_expect_tx(&sm.full[s], 2 * kSlabBytes);
    bulk_g2s(sm.k[s], p.k_cache + off, kSlabBytes, &sm.full[s]);
    bulk_g2s(sm.v[s], p.v_cache + off, kSlabBytes, &sm.full[s]);
    if (kL2Ahead > 0 && i + kL2Ahead < npg) {
      const size_t poff = slab_off(i + kL2Ahead);
      bulk_prefetch_l2(p.k_cache + poff, kSlabBytes);
      bulk_prefetch_l2(p.v_cache + poff, kSlabBytes);
    }
  };
  const bool producer = (tid == 0);
  int issued = 0;
  if (producer) {
    issued = min(npg, kStages);
    for (int i = 0; i < issued; ++i) issue(i);
  }

  // q of the 4 heads of this group, scaled into the log2 domain, as float2
  // pairs matching the K layout this thread reads.
  float2 q2[kGroup][8];
  {
    const uint16_t* qrow = p.q + ((size_t)tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
    const float2 sc = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const uint4 a = *reinterpret_cast<const uint4*>(qrow + g * kHeadDim + 8 * c);
      const uint4 b = *reinterpret_cast<const uint4*>(qrow + g * kHeadDim + 64 + 8 * c);
      unpack16(a, b, q2[g]);
#pragma unroll
      for (int j = 0; j < 8; ++j) q2[g][j] = __fmul2_rn(q2[g][j], sc);
    }
  }

  float2 acc[kGroup][8];
#pragma unroll
  for (int g = 0; g < kGroup; ++g)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[g][j] = make_float2(0.f, 0.f);
  // running max and sum of head hd for this token slot (kept by the lanes
  // that own hd after the reduction)
  float m_own = -INFINITY, l_own = 0.f;

  bool aborted = false;
  for (int i = 0; i < npg; ++i) {
    if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) {
      aborted = true;
      break;
    }
    const int s = i % kStages;
    if (!mbar_wait_bounded(&sm.full[s], (uint32_t)(i / kStages) & 1u)) {
      record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
      aborted = true;
      break;
    }
    const uint8_t* krow = sm.k[s] + ts * (kHeadDim * 2);
    const uint4 ka = *reinterpret_cast<const uint4*>(krow + 16 * c);
    const uint4 kb = *reinterpret_cast<const uint4*>(krow + 128 + 16 * c);
    const bool valid = ((pg0 + i) * kPage + ts < L) && (sm.ids[i] >= 0);

    // partial scores over this thread's 16 dims: (h0, h1) and (h2, h3)
    float2 sp0, sp1;
    {
      float2 k2[8];
      unpack16(ka, kb, k2);
      float2 a0 = __fmul2_rn(q2[0][0], k2[0]), a1 = __fmul2_rn(q2[0][1], k2[1]);
      float2 b0 = __fmul2_rn(q2[1][0], k2[0]), b1 = __fmul2_rn(q2[1][1], k2[1]);
      float2 c0 = __fmul2_rn(q2[2][0], k2[0]), c1 = __fmul2_rn(q2[2][1], k2[1]);
      float2 d0 = __fmul2_rn(q2[3][0], k2[0]), d1 = __fmul2_rn(q2[3][1], k2[1]);
#pragma unroll
      for (int j = 2; j < 8; j += 2) {
        a0 = __ffma2_rn(q2[0][j], k2[j], a0);
        a1 = __ffma2_rn(q2[0][j + 1], k2[j + 1], a1);
        b0 = __ffma2_rn(q2[1][j], k2[j], b0);
        b1 = __ffma2_rn(q2[1][j + 1], k2[j + 1], b1);
        c0 = __ffma2_rn(q2[2][j], k2[j], c0);
        c1 = __ffma2_rn(q2[2][j + 1], k2[j + 1], c1);
        d0 = __ffma2_rn(q2[3][j], k2[j], d0);
        d1 = __ffma2_rn(q2[3][j + 1], k2[j + 1], d1);
      }
      a0 = __fadd2_rn(a0, a1);
      b0 = __fadd2_rn(b0, b1);
      c0 = __fadd2_rn(c0, c1);
      d0 = __fadd2_rn(d0, d1);
      sp0 = make_float2(a0.x + a0.y, b0.x + b0.y);
      sp1 = make_float2(c0.x + c0.y, d0.x + d0.y);
    }
    // transposed reduction over the 8 lanes of the slot: each step halves
    // the values a lane keeps, so lane c ends with the full score of head hd
    float sc;
    {
      const bool b2 = (c >> 2) & 1;
      const float2 send = b2 ? sp0 : sp1;
      float2 keep = b2 ? sp1 : sp0;
      keep = __fadd2_rn(keep, make_float2(__shfl_xor_sync(0xffffffffu, send.x, 4),
                                          __shfl_xor_sync(0xffffffffu, send.y, 4)));
      const bool b1 = (c >> 1) & 1;
      const float snd = b1 ? keep.x : keep.y;
      sc = (b1 ? keep.y : keep.x) + __shfl_xor_sync(0xffffffffu, snd, 2);
      sc += __shfl_xor_sync(0xffffffffu, sc, 1);
    }

    // online softmax of head hd; the rescale (rare) is warp-uniform
    const float sv = valid ? sc : -INFINITY;
    const bool grow = sv > m_own + kRescaleSlack;
    if (__any_sync(0xffffffffu, grow)) {
      const float corr = grow ? fast_exp2(m_own - sv) : 1.f;  // m_own = -inf -> 0
      if (grow) m_own = sv;
      l_own *= corr;
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const float cg = __shfl_sync(0xffffffffu, corr, slot_base + (g >> 1) * 4 + (g & 1) * 2);
        const float2 c2 = make_float2(cg, cg);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[g][j] = __fmul2_rn(acc[g][j], c2);
      }
    }
    const float pown = valid ? fast_exp2(sv - m_own) : 0.f;
    l_own += pown;

    // values: acc[g] += p_g * V, p_g broadcast from the lane owning head g
    // (all lanes shuffle; only valid tokens touch V)
    float pg[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) pg[g] = __shfl_sync(0xffffffffu, pown, slot_base + (g >> 1) * 4 + (g & 1) * 2);
    if (valid) {
      const uint8_t* vrow = sm.v[s] + ts * (kHeadDim * 2);
      const uint4 va = *reinterpret_cast<const uint4*>(vrow + 16 * c);
      const uint4 vb = *reinterpret_cast<const uint4*>(vrow + 128 + 16 * c);
      float2 v2[8];
      unpack16(va, vb, v2);
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const float2 p2 = make_float2(pg[g], pg[g]);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[g][j] = __ffma2_rn(p2, v2[j], acc[g][j]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);  // this warp is done with stage s

    // producer: refill the stage consumed one page ago once every warp has
    // released it
    if (producer && i >= 1) {
      const int j = i - 1;
      if (j + kStages < npg) {
        if (!mbar_wait_bounded(&sm.empty[j % kStages], (uint32_t)(j / kStages) & 1u)) {
          record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
          *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
          aborted = true;
          break;
        }
        issue(j + kStages);
        issued = j + kStages + 1;
      }
    }
  }

  __syncthreads();  // every thread has left the loop
  if (aborted || *reinterpret_cast<volatile int*>(&sm.abort_flag)) {
    // A wait gave up: let the copies already issued land (bounded), then leave.
    if (producer) {
      for (int j = max(0, issued - kStages); j < issued; ++j)
        if (!mbar_wait_bounded(&sm.full[j % kStages], (uint32_t)(j / kStages) & 1u)) break;
    }
    return;
  }

  // Merge the 16 token slots: global max per head, then rescaled sums.
  if ((c & 1) == 0) {
    sm.red_m[ts][hd] = m_own;
    sm.red_l[ts][hd] = l_own;
  }
  __syncthreads();
  float* red = reinterpret_cast<float*>(&sm.k[0][0]);  // [16 slots][4 heads][128 dims]
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPage; ++j) mx = fmaxf(mx, sm.red_m[j][g]);
    const float mslot = sm.red_m[ts][g];
    const float f = (mslot == -INFINITY) ? 0.f : fast_exp2(mslot - mx);
    float* dst = red + (ts * kGroup + g) * kHeadDim;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      *reinterpret_cast<float4*>(dst + 8 * c + 2 * j) =
          make_float4(acc[g][j].x * f, acc[g][j].y * f, acc[g][j + 1].x * f, acc[g][j + 1].y * f);
      *reinterpret_cast<float4*>(dst + 64 + 8 * c + 2 * j) =
          make_float4(acc[g][4 + j].x * f, acc[g][4 + j].y * f, acc[g][5 + j].x * f, acc[g][5 + j].y * f);
    }
  }
  __syncthreads();
  // warp g finishes head g: lane owns dims [4 lane, 4 lane + 4)
  const int g = warp;
  float Mg = -INFINITY;
#pragma unroll
  for (int j = 0; j < kPage; ++j) Mg = fmaxf(Mg, sm.red_m[j][g]);
  float Lg = 0.f;
  if (Mg != -INFINITY) {
#pragma unroll
    for (int j = 0; j < kPage; ++j) {
      const float mj = sm.red_m[j][g];
      if (mj != -INFINITY) Lg += sm.red_l[j][g] * fast_exp2(mj - Mg);
    }
  }
  const int d0 = lane * 4;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(red + (j * kGroup + g) * kHeadDim + d0);
    o.x += x.x;
    o.y += x.y;
    o.z += x.z;
    o.w += x.w;
  }
  const float inv = Lg > 0.f ? 1.f / Lg : 0.f;
  o.x *= inv;
  o.y *= inv;
  o.z *= inv;
  o.w *= inv;
  const int head = kvh * kGroup + g;
  const float lse2 = Lg > 0.f ? Mg + log2f(Lg) : -INFINITY;
  if (p.num_splits == 1) {
    uint2 packed;
    packed.x = pack_bf16x2(o.x, o.y);
    packed.y = pack_bf16x2(o.z, o.w);
    *reinterpret_cast<uint2*>(p.out + ((size_t)tok * p.num_q_heads + head) * kHeadDim + d0) = packed;
    if (p.lse && lane == 0) p.lse[(size_t)tok * p.num_q_heads + head] = lse2 * kLn2;
  } else {
    const size_t row = ((size_t)split * p.total_q + tok) * p.num_q_heads + head;
    *reinterpret_cast<float4*>(p.part_o + row * kHeadDim + d0) = o;
    if (lane == 0) p.part_lse[row] = lse2;
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
