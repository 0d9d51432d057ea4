// Persistent flash-decode over a paged KV cache (decode rows, qo_len = 1).
//
// What is computed: for a decode row, every q head attends to all seq_len
// keys of its kv head, read through the block table ("Inference
// optimisation", AI-infra book ch. 8, §8.3.1 / Fig. 8-10; "vLLM, SGLang and
// continuous batching", section "PagedAttention").  The softmax is computed
// online in fp32 (log2 domain); partial results over disjoint key ranges
// are merged by the log-sum-exp identity.
//
// Design for GB300 (HBM-bound; 2 FMA per byte of K/V for the 4-head group):
//   * Work stream.  For each kv head the decode rows' pages are laid end to
//     end as one stream, cut into equal contiguous segments; CTA b takes kv
//     head b % Hkv and segment b / Hkv, with one CTA per resident slot (3 per
//     SM).  A CTA streams its segment through one TMA ring without
//     restarting at row boundaries, so there is no tail of short CTAs and no
//     per-CTA start-up latency beyond the first page.  The Hkv CTAs of a
//     segment read the Hkv head slabs of the same blocks (one contiguous
//     32 KiB block for 8 kv heads) at the same time.
//   * Each page's K slab and V slab (4 KiB each, contiguous in the HND pool)
//     are fetched by two 1-D bulk copies into an 8-deep shared-memory ring
//     guarded by mbarriers.  The 4 q heads of the GQA group share every K/V
//     element read.
//   * 128 threads = 16 token slots x 8 dim chunks.  Thread (t, c) owns dims
//     [8c, 8c+8) and [64+8c, 64+8c+8) of token t of a page (conflict-free
//     16-byte shared loads).  Two pages per loop iteration.  Scores use
//     packed fp32x2 FMA on head pairs: q is held as (head 0, head 1) and
//     (head 2, head 3) pairs per dim and each k element is used in both
//     lanes, so the products come out as (h0, h1), (h2, h3) score pairs with
//     no final lane sum.  A transposed 8-lane reduction then leaves each
//     lane one complete (token, head) score, one exp2 per lane, weights
//     broadcast back by shuffles.  The running max is re-based only when it
//     grows by more than 2^8.
//   * No CTA-wide barrier and no producer thread: each warp counts itself
//     out of a stage (a shared-memory atomic) when it has read it, and the
//     last of the 4 warps issues that stage's next page at once, so the
//     ring stays 8 pages deep and the TMA issue work is spread over warps.
//   * Item end: the 16 token slots are merged (a transposed shuffle
//     reduction inside each warp, then across the 4 warps through 4 KiB of
//     shared memory, two heads per round: three CTAs per SM leave no room
//     for all four at once).  With bf16 pages and the host plan the next
//     item's q is bulk-copied into shared memory at the item end, so the
//     next item starts without a global-memory round trip.  An item that
//     lies inside one segment is written out at once;
//     an item cut by segment boundaries leaves one partial per CTA in the
//     workspace, and the last of those CTAs to finish (a counter it resets)
//     merges them into out / lse.
#include <math.h>
#include <stddef.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 8;  // pages in the shared-memory ring (a power of two)
// Rescale the running sums only when the running max grows by more than
// 2^kRescaleSlack; until then exp2(s - m) stays below 2^kRescaleSlack.
constexpr float kRescaleSlack = 8.f;

struct Item {        // one request's pages within this CTA's segment
  int32_t q_start;  // first page of the item in this segment
  int32_t n;        // pages of the item in this segment
  int32_t p0;       // row page index of the item's first page in this segment
  int32_t r;        // request
  int32_t L;        // seq_len of the request
  int32_t tok;      // its query token
  int32_t A;        // stream position of the row's start (its cost units, then its pages)
};

// Bytes of one (page, kv head) slab: bf16 pages, or q8_0 pages (16 x 128
// int8 codes, then 16 x 4 binary16 group scales).
constexpr int kQ8SlabBytes = kPage * kHeadDim + kPage * (kHeadDim / 32) * 2;  // 2176
static_assert(kQ8SlabBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

template <int kSlab>
struct __align__(128) DecodeSmem {
  uint8_t k[kStages][kSlab];
  uint8_t v[kStages][kSlab];
  uint16_t qs[kGroup * kHeadDim];        // the current item's q (bulk copy)
  float mrg_o[kWarps][2][kHeadDim];      // cross-warp merge: two heads per round
  float mrg_m[kWarps][2], mrg_l[kWarps][2];
  uint64_t full[kStages];   // TMA landed
  uint64_t q_full;          // q landed
  int q_issued;             // q copies issued
  int readers[kStages];     // warps done reading the stage's current page
  int32_t ids[kDecodeMaxPagesPerCta];
  Item items[kDecodeMaxItemsPerCta];
  int n_cov;                 // end of the pages the current window's items cover
  int seg_pages;             // pages of the segment (self-planned)
  int n_items;               // items of the current window
  int n_items_all;           // items of the segment
  int seg_cost;              // segment length in stream units (self-planned)
  int scan[kThreads / 32];   // per-warp totals of the planning scans
  int stage_page[kStages];   // last page issued into each stage (-1: none)
  int abort_flag;
  int is_last;
};

static_assert(offsetof(DecodeSmem<kSlabBytes>, k) % 128 == 0 && offsetof(DecodeSmem<kSlabBytes>, v) % 128 == 0 &&
                  offsetof(DecodeSmem<kQ8SlabBytes>, v) % 16 == 0 && offsetof(DecodeSmem<kSlabBytes>, qs) % 16 == 0 &&
                  offsetof(DecodeSmem<kQ8SlabBytes>, qs) % 16 == 0,
              "bulk copies land on 16-byte boundaries");
// three CTAs per SM: 228 KiB of shared memory per SM, 1 KiB of it reserved per CTA
static_assert(3 * (sizeof(DecodeSmem<kSlabBytes>) + 1024) <= 228 * 1024, "three decode CTAs per SM");

// 8 packed bf16 pairs (two 16-byte loads) -> 8 float2
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float2* f) {
  f[0] = bf16x2_to_f2(a.x); f[1] = bf16x2_to_f2(a.y); f[2] = bf16x2_to_f2(a.z); f[3] = bf16x2_to_f2(a.w);
  f[4] = bf16x2_to_f2(b.x); f[5] = bf16x2_to_f2(b.y); f[6] = bf16x2_to_f2(b.z); f[7] = bf16x2_to_f2(b.w);
}

// 8 packed bf16 pairs -> 16 scalars (element order kept)
__device__ __forceinline__ void unpack16s(const uint4& a, const uint4& b, float* f) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16lo(w[i]);
    f[2 * i + 1] = bf16hi(w[i]);
  }
}

// Partial scores of one token over this thread's 16 dims (bf16 pages), with
// the dims paired: qp[hp][8 e + j] = (q[2 hp + e][dim 2j], q[2 hp + e][dim
// 2j + 1]).  A K word holds two consecutive dims, so it unpacks straight into
// the operand pair of a packed fp32x2 FMA; each head's two lanes are added
// at the end.  Returns the (h0, h1) and (h2, h3) score pairs.
__device__ __forceinline__ void qk16(const float2 (&qp)[2][16], const uint4& ka, const uint4& kb, float2& s01,
                                     float2& s23) {
  float2 k2[8];
  unpack16(ka, kb, k2);
  float2 a0 = __fmul2_rn(qp[0][0], k2[0]);
  float2 a1 = __fmul2_rn(qp[0][8], k2[0]);
  float2 a2 = __fmul2_rn(qp[1][0], k2[0]);
  float2 a3 = __fmul2_rn(qp[1][8], k2[0]);
#pragma unroll
  for (int j = 1; j < 8; ++j) {
    a0 = __ffma2_rn(qp[0][j], k2[j], a0);
    a1 = __ffma2_rn(qp[0][8 + j], k2[j], a1);
    a2 = __ffma2_rn(qp[1][j], k2[j], a2);
    a3 = __ffma2_rn(qp[1][8 + j], k2[j], a3);
  }
  s01 = make_float2(a0.x + a0.y, a1.x + a1.y);
  s23 = make_float2(a2.x + a2.y, a3.x + a3.y);
}

// q8_0 pages: 8 int8 codes (dims 8c..8c+7 or 64+8c..) -> 8 floats, without
// integer-to-float conversion instructions (exponent-bias construction): a
// code c biased to c + 128 (flipping each byte's top bit) becomes the low
// mantissa byte of a binary32 with exponent 2^23 (a byte permute), whose value
// is 2^23 + c + 128 exactly; subtracting 2^23 + 128 gives c exactly.  Two
// codes share one packed subtraction.
__device__ __forceinline__ void codes8(const uint2& w, float* f) {
  const uint32_t x = w.x ^ 0x80808080u, y = w.y ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    // byte 0 from the word (selector nibble i), bytes 1-2 zero, byte 3 = 0x4B
    const float2 a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u + i)),
                                            __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7441u + i))),
                                bias);
    const float2 b = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(y, 0x4B000000u, 0x7440u + i)),
                                            __uint_as_float(__byte_perm(y, 0x4B000000u, 0x7441u + i))),
                                bias);
    f[i] = a.x;
    f[i + 1] = a.y;
    f[4 + i] = b.x;
    f[5 + i] = b.y;
  }
}

// qk16 over q8_0 codes, with q as head pairs per dim: qp[hp][i] =
// (q[2 hp][dim i], q[2 hp + 1][dim i]).  The dims of ka lie in one 32-value
// group (scale dA), those of kb in another (dB); each group's partial dot
// product is scaled once.  (The dim-pair layout of qk16 measured ~1% slower
// here: the int8 conversions, not the operand pairing, dominate.)
__device__ __forceinline__ void qk16_q8(const float2 (&qp)[2][16], const uint2& ka, const uint2& kb, float dA,
                                        float dB, float2& s01, float2& s23) {
  float kf[16];
  codes8(ka, kf);
  codes8(kb, kf + 8);
  float2 a0 = __fmul2_rn(qp[0][0], make_float2(kf[0], kf[0]));
  float2 a1 = __fmul2_rn(qp[0][1], make_float2(kf[1], kf[1]));
  float2 c0 = __fmul2_rn(qp[1][0], make_float2(kf[0], kf[0]));
  float2 c1 = __fmul2_rn(qp[1][1], make_float2(kf[1], kf[1]));
  float2 e0 = __fmul2_rn(qp[0][8], make_float2(kf[8], kf[8]));
  float2 e1 = __fmul2_rn(qp[0][9], make_float2(kf[9], kf[9]));
  float2 g0 = __fmul2_rn(qp[1][8], make_float2(kf[8], kf[8]));
  float2 g1 = __fmul2_rn(qp[1][9], make_float2(kf[9], kf[9]));
#pragma unroll
  for (int i = 2; i < 8; i += 2) {
    a0 = __ffma2_rn(qp[0][i], make_float2(kf[i], kf[i]), a0);
    a1 = __ffma2_rn(qp[0][i + 1], make_float2(kf[i + 1], kf[i + 1]), a1);
    c0 = __ffma2_rn(qp[1][i], make_float2(kf[i], kf[i]), c0);
    c1 = __ffma2_rn(qp[1][i + 1], make_float2(kf[i + 1], kf[i + 1]), c1);
    e0 = __ffma2_rn(qp[0][8 + i], make_float2(kf[8 + i], kf[8 + i]), e0);
    e1 = __ffma2_rn(qp[0][9 + i], make_float2(kf[9 + i], kf[9 + i]), e1);
    g0 = __ffma2_rn(qp[1][8 + i], make_float2(kf[8 + i], kf[8 + i]), g0);
    g1 = __ffma2_rn(qp[1][9 + i], make_float2(kf[9 + i], kf[9 + i]), g1);
  }
  const float2 dA2 = make_float2(dA, dA), dB2 = make_float2(dB, dB);
  s01 = __ffma2_rn(dA2, __fadd2_rn(a0, a1), __fmul2_rn(dB2, __fadd2_rn(e0, e1)));
  s23 = __ffma2_rn(dA2, __fadd2_rn(c0, c1), __fmul2_rn(dB2, __fadd2_rn(g0, g1)));
}

// pv16 over q8_0 codes: each head's weight is scaled by the group scale of
// the dims it multiplies.
__device__ __forceinline__ void pv16_q8(float2 (&acc)[kGroup][8], const float (&pg)[kGroup], const uint2& va,
                                        const uint2& vb, float dA, float dB) {
  float vf[16];
  codes8(va, vf);
  codes8(vb, vf + 8);
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    const float2 pa2 = make_float2(pg[g] * dA, pg[g] * dA), pb2 = make_float2(pg[g] * dB, pg[g] * dB);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[g][j] = __ffma2_rn(pa2, make_float2(vf[2 * j], vf[2 * j + 1]), acc[g][j]);
      acc[g][4 + j] = __ffma2_rn(pb2, make_float2(vf[8 + 2 * j], vf[9 + 2 * j]), acc[g][4 + j]);
    }
  }
}

// The group scales of token slot ts of a q8_0 slab that thread chunk c
// needs: dims 8c.. lie in group c / 4, dims 64 + 8c.. in group 2 + c / 4.
__device__ __forceinline__ void q8_scales(const uint8_t* slab, int ts, int c, float& dA, float& dB) {
  const uint2 w = *reinterpret_cast<const uint2*>(slab + kPage * kHeadDim + ts * 8);
  const uint32_t lo = (c >> 2) ? (w.x >> 16) : (w.x & 0xffffu);
  const uint32_t hi = (c >> 2) ? (w.y >> 16) : (w.y & 0xffffu);
  dA = __half2float(__ushort_as_half((unsigned short)lo));
  dB = __half2float(__ushort_as_half((unsigned short)hi));
}

__device__ __forceinline__ void pv16(float2 (&acc)[kGroup][8], const float (&pg)[kGroup], const uint4& va,
                                     const uint4& vb) {
  float2 v2[8];
  unpack16(va, vb, v2);
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    const float2 p2 = make_float2(pg[g], pg[g]);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[g][j] = __ffma2_rn(p2, v2[j], acc[g][j]);
  }
}

__device__ __forceinline__ float2 shfl_xor2(float2 v, int o) {
  return make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
}

__device__ __forceinline__ void bar_all() { __syncthreads(); }

// Whole warp (lane = 4 dims at d0): folds the shared-prefix partials of
// output row orow (p.prefix_n key-chunk partials, or the merged one) into
// the normalised partial o with log2 lse lse2 by log-sum-exp; returns the
// merged lse.  Eight partials per round, every load of the round (lane i:
// partial i's lse; all lanes: 4 dims of each) in flight at once, with a
// running max across rounds.
__device__ __forceinline__ float fold_prefix(const DecodeParams& p, float4& o, float lse2, size_t orow, int d0,
                                             int lane) {
  constexpr int kRound = 8;
  const int n = p.prefix_n;
  float M = lse2;
  float wsum = lse2 == -INFINITY ? 0.f : 1.f;
  float4 a = lse2 == -INFINITY ? make_float4(0.f, 0.f, 0.f, 0.f) : o;
  for (int c0 = 0; c0 < n; c0 += kRound) {
    const int nc = min(kRound, n - c0);
    const float lv = lane < nc ? p.prefix_lse[(size_t)(c0 + lane) * p.prefix_rows + orow] : -INFINITY;
    float4 y[kRound];
#pragma unroll
    for (int i = 0; i < kRound; ++i)
      y[i] = i < nc ? *reinterpret_cast<const float4*>(p.prefix_o + ((size_t)(c0 + i) * p.prefix_rows + orow) * kHeadDim +
                                                       d0)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    float mb = lv;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, s));
    const float mn = fmaxf(M, mb);
    if (mn == -INFINITY) continue;  // every partial so far is empty
    const float sc = exp2f(M - mn);  // M = -inf -> 0
    wsum *= sc;
    a = make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
    const float w = exp2f(lv - mn);  // -inf -> 0
    float ws = w;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, s);
    wsum += ws;
#pragma unroll
    for (int i = 0; i < kRound; ++i) {
      const float wi = __shfl_sync(0xffffffffu, w, i);
      a.x = fmaf(wi, y[i].x, a.x);
      a.y = fmaf(wi, y[i].y, a.y);
      a.z = fmaf(wi, y[i].z, a.z);
      a.w = fmaf(wi, y[i].w, a.w);
    }
    M = mn;
  }
  if (M == -INFINITY) return -INFINITY;
  const float inv = 1.f / wsum;
  o = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  return M + log2f(wsum);
}

// Decode step: each CTA plans its own segment from the device seq_lens.
// Row r of the padded batch costs pages_r + kStepItemCost units (0 for a
// padding row: seq_len 0, or a length outside the call's bounds), the rows'
// costs are laid end to end and cut into n_eff equal segments of C units;
// a row's pages sit after its fixed cost, and segment s holds the pages
// whose units fall in [s C, (s + 1) C).  The fixed cost stands for the item-
// end merge work, so segments with many short rows hold fewer pages.  Fills
// the items win0 .. win0 + kMaxItems - 1 of this CTA's segment (kNThreads
// threads, all of which call it; it ends with a barrier).  Also writes the outputs of
// padding rows (zero, lse -inf) and records rows outside the bounds.
template <int kUnit, int kNThreads, int kMaxItems, int kMaxPages, class Smem>
__device__ void step_window(const DecodeParams& p, const StepPlan& plan, Smem& sm, int kvh, int sidx, int nseg_grid,
                            int win0) {
  constexpr int kRows = (kPlanMaxRows + kNThreads - 1) / kNThreads;  // rows per thread, consecutive
  constexpr int kNWarps = kNThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.num_kv_heads;
  int pg[kRows], len[kRows];
  int tsum = 0;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int r = tid * kRows + i;
    const int L = r < plan.n_rows ? __ldg(p.seq_lens + r) : 0;
    const int pages = (L + kPage - 1) / kPage;
    const bool bad = r < plan.n_rows && (L < 0 || L > plan.max_seq_len || pages > p.max_blocks_per_req);
    len[i] = L;
    pg[i] = (bad || L <= 0) ? 0 : pages;
    tsum += pg[i] > 0 ? pg[i] + kStepItemCost : 0;
    if (win0 == 0 && r < plan.n_rows && pg[i] == 0 && sidx == r % nseg_grid) {
      // padding (or invalid) row: defined outputs for this kv head's 4 q heads
      if (bad) record_error(p.err, PA_ERR_DEVICE_INDEX);
      uint4* o = reinterpret_cast<uint4*>(p.out + ((size_t)r * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim);
      for (int j = 0; j < kGroup * kHeadDim * 2 / 16; ++j) o[j] = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse)
        for (int g = 0; g < kGroup; ++g) p.lse[(size_t)r * p.num_q_heads + kvh * kGroup + g] = -INFINITY;
    }
  }
  // exclusive scan of the row costs (thread-local, then across the block)
  int incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.scan[warp] = incl;
  __syncthreads();
  int total = 0, woff = 0;
#pragma unroll
  for (int w = 0; w < kNWarps; ++w) {
    const int v = sm.scan[w];
    woff += (w < warp) ? v : 0;
    total += v;
  }
  int A = woff + incl - tsum;  // cost position of this thread's first row
  const int n_eff = max(1, min(nseg_grid, (total + kStepMinSegCost - 1) / kStepMinSegCost));
  // segment length in stream units, whole warp segments for the warp-granular kernel (kUnit warps)
  const int C = (max(1, (total + n_eff - 1) / n_eff) + kUnit - 1) / kUnit * kUnit;
  const int S = sidx * C, E = min(S + C, total);
  // this segment's part of each row: (first page p0, pages nn), packed with
  // an item count for the second scan: (pages << 16) | 1
  int p0v[kRows], nnv[kRows], Av[kRows];
  int t2 = 0;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int u0 = A + kStepItemCost, u1 = u0 + pg[i];
    const bool in = pg[i] > 0 && u1 > S && u0 < E;
    p0v[i] = in ? max(0, S - u0) : 0;
    nnv[i] = in ? min(u1, E) - u0 - p0v[i] : 0;
    Av[i] = A;
    t2 += in ? ((nnv[i] << 16) | 1) : 0;
    A += pg[i] > 0 ? pg[i] + kStepItemCost : 0;
  }
  __syncthreads();  // sm.scan is reused
  int incl2 = t2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl2, o);
    if (lane >= o) incl2 += y;
  }
  if (lane == 31) sm.scan[warp] = incl2;
  __syncthreads();
  int tot2 = 0, woff2 = 0;
#pragma unroll
  for (int w = 0; w < kNWarps; ++w) {
    const int v = sm.scan[w];
    woff2 += (w < warp) ? v : 0;
    tot2 += v;
  }
  int e2 = woff2 + incl2 - t2;
  const int n_all = tot2 & 0xffff;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    if (nnv[i] > 0) {
      const int idx = (e2 & 0xffff) - win0;
      if (idx >= 0 && idx < kMaxItems) {
        const int r = tid * kRows + i;
        Item& it = sm.items[idx];
        it.q_start = e2 >> 16;
        it.n = nnv[i];
        it.p0 = p0v[i];
        it.r = r;
        it.L = len[i];
        it.tok = r;
        it.A = Av[i];
        const size_t qoff = ((size_t)r * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
        bulk_prefetch_l2(p.q + qoff, kGroup * kHeadDim * 2);
        if (p0v[i] + nnv[i] == pg[i]) {  // this CTA appends the row's new token
          const size_t noff = ((size_t)r * Hkv + kvh) * kHeadDim;
          bulk_prefetch_l2(p.k_new + noff, kHeadDim * 2);
          bulk_prefetch_l2(p.v_new + noff, kHeadDim * 2);
        }
      }
      e2 += (nnv[i] << 16) | 1;
    }
  }
  if (tid == 0) {
    sm.n_items = max(0, min(n_all - win0, kMaxItems));
    sm.n_items_all = n_all;
    sm.seg_cost = C;
    sm.seg_pages = tot2 >> 16;
    if (tot2 >> 16 > kMaxPages) {  // bounded by the host's grid choice
      record_error(p.err, PA_ERR_DEVICE_INDEX);
      sm.n_items = 0;
    }
  }
  __syncthreads();
}

// kDiag: the diagnostic instantiation that tests the timeout path (bf16
// pages, host plan).  CTA 0 arms the barrier of its segment's second page
// without issuing that page's copies, so the wait on it runs out; every wait
// of this instantiation gives up after 1 ms instead of kWaitLimitNs.  No
// copy is dropped anywhere else, and nothing is read out of bounds.
template <bool kQ8, bool kStep, bool kDiag = false>
__global__ void __launch_bounds__(kThreads, 3)
    decode_kernel(const DecodeParams p, const __grid_constant__ typename PlanOf<kStep>::type plan) {
  static_assert(!(kQ8 && kStep), "the decode step serves bf16 pages");
  static_assert(!(kDiag && (kQ8 || kStep)), "the diagnostic instantiation is the bf16 host-plan kernel");
  constexpr unsigned long long kLimit = kDiag ? 1000000ull : kWaitLimitNs;
  // the fixed cost of a row in the stream's units (the host plan cuts in
  // pages, with no fixed cost)
  constexpr int kAlpha = kStep ? kStepItemCost : 0;
  constexpr int kSlab = kQ8 ? kQ8SlabBytes : kSlabBytes;
  using Smem = DecodeSmem<kSlab>;
  // q of each item by a bulk copy into shared memory, issued an item ahead
  // (bf16 pages, host plan), else read from global memory at the item's
  // start: measured, the copy shortens the first and lengthens the others
  constexpr bool kQSmem = !kQ8 && !kStep;
  // No early launch of the next kernel: this grid is one wave sized to fill
  // every SM, and CTAs of a dependent kernel arriving early would take slots
  // its own CTAs need.  The next kernel is released as the CTAs exit.  The
  // host plan's item table comes from the kernel parameters alone, so it is
  // built before the wait for the previous kernel (which may still run).
  if constexpr (kStep) pdl_wait();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.num_kv_heads;
  const int kvh = b % Hkv, sidx = b / Hkv;
  int npg;  // pages of this CTA's segment
  if constexpr (kStep) {
    if (tid == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&sm.full[s], 1);
        sm.readers[s] = 0;
        sm.stage_page[s] = -1;
      }
      mbar_init(&sm.q_full, 1);
      sm.q_issued = 0;
      sm.abort_flag = 0;
      fence_mbar_init();
    }
    step_window<1, kThreads, kDecodeMaxItemsPerCta, kDecodeMaxPagesPerCta>(p, plan, sm, kvh, sidx,
                                                                          (int)gridDim.x / Hkv, 0);
    npg = sm.seg_pages;
  } else {
    const int S0 = sidx * plan.seg;
    npg = min(plan.total, S0 + plan.seg) - S0;
    if (npg <= 0) return;
    if (tid == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&sm.full[s], 1);
        sm.readers[s] = 0;
        sm.stage_page[s] = -1;
      }
      mbar_init(&sm.q_full, 1);
      sm.q_issued = 0;
      sm.abort_flag = 0;
      fence_mbar_init();
    }
    const int n_items_all = plan.n_rows;

    // ---- item table of this segment (warp 0), 32 items per round
    if (warp == 0) {
      int base_q = 0, n_it = 0;
      for (int k0 = 0; k0 < kDecodeMaxItemsPerCta; k0 += 32) {
        const int item = plan.first_row[sidx] + k0 + lane;
        const bool exists = item < n_items_all;
        int r = 0, L = 0, size = 0, tok = 0;
        const int p0 = (k0 + lane == 0) ? plan.first_page[sidx] : 0;
        if (exists) {
          // the plan's copies of seq_lens[r] and qo_indptr[r] (no device read)
          r = plan.rows[item];
          L = plan.seq[item];
          tok = plan.tok[item];
          size = max((L + kPage - 1) / kPage - p.page_offset - p0, 0);
        }
        int incl = size;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int start = base_q + incl - size;
        const bool in_seg = size > 0 && start < npg;
        if (in_seg && k0 + lane < kDecodeMaxItemsPerCta) {
          Item& it = sm.items[k0 + lane];
          it.q_start = start;
          it.n = min(size, npg - start);
          it.p0 = p0;
          it.r = r;
          it.L = L;
          it.tok = tok;
          it.A = S0 + start - p0;  // stream position of the row's page 0
          // the item's q (4 heads x 256 B) into L2 now; it is read at the item's start
          bulk_prefetch_l2(p.q + ((size_t)tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim,
                           kGroup * kHeadDim * 2);
        }
        // the table is the leading run of covered items (a gap can only come
        // from metadata that differ from the plan)
        const unsigned covered = __ballot_sync(0xffffffffu, in_seg);
        const int prefix = (~covered == 0u) ? 32 : (__ffs((int)~covered) - 1);
        n_it = k0 + prefix;
        base_q += __shfl_sync(0xffffffffu, incl, 31);
        if (prefix < 32 || base_q >= npg) break;
      }
      if (lane == 0) {
        if (base_q < npg) record_error(p.err, PA_ERR_DEVICE_INDEX);  // metadata differ from the plan
        sm.n_items = min(n_it, kDecodeMaxItemsPerCta);
      }
    }
    __syncthreads();
    pdl_wait();
  }
  int n_cov = 0;
  const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k_cache);
  const uint8_t* vbase = reinterpret_cast<const uint8_t*>(p.v_cache);
  // segment page i -> stage i % kStages (K and V slabs of kv head kvh)
  auto issue = [&](int i) {
    const int s = i & (kStages - 1);
    const size_t off = ((size_t)max(sm.ids[i], 0) * Hkv + kvh) * kSlab;
    mbar_arrive_expect_tx(&sm.full[s], 2 * kSlab);
    if (!(kDiag && b == 0 && i == 1)) {  // (diagnostic: CTA 0's page 1 is armed, never copied)
      bulk_g2s(sm.k[s], kbase + off, kSlab, &sm.full[s]);
      bulk_g2s(sm.v[s], vbase + off, kSlab, &sm.full[s]);
    }
    sm.stage_page[s] = i;  // one issuer per stage at a time
  };
  // q of item k of the window (4 heads x 256 B) -> sm.qs
  auto issue_q = [&](int k) {
    const size_t qoff = ((size_t)sm.items[k].tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
    mbar_arrive_expect_tx(&sm.q_full, kGroup * kHeadDim * 2);
    bulk_g2s(sm.qs, p.q + qoff, kGroup * kHeadDim * 2, &sm.q_full);
    sm.q_issued += 1;
  };
  // a warp is done with page i: the last of the 4 warps refills its stage
  // with page i + kStages
  auto release = [&](int i) {
    const int s = i & (kStages - 1);
    if (atomicAdd(&sm.readers[s], 1) == kWarps - 1) {
      atomicExch(&sm.readers[s], 0);
      if (i + kStages < n_cov) {
        fence_proxy_async_smem();
        issue(i + kStages);
      }
    }
  };

  const int ts = tid >> 3;  // token slot within a page
  const int c = tid & 7;    // dim chunk: dims [8c, 8c+8) and [64+8c, 64+8c+8)
  // After the transposed reduction lane c holds token u = bit0(c) of the
  // iteration and head hd = 2 bit2(c) + bit1(c).
  const int slot_base = lane & ~7;
  bool aborted = false;
  int qg = 0;    // segment page counter at the current item's start
  int win0 = 0;  // the window's first item within the segment

  // Windows of up to kDecodeMaxItemsPerCta items: one for the host plan;
  // the self-planned step walks a segment with more items in several.  The
  // host path keeps the shape of the single-window loop (its register
  // allocation, and so its speed, is sensitive to the code around the page
  // loop).
  for (;;) {
  const int n_items = sm.n_items;
  if (n_items == 0) break;  // nothing covered (recorded above); no copy was issued

  // ---- block ids of the window's pages; an id outside the pool (or a page
  // past the table) is recorded and masked, and fetched from block 0
  const int q_lo = kStep ? sm.items[0].q_start : 0;
  const int q_hi = kStep ? sm.items[n_items - 1].q_start + sm.items[n_items - 1].n : npg;
  int ok = 1;
  for (int q = q_lo + tid; q < q_hi; q += kThreads) {
    int lo = 0, hi = n_items - 1;
    while (lo < hi) {  // last item with q_start <= q
      const int mid = (lo + hi + 1) >> 1;
      if (sm.items[mid].q_start <= q) lo = mid; else hi = mid - 1;
    }
    int32_t blk = -1;
    const Item& it = sm.items[lo];
    const int page = p.page_offset + it.p0 + (q - it.q_start);
    if (q < it.q_start + it.n && page < p.max_blocks_per_req)
      blk = p.block_tables[(size_t)it.r * p.max_blocks_per_req + page];
    if (blk < 0 || blk >= p.num_blocks) {
      record_error(p.err, PA_ERR_DEVICE_INDEX);
      blk = -1;
      ok = 0;
    }
    sm.ids[q] = blk;
  }
  if (tid == 0) {
    // pages the items cover: exactly these are issued, and every one of
    // them is consumed, so no copy is in flight when the window ends
    sm.n_cov = sm.items[n_items - 1].q_start + sm.items[n_items - 1].n;
  }
  if constexpr (kStep) {
    // decode step: the CTA that streams a row's last page appends the row's
    // new token (position L - 1) for its kv head before any copy of the
    // window is issued; the proxy fence and the barrier below order the
    // stores before the bulk copies that read the page.  32 threads move one
    // row's 256 bytes of K and of V.
    for (int w = tid; w < n_items * 32; w += kThreads) {
      const Item& it = sm.items[w >> 5];
      if (it.p0 + it.n != (it.L + kPage - 1) / kPage) continue;  // not the row's last page
      const int pos = it.L - 1;
      const int blk = p.block_tables[(size_t)it.r * p.max_blocks_per_req + pos / kPage];
      if (blk < 0 || blk >= p.num_blocks) continue;  // recorded by the id check above
      const int j = w & 31;
      const size_t src = ((size_t)it.r * Hkv + kvh) * kHeadDim;
      const size_t dst = (((size_t)blk * Hkv + kvh) * kPage + pos % kPage) * kHeadDim;
      const uint4 x = reinterpret_cast<const uint4*>((j < 16 ? p.k_new : p.v_new) + src)[j & 15];
      reinterpret_cast<uint4*>((j < 16 ? p.k_store : p.v_store) + dst)[j & 15] = x;
    }
    fence_proxy_async_global();
  }
  const bool ids_ok = __syncthreads_and(ok) != 0;
  n_cov = sm.n_cov;


  if (tid == 0) {
    // a later window refills stages the warps have read (generic proxy)
    if (kStep && q_lo > 0) fence_proxy_async_smem();
    if constexpr (kQSmem) issue_q(0);
    const int n0 = min(n_cov, q_lo + kStages);
    for (int i = q_lo; i < n0; ++i) issue(i);
  }
  for (int k = 0; k < n_items && !aborted; ++k) {
    const Item& it = sm.items[k];
    const int tok = it.tok;
    const int qend = qg + it.n;
    const int pages_abs = (it.L + kPage - 1) / kPage;
    const int pages_r = pages_abs - p.page_offset;  // pages of the row in the stream
    const int tail_tokens = it.L - (pages_abs - 1) * kPage;
    // segment page at which this token slot is past the row's end (the
    // row's last page, when this slot is beyond its tokens), else none
    const int q_inv = (ts < tail_tokens) ? -1 : qg + (pages_r - 1 - it.p0);
    // q of the 4 heads of this group, scaled into the log2 domain: for bf16
    // pages as dim pairs per head (see qk16), for q8_0 pages as head pairs
    // per dim (see qk16_q8)
    float2 qp[2][16];
    if (kQSmem && !mbar_wait_bounded(&sm.q_full, (uint32_t)k & 1u, kLimit)) {
      // the page loop's first abort check ends the item
      record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
    }
    {
      const uint16_t* qrow =
          kQSmem ? sm.qs : p.q + ((size_t)tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
#pragma unroll
      for (int hp = 0; hp < 2; ++hp) {
        float f0[16], f1[16];
        unpack16s(*reinterpret_cast<const uint4*>(qrow + (2 * hp) * kHeadDim + 8 * c),
                  *reinterpret_cast<const uint4*>(qrow + (2 * hp) * kHeadDim + 64 + 8 * c), f0);
        unpack16s(*reinterpret_cast<const uint4*>(qrow + (2 * hp + 1) * kHeadDim + 8 * c),
                  *reinterpret_cast<const uint4*>(qrow + (2 * hp + 1) * kHeadDim + 64 + 8 * c), f1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if constexpr (kQ8) {
            qp[hp][i] = make_float2(f0[i] * p.scale_log2, f1[i] * p.scale_log2);
          } else {
            const float* f = (i < 8) ? f0 : f1;
            const int j = i & 7;
            qp[hp][i] = make_float2(f[2 * j] * p.scale_log2, f[2 * j + 1] * p.scale_log2);
          }
        }
      }
    }
    float2 acc[kGroup][8];
#pragma unroll
    for (int g = 0; g < kGroup; ++g)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[g][j] = make_float2(0.f, 0.f);
    // running max of head hd (the same in lanes c and c ^ 1) and the sum of
    // this lane's own weights
    float m_own = -INFINITY, l_own = 0.f;

    for (int qa = qg; qa < qend; qa += 2) {
      const int qb = qa + 1;
      const bool has1 = qb < qend;
      const int sa = qa & (kStages - 1), sb = qb & (kStages - 1);
      const uint32_t pa = (uint32_t)(qa / kStages) & 1u, pb = (uint32_t)(qb / kStages) & 1u;
      if (!mbar_wait_bounded(&sm.full[sa], pa, kLimit) || (has1 && !mbar_wait_bounded(&sm.full[sb], pb, kLimit))) {
        record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
        aborted = true;
        break;
      }
      bool valid0 = qa != q_inv;
      bool valid1 = has1 && (qb != q_inv);
      if (!ids_ok) {
        valid0 = valid0 && sm.ids[qa] >= 0;
        valid1 = valid1 && sm.ids[min(qb, (kStep ? kDecodeMaxPagesPerCta : npg) - 1)] >= 0;
      }
      // a missing second page reads whatever stage sb holds; its scores are
      // masked below and its V is not read
      float2 sA01, sA23, sB01, sB23;
      float vdA0 = 0.f, vdB0 = 0.f, vdA1 = 0.f, vdB1 = 0.f;  // q8_0: V group scales of the two pages
      if constexpr (kQ8) {
        const uint8_t* kr0 = sm.k[sa] + ts * kHeadDim;
        const uint8_t* kr1 = sm.k[sb] + ts * kHeadDim;
        float kdA0, kdB0, kdA1, kdB1;
        q8_scales(sm.k[sa], ts, c, kdA0, kdB0);
        q8_scales(sm.k[sb], ts, c, kdA1, kdB1);
        q8_scales(sm.v[sa], ts, c, vdA0, vdB0);
        q8_scales(sm.v[sb], ts, c, vdA1, vdB1);
        qk16_q8(qp, *reinterpret_cast<const uint2*>(kr0 + 8 * c), *reinterpret_cast<const uint2*>(kr0 + 64 + 8 * c),
                kdA0, kdB0, sA01, sA23);
        qk16_q8(qp, *reinterpret_cast<const uint2*>(kr1 + 8 * c), *reinterpret_cast<const uint2*>(kr1 + 64 + 8 * c),
                kdA1, kdB1, sB01, sB23);
      } else {
        const uint8_t* kr0 = sm.k[sa] + ts * (kHeadDim * 2);
        const uint8_t* kr1 = sm.k[sb] + ts * (kHeadDim * 2);
        const uint4 ka0 = *reinterpret_cast<const uint4*>(kr0 + 16 * c);
        const uint4 kb0 = *reinterpret_cast<const uint4*>(kr0 + 128 + 16 * c);
        const uint4 ka1 = *reinterpret_cast<const uint4*>(kr1 + 16 * c);
        const uint4 kb1 = *reinterpret_cast<const uint4*>(kr1 + 128 + 16 * c);
        qk16(qp, ka0, kb0, sA01, sA23);
        qk16(qp, ka1, kb1, sB01, sB23);
      }
      // transposed reduction: 8 values per lane -> 1 complete (token, head)
      float sc;
      {
        const bool b2 = (c >> 2) & 1, b1 = (c >> 1) & 1, b0 = c & 1;
        float2 kA = b2 ? sA23 : sA01, kB = b2 ? sB23 : sB01;
        const float2 oA = shfl_xor2(b2 ? sA01 : sA23, 4), oB = shfl_xor2(b2 ? sB01 : sB23, 4);
        kA = __fadd2_rn(kA, oA);
        kB = __fadd2_rn(kB, oB);
        float2 kk = b1 ? make_float2(kA.y, kB.y) : make_float2(kA.x, kB.x);
        const float2 send = b1 ? make_float2(kA.x, kB.x) : make_float2(kA.y, kB.y);
        kk = __fadd2_rn(kk, shfl_xor2(send, 2));
        sc = (b0 ? kk.y : kk.x) + __shfl_xor_sync(0xffffffffu, b0 ? kk.x : kk.y, 1);
      }
      const bool my_valid = (c & 1) ? valid1 : valid0;
      const float sv = my_valid ? sc : -INFINITY;
      const float mx = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, 1));  // both tokens of head hd
      const bool grow = mx > m_own + kRescaleSlack;
      if (__any_sync(0xffffffffu, grow)) {  // running max grew a lot: rescale (rare)
        const float corr = grow ? fast_exp2(m_own - mx) : 1.f;  // m_own = -inf -> 0
        if (grow) m_own = mx;
        l_own *= corr;
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
          const float cg = __shfl_sync(0xffffffffu, corr, slot_base + (g >> 1) * 4 + (g & 1) * 2);
          const float2 c2 = make_float2(cg, cg);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[g][j] = __fmul2_rn(acc[g][j], c2);
        }
      }
      const float pown = my_valid ? fast_exp2(sv - m_own) : 0.f;
      l_own += pown;
      float pA[kGroup], pB[kGroup];
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int src = slot_base + (g >> 1) * 4 + (g & 1) * 2;
        pA[g] = __shfl_sync(0xffffffffu, pown, src);
        pB[g] = __shfl_sync(0xffffffffu, pown, src + 1);
      }
      if constexpr (kQ8) {
        if (valid0) {
          const uint8_t* vr = sm.v[sa] + ts * kHeadDim;
          pv16_q8(acc, pA, *reinterpret_cast<const uint2*>(vr + 8 * c),
                  *reinterpret_cast<const uint2*>(vr + 64 + 8 * c), vdA0, vdB0);
        }
        if (valid1) {
          const uint8_t* vr = sm.v[sb] + ts * kHeadDim;
          pv16_q8(acc, pB, *reinterpret_cast<const uint2*>(vr + 8 * c),
                  *reinterpret_cast<const uint2*>(vr + 64 + 8 * c), vdA1, vdB1);
        }
      } else {
        if (valid0) {
          const uint8_t* vr = sm.v[sa] + ts * (kHeadDim * 2);
          pv16(acc, pA, *reinterpret_cast<const uint4*>(vr + 16 * c),
               *reinterpret_cast<const uint4*>(vr + 128 + 16 * c));
        }
        if (valid1) {
          const uint8_t* vr = sm.v[sb] + ts * (kHeadDim * 2);
          pv16(acc, pB, *reinterpret_cast<const uint4*>(vr + 16 * c),
               *reinterpret_cast<const uint4*>(vr + 128 + 16 * c));
        }
      }
      __syncwarp();
      if (lane == 0) {  // this warp is done with the iteration's pages
        release(qa);
        if (has1) release(qb);
      }
      if (((qa - qg) & 15) == 0 && *reinterpret_cast<volatile int*>(&sm.abort_flag)) {
        aborted = true;
        break;
      }
    }
    qg = qend;

    // ---- item end: merge the 16 token slots (all threads take part)
    bar_all();
    if (aborted || *reinterpret_cast<volatile int*>(&sm.abort_flag)) {
      aborted = true;
      break;
    }
    // every warp has read the item's q: the next item's q can land
    if (kQSmem && tid == 0 && k + 1 < n_items) {
      fence_proxy_async_smem();
      issue_q(k + 1);
    }
    // merge across the 4 warps in two rounds of two heads (shared memory);
    // warp g ends with head g
    const int g = warp;
    const int d0 = lane * 4;
    float M = -INFINITY, Ls = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    {
      const float l_pair = l_own + __shfl_xor_sync(0xffffffffu, l_own, 1);
      float mh[kGroup], lh[kGroup], Mw[kGroup], Lw[kGroup];
#pragma unroll
      for (int gg = 0; gg < kGroup; ++gg) {
        const int src = slot_base + (gg >> 1) * 4 + (gg & 1) * 2;
        mh[gg] = __shfl_sync(0xffffffffu, m_own, src);
        lh[gg] = __shfl_sync(0xffffffffu, l_pair, src);
        float Mg = fmaxf(mh[gg], __shfl_xor_sync(0xffffffffu, mh[gg], 8));
        Mg = fmaxf(Mg, __shfl_xor_sync(0xffffffffu, Mg, 16));
        Mw[gg] = Mg;
        const float f = (mh[gg] == -INFINITY) ? 0.f : fast_exp2(mh[gg] - Mg);
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[gg][j] = __fmul2_rn(acc[gg][j], f2);
        float lsum = lh[gg] * f;
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
        Lw[gg] = lsum;
      }
      // sum over the warp's 4 token slots, transposed: the slot with bits
      // (s1, s0) ends with head 2 s1 + s0
      const bool s1 = (lane >> 4) & 1, s0 = (lane >> 3) & 1;
      float2 h0[8], h1[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // xor 16: keep heads {2 s1, 2 s1 + 1}
        const float2 keep0 = s1 ? acc[2][j] : acc[0][j], send0 = s1 ? acc[0][j] : acc[2][j];
        const float2 keep1 = s1 ? acc[3][j] : acc[1][j], send1 = s1 ? acc[1][j] : acc[3][j];
        h0[j] = __fadd2_rn(keep0, shfl_xor2(send0, 16));
        h1[j] = __fadd2_rn(keep1, shfl_xor2(send1, 16));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // xor 8: keep head 2 s1 + s0
        const float2 keep = s0 ? h1[j] : h0[j], send = s0 ? h0[j] : h1[j];
        h0[j] = __fadd2_rn(keep, shfl_xor2(send, 8));
      }
#pragma unroll
      for (int rnd = 0; rnd < 2; ++rnd) {  // heads 2 rnd and 2 rnd + 1
        if (rnd) bar_all();                // round 0's reads are done
        if ((int)s1 == rnd) {
          float* dst = sm.mrg_o[warp][s0 ? 1 : 0];
          *reinterpret_cast<float4*>(dst + 8 * c) = make_float4(h0[0].x, h0[0].y, h0[1].x, h0[1].y);
          *reinterpret_cast<float4*>(dst + 8 * c + 4) = make_float4(h0[2].x, h0[2].y, h0[3].x, h0[3].y);
          *reinterpret_cast<float4*>(dst + 64 + 8 * c) = make_float4(h0[4].x, h0[4].y, h0[5].x, h0[5].y);
          *reinterpret_cast<float4*>(dst + 64 + 8 * c + 4) = make_float4(h0[6].x, h0[6].y, h0[7].x, h0[7].y);
        }
        if (lane == 0) {
          sm.mrg_m[warp][0] = Mw[2 * rnd];
          sm.mrg_m[warp][1] = Mw[2 * rnd + 1];
          sm.mrg_l[warp][0] = Lw[2 * rnd];
          sm.mrg_l[warp][1] = Lw[2 * rnd + 1];
        }
        bar_all();
        if ((g >> 1) == rnd) {  // head g: lane owns dims [4 lane, +4)
          const int j = g & 1;
          float mwv[kWarps];
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            mwv[w] = sm.mrg_m[w][j];
            M = fmaxf(M, mwv[w]);
          }
          if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
              const float f = (mwv[w] == -INFINITY) ? 0.f : fast_exp2(mwv[w] - M);
              const float4 x = *reinterpret_cast<const float4*>(&sm.mrg_o[w][j][d0]);
              Ls += sm.mrg_l[w][j] * f;
              o.x = fmaf(f, x.x, o.x);
              o.y = fmaf(f, x.y, o.y);
              o.z = fmaf(f, x.z, o.z);
              o.w = fmaf(f, x.w, o.w);
            }
          }
        }
      }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
    float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
    const int head = kvh * kGroup + g;
    const size_t orow = (size_t)tok * p.num_q_heads + head;
    const bool complete = (it.p0 == 0) && (it.n == pages_r);
    if (complete) {
      if (p.prefix_o) lse2 = fold_prefix(p, o, lse2, orow, d0, lane);
      uint2 packed;
      packed.x = pack_bf16x2(o.x, o.y);
      packed.y = pack_bf16x2(o.z, o.w);
      *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + d0) = packed;
      if (p.lse && lane == 0) p.lse[orow] = lse2 * kLn2;
      bar_all();  // warps leave the item together (measured faster than without)
      continue;
    }
    // the item is cut by segment boundaries: publish this CTA's partial
    const int A = it.A;
    // segments holding the row's pages: the row starts at stream position A,
    // its pages at A + kAlpha.  Its piece in segment b0 is that CTA's last
    // item (slot 1) when the segment starts before the row, else its first
    int seg_len;
    if constexpr (kStep) seg_len = sm.seg_cost; else seg_len = plan.seg;
    const int b0 = (A + kAlpha) / seg_len, b1 = (A + kAlpha + pages_r - 1) / seg_len;
    const int jslot = ((kStep ? win0 : 0) + k == 0) ? 0 : 1;
    const size_t slot = ((size_t)b * 2 + jslot) * kGroup + g;
    if ((int64_t)slot < p.piece_slots) {
      *reinterpret_cast<float4*>(p.piece_o + slot * kHeadDim + d0) = o;
      if (lane == 0) p.piece_lse[slot] = lse2;
    } else if (lane == 0) {
      record_error(p.err, PA_ERR_DEVICE_INDEX);  // the host sized the workspace for fewer pieces
    }
    bar_all();  // every piece write of the CTA precedes tid 0's release below
    if (tid == 0) {
      int* cnt = p.counters + (size_t)it.r * Hkv + kvh;
      const int done = atom_add_acq_rel_gpu(cnt, 1);
      sm.is_last = (done == b1 - b0);
      if (sm.is_last) *cnt = 0;  // every piece has arrived: ready for the next call
    }
    bar_all();  // tid 0's acquire orders the piece reads below
    if (sm.is_last) {
      // kRound pieces per round with every load of the round (lane i: the
      // lse of piece i; all lanes: 4 dims of each piece) in flight at once,
      // merged by log-sum-exp with a running max across rounds
      constexpr int kRound = 16;
      const int n_pc = b1 - b0 + 1;
      auto piece_slot = [&](int bb) {
        const int jj = (bb == b0 && b0 * seg_len < A) ? 1 : 0;
        return ((size_t)(bb * Hkv + kvh) * 2 + jj) * kGroup + g;
      };
      float Mx = -INFINITY, wsum = 0.f;
      float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c0 = 0; c0 < n_pc; c0 += kRound) {
        const int nc = min(kRound, n_pc - c0);
        const float lv = lane < nc ? __ldcg(p.piece_lse + piece_slot(b0 + c0 + lane)) : -INFINITY;
        float4 x[kRound];
#pragma unroll
        for (int i = 0; i < kRound; ++i)
          x[i] = i < nc ? __ldcg(reinterpret_cast<const float4*>(p.piece_o + piece_slot(b0 + c0 + i) * kHeadDim + d0))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        float mb = lv;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o2));
        const float mn = fmaxf(Mx, mb);
        if (mn == -INFINITY) continue;  // every piece so far is empty
        const float sc = fast_exp2(Mx - mn);  // Mx = -inf -> 0
        wsum *= sc;
        a4 = make_float4(a4.x * sc, a4.y * sc, a4.z * sc, a4.w * sc);
        const float w = fast_exp2(lv - mn);  // -inf -> 0
        float ws = w;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o2);
        wsum += ws;
#pragma unroll
        for (int i = 0; i < kRound; ++i) {
          const float wi = __shfl_sync(0xffffffffu, w, i);
          a4.x = fmaf(wi, x[i].x, a4.x);
          a4.y = fmaf(wi, x[i].y, a4.y);
          a4.z = fmaf(wi, x[i].z, a4.z);
          a4.w = fmaf(wi, x[i].w, a4.w);
        }
        Mx = mn;
      }
      const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
      a4.x *= winv;
      a4.y *= winv;
      a4.z *= winv;
      a4.w *= winv;
      float l2 = wsum > 0.f ? Mx + log2f(wsum) : -INFINITY;
      if (p.prefix_o) l2 = fold_prefix(p, a4, l2, orow, d0, lane);
      uint2 packed;
      packed.x = pack_bf16x2(a4.x, a4.y);
      packed.y = pack_bf16x2(a4.z, a4.w);
      *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + d0) = packed;
      if (p.lse && lane == 0) p.lse[orow] = l2 * kLn2;
    }
    bar_all();  // is_last is free again
  }
  if (aborted || !kStep) break;
  // next window: every item of this one is done (the barrier at its end)
  // and its pages are consumed, so the ring is empty
  win0 += n_items;
  if (win0 >= sm.n_items_all) break;
  if constexpr (kStep)
    step_window<1, kThreads, kDecodeMaxItemsPerCta, kDecodeMaxPagesPerCta>(p, plan, sm, kvh, sidx,
                                                                          (int)gridDim.x / Hkv, win0);
  }

  __syncthreads();  // every thread has left the item loop
  if (*reinterpret_cast<volatile int*>(&sm.abort_flag) && tid == 0) {
    // A wait gave up: let the last copy issued into each stage land
    // (bounded), then leave.  A stage whose copies never land is passed
    // over after the bound, and the others are still waited for, so no
    // copy that can land is still in flight when the CTA leaves.
    for (int s = 0; s < kStages; ++s) {
      const int j = *reinterpret_cast<volatile int*>(&sm.stage_page[s]);
      if (j >= 0) mbar_wait_bounded(&sm.full[s], (uint32_t)(j / kStages) & 1u, kLimit);
    }
    if (sm.q_issued > 0) mbar_wait_bounded(&sm.q_full, (uint32_t)(sm.q_issued - 1) & 1u, kLimit);
  }
}


// ---------------------------------------------------- warp-granular kernel
// One CTA of kWgWarps warps per SM.  Every CTA segment is cut into kWgWarps
// equal warp segments: warp w of CTA b streams pages [w sw, (w + 1) sw) of
// the CTA's segment (sw = seg / kWgWarps) through its own kWgStages-deep
// ring and finishes its items on its own.  A warp's item end (the merge of
// its 4 token slots, the partial of a cut row, the count of finished pieces,
// the merge of all pieces by the last one) then stalls only that warp: the
// other warps of the SM keep streaming, and no CTA-wide barrier follows the
// prologue.  The page loop is the same arithmetic as above; a warp takes the
// 16 tokens of a page as two pairs per lane (tokens ts + 8 h and ts + 4 + 8
// h, h = 0, 1).
constexpr int kWgStages = 2;  // pages in flight per warp
constexpr int kWgThreads = kWgWarps * 32;

template <int kSlab>
struct __align__(128) WgSmem {
  uint8_t k[kWgWarps][kWgStages][kSlab];
  uint8_t v[kWgWarps][kWgStages][kSlab];
  uint16_t qs[kWgWarps][kGroup * kHeadDim];  // each warp's current item's q (bulk copy)
  uint64_t full[kWgWarps][kWgStages];        // TMA landed
  uint64_t q_full[kWgWarps];                 // q landed
  int32_t ids[kWgMaxPagesPerCta];
  Item items[kWgMaxItemsPerCta];
  int stage_page[kWgWarps][kWgStages];  // last warp page issued into each stage (-1: none)
  int q_issued[kWgWarps];
  int n_items;
  int abort_flag;
  // decode step (self-planned): see step_window
  int scan[kWgWarps];
  int n_items_all;
  int seg_cost;
  int seg_pages;
};

static_assert(offsetof(WgSmem<kSlabBytes>, v) % 128 == 0 && offsetof(WgSmem<kQ8SlabBytes>, v) % 16 == 0 &&
                  offsetof(WgSmem<kSlabBytes>, qs) % 16 == 0 && offsetof(WgSmem<kQ8SlabBytes>, qs) % 16 == 0 &&
                  (kWgStages * kSlabBytes) % 16 == 0 && (kWgStages * kQ8SlabBytes) % 16 == 0,
              "bulk copies land on 16-byte boundaries");
static_assert(sizeof(WgSmem<kSlabBytes>) <= 227 * 1024, "one decode CTA per SM");

// Online log-sum-exp merge of normalised partials (log2-domain lse) for one
// head per 8-lane group (head g = lane >> 3), 16 dims per lane (dims
// 8c .. 8c + 7 and 64 + 8c .. 64 + 8c + 7): m is the running max, w the sum
// of weights relative to it and a the weighted sum of the partials.
struct LseAcc {
  float m, w;
  float a[16];
};

__device__ __forceinline__ void lse_acc_init(LseAcc& s, const float (&o)[16], float lse2) {
  s.m = lse2;
  s.w = lse2 == -INFINITY ? 0.f : 1.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) s.a[i] = lse2 == -INFINITY ? 0.f : o[i];
}

// Adds up to 4 partials: row(u) points at partial u's 128 fp32 of this head,
// lse_at(u) at its lse; every load of the batch is issued before any is used.
template <bool kL2Only, class Row, class Lse>
__device__ __forceinline__ void lse_acc_batch(LseAcc& s, int nb, int c, Row&& row, Lse&& lse_at) {
  float l[4];
  float4 y[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (u < nb) {
      const float* yr = row(u);
      const float* lp = lse_at(u);
      if constexpr (kL2Only) {
        l[u] = __ldcg(lp);
        y[u][0] = __ldcg(reinterpret_cast<const float4*>(yr + 8 * c));
        y[u][1] = __ldcg(reinterpret_cast<const float4*>(yr + 8 * c + 4));
        y[u][2] = __ldcg(reinterpret_cast<const float4*>(yr + 64 + 8 * c));
        y[u][3] = __ldcg(reinterpret_cast<const float4*>(yr + 64 + 8 * c + 4));
      } else {
        l[u] = *lp;
        y[u][0] = *reinterpret_cast<const float4*>(yr + 8 * c);
        y[u][1] = *reinterpret_cast<const float4*>(yr + 8 * c + 4);
        y[u][2] = *reinterpret_cast<const float4*>(yr + 64 + 8 * c);
        y[u][3] = *reinterpret_cast<const float4*>(yr + 64 + 8 * c + 4);
      }
    } else {
      l[u] = -INFINITY;
      y[u][0] = y[u][1] = y[u][2] = y[u][3] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const float mb = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
  const float mn = fmaxf(s.m, mb);
  if (mn == -INFINITY) return;  // every partial so far is empty
  const float sc = fast_exp2(s.m - mn);  // s.m = -inf -> 0
  s.w *= sc;
#pragma unroll
  for (int i = 0; i < 16; ++i) s.a[i] *= sc;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float wu = fast_exp2(l[u] - mn);  // -inf -> 0
    s.w += wu;
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      s.a[4 * v4 + 0] = fmaf(wu, y[u][v4].x, s.a[4 * v4 + 0]);
      s.a[4 * v4 + 1] = fmaf(wu, y[u][v4].y, s.a[4 * v4 + 1]);
      s.a[4 * v4 + 2] = fmaf(wu, y[u][v4].z, s.a[4 * v4 + 2]);
      s.a[4 * v4 + 3] = fmaf(wu, y[u][v4].w, s.a[4 * v4 + 3]);
    }
  }
  s.m = mn;
}

// Normalises the merged partial into o; returns its log2 lse.
__device__ __forceinline__ float lse_acc_done(const LseAcc& s, float (&o)[16]) {
  const float inv = s.w > 0.f ? 1.f / s.w : 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = s.a[i] * inv;
  return s.w > 0.f ? s.m + log2f(s.w) : -INFINITY;
}

// Folds the shared-prefix partials of output row orow (p.prefix_n key-chunk
// partials, or the merged one) into the merge state, four at a time.
__device__ __forceinline__ void lse_acc_prefix(LseAcc& s, const DecodeParams& p, size_t orow, int c) {
  for (int c0 = 0; c0 < p.prefix_n; c0 += 4)
    lse_acc_batch<false>(
        s, min(4, p.prefix_n - c0), c,
        [&](int u) { return p.prefix_o + ((size_t)(c0 + u) * p.prefix_rows + orow) * kHeadDim; },
        [&](int u) { return p.prefix_lse + (size_t)(c0 + u) * p.prefix_rows + orow; });
}

// A prefix pass running beside the decode launch (p.prefix_done set): the
// count of key chunks written for token tok's query tile and kv head.
__device__ __forceinline__ const int* prefix_flag(const DecodeParams& p, int tok, int kvh) {
  return p.prefix_done ? p.prefix_done + (size_t)(tok / kPrefillQTile) * p.num_kv_heads + kvh : nullptr;
}

// Whole warp, before a fold: completes the wait for every key chunk of the
// tile, begun by lane 0's relaxed read `peek` of the count (issued early, so
// its latency hides behind other loads): a bounded acquire spin if the count
// was short, else an acquire fence.  False on a timeout (recorded; the fold
// is left out).  Then counts this reader, its result (lane 0) in *readers_old
// for prefix_read_done: every reader has passed its wait when the count is
// full, so the last one may return the counters to zero while the others
// still read the partials (which the counters do not guard).
__device__ __forceinline__ bool prefix_ready(const DecodeParams& p, int tok, int kvh, int lane, int peek,
                                             int* readers_old) {
  if (!p.prefix_done) return true;
  int ok = 1;
  if (lane == 0) {
    const int* f = prefix_flag(p, tok, kvh);
    if (peek >= p.prefix_n) {
      fence_acq_rel_gpu();
    } else if (ld_acquire_gpu(f) < p.prefix_n) {
      const unsigned long long t0 = globaltimer();
      while (ld_acquire_gpu(f) < p.prefix_n) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(128);
      }
    }
    *readers_old = atomicAdd(p.prefix_readers + (size_t)(tok / kPrefillQTile) * p.num_kv_heads + kvh, 1);
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();  // lane 0's acquire orders every lane's partial reads
  return ok != 0;
}

// After a fold (lane 0's count from prefix_ready): the last reader of a
// tile's kv head (one per query token of the tile) returns both counters to
// zero for the next call.
__device__ __forceinline__ void prefix_read_done(const DecodeParams& p, int tok, int kvh, int lane, int readers_old) {
  if (!p.prefix_done || lane != 0) return;
  const int t = tok / kPrefillQTile;
  const int readers = min(kPrefillQTile, p.total_q - t * kPrefillQTile);
  if (readers_old == readers - 1) {
    const size_t idx = (size_t)t * p.num_kv_heads + kvh;
    p.prefix_readers[idx] = 0;
    p.prefix_done[idx] = 0;
  }
}

// bf16 store of a lane's 16 dims (dims 8c .. 8c + 7 and 64 + 8c .. 64 + 8c + 7)
__device__ __forceinline__ void store_row16(uint16_t* row, const float (&o)[16], int c) {
  uint4 lo, hi;
  lo.x = pack_bf16x2(o[0], o[1]);
  lo.y = pack_bf16x2(o[2], o[3]);
  lo.z = pack_bf16x2(o[4], o[5]);
  lo.w = pack_bf16x2(o[6], o[7]);
  hi.x = pack_bf16x2(o[8], o[9]);
  hi.y = pack_bf16x2(o[10], o[11]);
  hi.z = pack_bf16x2(o[12], o[13]);
  hi.w = pack_bf16x2(o[14], o[15]);
  *reinterpret_cast<uint4*>(row + 8 * c) = lo;
  *reinterpret_cast<uint4*>(row + 64 + 8 * c) = hi;
}

// The merge of a cut row's pieces by its last piece (whole warp), four
// partials per batch with all their loads in flight; kept out of line so that
// its registers do not weigh on the page loop.  With a prefix pass beside
// the launch, lane 0 first reads the row's prefix chunk count (relaxed; its
// latency hides behind the piece loads) and returns it.
__device__ __noinline__ int wg_merge_pieces(const float* piece_o, const float* piece_lse, int64_t piece_slots, int b0,
                                            int b1, int A, int sw, int Hkv, int kvh, int g, int c, int lane,
                                            const int* flag, LseAcc& out) {
  const int peek = (flag && lane == 0) ? ld_relaxed_gpu(flag) : 0;
  const int n_pc = b1 - b0 + 1;
  auto piece_slot = [&](int bb) {  // (a slot past the workspace was recorded and is read clamped)
    const int jj = (bb == b0 && b0 * sw < A) ? 1 : 0;
    return min(((size_t)(bb * Hkv + kvh) * 2 + jj) * kGroup + g, (size_t)piece_slots - 1);
  };
  LseAcc acc;
  acc.m = -INFINITY;
  acc.w = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc.a[i] = 0.f;
  for (int c0 = 0; c0 < n_pc; c0 += 4)
    lse_acc_batch<true>(
        acc, min(4, n_pc - c0), c, [&](int u) { return piece_o + piece_slot(b0 + c0 + u) * kHeadDim; },
        [&](int u) { return piece_lse + piece_slot(b0 + c0 + u); });
  out = acc;
  return peek;
}

// kDiag: the diagnostic instantiation that tests the timeout path (bf16
// pages).  Warp 0 of CTA 0 arms the barrier of its second page without
// issuing that page's copies, so the wait on it runs out; every wait of this
// instantiation gives up after 1 ms instead of kWaitLimitNs.  No copy is
// dropped anywhere else, and nothing is read out of bounds.
template <bool kQ8, bool kDiag, bool kStep = false>
__global__ void __launch_bounds__(kWgThreads, 1)
    decode_wg_kernel(const DecodeParams p, const __grid_constant__ typename PlanOf<kStep>::type plan) {
  static_assert(!(kDiag && kQ8), "the diagnostic instantiation reads bf16 pages");
  static_assert(!(kStep && (kQ8 || kDiag)), "the decode step serves bf16 pages");
  // the fixed cost of a row in the stream's units (the host plan cuts in
  // pages, with no fixed cost)
  constexpr int kAlpha = kStep ? kStepItemCost : 0;
  constexpr unsigned long long kLimit = kDiag ? 1000000ull : kWaitLimitNs;
  constexpr int kSlab = kQ8 ? kQ8SlabBytes : kSlabBytes;
  using Smem = WgSmem<kSlab>;
  // q of each item by a bulk copy into the warp's shared-memory slot, issued
  // an item ahead (bf16 pages); q8_0 pages read q from global memory
  constexpr bool kQSmem = !kQ8;
  // the self-planned step reads lengths and tables that earlier kernels may
  // write: it waits for them before anything else
  if constexpr (kStep) pdl_wait();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.num_kv_heads;
  const int kvh = b % Hkv, sidx = b / Hkv;
  if (tid == 0) {
    for (int w = 0; w < kWgWarps; ++w) {
      for (int s = 0; s < kWgStages; ++s) {
        mbar_init(&sm.full[w][s], 1);
        sm.stage_page[w][s] = -1;
      }
      mbar_init(&sm.q_full[w], 1);
      sm.q_issued[w] = 0;
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  int seg_units;  // segment length in stream units (pages, or pages plus row costs)
  if constexpr (kStep) {
    // the CTA plans its own segment from the device seq_lens; a segment with
    // more than kWgMaxItemsPerCta rows cannot occur for the launches the
    // host sends here (it checks the bound) and is recorded
    step_window<kWgWarps, kWgThreads, kWgMaxItemsPerCta, kWgMaxPagesPerCta>(p, plan, sm, kvh, sidx,
                                                                           (int)gridDim.x / Hkv, 0);
    seg_units = sm.seg_cost;
    if (tid == 0 && sm.n_items_all > kWgMaxItemsPerCta) record_error(p.err, PA_ERR_DEVICE_INDEX);
  } else {
    const int S0 = sidx * plan.seg;
    const int npg = min(plan.total, S0 + plan.seg) - S0;  // pages of this CTA's segment
    if (npg <= 0) return;
    seg_units = plan.seg;
    const int n_items_all = plan.n_rows;
    // ---- item table of the CTA's segment (warp 0), 32 items per round; it
    // comes from the kernel parameters alone, so it is built before the wait
    // for the previous kernel
    if (warp == 0) {
      int base_q = 0, n_it = 0;
      for (int k0 = 0; k0 < kWgMaxItemsPerCta; k0 += 32) {
        const int item = plan.first_row[sidx] + k0 + lane;
        const bool exists = item < n_items_all;
        int r = 0, L = 0, size = 0, tok = 0;
        const int p0 = (k0 + lane == 0) ? plan.first_page[sidx] : 0;
        if (exists) {
          r = plan.rows[item];
          L = plan.seq[item];
          tok = plan.tok[item];
          size = max((L + kPage - 1) / kPage - p.page_offset - p0, 0);
        }
        int incl = size;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int start = base_q + incl - size;
        const bool in_seg = size > 0 && start < npg;
        if (in_seg && k0 + lane < kWgMaxItemsPerCta) {
          Item& it = sm.items[k0 + lane];
          it.q_start = start;
          it.n = min(size, npg - start);
          it.p0 = p0;
          it.r = r;
          it.L = L;
          it.tok = tok;
          it.A = S0 + start - p0;  // stream position of the row's page 0
          bulk_prefetch_l2(p.q + ((size_t)tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim,
                           kGroup * kHeadDim * 2);
        }
        const unsigned covered = __ballot_sync(0xffffffffu, in_seg);
        const int prefix = (~covered == 0u) ? 32 : (__ffs((int)~covered) - 1);
        n_it = k0 + prefix;
        base_q += __shfl_sync(0xffffffffu, incl, 31);
        if (prefix < 32 || base_q >= npg) break;
      }
      if (lane == 0) {
        if (base_q < npg) record_error(p.err, PA_ERR_DEVICE_INDEX);  // metadata differ from the plan
        sm.n_items = min(n_it, kWgMaxItemsPerCta);
      }
    }
    __syncthreads();
    // Beside a tile kernel (p.beside) this launch starts once every CTA of
    // that kernel has passed its own wait, so the kernels before it are
    // complete; waiting here would wait for the tile kernel itself.
    if (!p.beside) pdl_wait();
  }
  const int n_items = sm.n_items;
  if (n_items == 0) return;  // nothing covered (recorded above); no copy was issued
  // ---- block ids of the segment's pages; an id outside the pool (or a page
  // past the table) is recorded and masked, and fetched from block 0
  const int n_cov = sm.items[n_items - 1].q_start + sm.items[n_items - 1].n;
  int ok = 1;
  for (int q = tid; q < n_cov; q += kWgThreads) {
    int lo = 0, hi = n_items - 1;
    while (lo < hi) {  // last item with q_start <= q
      const int mid = (lo + hi + 1) >> 1;
      if (sm.items[mid].q_start <= q) lo = mid; else hi = mid - 1;
    }
    int32_t blk = -1;
    const Item& it = sm.items[lo];
    const int page = p.page_offset + it.p0 + (q - it.q_start);
    if (page < p.max_blocks_per_req) blk = p.block_tables[(size_t)it.r * p.max_blocks_per_req + page];
    if (blk < 0 || blk >= p.num_blocks) {
      record_error(p.err, PA_ERR_DEVICE_INDEX);
      blk = -1;
      ok = 0;
    }
    sm.ids[q] = blk;
  }
  const bool ids_ok = __syncthreads_and(ok) != 0;

  // ---- this warp's part of the segment: stream units [cs, cs + sw), its
  // pages [a, e) of the segment (with the host plan a unit is a page)
  const int sw = seg_units / kWgWarps;
  int a, e;
  if constexpr (kStep) {
    const int cs = sidx * seg_units + warp * sw, ce = cs + sw;
    a = n_cov;
    e = n_cov;
    for (int kk = n_items - 1; kk >= 0; --kk) {  // the first page at or past cs, resp. ce
      const Item& it = sm.items[kk];
      const int u0 = it.A + kAlpha + it.p0;  // stream position of the item's first page
      if (u0 + it.n > cs) a = it.q_start + max(0, cs - u0);
      if (u0 + it.n > ce) e = it.q_start + max(0, ce - u0);
    }
  } else {
    a = warp * sw;
    e = min(a + sw, n_cov);
  }
  if (a >= e) return;
  int k = 0;  // first item holding page a
  {
    int lo = 0, hi = n_items - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sm.items[mid].q_start <= a) lo = mid; else hi = mid - 1;
    }
    k = lo;
  }
  const int k_first = k;
  const int gw = sidx * kWgWarps + warp;  // warp segment of the stream
  const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k_cache);
  const uint8_t* vbase = reinterpret_cast<const uint8_t*>(p.v_cache);
  // segment page q in [a, e) -> warp page j = q - a -> stage j % kWgStages
  auto issue = [&](int q) {
    const int j = q - a;
    const int s = j & (kWgStages - 1);
    const size_t off = ((size_t)max(sm.ids[q], 0) * Hkv + kvh) * kSlab;
    mbar_arrive_expect_tx(&sm.full[warp][s], 2 * kSlab);
    if (!(kDiag && b == 0 && warp == 0 && j == 1)) {  // (diagnostic: armed, never copied)
      bulk_g2s(sm.k[warp][s], kbase + off, kSlab, &sm.full[warp][s]);
      bulk_g2s(sm.v[warp][s], vbase + off, kSlab, &sm.full[warp][s]);
    }
    sm.stage_page[warp][s] = j;  // only lane 0 of this warp writes it
  };
  auto issue_q = [&](int kk) {
    const size_t qoff = ((size_t)sm.items[kk].tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
    mbar_arrive_expect_tx(&sm.q_full[warp], kGroup * kHeadDim * 2);
    bulk_g2s(sm.qs[warp], p.q + qoff, kGroup * kHeadDim * 2, &sm.q_full[warp]);
    sm.q_issued[warp] += 1;
  };
  if constexpr (kStep) {
    // decode step: the warp that reads a row's last page stores the row's
    // new token (position L - 1) for its kv head before any copy it issues;
    // the proxy fence orders the stores before those bulk copies
    for (int kk = k; kk < n_items; ++kk) {
      const Item& it = sm.items[kk];
      if (it.q_start >= e) break;
      if (it.p0 + it.n != (it.L + kPage - 1) / kPage) continue;  // not the row's last page
      const int qlast = it.q_start + it.n - 1;
      if (qlast < a || qlast >= e) continue;  // another warp's page
      const int pos = it.L - 1;
      const int blk = p.block_tables[(size_t)it.r * p.max_blocks_per_req + pos / kPage];
      if (blk < 0 || blk >= p.num_blocks) continue;  // recorded by the id check above
      const size_t src = ((size_t)it.r * Hkv + kvh) * kHeadDim;
      const size_t dst = (((size_t)blk * Hkv + kvh) * kPage + pos % kPage) * kHeadDim;
      const uint4 x = reinterpret_cast<const uint4*>((lane < 16 ? p.k_new : p.v_new) + src)[lane & 15];
      reinterpret_cast<uint4*>((lane < 16 ? p.k_store : p.v_store) + dst)[lane & 15] = x;
    }
    fence_proxy_async_global();
    __syncwarp();
  }
  if (lane == 0) {
    if constexpr (kQSmem) issue_q(k);
    for (int q = a; q < min(e, a + kWgStages); ++q) issue(q);
  }

  const int ts = lane >> 3;  // token slot: tokens ts + 4 u of every page
  const int c = lane & 7;    // dim chunk: dims [8c, 8c+8) and [64+8c, 64+8c+8)
  // After the transposed reduction lane c holds token u = bit0(c) of the
  // pair and head hd = 2 bit2(c) + bit1(c).
  const int slot_base = lane & ~7;
  bool aborted = false;
  int nq = 0;  // q copies this warp has consumed

  for (; k < n_items && !aborted; ++k) {
    const Item& it = sm.items[k];
    const int i0 = max(it.q_start, a);
    const int i1 = min(it.q_start + it.n, e);
    if (i0 >= i1) break;  // past this warp's pages
    const int tok = it.tok;
    const int p0w = it.p0 + (i0 - it.q_start);  // row page of the warp's first page of the item
    const int pages_abs = (it.L + kPage - 1) / kPage;
    const int pages_r = pages_abs - p.page_offset;  // pages of the row in the stream
    const int tail_tokens = it.L - (pages_abs - 1) * kPage;
    const int q_last = i0 + (pages_r - 1 - p0w);  // segment page holding the row's last token
    // q of the 4 heads of this group, scaled into the log2 domain (see qk16 /
    // qk16_q8 for the two layouts)
    float2 qp[2][16];
    if (kQSmem && !mbar_wait_bounded(&sm.q_full[warp], (uint32_t)nq & 1u, kLimit)) {
      record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
      aborted = true;
      break;
    }
    ++nq;
    {
      const uint16_t* qrow =
          kQSmem ? sm.qs[warp] : p.q + ((size_t)tok * p.num_q_heads + (size_t)kvh * kGroup) * kHeadDim;
#pragma unroll
      for (int hp = 0; hp < 2; ++hp) {
        float f0[16], f1[16];
        unpack16s(*reinterpret_cast<const uint4*>(qrow + (2 * hp) * kHeadDim + 8 * c),
                  *reinterpret_cast<const uint4*>(qrow + (2 * hp) * kHeadDim + 64 + 8 * c), f0);
        unpack16s(*reinterpret_cast<const uint4*>(qrow + (2 * hp + 1) * kHeadDim + 8 * c),
                  *reinterpret_cast<const uint4*>(qrow + (2 * hp + 1) * kHeadDim + 64 + 8 * c), f1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if constexpr (kQ8) {
            qp[hp][i] = make_float2(f0[i] * p.scale_log2, f1[i] * p.scale_log2);
          } else {
            const float* f = (i < 8) ? f0 : f1;
            const int j = i & 7;
            qp[hp][i] = make_float2(f[2 * j] * p.scale_log2, f[2 * j + 1] * p.scale_log2);
          }
        }
      }
    }
    if constexpr (kQSmem) {
      // every lane holds its q: the warp's next item's q can land
      __syncwarp();
      if (lane == 0 && k + 1 < n_items && sm.items[k + 1].q_start < e) {
        fence_proxy_async_smem();
        issue_q(k + 1);
      }
    }
    float2 acc[kGroup][8];
#pragma unroll
    for (int g = 0; g < kGroup; ++g)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[g][j] = make_float2(0.f, 0.f);
    // running max of head hd (the same in lanes c and c ^ 1) and the sum of
    // this lane's own weights
    float m_own = -INFINITY, l_own = 0.f;

    for (int q = i0; q < i1; ++q) {
      const int j = q - a;
      const int s = j & (kWgStages - 1);
      if (!mbar_wait_bounded(&sm.full[warp][s], (uint32_t)(j / kWgStages) & 1u, kLimit)) {
        record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
        aborted = true;
        break;
      }
      const bool last_pg = q == q_last;
      const bool pg_ok = ids_ok || sm.ids[q] >= 0;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int t0 = ts + 8 * h, t1 = t0 + 4;  // the pair's two tokens of the page
        const bool valid0 = pg_ok && (!last_pg || t0 < tail_tokens);
        const bool valid1 = pg_ok && (!last_pg || t1 < tail_tokens);
        float2 sA01, sA23, sB01, sB23;
        float vdA0 = 0.f, vdB0 = 0.f, vdA1 = 0.f, vdB1 = 0.f;  // q8_0: V group scales of the two tokens
        if constexpr (kQ8) {
          const uint8_t* kr0 = sm.k[warp][s] + t0 * kHeadDim;
          const uint8_t* kr1 = sm.k[warp][s] + t1 * kHeadDim;
          float kdA0, kdB0, kdA1, kdB1;
          q8_scales(sm.k[warp][s], t0, c, kdA0, kdB0);
          q8_scales(sm.k[warp][s], t1, c, kdA1, kdB1);
          q8_scales(sm.v[warp][s], t0, c, vdA0, vdB0);
          q8_scales(sm.v[warp][s], t1, c, vdA1, vdB1);
          qk16_q8(qp, *reinterpret_cast<const uint2*>(kr0 + 8 * c),
                  *reinterpret_cast<const uint2*>(kr0 + 64 + 8 * c), kdA0, kdB0, sA01, sA23);
          qk16_q8(qp, *reinterpret_cast<const uint2*>(kr1 + 8 * c),
                  *reinterpret_cast<const uint2*>(kr1 + 64 + 8 * c), kdA1, kdB1, sB01, sB23);
        } else {
          const uint8_t* kr0 = sm.k[warp][s] + t0 * (kHeadDim * 2);
          const uint8_t* kr1 = sm.k[warp][s] + t1 * (kHeadDim * 2);
          const uint4 ka0 = *reinterpret_cast<const uint4*>(kr0 + 16 * c);
          const uint4 kb0 = *reinterpret_cast<const uint4*>(kr0 + 128 + 16 * c);
          const uint4 ka1 = *reinterpret_cast<const uint4*>(kr1 + 16 * c);
          const uint4 kb1 = *reinterpret_cast<const uint4*>(kr1 + 128 + 16 * c);
          qk16(qp, ka0, kb0, sA01, sA23);
          qk16(qp, ka1, kb1, sB01, sB23);
        }
        // transposed reduction: 8 values per lane -> 1 complete (token, head)
        float sc;
        {
          const bool b2 = (c >> 2) & 1, b1 = (c >> 1) & 1, b0 = c & 1;
          float2 kA = b2 ? sA23 : sA01, kB = b2 ? sB23 : sB01;
          const float2 oA = shfl_xor2(b2 ? sA01 : sA23, 4), oB = shfl_xor2(b2 ? sB01 : sB23, 4);
          kA = __fadd2_rn(kA, oA);
          kB = __fadd2_rn(kB, oB);
          float2 kk = b1 ? make_float2(kA.y, kB.y) : make_float2(kA.x, kB.x);
          const float2 send = b1 ? make_float2(kA.x, kB.x) : make_float2(kA.y, kB.y);
          kk = __fadd2_rn(kk, shfl_xor2(send, 2));
          sc = (b0 ? kk.y : kk.x) + __shfl_xor_sync(0xffffffffu, b0 ? kk.x : kk.y, 1);
        }
        const bool my_valid = (c & 1) ? valid1 : valid0;
        const float sv = my_valid ? sc : -INFINITY;
        const float mx = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, 1));  // both tokens of head hd
        const bool grow = mx > m_own + kRescaleSlack;
        if (__any_sync(0xffffffffu, grow)) {  // running max grew a lot: rescale (rare)
          const float corr = grow ? fast_exp2(m_own - mx) : 1.f;  // m_own = -inf -> 0
          if (grow) m_own = mx;
          l_own *= corr;
#pragma unroll
          for (int g = 0; g < kGroup; ++g) {
            const float cg = __shfl_sync(0xffffffffu, corr, slot_base + (g >> 1) * 4 + (g & 1) * 2);
            const float2 c2 = make_float2(cg, cg);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) acc[g][jj] = __fmul2_rn(acc[g][jj], c2);
          }
        }
        const float pown = my_valid ? fast_exp2(sv - m_own) : 0.f;
        l_own += pown;
        float pA[kGroup], pB[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
          const int src = slot_base + (g >> 1) * 4 + (g & 1) * 2;
          pA[g] = __shfl_sync(0xffffffffu, pown, src);
          pB[g] = __shfl_sync(0xffffffffu, pown, src + 1);
        }
        if constexpr (kQ8) {
          if (valid0) {
            const uint8_t* vr = sm.v[warp][s] + t0 * kHeadDim;
            pv16_q8(acc, pA, *reinterpret_cast<const uint2*>(vr + 8 * c),
                    *reinterpret_cast<const uint2*>(vr + 64 + 8 * c), vdA0, vdB0);
          }
          if (valid1) {
            const uint8_t* vr = sm.v[warp][s] + t1 * kHeadDim;
            pv16_q8(acc, pB, *reinterpret_cast<const uint2*>(vr + 8 * c),
                    *reinterpret_cast<const uint2*>(vr + 64 + 8 * c), vdA1, vdB1);
          }
        } else {
          if (valid0) {
            const uint8_t* vr = sm.v[warp][s] + t0 * (kHeadDim * 2);
            pv16(acc, pA, *reinterpret_cast<const uint4*>(vr + 16 * c),
                 *reinterpret_cast<const uint4*>(vr + 128 + 16 * c));
          }
          if (valid1) {
            const uint8_t* vr = sm.v[warp][s] + t1 * (kHeadDim * 2);
            pv16(acc, pB, *reinterpret_cast<const uint4*>(vr + 16 * c),
                 *reinterpret_cast<const uint4*>(vr + 128 + 16 * c));
          }
        }
      }
      // the warp is done with page q: refill its stage with page q + kWgStages
      __syncwarp();
      if (lane == 0 && q + kWgStages < e) {
        fence_proxy_async_smem();
        issue(q + kWgStages);
      }
      if (((q - i0) & 15) == 15 && *reinterpret_cast<volatile int*>(&sm.abort_flag)) {
        aborted = true;
        break;
      }
    }
    if (aborted) break;

    // ---- item end: merge the warp's 4 token slots (shuffles only); lane
    // (ts, c) ends with head g = ts, dims of chunk c
    const int g = ts;
    float o[16];
    float lse2;
    {
      const float l_pair = l_own + __shfl_xor_sync(0xffffffffu, l_own, 1);
      float Mw[kGroup], Lw[kGroup];
#pragma unroll
      for (int gg = 0; gg < kGroup; ++gg) {
        const int src = slot_base + (gg >> 1) * 4 + (gg & 1) * 2;
        const float mh = __shfl_sync(0xffffffffu, m_own, src);
        const float lh = __shfl_sync(0xffffffffu, l_pair, src);
        float Mg = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 8));
        Mg = fmaxf(Mg, __shfl_xor_sync(0xffffffffu, Mg, 16));
        Mw[gg] = Mg;
        const float f = (mh == -INFINITY) ? 0.f : fast_exp2(mh - Mg);
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[gg][jj] = __fmul2_rn(acc[gg][jj], f2);
        float lsum = lh * f;
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
        Lw[gg] = lsum;
      }
      // sum over the 4 token slots, transposed: slot (s1, s0) ends with head 2 s1 + s0
      const bool s1 = (lane >> 4) & 1, s0 = (lane >> 3) & 1;
      float2 h0[8], h1[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {  // xor 16: keep heads {2 s1, 2 s1 + 1}
        const float2 keep0 = s1 ? acc[2][jj] : acc[0][jj], send0 = s1 ? acc[0][jj] : acc[2][jj];
        const float2 keep1 = s1 ? acc[3][jj] : acc[1][jj], send1 = s1 ? acc[1][jj] : acc[3][jj];
        h0[jj] = __fadd2_rn(keep0, shfl_xor2(send0, 16));
        h1[jj] = __fadd2_rn(keep1, shfl_xor2(send1, 16));
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {  // xor 8: keep head 2 s1 + s0
        const float2 keep = s0 ? h1[jj] : h0[jj], send = s0 ? h0[jj] : h1[jj];
        h0[jj] = __fadd2_rn(keep, shfl_xor2(send, 8));
      }
      const float M = g == 0 ? Mw[0] : g == 1 ? Mw[1] : g == 2 ? Mw[2] : Mw[3];
      const float Ls = g == 0 ? Lw[0] : g == 1 ? Lw[1] : g == 2 ? Lw[2] : Lw[3];
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        o[2 * jj] = h0[jj].x * inv;
        o[2 * jj + 1] = h0[jj].y * inv;
      }
      lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
    }
    const int head = kvh * kGroup + g;
    const size_t orow = (size_t)tok * p.num_q_heads + head;
    if (p0w == 0 && i1 - i0 == pages_r) {  // the whole row in this warp
      int rd = 0;
      if (p.prefix_o) {
        const int* f = prefix_flag(p, tok, kvh);
        const int peek = (f && lane == 0) ? ld_relaxed_gpu(f) : 0;
        if (prefix_ready(p, tok, kvh, lane, peek, &rd)) {
          LseAcc acc;
          lse_acc_init(acc, o, lse2);
          lse_acc_prefix(acc, p, orow, c);
          lse2 = lse_acc_done(acc, o);
        }
      }
      store_row16(p.out + orow * kHeadDim, o, c);
      if (p.lse && c == 0) p.lse[orow] = lse2 * kLn2;
      if (p.prefix_o) prefix_read_done(p, tok, kvh, lane, rd);
      continue;
    }
    // the item is cut by warp-segment boundaries: publish this warp's partial
    const int A = it.A;  // stream position of the row's start; its pages start at A + kAlpha
    const int b0 = (A + kAlpha) / sw, b1 = (A + kAlpha + pages_r - 1) / sw;  // warp segments holding them
    const int jslot = (k == k_first) ? 0 : 1;
    {
      const size_t slot = ((size_t)(gw * Hkv + kvh) * 2 + jslot) * kGroup + g;
      if ((int64_t)slot < p.piece_slots) {
        float* dst = p.piece_o + slot * kHeadDim;
        *reinterpret_cast<float4*>(dst + 8 * c) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(dst + 8 * c + 4) = make_float4(o[4], o[5], o[6], o[7]);
        *reinterpret_cast<float4*>(dst + 64 + 8 * c) = make_float4(o[8], o[9], o[10], o[11]);
        *reinterpret_cast<float4*>(dst + 64 + 8 * c + 4) = make_float4(o[12], o[13], o[14], o[15]);
        if (c == 0) p.piece_lse[slot] = lse2;
      } else if (c == 0) {
        record_error(p.err, PA_ERR_DEVICE_INDEX);  // the host sized the workspace for fewer pieces
      }
    }
    __syncwarp();  // every lane's piece write precedes lane 0's release below
    int last = 0;
    if (lane == 0) {
      int* cnt = p.counters + (size_t)it.r * Hkv + kvh;
      const int done = atom_add_acq_rel_gpu(cnt, 1);
      last = done == b1 - b0;
      if (last) *cnt = 0;  // every piece has arrived: ready for the next call
    }
    __syncwarp();  // lane 0's acquire orders the piece reads below
    if (!__shfl_sync(0xffffffffu, last, 0)) continue;
    // the last piece to finish: merge every piece of the row (and the
    // prefix partials)
    {
      LseAcc acc;
      const int peek =
          wg_merge_pieces(p.piece_o, p.piece_lse, p.piece_slots, b0, b1, A, sw, Hkv, kvh, g, c, lane,
                          prefix_flag(p, tok, kvh), acc);
      int rd = 0;
      if (p.prefix_o && prefix_ready(p, tok, kvh, lane, peek, &rd)) lse_acc_prefix(acc, p, orow, c);
      float a4[16];
      const float l2 = lse_acc_done(acc, a4);
      store_row16(p.out + orow * kHeadDim, a4, c);
      if (p.lse && c == 0) p.lse[orow] = l2 * kLn2;
      if (p.prefix_o) prefix_read_done(p, tok, kvh, lane, rd);
    }
  }

  if (aborted && lane == 0) {
    // A wait gave up: let the last copy issued into each of this warp's
    // stages land (bounded), then leave.  A stage whose copies never land is
    // passed over after the bound; the others are still waited for, so no
    // copy that can land is in flight when the warp leaves.
    for (int s = 0; s < kWgStages; ++s) {
      const int j = sm.stage_page[warp][s];
      if (j >= 0) mbar_wait_bounded(&sm.full[warp][s], (uint32_t)(j / kWgStages) & 1u, kLimit);
    }
    if (sm.q_issued[warp] > 0) mbar_wait_bounded(&sm.q_full[warp], (uint32_t)(sm.q_issued[warp] - 1) & 1u, kLimit);
  }
  // beside a tile kernel: this launch completes after it (a warp that ends
  // here waits for it; it never waits on this launch, so this ends)
  if (p.beside) pdl_wait();
}

std::atomic<bool> g_decode_attr_set[4][kMaxDevices];

std::atomic<bool> g_decode_cta_attr_set[3][kMaxDevices];

template <bool kQ8, bool kStep, bool kDiag = false>
cudaError_t launch_decode_as(const DecodeParams& p, const typename PlanOf<kStep>::type& plan, int grid,
                             bool overlap, cudaStream_t stream) {
  constexpr size_t kSmem = sizeof(DecodeSmem<kQ8 ? kQ8SlabBytes : kSlabBytes>);
  constexpr int kVariant = kStep ? 2 : (kQ8 ? 1 : 0);
  const cudaError_t e = set_smem_limit_once((const void*)decode_kernel<kQ8, kStep, kDiag>, (int)kSmem,
                                            g_decode_cta_attr_set[kVariant]);
  if (e != cudaSuccess) return e;
  return launch_maybe_pdl(overlap, decode_kernel<kQ8, kStep, kDiag>, dim3(grid), dim3(kThreads), kSmem, stream, p,
                          plan);
}

template <bool kQ8, bool kDiag, bool kStep = false>
cudaError_t launch_decode_wg(const DecodeParams& p, const typename PlanOf<kStep>::type& plan, int grid, bool overlap,
                             cudaStream_t stream) {
  constexpr size_t kSmem = sizeof(WgSmem<kQ8 ? kQ8SlabBytes : kSlabBytes>);
  constexpr int kVariant = kStep ? 2 : kDiag ? 3 : (kQ8 ? 1 : 0);
  const cudaError_t e = set_smem_limit_once((const void*)decode_wg_kernel<kQ8, kDiag, kStep>, (int)kSmem,
                                            g_decode_attr_set[kVariant]);
  if (e != cudaSuccess) return e;
  return launch_maybe_pdl(overlap, decode_wg_kernel<kQ8, kDiag, kStep>, dim3(grid), dim3(kWgThreads), kSmem, stream,
                          p, plan);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, const DecodePlan& plan, int grid, bool q8, bool overlap,
                          bool diag, bool cta_granular, cudaStream_t stream) {
  if (cta_granular)  // short segments: the CTA-granular kernel (bf16 or q8_0 pages)
    return q8 ? launch_decode_as<true, false>(p, plan, grid, overlap, stream)
              : launch_decode_as<false, false>(p, plan, grid, overlap, stream);
  if (q8) return launch_decode_wg<true, false>(p, plan, grid, overlap, stream);
  return diag ? launch_decode_wg<false, true>(p, plan, grid, overlap, stream)
              : launch_decode_wg<false, false>(p, plan, grid, overlap, stream);
}

cudaError_t launch_decode_step(const DecodeParams& p, const StepPlan& plan, int grid, bool warp_granular,
                               cudaStream_t stream) {
  return warp_granular ? launch_decode_wg<false, false, true>(p, plan, grid, true, stream)
                       : launch_decode_as<false, true>(p, plan, grid, true, stream);
}

}  // namespace pa
