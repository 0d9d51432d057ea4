// Tensor-core tiles of paged attention: chunked-prefill rows (qo_len > 1)
// and the shared-prefix pass of a batch whose requests share leading pages.
//
// What is computed: a chunk of c new tokens after h cached ones; new token j
// sits at position h + j and attends to keys 0 .. h + j ("Inference
// optimisation", AI-infra book ch. 8, §8.2.3, the N_pair equation and Fig.
// 8-8/8-9: a rectangle of c x h pairs plus a causal triangle).  Keys are read
// through the block table (§8.3.1).  Here h = seq_len - qo_len.  Pages shared
// by several requests are stored once (§8.3.2, Fig. 8-13); when every query
// of the batch comes after such a shared prefix, the prefix is attended once
// for all queries together (no mask: every prefix key is visible to every
// query) and merged with each request's own part by log-sum-exp.
//
// Design: both products are dense contractions (QK^T and PV), so they run on
// the tensor cores (mma.sync m16n8k16, bf16 inputs, fp32 accumulators).
//   * One CTA per (16-query tile, kv head [, key chunk]).  The 4 q heads of
//     the GQA group are packed into the M dimension: 16 tokens x 4 heads = 64
//     rows, so every K/V tile staged in shared memory serves all four heads.
//   * 4 warps x 16 rows; each warp keeps its Q fragments in registers for
//     the whole key loop.
//   * K/V tiles of 64 keys (4 pages) are staged with cp.async (16 B per
//     request) into XOR-swizzled rows (16-byte chunk c of row r lands at
//     chunk c ^ (r & 7)), double buffered, so ldmatrix reads are
//     conflict-free.
//   * Online softmax in the log2 domain on the fp32 S fragments; P is
//     rounded to bf16 for the PV product.  Only tiles that cross the causal
//     diagonal or the end of the key range evaluate a mask.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kQT = kPrefillQTile;     // query tokens per CTA
constexpr int kRows = kQT * kGroup;    // 64 MMA rows
constexpr int kKT = 64;                // keys per tile
constexpr int kThreads = 128;
constexpr int kChunksPerRow = kHeadDim * 2 / 16;  // 16 chunks of 16 B

struct __align__(128) PrefillSmem {
  uint16_t q[kRows * kHeadDim];
  uint16_t k[2][kKT * kHeadDim];
  uint16_t v[2][kKT * kHeadDim];
};

// element offset of 16-byte chunk `ch` of row `row` in a swizzled tile
__device__ __forceinline__ int swz(int row, int ch) { return (row * kChunksPerRow + (ch ^ (row & 7))) * 8; }

__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The 64 rows of one CTA (tokens tok0 .. tok0 + nq - 1 of q, 4 heads of kv
// head kvh) against keys [k_lo, k_hi) of one block table; k_lo is a multiple
// of 16.  Causal: the row of token l (position pos0 + l) sees keys <= that
// position.  Leaves per thread the O fragments of its two rows (gq, gq + 8 of
// the warp's 16) and their running max (log2 domain) and partial sum.
template <bool kCausal>
__device__ __forceinline__ void attend_rows(PrefillSmem& sm, const uint16_t* q, int64_t tok0, int nq, int num_q_heads,
                                            int kvh, const uint16_t* k_cache, const uint16_t* v_cache,
                                            int num_kv_heads, int64_t num_blocks, const int32_t* table, int k_lo,
                                            int k_hi, int pos0, float scale_log2, int* err, float (&o)[16][4],
                                            float (&m_run)[2], float (&l_run)[2]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (k_hi - k_lo + kKT - 1) / kKT;
  const int last_page = (k_hi - 1) / kPage;

  // Q: row m = 4 * token + head-in-group; invalid tokens are zero rows.
#pragma unroll
  for (int it = 0; it < kRows * kChunksPerRow / kThreads; ++it) {
    const int ci = tid + it * kThreads;
    const int row = ci / kChunksPerRow, ch = ci % kChunksPerRow;
    const int tokl = row >> 2, g = row & 3;
    uint16_t* dst = sm.q + swz(row, ch);
    if (tokl < nq) {
      cp_async16(dst, q + ((size_t)(tok0 + tokl) * num_q_heads + kvh * kGroup + g) * kHeadDim + ch * 8);
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  }

  auto load_kv = [&](int kt, int buf) {
#pragma unroll
    for (int it = 0; it < kKT * kChunksPerRow / kThreads; ++it) {
      const int ci = tid + it * kThreads;
      const int row = ci / kChunksPerRow, ch = ci % kChunksPerRow;
      // keys past the range read the last page again (finite data, masked)
      const int page = min((k_lo + kt * kKT) / kPage + row / kPage, last_page);
      int32_t b = table[page];
      if (b < 0 || b >= num_blocks) {
        record_error(err, PA_ERR_DEVICE_INDEX);
        b = 0;
      }
      const size_t src = (((size_t)b * num_kv_heads + kvh) * kPage + (row % kPage)) * kHeadDim + ch * 8;
      cp_async16(sm.k[buf] + swz(row, ch), k_cache + src);
      cp_async16(sm.v[buf] + swz(row, ch), v_cache + src);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  uint32_t qa[kHeadDim / 16][4];
#pragma unroll
  for (int i = 0; i < kHeadDim / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  m_run[0] = m_run[1] = -INFINITY;
  l_run[0] = l_run[1] = 0.f;
  const int gq = lane >> 2, tq = lane & 3;
  // positions of this thread's two rows (gq and gq + 8 of the warp's 16)
  const int row_pos[2] = {pos0 + ((warp * 16 + gq) >> 2), pos0 + ((warp * 16 + gq + 8) >> 2)};

  for (int kt = 0; kt < n_tiles; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < n_tiles) load_kv(kt + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kt == 0) {
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        ldsm_x4(qa[kk], sm.q + swz(warp * 16 + (mi & 1) * 8 + ri, 2 * kk + (mi >> 1)));
    }

    // S = Q K^T for 16 rows x 64 keys
    float s[kKT / 8][4];
#pragma unroll
    for (int i = 0; i < kKT / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    {
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < kKT / 16; ++np) {
          uint32_t b[4];
          ldsm_x4(b, sm.k[buf] + swz(16 * np + (mi >> 1) * 8 + ri, 2 * kk + (mi & 1)));
          mma16816(s[2 * np], qa[kk], b[0], b[1]);
          mma16816(s[2 * np + 1], qa[kk], b[2], b[3]);
        }
      }
    }

    // scale, mask (only where the tile crosses the diagonal or the range end)
    const int kbase = k_lo + kt * kKT;
    const bool need_mask = (kCausal && kbase + kKT - 1 > pos0) || (kbase + kKT > k_hi);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < kKT / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e] * scale_log2;
        if (need_mask) {
          const int key = kbase + nt * 8 + 2 * tq + (e & 1);
          if (key >= k_hi || (kCausal && key > row_pos[e >> 1])) x = -INFINITY;
        }
        s[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
    float corr[2], mref[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float m_new = fmaxf(m_run[h], mx[h]);
      mref[h] = (m_new == -INFINITY) ? 0.f : m_new;
      corr[h] = exp2f(m_run[h] - mref[h]);
      m_run[h] = m_new;
      l_run[h] *= corr[h];
    }
#pragma unroll
    for (int i = 0; i < kHeadDim / 8; ++i) {
      o[i][0] *= corr[0];
      o[i][1] *= corr[0];
      o[i][2] *= corr[1];
      o[i][3] *= corr[1];
    }
    uint32_t pa[kKT / 16][4];
#pragma unroll
    for (int nt = 0; nt < kKT / 8; ++nt) {
      const float p0 = exp2f(s[nt][0] - mref[0]);
      const float p1 = exp2f(s[nt][1] - mref[0]);
      const float p2 = exp2f(s[nt][2] - mref[1]);
      const float p3 = exp2f(s[nt][3] - mref[1]);
      l_run[0] += p0 + p1;
      l_run[1] += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }

    // O += P V
    {
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int kk = 0; kk < kKT / 16; ++kk) {
#pragma unroll
        for (int dp = 0; dp < kHeadDim / 16; ++dp) {
          uint32_t b[4];
          ldsm_x4_t(b, sm.v[buf] + swz(16 * kk + (mi & 1) * 8 + ri, 2 * dp + (mi >> 1)));
          mma16816(o[2 * dp], pa[kk], b[0], b[1]);
          mma16816(o[2 * dp + 1], pa[kk], b[2], b[3]);
        }
      }
    }
    __syncthreads();  // buffer `buf` is refilled by the next iteration
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const PrefillParams p, const __grid_constant__ PrefillItems items) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw);
  const int r = items.req[blockIdx.x];
  const int j0 = items.q_start[blockIdx.x];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int qo0 = p.qo_indptr[r];
  const int c = p.qo_indptr[r + 1] - qo0;
  const int L = p.seq_lens[r];
  const int nq = min(kQT, c - j0);  // valid query tokens in this tile
  const int pos0 = L - c + j0;      // position of the tile's first query
  const int kv_end = pos0 + nq;     // keys [0, kv_end) are visible to some row
  const int32_t* table = p.block_tables + (size_t)r * p.max_blocks_per_req;

  float o[kHeadDim / 8][4], m_run[2], l_run[2];
  attend_rows<true>(sm, p.q, (int64_t)qo0 + j0, nq, p.num_q_heads, kvh, p.k_cache, p.v_cache, p.num_kv_heads,
                    p.num_blocks, table, p.kv_key_offset, kv_end, pos0, p.scale_log2, p.err, o, m_run, l_run);

  // normalise, fold in the shared prefix (if any) and write the valid rows
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = warp * 16 + gq + 8 * h;
    const int tokl = row >> 2;
    if (tokl >= nq) continue;
    const int head = kvh * kGroup + (row & 3);
    const size_t orow = (size_t)(qo0 + j0 + tokl) * p.num_q_heads + head;
    float lse2 = l_run[h] > 0.f ? m_run[h] + log2f(l_run[h]) : -INFINITY;
    float ws = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f, wp = 0.f;
    const float* po = nullptr;
    if (p.prefix_o) {
      float wo;
      lse2 = merge2_weights(lse2, p.prefix_lse[orow], wo, wp);
      ws *= wo;
      po = p.prefix_o + orow * kHeadDim + 2 * tq;
    }
#pragma unroll
    for (int nt = 0; nt < kHeadDim / 8; ++nt) {
      float x0 = o[nt][2 * h] * ws, x1 = o[nt][2 * h + 1] * ws;
      if (po) {
        const float2 y = *reinterpret_cast<const float2*>(po + nt * 8);
        x0 = fmaf(wp, y.x, x0);
        x1 = fmaf(wp, y.y, x1);
      }
      *reinterpret_cast<uint32_t*>(p.out + orow * kHeadDim + nt * 8 + 2 * tq) = pack_bf16x2(x0, x1);
    }
    if (p.lse && tq == 0) p.lse[orow] = lse2 * kLn2;
  }
}

// Shared-prefix pass: grid (key chunk, kv head, 16-token tile of all the
// batch's queries).  Each CTA leaves a chunk partial (prefix_merge_kernel
// merges them); with a single chunk it writes the prefix partial itself.
__global__ void __launch_bounds__(kThreads, 2) prefix_kernel(const PrefixParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw);
  const int chunk = blockIdx.x, kvh = blockIdx.y, qt = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tok0 = qt * kQT;
  const int nq = min(kQT, p.total_q - tok0);
  const int k_lo = chunk * p.chunk_keys;
  const int k_hi = min(p.prefix_keys, k_lo + p.chunk_keys);
  const int32_t* table = p.block_tables + (size_t)p.table_row * p.max_blocks_per_req;

  float o[kHeadDim / 8][4], m_run[2], l_run[2];
  attend_rows<false>(sm, p.q, tok0, nq, p.num_q_heads, kvh, p.k_cache, p.v_cache, p.num_kv_heads, p.num_blocks,
                     table, k_lo, k_hi, 0, p.scale_log2, p.err, o, m_run, l_run);

  // chunk partial (normalised o, log2 lse per row); a single chunk is the
  // prefix partial itself
  const bool direct = gridDim.x == 1;
  float* dst_o = direct ? p.prefix_o : p.chunk_o;
  float* dst_lse = direct ? p.prefix_lse : p.chunk_lse;
  const int gq = lane >> 2, tq = lane & 3;
  const size_t chunk_stride = (size_t)p.total_q * p.num_q_heads;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = warp * 16 + gq + 8 * h;
    const int tokl = row >> 2;
    if (tokl >= nq) continue;
    const size_t orow = (size_t)(tok0 + tokl) * p.num_q_heads + kvh * kGroup + (row & 3);
    const size_t prow = (size_t)chunk * chunk_stride + orow;
    const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
#pragma unroll
    for (int nt = 0; nt < kHeadDim / 8; ++nt)
      *reinterpret_cast<float2*>(dst_o + prow * kHeadDim + nt * 8 + 2 * tq) =
          make_float2(o[nt][2 * h] * inv, o[nt][2 * h + 1] * inv);
    if (tq == 0) dst_lse[prow] = l_run[h] > 0.f ? m_run[h] + log2f(l_run[h]) : -INFINITY;
  }
}

// Merge of the prefix pass's key-chunk partials: one warp per (query token,
// q head) row, two rows per CTA so the merge spreads over the SMs.  Lanes
// read the chunks' lse in parallel; then each lane issues the loads of its 4
// dims of up to 32 chunks at once and sums them with the broadcast weights.
constexpr int kMergeWarps = 2;
__global__ void __launch_bounds__(kMergeWarps * 32) prefix_merge_kernel(const PrefixParams p, int n_chunks) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int64_t rows = (int64_t)p.total_q * p.num_q_heads;
  if (row >= rows) return;
  float M = -INFINITY;
  for (int c0 = 0; c0 < n_chunks; c0 += 32)
    if (c0 + lane < n_chunks) M = fmaxf(M, p.chunk_lse[(c0 + lane) * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float wsum = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int c0 = 0; c0 < n_chunks; c0 += 32) {
      const int nc = min(32, n_chunks - c0);
      const float* src = p.chunk_o + ((int64_t)c0 * rows + row) * kHeadDim + 4 * lane;
      float4 x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nc) x[j] = *reinterpret_cast<const float4*>(src + (int64_t)j * rows * kHeadDim);
      const float w = lane < nc ? exp2f(p.chunk_lse[(c0 + lane) * rows + row] - M) : 0.f;
      float ws = w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
      wsum += ws;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, j);
        if (j < nc) {
          a.x = fmaf(wj, x[j].x, a.x);
          a.y = fmaf(wj, x[j].y, a.y);
          a.z = fmaf(wj, x[j].z, a.z);
          a.w = fmaf(wj, x[j].w, a.w);
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  *reinterpret_cast<float4*>(p.prefix_o + row * kHeadDim + 4 * lane) =
      make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  if (lane == 0) p.prefix_lse[row] = wsum > 0.f ? M + log2f(wsum) : -INFINITY;
}

bool g_prefill_attr_set[64] = {};
bool g_prefix_attr_set[64] = {};

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const PrefillItems& items, cudaStream_t stream) {
  if (items.count <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !g_prefill_attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(PrefillSmem));
    if (e != cudaSuccess) return e;
    g_prefill_attr_set[dev] = true;
  }
  dim3 grid(items.count, p.num_kv_heads);
  prefill_kernel<<<grid, kThreads, sizeof(PrefillSmem), stream>>>(p, items);
  return cudaGetLastError();
}

cudaError_t launch_prefix(const PrefixParams& p, int n_chunks, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !g_prefix_attr_set[dev]) {
    e = cudaFuncSetAttribute(prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(PrefillSmem));
    if (e != cudaSuccess) return e;
    g_prefix_attr_set[dev] = true;
  }
  dim3 grid(n_chunks, p.num_kv_heads, (p.total_q + kQT - 1) / kQT);
  prefix_kernel<<<grid, kThreads, sizeof(PrefillSmem), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefix_merge(const PrefixParams& p, int n_chunks, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.total_q * p.num_q_heads;
  prefix_merge_kernel<<<(unsigned)((rows + kMergeWarps - 1) / kMergeWarps), kMergeWarps * 32, 0, stream>>>(p, n_chunks);
  return cudaGetLastError();
}

}  // namespace pa
