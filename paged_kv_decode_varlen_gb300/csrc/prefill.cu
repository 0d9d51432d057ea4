// Chunked-prefill rows (qo_len > 1): causal GQA attention over the paged KV
// cache on tensor cores.
//
// What is computed: a chunk of c new tokens after h cached ones; new token j
// sits at position h + j and attends to keys 0 .. h + j ("Inference
// optimisation", AI-infra book ch. 8, §8.2.3, the N_pair equation and Fig.
// 8-8/8-9: a rectangle of c x h pairs plus a causal triangle).  Keys are read
// through the block table (§8.3.1).  Here h = seq_len - qo_len.
//
// Design: both products are dense contractions (QK^T and PV), so they run on
// the tensor cores (mma.sync m16n8k16, bf16 inputs, fp32 accumulators).
//   * One CTA per (16-query tile, kv head).  The 4 q heads of the GQA group
//     are packed into the M dimension: 16 tokens x 4 heads = 64 rows, so
//     every K/V tile staged in shared memory serves all four heads.
//   * 4 warps x 16 rows; each warp keeps its Q fragments in registers for
//     the whole key loop.
//   * K/V tiles of 64 keys (4 pages) are staged with cp.async (16 B per
//     request) into XOR-swizzled rows (16-byte chunk c of row r lands at
//     chunk c ^ (r & 7)), double buffered, so ldmatrix reads are
//     conflict-free.
//   * Online softmax in the log2 domain on the fp32 S fragments; P is
//     rounded to bf16 for the PV product.  Only tiles that cross the
//     diagonal evaluate the causal mask.
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

__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const PrefillParams p, const __grid_constant__ PrefillItems items) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw);
  const int r = items.req[blockIdx.x];
  const int j0 = items.q_start[blockIdx.x];
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int qo0 = p.qo_indptr[r];
  const int c = p.qo_indptr[r + 1] - qo0;
  const int L = p.seq_lens[r];
  const int nq = min(kQT, c - j0);       // valid query tokens in this tile
  const int pos0 = L - c + j0;           // position of the tile's first query
  const int kv_end = pos0 + nq;          // keys [0, kv_end) are visible to some row
  const int n_tiles = (kv_end + kKT - 1) / kKT;
  const int last_page = (kv_end - 1) / kPage;
  const int32_t* table = p.block_tables + (size_t)r * p.max_blocks_per_req;

  // Q: row m = 4 * token + head-in-group; invalid tokens are zero rows.
#pragma unroll
  for (int it = 0; it < kRows * kChunksPerRow / kThreads; ++it) {
    const int ci = tid + it * kThreads;
    const int row = ci / kChunksPerRow, ch = ci % kChunksPerRow;
    const int tokl = row >> 2, g = row & 3;
    uint16_t* dst = sm.q + swz(row, ch);
    if (tokl < nq) {
      cp_async16(dst, p.q + ((size_t)(qo0 + j0 + tokl) * p.num_q_heads + kvh * kGroup + g) * kHeadDim + ch * 8);
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  }

  auto load_kv = [&](int kt, int buf) {
#pragma unroll
    for (int it = 0; it < kKT * kChunksPerRow / kThreads; ++it) {
      const int ci = tid + it * kThreads;
      const int row = ci / kChunksPerRow, ch = ci % kChunksPerRow;
      const int page = min(kt * (kKT / kPage) + row / kPage, last_page);
      int32_t b = table[page];
      if (b < 0 || b >= p.num_blocks) {
        record_error(p.err, PA_ERR_DEVICE_INDEX);
        b = 0;
      }
      const size_t src = (((size_t)b * p.num_kv_heads + kvh) * kPage + (row % kPage)) * kHeadDim + ch * 8;
      cp_async16(sm.k[buf] + swz(row, ch), p.k_cache + src);
      cp_async16(sm.v[buf] + swz(row, ch), p.v_cache + src);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  uint32_t qa[kHeadDim / 16][4];
  float o[kHeadDim / 8][4];
#pragma unroll
  for (int i = 0; i < kHeadDim / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
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

    // scale, causal mask (only where the tile crosses the diagonal), row max
    const int kbase = kt * kKT;
    const bool need_mask = kbase + kKT - 1 > pos0;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < kKT / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e] * p.scale_log2;
        if (need_mask) {
          const int key = kbase + nt * 8 + 2 * tq + (e & 1);
          if (key > row_pos[e >> 1]) x = -INFINITY;
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

  // normalise and write the valid rows
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = warp * 16 + gq + 8 * h;
    const int tokl = row >> 2;
    if (tokl >= nq) continue;
    const int head = kvh * kGroup + (row & 3);
    const size_t orow = (size_t)(qo0 + j0 + tokl) * p.num_q_heads + head;
    const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
#pragma unroll
    for (int nt = 0; nt < kHeadDim / 8; ++nt) {
      const uint32_t v = pack_bf16x2(o[nt][2 * h] * inv, o[nt][2 * h + 1] * inv);
      *reinterpret_cast<uint32_t*>(p.out + orow * kHeadDim + nt * 8 + 2 * tq) = v;
    }
    if (p.lse && tq == 0) p.lse[orow] = l_run[h] > 0.f ? (m_run[h] + log2f(l_run[h])) * kLn2 : -INFINITY;
  }
}

bool g_prefill_attr_set[64] = {};

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

}  // namespace pa
