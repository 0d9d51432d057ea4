// Tensor-core tiles of paged attention on the 5th-generation tensor cores:
// chunked-prefill rows (qo_len > 1) and the shared-prefix pass of a batch
// whose requests share leading pages.
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
// Design (QK^T and PV are dense contractions):
//   * One CTA per (32-query tile, kv head [, key chunk]), or, for the
//     chunked-prefill jobs of a batch that also has decode rows, a few
//     persistent CTAs that run the jobs one after another beside the decode
//     launch on the other SMs (a chunked-prefill step mixes compute-bound
//     and memory-bound work: the serving page "vLLM, SGLang и непрерывный
//     батчинг", section "Непрерывный батчинг").  The 4 q heads of the GQA
//     group are packed into the M dimension: 32 tokens x 4 heads = 128 rows
//     = the M of one tcgen05.mma, so every K/V tile serves all four heads.
//     Keys go in tiles of 128 (8 pages).
//   * Warp roles: warps 4 and 6 issue tiled TMA copies (Q once; per key tile
//     the two 64-dim halves of each page's K slab, resp. V slab, 128-byte
//     swizzled, into a 4-stage K ring and a 2-stage V ring: a K stage is
//     refilled as soon as its S product is done); warp 5 owns the tensor memory and one of its
//     threads issues the MMAs; warps 0-3 run the softmax, one thread per row
//     (tensor-memory lane = row).
//   * Tensor memory: two S buffers of 128 fp32 columns, the O accumulator
//     (128 columns) and two P buffers of 64 columns (bf16 key pairs: P is the
//     A operand of the PV product, read from tensor memory, which leaves the
//     shared memory to the K ring).  S of tile j + 1 is queued before PV of
//     tile j, so it runs while the softmax of tile j does; PV of tile j
//     follows the softmax that wrote its P.  The softmax of tile j waits only for PV of
//     tile j - 2 (the last reader of its P buffer) unless it must rescale O,
//     so its exponentials overlap PV of tile j - 1.
//   * Online softmax in the log2 domain; the running max is re-based (and O
//     in tensor memory rescaled) only when it grows by more than 2^8, so P
//     stays below 256 and the rescale is rare.
//   * Every wait is bounded; on a timeout the CTA records the error, lets
//     its copies and MMAs finish (bounded), frees its tensor memory and
//     returns.
#include <math.h>
#include <stddef.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kTok = kPrefillQTile;              // 32 query tokens per CTA
constexpr int kRows = kTok * kGroup;             // 128 MMA rows
constexpr int kKeys = kTcKeyTile;                // 128 keys per tile
constexpr int kPagesPerTile = kKeys / kPage;     // 8
constexpr int kHalf = 128 * 128;                 // 128 rows x 64 bf16 (one 64-column half): 16 KiB
constexpr int kTileBytes = 2 * kHalf;            // 32 KiB
constexpr int kPageHalfBytes = kPage * 128;      // one page's rows of one half: 2 KiB
constexpr int kKStages = 4;  // K ring: S of a tile waits for its K, so it runs deep
constexpr int kVStages = 2;  // V ring: PV of a tile comes a softmax later
constexpr int kSoftmaxWarps = 4;
constexpr int kKWarp = 4, kMmaWarp = 5, kVWarp = 6;  // Q/K copies, MMA issue, V copies
constexpr int kThreads = 7 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 128
constexpr uint32_t kColO = 256;  // O accumulator
constexpr uint32_t kColP = 384;  // two P buffers of 64 columns (128 bf16 keys per lane, in pairs)
constexpr float kRescaleSlack = 8.f;
constexpr uint32_t kIdescS = idesc_bf16_f32(kRows, kKeys, false);     // Q (K-major) x K^T (K-major)
constexpr uint32_t kIdescO = idesc_bf16_f32(kRows, kHeadDim, true);   // P (K-major) x V (MN-major)
static_assert(kRows == 128 && kKeys == 128, "tile shape");

struct __align__(1024) TcSmem {
  uint8_t q[kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[kVStages][kTileBytes];
  uint64_t bar_q;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];  // S of the stage's tile done: the stage may be refilled
  uint64_t v_full[kVStages];
  uint64_t pv_done[2];  // PV of tile j done: phase j / 2 of pv_done[j % 2]
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t q_free;  // a job's last S product done: Q may be reloaded (jobs in turn without a CTA barrier)
  uint64_t o_free;  // the softmax warps have read a job's O: the next job's first PV may overwrite it
  uint32_t tmem;
  int abort;
};
constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;  // + slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kKStages >= 2, "staging area = the first two K stages (64 KiB)");

__device__ __forceinline__ TcSmem& tc_smem() {
  extern __shared__ uint8_t tc_smem_raw[];
  return *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
}

// Bounded wait that also gives up once another thread of the CTA has given
// up (the abort flag).
__device__ __forceinline__ bool tc_wait(TcSmem& sm, uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(&sm.abort)) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        record_error(err, PA_ERR_DEVICE_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sm.abort) = 1;
        return false;
      }
    }
  }
}

// One CTA's work: rows = tokens tok0 .. tok0 + nq - 1 of q (4 heads of kv
// head kvh each) against keys [k_lo, k_hi) of one block-table row; k_lo is a
// multiple of 16.  Causal: token l (position pos0 + l) sees keys <= pos0 + l.
struct TcJob {
  int32_t tok0;
  int32_t nq;
  int32_t kvh;
  int32_t k_lo;
  int32_t k_hi;
  int32_t pos0;
  const int32_t* table;
};

// A CTA's place in its pipelines, carried from one job to the next: the key
// tiles and jobs it has run.  Every ring stage, barrier phase and tensor-
// memory buffer is indexed by the CTA's running tile count J (tile j of a
// job is J = tiles + j) and bar_q by the job count, so a persistent CTA runs
// job after job without re-initialising anything.
struct TcPos {
  int tiles = 0;
  int jobs = 0;
};

// Runs one job.  Each softmax thread calls `stage(row, o, m, l, smem)` with
// its row's unnormalised O (4 x 32 fp32), running max (log2 domain) and
// sum, to leave its output row in the 64 KiB staging area `smem`; after a
// barrier of the softmax warps each of their threads calls `store(t, smem)`
// (t = 0 .. 127) to copy the staged rows out with contiguous stores.  The
// CTA's first job initialises the barriers and allocates the tensor memory
// (tc_finish frees it); every job ends with a CTA barrier, after which the
// staging area, Q and the tensor memory are free for the next.
//
// kOverlap (several jobs per CTA): no barrier between jobs, so the next
// job's block ids, Q, first K and V tiles and first S product overlap this
// job's last tile and epilogue.  Q is reloaded once the job's last S product
// has completed (q_free), the next job's first PV overwrites O once every
// softmax thread has read it (o_free), and the epilogue stores each row from
// registers (`stage(row, o, m, l, nullptr)`, no staging area: the K and V
// stages already hold the next job's tiles; `store` is not called).  The
// caller ends the last job with a CTA barrier before tc_finish.
template <bool kCausal, bool kOverlap, class Stage, class Store>
__device__ __forceinline__ void run_tile(const TcJob& job, const TcMaps& maps, int num_kv_heads, int64_t num_blocks,
                                         float scale_log2, int* err, TcPos& pos, Stage&& stage, Store&& store) {
  TcSmem& sm = tc_smem();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int J0 = pos.tiles;
  const bool first = pos.jobs == 0;
  const uint32_t q_par = (uint32_t)pos.jobs & 1u;
  const int n_tiles = (job.k_hi - job.k_lo + kKeys - 1) / kKeys;
  const int first_page = job.k_lo / kPage;
  const int last_page = (job.k_hi - 1) / kPage;
  const bool is_producer = warp == kKWarp || warp == kVWarp;
  const bool is_k = warp == kKWarp;

  // Block ids are read four tiles at a time, one group ahead: lane l of a
  // producer warp holds the pool row of page l % 8 of tile 4 g + l / 8.
  auto load_group = [&](int g) -> int {
    const int t = 4 * g + (lane >> 3);
    if (t >= n_tiles) return 0;
    // pages past the range repeat the last page (finite data; masked)
    const int page = min(first_page + t * kPagesPerTile + (lane & 7), last_page);
    int32_t b = job.table[page];
    if (b < 0 || b >= num_blocks) {
      if (is_k) record_error(err, PA_ERR_DEVICE_INDEX);
      b = 0;
    }
    return (b * num_kv_heads + job.kvh) * kPage;
  };
  int grp_cur = 0, grp_next = 0;
  bool q_pending = false;  // (K warp, lane 0) this job's Q copy was issued
  if (is_producer) {  // in flight during the set-up below
    grp_cur = load_group(0);
    grp_next = load_group(1);
  }

  if (is_k && lane == 0) {
    if (first) {
      mbar_init(&sm.bar_q, 1);
      for (int s = 0; s < kKStages; ++s) {
        mbar_init(&sm.k_full[s], 1);
        mbar_init(&sm.k_empty[s], 1);
      }
      for (int s = 0; s < kVStages; ++s) mbar_init(&sm.v_full[s], 1);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&sm.s_full[b], 1);
        mbar_init(&sm.p_full[b], kSoftmaxWarps * 32);
        mbar_init(&sm.pv_done[b], 1);
      }
      mbar_init(&sm.q_free, 1);
      mbar_init(&sm.o_free, kSoftmaxWarps * 32);
      sm.abort = 0;
      fence_mbar_init();
      prefetch_tensormap(&maps.q);
    }
    // Q first: its copy overlaps the rest of the set-up (the previous job's
    // closing barrier freed the buffer; with kOverlap its last S product)
    if (first || !kOverlap || tc_wait(sm, &sm.q_free, ((uint32_t)pos.jobs - 1u) & 1u, err)) {
      fence_after_sync();
      mbar_arrive_expect_tx(&sm.bar_q, kTileBytes);
      tma_load_3d(sm.q, &maps.q, 0, job.kvh * kGroup, job.tok0, &sm.bar_q);
      tma_load_3d(sm.q + kHalf, &maps.q, 64, job.kvh * kGroup, job.tok0, &sm.bar_q);
      q_pending = true;
    }
  }
  if (first) {
    if (warp == kMmaWarp) tmem_alloc(&sm.tmem, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
  }
  const uint32_t tmem = sm.tmem;

  if (is_producer) {
    // ----------------------------------------------------------- producers
    // warp kKWarp: Q (above), then the K ring; warp kVWarp: the V ring.  A K
    // stage is free once its S product is done (k_empty), a V stage once its
    // PV product is (pv_done); stage s serves tiles s, s + n, ... (n stages),
    // so tile j waits for phase j / n - 1 of the stage's barrier.
    const CUtensorMap* map = is_k ? &maps.k : &maps.v;
    uint64_t* full = is_k ? sm.k_full : sm.v_full;
    uint64_t* empty = is_k ? sm.k_empty : sm.pv_done;
    const int n_st = is_k ? kKStages : kVStages;
    int last_issued[kKStages];
#pragma unroll
    for (int s = 0; s < kKStages; ++s) last_issued[s] = -1;
    if (lane == 0) prefetch_tensormap(map);
    for (int j = 0; j < n_tiles; ++j) {
      const int J = J0 + j;
      const int s = J % n_st;
      if (J >= n_st && !__all_sync(0xffffffffu, tc_wait(sm, &empty[s], ((J / n_st) - 1) & 1, err))) break;
      if (j > 0 && (j & 3) == 0) {
        grp_cur = grp_next;
        grp_next = load_group((j >> 2) + 1);
      }
      const int row = __shfl_sync(0xffffffffu, grp_cur, ((j & 3) << 3) + (lane & 7));
      if (lane == 0) mbar_arrive_expect_tx(&full[s], kTileBytes);
      __syncwarp();
      uint8_t* dst = is_k ? sm.k[s] : sm.v[s];
      if (lane < kPagesPerTile) {
        const int off = lane * kPageHalfBytes;
        tma_load_2d(dst + off, map, 0, row, &full[s]);
        tma_load_2d(dst + kHalf + off, map, 64, row, &full[s]);
      }
      last_issued[s] = J;
    }
    if (*reinterpret_cast<volatile int*>(&sm.abort) && lane == 0) {
      // let the copies in flight land before the CTA leaves (bounded)
      if (is_k && q_pending) mbar_wait_bounded(&sm.bar_q, q_par);
      for (int s = 0; s < n_st; ++s)
        if (last_issued[s] >= 0) mbar_wait_bounded(&full[s], (last_issued[s] / n_st) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t qb = smem_addr(sm.q);
      int last_s = -1, last_pv = -1;  // last S / PV issued
      auto issue_s = [&](int j) -> bool {
        const int J = J0 + j;
        const int s = J % kKStages;
        if (!tc_wait(sm, &sm.k_full[s], (J / kKStages) & 1, err)) return false;
        fence_after_sync();
        last_s = J;
        const uint32_t kb = smem_addr(sm.k[s]);
        const uint32_t d = tmem + kColS + (uint32_t)(J & 1) * kKeys;
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;  // 64-dim half, 16-dim step in it
          mma_bf16(d, desc_sw128(qb + off, 16, 1024), desc_sw128(kb + off, 16, 1024), kIdescS, ks > 0);
        }
        commit(&sm.s_full[J & 1]);  // one commit per MMA group and barrier
        commit(&sm.k_empty[s]);
        if (kOverlap && j == n_tiles - 1) commit(&sm.q_free);  // the job's last read of Q
        return true;
      };
      // S runs one tile ahead: S(j + 1) is queued before PV(j), which waits
      // for the softmax of tile j
      bool ok = tc_wait(sm, &sm.bar_q, q_par, err) && issue_s(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles && !issue_s(j + 1)) break;
        const int J = J0 + j;
        const int s = J % kVStages;
        ok = tc_wait(sm, &sm.p_full[J & 1], (J >> 1) & 1, err) && tc_wait(sm, &sm.v_full[s], (J / kVStages) & 1, err);
        // the first PV overwrites O: the previous job's epilogue has read it
        if (kOverlap && ok && j == 0 && !first)
          ok = tc_wait(sm, &sm.o_free, ((uint32_t)pos.jobs - 1u) & 1u, err);
        if (!ok) break;
        fence_after_sync();
        const uint32_t pt = tmem + kColP + (uint32_t)(J & 1) * (kKeys / 2), vb = smem_addr(sm.v[s]);
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const uint32_t va = vb + ks * 2 * 1024;  // 16 keys = two 8-row groups
          // A = P in tensor memory: 16 keys = 8 columns of bf16 pairs
          mma_bf16_ts(tmem + kColO, pt + 8 * ks, desc_sw128(va, kHalf, 1024), kIdescO, (j > 0 || ks > 0) ? 1u : 0u);
        }
        commit(&sm.pv_done[J & 1]);
        last_pv = J;
      }
      // every MMA issued has completed before the CTA frees its tensor memory:
      // the PVs form one chain on O, and the S products were each waited for
      // by the softmax unless it gave up
      if (last_pv >= 0) mbar_wait_bounded(&sm.pv_done[last_pv & 1], (last_pv >> 1) & 1);
      if (last_s >= 0) mbar_wait_bounded(&sm.s_full[last_s & 1], (last_s >> 1) & 1);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;  // row = 4 * token + head in group
    const int pos = job.pos0 + (r >> 2);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int J = J0 + j;
      ok = __all_sync(0xffffffffu, tc_wait(sm, &sm.s_full[J & 1], (J >> 1) & 1, err));
      if (!ok) break;
      fence_after_sync();
      // scores of this row, scaled into the log2 domain in pairs
      float2 x[64];
      {
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_async(lane_base + kColS + (uint32_t)(J & 1) * kKeys + 32 * c, raw[c]);
        tmem_wait_ld(raw[0], raw[1], raw[2], raw[3]);
        const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
        for (int i = 0; i < 64; ++i)
          x[i] = __fmul2_rn(make_float2(__uint_as_float(raw[i >> 4][(2 * i) & 31]),
                                        __uint_as_float(raw[i >> 4][(2 * i + 1) & 31])),
                            sc2);
      }
      const int kbase = job.k_lo + j * kKeys;
      const bool need_mask = (kCausal && kbase + kKeys - 1 > job.pos0) || (kbase + kKeys > job.k_hi);
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int key = kbase + 2 * i;
          if (key >= job.k_hi || (kCausal && key > pos)) x[i].x = -INFINITY;
          if (key + 1 >= job.k_hi || (kCausal && key + 1 > pos)) x[i].y = -INFINITY;
        }
      }
      float mx8[8];  // 8 independent max chains
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], fmaxf(x[i].x, x[i].y));
      const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const bool grow = mt > m_run + kRescaleSlack;  // always true for the first finite max
      float corr = 1.f;
      if (grow) {
        corr = exp2f(m_run - mt);  // m_run = -inf -> 0
        l_run *= corr;
        m_run = mt;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O is rescaled: PV of tile j - 1 must be done (and with it every
        // earlier PV: they form one chain on O), so O is stable
        ok = __all_sync(0xffffffffu, tc_wait(sm, &sm.pv_done[(J - 1) & 1], ((J - 1) >> 1) & 1, err));
        if (!ok) break;
        fence_after_sync();
        // rescale the rows of O whose running max grew
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(lane_base + kColO + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(lane_base + kColO + 32 * c, o);
        }
      } else if (j >= 2) {
        // P buffer J & 1 was last read by PV of tile J - 2, which must be done
        // before it is rewritten (an S product goes to another accumulator
        // and may finish before it).  PV of tile J - 1 may still run: the
        // exponentials below overlap it.  (The previous job's PVs are all
        // done: its softmax waited for the last one before its closing
        // barrier.)
        ok = __all_sync(0xffffffffu, tc_wait(sm, &sm.pv_done[J & 1], ((J - 2) >> 1) & 1, err));
        if (!ok) break;
        fence_after_sync();
      }
      const float nm = (m_run == -INFINITY) ? 0.f : -m_run;
      const float2 nm2 = make_float2(nm, nm);
      float2 ls4[4];  // 4 independent pair-sum chains
#pragma unroll
      for (int i = 0; i < 4; ++i) ls4[i] = make_float2(0.f, 0.f);
      // P of this row: 128 bf16 keys as 64 pairs, into this lane's P columns
      const uint32_t prow = lane_base + kColP + (uint32_t)(J & 1) * (kKeys / 2);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // keys 64 hf .. + 63 = P columns 32 hf .. + 31
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 d = __fadd2_rn(x[32 * hf + i], nm2);
          const float2 e = make_float2(fast_exp2(d.x), fast_exp2(d.y));
          ls4[i & 3] = __fadd2_rn(ls4[i & 3], e);
          w[i] = pack_bf16x2(e.x, e.y);
        }
        tmem_st32u(prow + 32 * hf, w);
      }
      const float2 l2 = __fadd2_rn(__fadd2_rn(ls4[0], ls4[1]), __fadd2_rn(ls4[2], ls4[3]));
      l_run += l2.x + l2.y;
      fence_before_sync();  // the tensor-memory reads / writes above precede the arrive
      mbar_arrive(&sm.p_full[J & 1]);
    }
    const int J_last = J0 + n_tiles - 1;
    if (ok) ok = __all_sync(0xffffffffu, tc_wait(sm, &sm.pv_done[J_last & 1], (J_last >> 1) & 1, err));
    if (ok) {
      fence_after_sync();
      float o[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + kColO + 32 * c, o[c]);
      if constexpr (kOverlap) {
        fence_before_sync();  // the tensor-memory reads above precede the arrive
        mbar_arrive(&sm.o_free);
        stage(r, o, m_run, l_run, nullptr);
      } else {
        // the K stages are free (every S and PV is done, no copy is in
        // flight): the first two are the staging area
        stage(r, o, m_run, l_run, sm.k[0]);
      }
    }
    if constexpr (!kOverlap) {
      asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxWarps * 32) : "memory");
      if (!*reinterpret_cast<volatile int*>(&sm.abort)) store(r, sm.k[0]);
    }
  }

  if constexpr (!kOverlap) {
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
  }
  pos.tiles += n_tiles;
  pos.jobs += 1;
}

// After a CTA's last job (all threads): frees the tensor memory.
__device__ __forceinline__ void tc_finish(const TcPos& pos) {
  if (pos.jobs > 0 && (threadIdx.x >> 5) == kMmaWarp) tmem_dealloc(tc_smem().tmem, kTmemCols);
}

// Chunked-prefill rows: jobs (work item, kv head), item = (request, first
// query of a 32-token tile), items sorted by key extent, longest first.  Keys
// [kv_key_offset, position of the tile's last query] with the causal mask;
// the shared-prefix partial, if given, is folded in before the bf16
// rounding.  One CTA per job, or fewer CTAs that run several jobs each (a
// prefill pass beside a decode launch on the other SMs): CTA b takes job b
// of every round of gridDim.x jobs, in reverse order on odd rounds, so the
// long and the short jobs even out.
// kPersist: a grid of fewer CTAs than jobs (a separate instantiation: the
// job loop's registers would weigh on the one-job launches).
template <bool kPersist>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ PrefillItems items,
                   const __grid_constant__ TcMaps maps) {
  // the wait comes first: a decode launch that runs beside this pass starts
  // once every CTA here has released it, and so after the kernels before
  // this one have completed
  pdl_wait();
  pdl_launch_dependents();
  const int n_jobs = items.count * p.num_kv_heads;
  const int G = kPersist ? (int)gridDim.x : n_jobs;
  TcPos pos;
  for (int rnd = 0; rnd * G < n_jobs; ++rnd) {
    const int u = kPersist ? rnd * G + ((rnd & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x) : (int)blockIdx.x;
    if (u >= n_jobs) continue;
    // one job per CTA: (item, kv head), kv head fastest (dispatch order:
    // the longest items first); several per CTA: kv-head-major, so the jobs
    // running at the same time share a kv head's keys in L2
    const int it = kPersist ? u % items.count : u / p.num_kv_heads;
    const int r = items.req[it];
    const int j0 = items.q_start[it];
    const int qo0 = p.qo_indptr[r];
    const int c = p.qo_indptr[r + 1] - qo0;
    const int L = p.seq_lens[r];
    TcJob job;
    job.tok0 = qo0 + j0;
    job.nq = min(kTok, c - j0);
    job.kvh = kPersist ? u / items.count : u % p.num_kv_heads;
    job.pos0 = L - c + j0;
    job.k_lo = p.kv_key_offset;
    job.k_hi = job.pos0 + job.nq;
    job.table = p.block_tables + (size_t)r * p.max_blocks_per_req;
    // metadata that differ from the host plan: record and skip the job
    // (uniformly: every thread of the CTA reads the same values)
    if (job.nq <= 0 || job.k_hi <= job.k_lo || (job.k_hi - 1) / kPage >= p.max_blocks_per_req) {
      if (threadIdx.x == 0) record_error(p.err, PA_ERR_DEVICE_INDEX);
      continue;
    }
    // staged bf16 rows: 256 B per row, 16-byte chunk c at c ^ (row & 15);
    // with several jobs per CTA each row straight from registers to out
    run_tile<true, kPersist>(
        job, maps, p.num_kv_heads, p.num_blocks, p.scale_log2, p.err, pos,
      [&](int row, float (&o)[4][32], float m, float l, uint8_t* stg) {
        const size_t orow = (size_t)(job.tok0 + (row >> 2)) * p.num_q_heads + job.kvh * kGroup + (row & 3);
        const bool valid = (row >> 2) < job.nq;
        float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
        float ws = l > 0.f ? 1.f / l : 0.f, wp = 0.f;
        const float* po = nullptr;
        if (p.prefix_o && valid) {
          float wo;
          lse2 = merge2_weights(lse2, p.prefix_lse[orow], wo, wp);
          ws *= wo;
          po = p.prefix_o + orow * kHeadDim;
        }
#pragma unroll
        for (int c8 = 0; c8 < kHeadDim / 8; ++c8) {
          float y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = o[c8 >> 2][(c8 & 3) * 8 + i] * ws;
          if (po) {
            const float4 a = *reinterpret_cast<const float4*>(po + 8 * c8);
            const float4 b = *reinterpret_cast<const float4*>(po + 8 * c8 + 4);
            y[0] = fmaf(wp, a.x, y[0]);
            y[1] = fmaf(wp, a.y, y[1]);
            y[2] = fmaf(wp, a.z, y[2]);
            y[3] = fmaf(wp, a.w, y[3]);
            y[4] = fmaf(wp, b.x, y[4]);
            y[5] = fmaf(wp, b.y, y[5]);
            y[6] = fmaf(wp, b.z, y[6]);
            y[7] = fmaf(wp, b.w, y[7]);
          }
          const uint4 w = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                     pack_bf16x2(y[6], y[7]));
          if (!kPersist)
            *reinterpret_cast<uint4*>(stg + row * 256 + ((c8 ^ (row & 15)) << 4)) = w;
          else if (valid)
            *reinterpret_cast<uint4*>(p.out + orow * kHeadDim + 8 * c8) = w;
        }
        if (p.lse && valid) p.lse[orow] = lse2 * kLn2;
      },
      [&](int t, const uint8_t* stg) {
        // 16 consecutive threads write one 256-byte row; the 4 rows of a
        // token are adjacent in out, so a warp writes 2 KiB contiguously
#pragma unroll 4
        for (int i = 0; i < kRows * 16 / (kSoftmaxWarps * 32); ++i) {
          const int L = i * kSoftmaxWarps * 32 + t;
          const int row = L >> 4, c = L & 15;
          if ((row >> 2) >= job.nq) continue;
          const size_t orow = (size_t)(job.tok0 + (row >> 2)) * p.num_q_heads + job.kvh * kGroup + (row & 3);
          *reinterpret_cast<uint4*>(p.out + orow * kHeadDim + 8 * c) =
              *reinterpret_cast<const uint4*>(stg + row * 256 + ((c ^ (row & 15)) << 4));
        }
      });
    if (!kPersist || *reinterpret_cast<volatile int*>(&tc_smem().abort)) break;  // (a wait gave up: recorded)
  }
  if (kPersist) {  // the jobs ran without a barrier between them: every warp is done before the free
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
  }
  tc_finish(pos);
}

// Shared-prefix pass: grid (key chunk, kv head, 32-token tile of all the
// batch's queries), no mask.  Each CTA leaves a chunk partial (normalised o,
// log2 lse) for prefix_merge_kernel; with a single chunk it writes the
// prefix partial itself.
__global__ void __launch_bounds__(kThreads, 1) prefix_kernel(const PrefixParams p, const __grid_constant__ TcMaps maps) {
  // the wait comes first: a decode launch that runs beside this pass (done
  // != null) starts once every CTA here has released it, and so after the
  // kernels before this one have completed
  pdl_wait();
  pdl_launch_dependents();
  TcJob job;
  job.tok0 = blockIdx.z * kTok;
  job.nq = min(kTok, p.total_q - job.tok0);
  job.kvh = blockIdx.y;
  job.pos0 = 0;
  job.k_lo = blockIdx.x * p.chunk_keys;
  job.k_hi = min(p.prefix_keys, job.k_lo + p.chunk_keys);
  job.table = p.block_tables + (size_t)p.table_row * p.max_blocks_per_req;
  int* done = p.done ? p.done + (size_t)blockIdx.z * p.num_kv_heads + blockIdx.y : nullptr;
  if (job.nq <= 0 || job.k_hi <= job.k_lo) {  // not planned on the host
    if (done && threadIdx.x == 0) {
      record_error(p.err, PA_ERR_DEVICE_INDEX);
      red_add_release_gpu(done, 1);  // a waiting fold gives up no later than its bound
    }
    return;
  }
  const bool direct = gridDim.x == 1;
  float* dst_o = direct ? p.prefix_o : p.chunk_o + (size_t)blockIdx.x * p.total_q * p.num_q_heads * kHeadDim;
  float* dst_lse = direct ? p.prefix_lse : p.chunk_lse + (size_t)blockIdx.x * p.total_q * p.num_q_heads;
  // staged fp32 rows: 512 B per row, 16-byte chunk c at c ^ (row & 31)
  TcPos pos;
  run_tile<false, false>(
      job, maps, p.num_kv_heads, p.num_blocks, p.scale_log2, p.err, pos,
      [&](int row, float (&o)[4][32], float m, float l, uint8_t* stg) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c4 = 0; c4 < kHeadDim / 4; ++c4)
          *reinterpret_cast<float4*>(stg + row * 512 + ((c4 ^ (row & 31)) << 4)) =
              make_float4(o[c4 >> 3][(c4 & 7) * 4] * inv, o[c4 >> 3][(c4 & 7) * 4 + 1] * inv,
                          o[c4 >> 3][(c4 & 7) * 4 + 2] * inv, o[c4 >> 3][(c4 & 7) * 4 + 3] * inv);
        if ((row >> 2) < job.nq) {
          const size_t orow = (size_t)(job.tok0 + (row >> 2)) * p.num_q_heads + job.kvh * kGroup + (row & 3);
          dst_lse[orow] = l > 0.f ? m + log2f(l) : -INFINITY;
        }
      },
      [&](int t, const uint8_t* stg) {
#pragma unroll 4
        for (int i = 0; i < kRows * 32 / (kSoftmaxWarps * 32); ++i) {
          const int L = i * kSoftmaxWarps * 32 + t;
          const int row = L >> 5, c = L & 31;
          if ((row >> 2) >= job.nq) continue;
          const size_t orow = (size_t)(job.tok0 + (row >> 2)) * p.num_q_heads + job.kvh * kGroup + (row & 3);
          *reinterpret_cast<float4*>(dst_o + orow * kHeadDim + 4 * c) =
              *reinterpret_cast<const float4*>(stg + row * 512 + ((c ^ (row & 31)) << 4));
        }
      });
  // every store of the partial precedes run_tile's closing CTA barrier; the
  // release publishes them to the folds that acquire the count (also after
  // a recorded timeout, so no fold waits for a chunk that will not come)
  if (done && threadIdx.x == 0) red_add_release_gpu(done, 1);
  tc_finish(pos);
}

// Merge of the prefix pass's key-chunk partials: one warp per (query token,
// q head) row, two rows per CTA so the merge spreads over the SMs.  Lanes
// read the chunks' lse in parallel; then each lane issues the loads of its 4
// dims of up to 32 chunks at once and sums them with the broadcast weights.
constexpr int kMergeWarps = 2;
__global__ void __launch_bounds__(kMergeWarps * 32) prefix_merge_kernel(const PrefixParams p, int n_chunks) {
  pdl_launch_dependents();
  pdl_wait();
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

std::atomic<bool> g_prefill_attr_set[2][kMaxDevices];
std::atomic<bool> g_prefix_attr_set[kMaxDevices];

cudaError_t set_smem_attr(const void* fn, std::atomic<bool>* done) {
  return set_smem_limit_once(fn, (int)kSmemBytes, done);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const PrefillItems& items, const TcMaps& maps, int ctas,
                           cudaStream_t stream) {
  if (items.count <= 0) return cudaSuccess;
  const int jobs = items.count * p.num_kv_heads;
  if (ctas > 0 && ctas < jobs) {
    cudaError_t e = set_smem_attr((const void*)prefill_kernel<true>, g_prefill_attr_set[1]);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_kernel<true>, dim3(ctas), dim3(kThreads), kSmemBytes, stream, p, items, maps);
  }
  cudaError_t e = set_smem_attr((const void*)prefill_kernel<false>, g_prefill_attr_set[0]);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_kernel<false>, dim3(jobs), dim3(kThreads), kSmemBytes, stream, p, items, maps);
}

cudaError_t launch_prefix(const PrefixParams& p, int n_chunks, const TcMaps& maps, cudaStream_t stream) {
  cudaError_t e = set_smem_attr((const void*)prefix_kernel, g_prefix_attr_set);
  if (e != cudaSuccess) return e;
  dim3 grid(n_chunks, p.num_kv_heads, (p.total_q + kTok - 1) / kTok);
  return launch_pdl(prefix_kernel, grid, dim3(kThreads), kSmemBytes, stream, p, maps);
}

cudaError_t launch_prefix_merge(const PrefixParams& p, int n_chunks, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.total_q * p.num_q_heads;
  return launch_pdl(prefix_merge_kernel, dim3((unsigned)((rows + kMergeWarps - 1) / kMergeWarps)),
                    dim3(kMergeWarps * 32), 0, stream, p, n_chunks);
}

}  // namespace pa
