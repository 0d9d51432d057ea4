// Host-side interface between the C ABI (pa_api.cu) and the kernel files.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pa.h"

namespace pa {

struct AppendParams {
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int64_t* slot_mapping;
  int64_t n_tokens;
  uint16_t* k_cache;
  uint16_t* v_cache;
  int64_t num_blocks;
  int32_t num_kv_heads;
  int* err;
};

struct CopyParams {
  uint16_t* k_cache;
  uint16_t* v_cache;
  int64_t num_blocks;
  const int32_t* src;
  const int32_t* dst;
  int64_t n_pairs;
  int64_t block_vecs;  // 16-byte words in one block of one cache
  int* err;
};

// Persistent decode launch plan (host-made, passed by value).  For each kv
// head the decode rows' pages are laid end to end as one stream (row d of
// the launch, then row d + 1, ...); every stream is cut into n_seg equal
// segments of seg pages.  CTA b takes kv head b % Hkv and segment b / Hkv,
// so the Hkv CTAs of a segment read the same blocks at the same time.
constexpr int kPlanMaxRows = 1024;   // decode rows per launch
constexpr int kPlanMaxCtas = 1024;   // CTAs per launch
constexpr int kDecodeMaxItemsPerCta = 64;
// Warps of the CTA-granular decode kernel (three CTAs per SM).  Workspaces
// hold kDecodeWarps pieces per CTA of the largest CTA-granular grid, which
// also covers the warp-granular launches (a third of the CTAs, kWgWarps
// pieces each).
constexpr int kDecodeWarps = 4;
// Host-planned launches whose warp segments would hold fewer pages than this
// run the CTA-granular kernel: a row cut into many short warp pieces costs
// its last piece a long merge, and few pages per warp leave its 2-page ring
// latency-bound (measured: one 2048-token row per layer 12.6 us CTA-granular
// against 18.6 us warp-granular; 32 rows 58.2 against 54.9 us).
constexpr int kMinWarpSegPages = 8;
// The warp-granular decode kernel runs one CTA of kWgWarps warps per SM,
// one warp segment per warp: the warps of an SM then share one CTA, which
// measured faster than three CTAs of four warps (the later CTAs on an SM
// streamed up to 9 % slower).  A segment may hold kWgMaxPagesPerCta pages and
// kWgMaxItemsPerCta rows.
constexpr int kWgWarps = 12;
constexpr int kWgMaxPagesPerCta = 3072;
constexpr int kWgMaxItemsPerCta = 192;
// Bytes of one (page, kv head) slab of K or V in bf16 (16 tokens x 128 dims).
constexpr int kSlabBytesHost = 16 * 128 * 2;
struct DecodePlan {
  int32_t n_rows;                     // decode rows of this launch
  int32_t seg;                        // pages per segment
  int32_t total;                      // pages of one kv head's stream
  int32_t rows[kPlanMaxRows];         // request index of decode row d
  int32_t seq[kPlanMaxRows];          // its seq_len (from the host copy)
  int32_t tok[kPlanMaxRows];          // its query token (qo_indptr, from the host copy)
  int32_t first_row[kPlanMaxCtas];    // row (index d) holding a segment's first page
  int32_t first_page[kPlanMaxCtas];   // that page's index within its row
};

// Decode step (self-planned launch): the kernel parameters carry only the
// padded batch size and the longest valid seq_len; each CTA plans its own
// segment from the device seq_lens, so one captured launch serves any
// lengths within these bounds.  A row costs its pages plus kStepItemCost
// stream units (the item-end merge work, in pages of streaming), and the
// stream is cut into segments of at least kStepMinSegCost units.
struct StepPlan {
  int32_t n_rows;       // rows of the padded batch (<= kPlanMaxRows)
  int32_t max_seq_len;  // rows with a longer seq_len are errors
};
constexpr int kStepItemCost = 8;
constexpr int kStepMinSegCost = 8;
template <bool kStep>
struct PlanOf {
  using type = DecodePlan;
};
template <>
struct PlanOf<true> {
  using type = StepPlan;
};

struct DecodeParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_req;
  const int32_t* seq_lens;
  const int32_t* qo_indptr;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  float scale_log2;      // sm_scale * log2(e)
  int32_t page_offset;   // leading pages of every row left out (a shared prefix attended elsewhere)
  const float* prefix_o;    // fp32 [prefix_n][total_q, Hq, D] normalised partials over those pages, or null
  const float* prefix_lse;  // fp32 [prefix_n][total_q, Hq] their log2-domain lse
  int32_t prefix_n;         // partials to fold in (key chunks of the prefix; 1 once merged)
  int64_t prefix_rows;      // total_q * Hq: the stride between two partials' rows
  // Prefix pass running at the same time as this launch (else null: its
  // partials are complete before the launch).  prefix_done[t * Hkv + kvh]
  // counts the key chunks of query tile t (kPrefillQTile tokens) written so
  // far; a row's fold waits for prefix_n of them.  prefix_readers counts the
  // folds done per (tile, kv head); the last of a tile's prefix_tile_rows(t)
  // readers returns both counters to zero.
  int* prefix_done;
  int* prefix_readers;
  // 1: the tile kernel launched just before runs beside this launch (a
  // prefix pass, or chunked-prefill jobs on SMs of their own).  Its CTAs
  // waited for the kernels before it and then released this launch, which
  // therefore skips its own wait at the start, and waits for that kernel at
  // its end, so that this launch completes after it (stream order).
  int32_t beside;
  int32_t total_q;
  uint16_t* out;         // bf16 [total_q, Hq, D]
  float* lse;            // [total_q, Hq] natural log, or null
  float* piece_o;        // fp32 [2 x warp segments (warp-granular) or CTAs (CTA-granular), 4, D]: the
                         // partial of a segment's first / last item
  float* piece_lse;      // fp32 [2 x the same, 4], log2 domain
  int64_t piece_slots;   // (piece, head) slots the two arrays hold; a write past them is recorded, not made
  int* counters;         // [num_reqs, Hkv] CTAs finished per item; zero between calls
  int* err;
  // decode step only: the new token of every row ([rows, Hkv, D] bf16) and
  // the pools it is appended to (the same memory as k_cache / v_cache)
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_store;
  uint16_t* v_store;
};

// Tiled TMA maps of the tensor-core tile kernels (host-encoded, passed by
// value): q as [total_q][Hq][D] with 64 x 4 x 32 boxes, the K and V pools as
// [num_blocks * Hkv * 16][D] rows with 64 x 16 boxes, all 128-byte swizzled.
struct TcMaps {
  CUtensorMap q;
  CUtensorMap k;
  CUtensorMap v;
};

// Prefill work items: (request, first query of the tile) pairs, passed by
// value in the kernel's parameter block.
constexpr int kMaxPrefillItems = 1536;
struct PrefillItems {
  int32_t count;
  int32_t req[kMaxPrefillItems];
  int32_t q_start[kMaxPrefillItems];
};

struct PrefillParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_req;
  const int32_t* seq_lens;
  const int32_t* qo_indptr;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  float scale_log2;
  int32_t kv_key_offset;    // keys [0, kv_key_offset) left out (a shared prefix, whole pages)
  const float* prefix_o;    // as in DecodeParams, or null
  const float* prefix_lse;
  uint16_t* out;
  float* lse;
  int* err;
};

// Shared-prefix pass: all total_q query tokens against the prefix keys
// [0, prefix_keys) of block-table row table_row, cut into key chunks of
// chunk_keys (a multiple of 64).  Chunk partials go to chunk_o / chunk_lse
// ([n_chunks][total_q][Hq] rows), merged into prefix_o / prefix_lse by the
// merge kernel.  With one chunk the CTAs write prefix_o / prefix_lse directly.
struct PrefixParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_req;
  int32_t table_row;
  int32_t total_q;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t prefix_keys;
  int32_t chunk_keys;
  float scale_log2;
  float* chunk_o;
  float* chunk_lse;
  float* prefix_o;
  float* prefix_lse;
  int* done;  // per (query tile, kv head): chunks written (release), or null
  int* err;
};

struct MergeParams {
  const uint16_t* o_a;
  const float* lse_a;
  const uint16_t* o_b;
  const float* lse_b;
  uint16_t* o_out;
  float* lse_out;
  int64_t rows;
  int32_t num_heads;
  int32_t head_dim;
};

// Raises the dynamic shared-memory limit of kernel `fn` to `bytes` once per
// device: done[dev] records that it was set.  Host threads may race on the
// first call of a device; each then sets the same value, which is harmless,
// and the flag is an atomic.
constexpr int kMaxDevices = 64;
inline cudaError_t set_smem_limit_once(const void* fn, int bytes, std::atomic<bool>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
  return e;
}

// Sets the calling thread's pa_last_error_message() text and returns s.
pa_status set_error(pa_status s, const char* fmt, ...);

// Each launcher enqueues one kernel on `stream` and returns its launch error.
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_kv_append_q8(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream);
// overlap: programmatic launch after the stream's previous kernel; diag:
// the timeout-path diagnostic instantiation (bf16 pages, warp-granular);
// cta_granular: the kernel whose 4 warps read every page of the CTA's
// segment (no prefix pass beside it), for plans with short segments; else
// the warp-granular kernel (plan in whole warp segments of kWgWarps warps)
cudaError_t launch_decode(const DecodeParams& p, const DecodePlan& plan, int grid, bool q8, bool overlap,
                          bool diag, bool cta_granular, cudaStream_t stream);
// warp_granular: the warp-granular kernel (grid: one CTA per SM at most; no
// segment may hold more than kWgMaxItemsPerCta rows or kWgMaxPagesPerCta
// pages), else the CTA-granular one (windows of rows)
cudaError_t launch_decode_step(const DecodeParams& p, const StepPlan& plan, int grid, bool warp_granular,
                               cudaStream_t stream);
// ctas: CTAs of the launch (0: one per (item, kv head) job; fewer run
// several jobs each)
cudaError_t launch_prefill(const PrefillParams& p, const PrefillItems& items, const TcMaps& maps, int ctas,
                           cudaStream_t stream);
cudaError_t launch_prefix(const PrefixParams& p, int n_chunks, const TcMaps& maps, cudaStream_t stream);
cudaError_t launch_prefix_merge(const PrefixParams& p, int n_chunks, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

// Query tile of the tensor-core tile kernels (query tokens per CTA: with the
// 4 heads of a GQA group, 128 rows = the MMA's M) and their key tile.
constexpr int kPrefillQTile = 32;
constexpr int kTcKeyTile = 128;
// Decode kernel: pages a CTA may hold block ids for (bounds the segment).
constexpr int kDecodeMaxPagesPerCta = 1024;

}  // namespace pa
