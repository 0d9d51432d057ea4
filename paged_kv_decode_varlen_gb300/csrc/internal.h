// Host-side interface between the C ABI (pa_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

struct DecodeParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_req;
  const int32_t* seq_lens;
  const int32_t* qo_indptr;
  int32_t num_reqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_splits;
  float scale_log2;      // sm_scale * log2(e)
  uint16_t* out;         // bf16 [total_q, Hq, D]
  float* lse;            // [total_q, Hq] natural log, or null
  float* part_o;         // fp32 [num_splits, total_q, Hq, D] (used when num_splits > 1)
  float* part_lse;       // fp32 [num_splits, total_q, Hq], log2 domain
  int32_t total_q;
  int* err;
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
  uint16_t* out;
  float* lse;
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

// Each launcher enqueues one kernel on `stream` and returns its launch error.
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillParams& p, const PrefillItems& items, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

// Query tile of the prefill kernel (query tokens per CTA).
constexpr int kPrefillQTile = 16;
// Decode kernel: pages of block ids a CTA may hold (bounds pages per split).
constexpr int kDecodeMaxPagesPerCta = 1024;
constexpr int kMaxSplits = 64;

}  // namespace pa
