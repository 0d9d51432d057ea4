/*
 * pa.h -- C ABI of libpa: paged varlen attention for GB300 (sm_103a).
 *
 * One iteration-level (continuous) batch mixes decode rows (qo_len = 1) and
 * chunked-prefill rows (qo_len > 1, causal, starting at an offset).  Every
 * row reads its keys and values through a block table of fixed 16-token
 * pages; pages holding a shared prefix are referenced by many block tables
 * and stored once.
 *
 * Sources for the semantics (page titles and sections):
 *   - "Inference optimisation" (AI-infra book ch. 8), §8.1.1: prefill stores
 *     the keys and values of each layer; decode reads the whole context.
 *   - same, §8.3.1 and Fig. 8-10: fixed-size blocks, per-request block table
 *     from logical to physical block, logical order recovered through it.
 *   - same, §8.3.2 and Fig. 8-13: shared prefix blocks referenced by several
 *     block tables, stored once.
 *   - same, §8.2.3 and Fig. 8-8/8-9: a chunk of c new tokens after h old ones;
 *     new token j (0-based) attends to h + j + 1 keys.
 *   - "vLLM, SGLang and continuous batching", section "PagedAttention":
 *     16-token blocks, block table, attention kernel reads K/V through it.
 *   - "Disaggregated prefill and decode": qo_len / kv_len per request
 *     (decode sends qo_len = 1), and the HND page layout (head before token
 *     inside a page, so one head's page is contiguous).
 *
 * Conventions shared by every call:
 *   - All tensors are device memory owned by the caller.  No call allocates
 *     device memory: scratch space is the caller's `workspace`, except for
 *     pa_attention_varlen_noalloc, whose scratch is one fixed array that the
 *     library holds in each device's memory while it is loaded.
 *   - All launches are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  A call that returns PA_OK has only enqueued
 *     work.
 *   - Arguments are validated on the host first; on any error nothing is
 *     launched and the status says why (pa_last_error_message() has detail).
 *   - bf16 means IEEE bfloat16 (torch.bfloat16).  Row-major, densely packed.
 *   - KV pool layout (HND): k_cache and v_cache are each
 *     [num_blocks, num_kv_heads, block_size, head_dim] bf16, so one
 *     (block, kv head) slab is block_size * head_dim * 2 bytes, contiguous.
 *     Base pointers must be 16-byte aligned.
 *   - Supported shapes: head_dim = 128, block_size = 16,
 *     num_q_heads = 4 * num_kv_heads (GQA groups of 4 consecutive query
 *     heads per kv head: q head h reads kv head h / 4), num_kv_heads <= 256.
 *     Others give PA_ERR_UNSUPPORTED.
 *   - Decode rows are planned in launches of up to 1024 rows; the rows of
 *     one launch may hold at most 1,048,576 / num_kv_heads key pages of 16
 *     tokens in all (131,072 pages, 2,097,152 tokens, with 8 kv heads: 1024
 *     CTA segments of at most 1024 pages, shared by the kv heads).  Beyond
 *     that the attention calls give PA_ERR_UNSUPPORTED; pa_plan_decode_grid
 *     answers the same on the host alone.
 *   - Kernels never trap.  A block id or slot outside the pool found on the
 *     device is skipped (its keys are masked out / its write is dropped) and
 *     recorded in the error word at the start of the workspace; read it with
 *     pa_get_device_error() after synchronising the stream.
 *   - Every wait inside a kernel is bounded in time; a wait that gives up
 *     records PA_ERR_DEVICE_TIMEOUT in the error word and the kernel returns.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* the same handle as cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,         /* null pointer, bad size, inconsistent metadata */
  PA_ERR_UNSUPPORTED = 2,         /* shape outside what the kernels implement */
  PA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the *_workspace_size() query */
  PA_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
  PA_ERR_DEVICE_INDEX = 5,        /* (error word) block id or slot outside the pool */
  PA_ERR_DEVICE_TIMEOUT = 6       /* (error word) a bounded in-kernel wait gave up */
} pa_status;

#define PA_ABI_VERSION 1
#define PA_HEAD_DIM 128
#define PA_BLOCK_SIZE 16
#define PA_GQA_GROUP 4
#define PA_ERROR_WORD_BYTES 256   /* the workspace's first bytes hold the device error word */
#define PA_MAX_SEQ_LEN (1 << 20)  /* longest supported sequence (tokens) */

int32_t pa_abi_version(void);
const char* pa_status_string(int32_t status);
/* Detail of the last host-side error on the calling thread ("" if none). */
const char* pa_last_error_message(void);

/*
 * pa_kv_append -- write this step's new keys and values into their slots
 * ("Inference optimisation", AI-infra book ch. 8, §8.1.1: the keys and values
 * of every layer are kept for later tokens; §8.3.1 and Fig. 8-10: a token's
 * slot is a (physical block, offset) pair, and a sequence that grows takes a
 * new block from the free pool; "vLLM, SGLang and continuous batching",
 * section "PagedAttention": 16-token blocks).
 *   For new token i with slot = slot_mapping[i] >= 0, block = slot / 16 and
 *   offset = slot % 16, and every kv head h:
 *     k_cache[block, h, offset, :] = k_new[i, h, :]   (v likewise)
 *   Bytes are copied exactly.  slot < 0 means "no write" (padding).  Slots
 *   must be distinct; with duplicates the surviving row is unspecified.
 * k_new, v_new   [n_tokens, num_kv_heads, head_dim] bf16, 16-byte aligned.
 * slot_mapping   [n_tokens] int64, device.
 * k_cache, v_cache  the HND pools, modified in place.
 * workspace      device, >= PA_ERROR_WORD_BYTES bytes; only the error word is
 *                used.  A slot >= num_blocks * 16 is skipped and recorded as
 *                PA_ERR_DEVICE_INDEX.
 * n_tokens = 0 is valid and launches nothing.
 */
pa_status pa_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                       void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                       int32_t head_dim, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * q8_0 KV pages ("Inference optimisation", AI-infra book ch. 8, §8.4.2 and
 * Fig. 8-23: every 32 values share one 2-byte scale next to their 8-bit
 * codes, 34 bytes instead of 64).  A q8_0 pool is
 * [num_blocks, num_kv_heads, PA_Q8_SLAB_BYTES] bytes: one (block, kv head)
 * slab holds block_size x head_dim int8 codes (token t, dim d at
 * t * head_dim + d), then block_size x head_dim / 32 little-endian binary16
 * scales (token t, group g = d / 32 at byte block_size * head_dim +
 * 2 * (t * head_dim / 32 + g)).  Per group: d = max|x| / 127 in binary32,
 * stored as binary16 rounded to nearest even; code = rint(x / d16) in
 * binary32 with d16 the stored scale, clamped to [-127, 127]; all codes 0
 * when d16 is 0.  A code stands for code * d16.  Inputs must be finite.
 */
#define PA_Q8_SLAB_BYTES (PA_BLOCK_SIZE * PA_HEAD_DIM + PA_BLOCK_SIZE * (PA_HEAD_DIM / 32) * 2) /* 2176 */

/*
 * pa_kv_append_q8 -- pa_kv_append into q8_0 pools: each (token, kv head)
 * row of k_new / v_new is quantized in groups of 32 as described above and
 * stored with its scales in the slot's page.  Same arguments, validation and
 * error word as pa_kv_append; k_cache and v_cache are q8_0 pools
 * (16-byte aligned).
 */
pa_status pa_kv_append_q8(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                          void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                          int32_t head_dim, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_attention_varlen_q8 -- pa_attention_varlen over q8_0 pools, for decode
 * rows: every K and V element is its code times its group's scale, the rest
 * of the definition is unchanged (fp32 arithmetic, bf16 out, natural-log
 * lse).  Rows with qo_len > 1 give PA_ERR_UNSUPPORTED; rows with qo_len = 0
 * are skipped.  Workspace as pa_attention_varlen
 * (pa_attention_workspace_size).  Reading 34 instead of 64 bytes per 32
 * values shortens the HBM-bound decode when the saved read time exceeds
 * the added dequantization (the pages' Delta T = Delta D / beta - T_c).
 */
pa_status pa_attention_varlen_q8(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                                 const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* seq_lens,
                                 const int32_t* qo_indptr, const int32_t* seq_lens_host,
                                 const int32_t* qo_indptr_host, int32_t num_reqs, int32_t total_q,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 float sm_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 pa_stream_t stream);

/*
 * pa_copy_blocks -- copy-on-write block copy ("Inference optimisation",
 * AI-infra book ch. 8, §8.3.2 and Fig. 8-15: before a branch writes into a
 * block it shares with another request, it gets its own copy of that block,
 * and the filled read-only blocks stay shared).
 *   For pair i, the whole block src_blocks[i] -- every kv head and token
 *   slot, of k_cache and of v_cache -- is copied into block dst_blocks[i].
 * src_blocks, dst_blocks  [n_pairs] int32, device.  The dst ids must be
 *                distinct and none may also be a src id of the call;
 *                otherwise which copy lands is undefined (no fault).
 * k_cache, v_cache  HND pools as for pa_kv_append, modified in place.
 * workspace      device, >= PA_ERROR_WORD_BYTES bytes; a pair naming a block
 *                outside [0, num_blocks) is skipped and PA_ERR_DEVICE_INDEX
 *                is recorded in its error word.
 * Errors: PA_ERR_INVALID_ARG (n_pairs < 0, null or misaligned pointers),
 *   PA_ERR_UNSUPPORTED (shape), PA_ERR_WORKSPACE_TOO_SMALL, PA_ERR_CUDA.
 */
pa_status pa_copy_blocks(const int32_t* src_blocks, const int32_t* dst_blocks, int64_t n_pairs, void* k_cache,
                         void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_attention_workspace_size -- bytes of device workspace that
 * pa_attention_varlen needs for a batch with at most these sizes.  The
 * workspace holds the error word and the split-KV partial results.
 */
size_t pa_attention_workspace_size(int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t head_dim,
                                   int32_t max_seq_len);

/*
 * pa_attention_varlen -- causal GQA softmax attention over a paged KV cache
 * for a varlen batch ("Inference optimisation", AI-infra book ch. 8: §8.1.1,
 * decode attends each new token to the whole cached context; §8.2.3, the
 * N_pair equation and Fig. 8-8/8-9, a chunk of c tokens after h cached ones,
 * token j seeing h + j + 1 keys; §8.3.1 and Fig. 8-10, keys found through the
 * block table; "Continuous batching architecture", iteration-level batches
 * mixing decode rows and prefill chunks; "Disaggregated prefill and decode",
 * per-request qo_len / kv_len).
 *   Request r has qo_len = qo_indptr[r+1] - qo_indptr[r] query tokens, rows
 *   qo_indptr[r] .. qo_indptr[r+1]-1 of q, and seq_len = seq_lens[r] keys
 *   (the KV length after this step's append, so 0 <= qo_len <= seq_len).
 *   Query j of request r sits at position p = seq_len - qo_len + j and, for
 *   every q head h with kv head g = h / 4:
 *     s_t  = sm_scale * <q[row, h, :], K_g[t, :]>      for t = 0 .. p
 *     out[row, h, :] = sum_t exp(s_t - m) V_g[t, :] / sum_t exp(s_t - m)
 *     lse[row, h]    = m + ln(sum_t exp(s_t - m)),  m = max_t s_t
 *   where K_g[t, :] = k_cache[block_tables[r, t / 16], g, t % 16, :].
 *   Decode rows (qo_len = 1) use the persistent split-KV decode kernel: the
 *   (row, kv head) key ranges are laid end to end and cut into one equal
 *   segment per CTA, and ranges cut between CTAs are merged by log-sum-exp
 *   inside the same kernel.  Rows with qo_len > 1 use the tensor-core
 *   prefill kernel; rows with qo_len = 0 are skipped.  Arithmetic is fp32 on
 *   bf16 data; out is rounded to bf16.  The launch plan is made on the host
 *   from seq_lens_host / qo_indptr_host and travels in the kernel
 *   parameters, so a CUDA graph captured around this call replays the plan
 *   of the lengths it was captured with (for graphs replayed with new
 *   lengths, decode-only batches use pa_decode_step, which plans on the
 *   device).
 * q              [total_q, num_q_heads, head_dim] bf16, 16-byte aligned.
 * block_tables   [num_reqs, max_blocks_per_req] int32, device.  Entries past
 *                ceil(seq_len / 16) are never read.
 * seq_lens       [num_reqs] int32, device.
 * qo_indptr      [num_reqs + 1] int32, device; qo_indptr[0] = 0, non-decreasing,
 *                qo_indptr[num_reqs] = total_q.
 * seq_lens_host, qo_indptr_host  host copies of the same two arrays; the
 *                launch plan (which rows decode, how many KV splits) is made
 *                from them on the host.  They must equal the device arrays.
 * out            [total_q, num_q_heads, head_dim] bf16, 16-byte aligned.
 * lse            [total_q, num_q_heads] float32 (natural log), or NULL.
 * workspace      device, >= pa_attention_workspace_size(num_reqs, total_q,
 *                num_q_heads, head_dim, max over r of seq_lens) bytes,
 *                256-byte aligned, ZERO-FILLED before its first use.  It
 *                holds the error word, per-(request, kv head) counters of
 *                finished key ranges and the partial results of key ranges
 *                cut between CTAs; every call leaves the counters at zero,
 *                so a workspace is reused without clearing.  Calls sharing a workspace must not run
 *                concurrently.  After a PA_ERR_DEVICE_* error, zero it again.
 *                The error word is not cleared by this call (see
 *                pa_clear_device_error).
 */
pa_status pa_attention_varlen(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                              const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* seq_lens,
                              const int32_t* qo_indptr, const int32_t* seq_lens_host, const int32_t* qo_indptr_host,
                              int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, float sm_scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Decode step for CUDA graphs ("Inference optimisation", AI-infra book ch. 8,
 * §8.2.4: graphs captured in advance for a few row counts, inputs padded up
 * to the next captured size; "Continuous batching architecture", section
 * "CUDA graphs": one recorded launch sequence replayed for batches whose
 * padded shape matches, which removes the per-step CPU launch work).
 *
 * pa_decode_step -- the KV append and the attention of a decode-only batch
 * in one kernel launch whose launch shape depends only on the scalars
 * (num_reqs, num_kv_heads, max_seq_len) and the device's SM count, and which
 * reads no array on the host.  A launch captured in a CUDA graph is therefore valid for every
 * batch within those scalars: between replays the caller rewrites q, k_new,
 * v_new, block_tables and seq_lens in place.
 *   Row r (0 <= r < num_reqs) is one decode request with L = seq_lens[r]
 *   keys after this step (L >= 1), its new token at position L - 1 and
 *   query q[r].  The call writes k_new[r, h, :] / v_new[r, h, :] into
 *   k_cache / v_cache at the slot of position L - 1 (block
 *   block_tables[r, (L-1) / 16], offset (L-1) % 16; no slot_mapping is
 *   taken) and computes, for every q head, the attention of
 *   pa_attention_varlen with qo_len = 1 over the L keys, the new token
 *   included (out bf16, lse natural log).
 *   Rows with L = 0 are padding: nothing is written to the cache, their out
 *   rows are zero and lse is -inf.  Padding a batch to a captured size
 *   means L = 0 for the extra rows (KV lengths need no padding: the kernel
 *   reads the exact lengths).
 *   A row with L < 0, L > max_seq_len or more than max_blocks_per_req pages
 *   is treated as padding and recorded as PA_ERR_DEVICE_INDEX; a block id
 *   outside the pool is masked and recorded as in pa_attention_varlen.
 *   Requirement (copy-on-write, §8.3.2): the block receiving a row's new
 *   token is read by no other row of the call.  The appending CTA uses the
 *   new K/V directly, so the result equals pa_kv_append followed by
 *   pa_attention_varlen whenever that holds.
 * q              [num_reqs, num_q_heads, head_dim] bf16, 16-byte aligned.
 * k_new, v_new   [num_reqs, num_kv_heads, head_dim] bf16, 16-byte aligned.
 * k_cache, v_cache  HND bf16 pools, modified in place (the new tokens).
 * block_tables   [num_reqs, max_blocks_per_req] int32, device.
 * seq_lens       [num_reqs] int32, device only.
 * num_reqs       rows of the padded batch, 0 .. 1024 (see pa_decode_step_bucket).
 * max_seq_len    largest L any replay will use, 1 .. PA_MAX_SEQ_LEN.
 * out, lse       as pa_attention_varlen with total_q = num_reqs.
 * workspace      device, >= pa_decode_step_workspace_size(num_reqs,
 *                num_q_heads, head_dim, max_seq_len) bytes, 256-byte aligned,
 *                zero-filled before first use, left reusable by every call.
 *                Calls sharing a workspace must not run concurrently.
 * Errors: PA_ERR_INVALID_ARG (null or misaligned pointers, max_seq_len
 *   outside its range), PA_ERR_UNSUPPORTED (shape, num_reqs > 1024, or
 *   num_reqs x max_seq_len too large for one launch),
 *   PA_ERR_WORKSPACE_TOO_SMALL, PA_ERR_CUDA.  num_reqs = 0 launches nothing.
 */
pa_status pa_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_req,
                         const int32_t* seq_lens, int32_t num_reqs, int32_t max_seq_len, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, float sm_scale, void* out,
                         float* lse, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_step_workspace_size -- bytes of workspace pa_decode_step needs
 * for these scalars on the current device; 0 when no launch exists for them (num_reqs outside
 * 0 .. 1024, max_seq_len outside 1 .. PA_MAX_SEQ_LEN, num_q_heads < 4, or
 * num_reqs x max_seq_len too large).
 */
size_t pa_decode_step_workspace_size(int32_t num_reqs, int32_t num_q_heads, int32_t head_dim, int32_t max_seq_len);

/*
 * pa_decode_step_bucket -- the padded row count for a batch of num_reqs
 * decode rows: the smallest power of two >= num_reqs (1 for 0), so that a
 * handful of captured graphs cover 1 .. 1024 rows with less than 2x rows of
 * padding (padding rows cost no key reads).  -1 outside 0 .. 1024.
 */
int32_t pa_decode_step_bucket(int32_t num_reqs);

/*
 * pa_shared_prefix_workspace_size -- bytes of device workspace that
 * pa_attention_varlen_shared_prefix needs for a batch with at most these
 * sizes: the pa_attention_workspace_size() layout followed by the prefix
 * partial ([total_q, num_q_heads, head_dim + 1] fp32) and the key-chunk
 * partials it is merged from.  shared_prefix_pages = 0 gives
 * pa_attention_workspace_size().  Returns 0 for negative arguments.
 */
size_t pa_shared_prefix_workspace_size(int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t head_dim,
                                       int32_t max_seq_len, int32_t shared_prefix_pages);

/*
 * pa_attention_varlen_shared_prefix -- pa_attention_varlen for a batch whose
 * requests all begin with the same shared_prefix_pages pages (the shared
 * prefix blocks of "Inference optimisation" ch. 8, §8.3.2 and Fig. 8-13,
 * referenced by every block table and stored once).
 *   Same computation, arguments and results as pa_attention_varlen (up to
 *   fp32 rounding order), with the work split by key range:
 *     1. one tensor-core pass attends every query token of the batch to the
 *        prefix keys [0, 16 * shared_prefix_pages), reading each prefix page
 *        once per kv head for all rows together (no mask is needed: every
 *        query comes after the prefix); key chunks of it run on separate CTAs
 *        and are merged by log-sum-exp;
 *     2. the decode and prefill kernels attend each row to its own keys
 *        after the prefix and fold the prefix partial into their result by
 *        log-sum-exp before rounding to bf16.
 *   With fewer than two requests that have queries, or shared_prefix_pages
 *   = 0, the call runs exactly as pa_attention_varlen.
 * shared_prefix_pages  0 <= P <= max_blocks_per_req.  The caller asserts
 *                that entries 0 .. P-1 of every block-table row hold the same
 *                block ids (the pass reads them from the first request that
 *                has queries; rows that differ get that request's prefix).
 *                Every request with qo_len > 0 must have
 *                seq_len - qo_len >= 16 * P (the prefix is cached before this
 *                step's queries), else PA_ERR_INVALID_ARG.
 * workspace      >= pa_shared_prefix_workspace_size(num_reqs, total_q,
 *                num_q_heads, head_dim, max seq_len, P) bytes, 256-byte
 *                aligned, zero-filled before its first use, as for
 *                pa_attention_varlen (its counters are left at zero too).
 * Errors: as pa_attention_varlen.
 */
pa_status pa_attention_varlen_shared_prefix(
    const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks, const int32_t* block_tables,
    int32_t max_blocks_per_req, const int32_t* seq_lens, const int32_t* qo_indptr, const int32_t* seq_lens_host,
    const int32_t* qo_indptr_host, int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int32_t shared_prefix_pages, float sm_scale, void* out, float* lse,
    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_attention_varlen_noalloc -- pa_attention_varlen for callers that cannot
 * allocate device memory.  The pages describe no counterpart of this call;
 * it exists for callers that cannot obtain a workspace: a real-time serving
 * loop that must not enter the allocator between steps, a host framework
 * whose device memory is all handed out to its own pool, or a plugin that is
 * handed only its input and output pointers.
 *   Same computation, arguments and results as pa_attention_varlen, except
 *   that there is no workspace argument: the scratch is a fixed array of
 *   PA_NOALLOC_SCRATCH_BYTES (24 MiB) inside the library, present on every
 *   GPU that loads the library until the process exits.  A batch whose
 *   pa_attention_workspace_size() exceeds it is rejected with
 *   PA_ERR_UNSUPPORTED (and a message in pa_last_error_message()).
 *   No device memory is allocated or freed by this call.
 * device_error   nullable device int32; if given, receives the call's device
 *                error word (PA_OK or PA_ERR_DEVICE_*) on `stream`.  With
 *                NULL the device error word of the call is not reported
 *                anywhere (the next call clears it).
 * num_reqs       0 .. 65535 as for pa_attention_varlen (PA_ERR_INVALID_ARG
 *                outside, checked before seq_lens_host is read).
 * Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture.
 * Sharing: every call on a device uses the same array and leaves its contents
 *   there; each call clears its error word and counters on `stream` first.
 *   Calls that overlap on the GPU race on the array, so issue them in order
 *   (e.g. on one stream).
 */
#define PA_NOALLOC_SCRATCH_BYTES (24u << 20)
pa_status pa_attention_varlen_noalloc(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                                      const int32_t* block_tables, int32_t max_blocks_per_req,
                                      const int32_t* seq_lens, const int32_t* qo_indptr,
                                      const int32_t* seq_lens_host, const int32_t* qo_indptr_host, int32_t num_reqs,
                                      int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, float sm_scale, void* out, float* lse,
                                      int32_t* device_error, pa_stream_t stream);

/*
 * pa_merge_lse -- combine two partial attentions of the same queries over
 * disjoint key sets A and B.  The pages do not define this operation; it is
 * part of this library's interface so that a caller can split one request's
 * keys (across calls or devices) and combine the results.  It is the
 * log-sum-exp identity of softmax over a union of key sets:
 *   M = max(lse_a, lse_b), w_a = exp(lse_a - M), w_b = exp(lse_b - M)
 *   o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = M + ln(w_a + w_b)
 *   A part with lse = -inf has weight 0 (its o is ignored); if both are
 *   -inf, o = 0 and lse = -inf.
 * o_a, o_b, o_out  [rows, num_heads, head_dim] bf16, 16-byte aligned;
 *                  o_out may alias o_a or o_b.
 * lse_a, lse_b     [rows, num_heads] float32.
 * lse_out          [rows, num_heads] float32 or NULL; must not overlap lse_a
 *                  or lse_b.
 * head_dim must be a multiple of 8.
 */
pa_status pa_merge_lse(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o_out,
                       float* lse_out, int64_t rows, int32_t num_heads, int32_t head_dim, pa_stream_t stream);

/*
 * Error word.  pa_get_device_error copies the word at the start of
 * `workspace` to the host (synchronous: call it after the stream that used
 * the workspace has been synchronised) and stores PA_OK or the first
 * PA_ERR_DEVICE_* recorded.  pa_clear_device_error zeroes it on `stream`.
 */
pa_status pa_get_device_error(const void* workspace, int32_t* code_out);
pa_status pa_clear_device_error(void* workspace, pa_stream_t stream);

/*
 * Tuning and diagnostics.
 *   pa_set_decode_ctas(n): n > 0 asks for a persistent decode grid of n CTAs
 *     (capped by the plan limits and the workspace bound), 0 restores the
 *     automatic plan (one CTA per SM for the warp-granular kernel, three
 *     per SM for the CTA-granular one).  Process-wide.  pa_decode_step and
 *     pa_decode_step_workspace_size use it too (rounded up to whole kv
 *     heads, and raised where a segment would exceed 1024 pages).
 *   pa_set_prefill_ctas(n): for a call whose batch has decode rows and rows
 *     with qo_len > 1 (bf16 pages, no shared prefix, no forced decode grid,
 *     at most 1536 query tiles of 32 and 1024 decode rows: one launch each):
 *     n > 0 runs the tensor-core jobs of the qo_len > 1 rows on n persistent
 *     CTAs beside the decode launch (at most one fewer than the jobs and
 *     half the SMs), -1 never (the jobs first, one CTA each, then the decode
 *     launch), 0 restores the automatic choice (a cost model).  For a call
 *     whose batch has only rows with qo_len > 1 (bf16 pages, no shared
 *     prefix, no forced decode grid, at most 1536 query tiles of 32), n > 0
 *     runs its jobs on n persistent CTAs (at most one fewer than the jobs),
 *     each running its jobs in turn with the next one's start overlapping
 *     this one's end; 0 does so when
 *     every such row has at most 32 queries (verify rows) and there are at
 *     least two jobs per SM, on a grid a cost model picks (at most one CTA
 *     per SM), else one CTA per job; -1 always one CTA per job.
 *     Process-wide; n outside [-1, 1024] gives PA_ERR_INVALID_ARG.
 *   pa_launch_count(): kernels this library has launched in this process.
 *   pa_trace_enable(1): from now on every launch records a CUDA event before
 *     and after itself on its stream (at most 16384 launches are kept; the
 *     events are created by this call, on the current device);
 *     pa_trace_read() waits for the recorded events, returns per launch the
 *     kernel kind (pa_kernel_kind) and its duration in milliseconds, and
 *     clears the trace.  pa_trace_enable(0) stops recording.
 */
typedef enum {
  PA_KERNEL_KV_APPEND = 1,
  PA_KERNEL_DECODE = 2,
  PA_KERNEL_COMBINE = 3, /* reserved: the split merge is fused into PA_KERNEL_DECODE */
  PA_KERNEL_PREFILL = 4,
  PA_KERNEL_MERGE = 5,
  PA_KERNEL_PREFIX = 6,      /* shared-prefix pass of pa_attention_varlen_shared_prefix */
  PA_KERNEL_PREFIX_MERGE = 7, /* merge of that pass's key-chunk partials */
  PA_KERNEL_COPY_BLOCKS = 8,  /* pa_copy_blocks */
  PA_KERNEL_DECODE_STEP = 9   /* pa_decode_step */
} pa_kernel_kind;

pa_status pa_set_decode_ctas(int32_t n);
pa_status pa_set_prefill_ctas(int32_t n);
/*
 * pa_plan_tile_grid(job_tiles, n_jobs, decode_slabs, sms, ctas) -- the
 * persistent CTA count the library picks for a batch's tensor-core jobs
 * (rows with qo_len > 1), computed on the host alone (no device is touched):
 * job_tiles[i] is job i's number of 128-key tiles in the kernel's job order
 * (for each kv head, the batch's 32-query tiles by decreasing key extent),
 * sms the device's SM count.  With decode_slabs > 0 (the batch's decode rows
 * hold that many 8 KiB (page, kv head) K+V slabs) it is the count beside the
 * decode launch that pa_set_prefill_ctas(0) leads to (0: the jobs first, one
 * CTA each); with decode_slabs = 0 the count for the jobs alone, which
 * pa_attention_varlen uses when every such row has at most 32 queries (0:
 * one CTA per job).  Ownership: job_tiles is read, *ctas written; both host
 * memory.  Errors: PA_ERR_INVALID_ARG for a null ctas, n_jobs outside
 * [0, 393216] (1536 query tiles x 256 kv heads), a null job_tiles with
 * n_jobs > 0, a tile count below 1, sms outside [1, 1024] or decode_slabs < 0
 * (*ctas is then 0).
 */
pa_status pa_plan_tile_grid(const int32_t* job_tiles, int32_t n_jobs, int64_t decode_slabs, int32_t sms,
                            int32_t* ctas);
/*
 * pa_plan_decode_grid(seq_lens, n_rows, num_kv_heads, sms, grid,
 * warp_granular) -- the decode launch pa_attention_varlen plans for a batch
 * of n_rows decode rows (qo_len 1, bf16 pages, no shared prefix, no rows with
 * qo_len > 1) of these seq_lens on a device of sms SMs, computed on the host
 * alone (no device is touched): *grid CTAs (0: nothing to do) of the
 * warp-granular decode kernel (*warp_granular = 1) or of the CTA-granular one
 * (0).  A grid forced by pa_set_decode_ctas applies here as in the call.
 * Ownership: seq_lens is read, *grid and *warp_granular written; all host
 * memory.  Errors: PA_ERR_INVALID_ARG for a null output, n_rows outside
 * [0, 1024], a null seq_lens with n_rows > 0, a seq_len below 1, num_kv_heads
 * outside [1, 256] or sms outside [1, 1024]; PA_ERR_UNSUPPORTED when no plan
 * fits the kernels' limits, as the call would return.
 */
pa_status pa_plan_decode_grid(const int32_t* seq_lens, int32_t n_rows, int32_t num_kv_heads, int32_t sms,
                              int32_t* grid, int32_t* warp_granular);
/*
 * pa_set_decode_fault_injection(on) -- a test of the bounded-wait path, off
 * (0) by default, process-wide.  With on = 1, decode launches of
 * pa_attention_varlen and pa_attention_varlen_shared_prefix over bf16 pages
 * use a diagnostic build of the decode kernel in which CTA 0 arms the
 * barrier of its second page without issuing that page's copies, and every
 * wait gives up after 1 ms instead of 2 s.  Nothing faults or hangs: the
 * waiting warps give up, record PA_ERR_DEVICE_TIMEOUT in the error word, let
 * the copies they did issue land and return; the other CTAs finish
 * normally.  What such a call leaves: the error word set; the outputs of
 * the rows whose keys CTA 0 holds undefined; for rows cut between CTAs, their
 * counters in the workspace non-zero -- zero the workspace before its next
 * use, as after any PA_ERR_DEVICE_* error.  on outside {0, 1} gives
 * PA_ERR_INVALID_ARG.
 */
pa_status pa_set_decode_fault_injection(int32_t on);
int64_t pa_launch_count(void);
pa_status pa_trace_enable(int32_t on);
pa_status pa_trace_read(int32_t* kinds, float* ms, int32_t capacity, int32_t* count);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
