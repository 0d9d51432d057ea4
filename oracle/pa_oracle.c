/*
 * CPU oracle for paged varlen attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference arm may load this code.  The product path (the CUDA library
 * under paged_kv_decode_varlen_gb300/) shares nothing with it: no header,
 * helper, table or constant.
 *
 * Everything here is the plain definition, computed in fp64 from inputs
 * that are exact bf16 values:
 *
 *   * Paged KV addressing.  A sequence is cut into fixed blocks of p tokens;
 *     a per-request block table maps logical block i to a physical block, and
 *     attention recovers the logical order through that table.
 *     ("Inference optimisation", AI-infra book ch. 8, §8.3.1 and Fig. 8-10;
 *     "vLLM, SGLang and continuous batching", section "PagedAttention":
 *     16-token blocks, block table, the attention kernel reads K and V
 *     through it.)
 *   * Page layout.  HND: inside one page the head index comes before the
 *     token index, so one (page, kv head) is a contiguous [p, D] slab
 *     ("Disaggregated prefill and decode", paragraph on NHD vs HND pages).
 *     The layout lives in one function, kv_offset(), below.
 *   * Causal chunk semantics.  With c new tokens over h old ones, the first
 *     new token attends to h+1 keys and the last to h+c (§8.2.3, the
 *     N_pair equation and Fig. 8-8/8-9).  With seq_len = h + c the total
 *     KV length after this step's append, query j (0-based) of the chunk
 *     sits at absolute position seq_len - qo_len + j and sees keys
 *     0 .. that position.  A decode row (qo_len = 1, "Disaggregated
 *     prefill and decode", qo_len/kv_len paragraph) sees all seq_len keys.
 *   * Softmax attention with scale, GQA grouping kv_head = q_head / G with
 *     G = Hq / Hkv (contiguous groups), and the natural-log LSE.  The pages
 *     name these only in passing (the attention of §8.2.3 and the GQA of
 *     §8.4.2); the definition used is the textbook one written out below.
 *   * KV append: the keys and values of each new token are stored in the
 *     cache slot assigned to it (§8.1.1: prefill "stores keys and values
 *     of each layer"; §8.3.1: a new block is taken when the sequence grows).
 *     slot = block * p + offset; a negative slot means "no write".
 *   * LSE merge of two partial results over disjoint key sets: the
 *     log-sum-exp identity written out.
 *
 * Nothing is blocked, fused or reordered beyond the definition: each output
 * element is one loop over its visible keys in increasing order.  OpenMP
 * only distributes independent (query, head) outputs over threads, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_INDEX 2

/* bf16 bit pattern -> exact value.  bf16 is the top half of an IEEE
 * binary32, so shifting the 16 bits up gives the binary32 pattern. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), straight from the
 * double so that no intermediate binary32 rounding happens.  bf16 keeps 8
 * significant bits; frexp gives x = m * 2^e with 0.5 <= |m| < 1, and
 * rint() (round-to-nearest-even in the default mode) rounds m * 2^8.
 * Values below the smallest normal bf16 are flushed to signed zero;
 * overflow gives infinity. */
uint16_t oracle_round_bf16(double x) {
  float f;
  uint32_t u;
  if (isnan(x)) return (uint16_t)0x7fc0;
  if (x == 0.0 || fabs(x) < 1.1754943508222875e-38) {
    f = signbit(x) ? -0.0f : 0.0f;
  } else {
    int e;
    double m = frexp(x, &e);
    double r = ldexp(rint(ldexp(m, 8)), e - 8);
    if (fabs(r) > 3.3895313892515355e+38) r = copysign(INFINITY, x);
    f = (float)r; /* exact: r has at most 8 significant bits */
  }
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

double oracle_bf16_value(uint16_t bits) { return bf16_to_double(bits); }

void oracle_round_bf16_array(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i]);
}

/* binary16 bit pattern -> exact value. */
static double f16_to_double(uint16_t h) {
  int e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                      /* zero, subnormal */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x400), e - 25);                 /* 1.m * 2^(e-15) */
  return (h & 0x8000) ? -v : v;
}

/* binary32 value -> binary16 bits, round to nearest even, gradual underflow,
 * overflow to infinity: rounded with rint() at the value's binary16 quantum
 * (2^(e-11) for normal numbers, 2^-24 below 2^-14), then encoded. */
static uint16_t f32_to_f16(float f) {
  double x = (double)f;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7e00;
  double r;
  if (a < ldexp(1.0, -14)) {
    r = ldexp(rint(ldexp(a, 24)), -24);
  } else {
    int e;
    double m = frexp(a, &e);
    r = ldexp(rint(ldexp(m, 11)), e - 11);
  }
  if (r >= 65520.0 || isinf(a)) return sign | 0x7c00;
  if (r < ldexp(1.0, -14)) return sign | (uint16_t)ldexp(r, 24);   /* subnormal (or 0) */
  int e;
  double m = frexp(r, &e);                                          /* r = m 2^e, 0.5 <= m < 1 */
  return sign | (uint16_t)((e + 14) << 10) | (uint16_t)(ldexp(m, 11) - 1024.0);
}

uint16_t oracle_f32_to_f16(float f) { return f32_to_f16(f); }
double oracle_f16_value(uint16_t h) { return f16_to_double(h); }

/*
 * q8_0 ("Inference optimisation", AI-infra book ch. 8, §8.4.2 and Fig.
 * 8-23): 32 values share one 2-byte scale and each keeps an 8-bit code, 34
 * bytes instead of 64.  The pages fix the grouping and the sizes, not the
 * arithmetic; the reading used here: the scale is d = max|x| / 127 in
 * binary32, stored as binary16 (round to nearest even); each code is
 * rint(x / d16) in binary32 with d16 the stored scale, clamped to
 * [-127, 127]; a group whose stored scale is 0 gets all-zero codes.  The
 * value a code stands for is code * d16 (exact in binary32).
 */
static void quantize_group_q8(const uint16_t* x, int8_t* codes, uint16_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float v = (float)fabs(bf16_to_double(x[i]));
    if (v > amax) amax = v;
  }
  float d = amax / 127.0f;
  uint16_t h = f32_to_f16(d);
  float d16 = (float)f16_to_double(h);
  for (int i = 0; i < 32; ++i) {
    int c = 0;
    if (d16 != 0.0f) {
      float t = rintf((float)bf16_to_double(x[i]) / d16);
      c = t > 127.0f ? 127 : (t < -127.0f ? -127 : (int)t);
    }
    codes[i] = (int8_t)c;
  }
  *scale = h;
}

void oracle_quantize_q8(const uint16_t* x, int64_t n_groups, int8_t* codes, uint16_t* scales) {
  for (int64_t g = 0; g < n_groups; ++g) quantize_group_q8(x + 32 * g, codes + 32 * g, scales + g);
}

/* q8_0 pages: one (block, kv head) slab of p tokens is p * D code bytes
 * (token t, dim d at t * D + d) followed by p * D / 32 little-endian
 * binary16 scales (token t, group g at 2 * (t * D / 32 + g)). */
static size_t q8_slab_bytes(int p, int D) { return (size_t)p * (size_t)D + (size_t)p * (size_t)(D / 32) * 2; }

static double q8_elem(const uint8_t* cache, int64_t block, int kvh, int off, int d, int Hkv, int p, int D) {
  const uint8_t* slab = cache + ((size_t)block * (size_t)Hkv + (size_t)kvh) * q8_slab_bytes(p, D);
  const uint8_t* sc = slab + (size_t)p * D + 2 * ((size_t)off * (D / 32) + d / 32);
  return (double)(int8_t)slab[(size_t)off * D + d] * f16_to_double((uint16_t)(sc[0] | (sc[1] << 8)));
}

/* Element offset of (physical block, kv head, token-in-block, dim) in one
 * HND pool [num_blocks, Hkv, p, D]. */
static size_t kv_offset(int64_t block, int kvh, int off, int d, int Hkv, int p, int D) {
  return (((size_t)block * (size_t)Hkv + (size_t)kvh) * (size_t)p + (size_t)off) * (size_t)D + (size_t)d;
}

/*
 * Decode-step slots.  A decode row with L = seq_lens[r] keys after the step
 * holds its new token at position L - 1, the last of its sequence; that
 * position lives in logical block (L - 1) / p at offset (L - 1) % p, and the
 * block table maps the logical block to its physical one (§8.3.1 and Fig.
 * 8-10: tokens fill the table's blocks in order, a new block being taken
 * when the last one is full).  Rows with L = 0 are padding (slot -1), and so
 * are rows with L < 0, L > max_seq_len or more than max_blocks_per_req
 * blocks, which are counted.  Returns the count of such invalid rows.
 */
int oracle_decode_step_slots(const int32_t* block_tables, int max_blocks_per_req, const int32_t* seq_lens,
                             int num_reqs, int block_size, int max_seq_len, int64_t* slots) {
  int bad = 0;
  for (int r = 0; r < num_reqs; ++r) {
    int64_t L = seq_lens[r];
    slots[r] = -1;
    if (L == 0) continue;
    if (L < 0 || L > max_seq_len || (L + block_size - 1) / block_size > max_blocks_per_req) {
      ++bad;
      continue;
    }
    int64_t pos = L - 1;
    int64_t block = block_tables[(size_t)r * (size_t)max_blocks_per_req + (size_t)(pos / block_size)];
    slots[r] = block * block_size + pos % block_size;
  }
  return bad;
}

/*
 * KV append: for new token i with slot s = slot_mapping[i] >= 0, write
 * k_new[i, h, :] and v_new[i, h, :] into block s / p, offset s % p, for
 * every kv head h.  Negative slots are skipped.  A slot beyond the pool is
 * an error and nothing further is written.
 */
int oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                     uint16_t* k_cache, uint16_t* v_cache, int64_t num_blocks, int block_size, int num_kv_heads,
                     int head_dim) {
  if (block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || n_tokens < 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    int64_t block = slot / block_size;
    int off = (int)(slot % block_size);
    if (block >= num_blocks) return ORACLE_ERR_INDEX;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int d = 0; d < head_dim; ++d) {
        size_t src = ((size_t)i * (size_t)num_kv_heads + (size_t)h) * (size_t)head_dim + (size_t)d;
        size_t dst = kv_offset(block, h, off, d, num_kv_heads, block_size, head_dim);
        k_cache[dst] = k_new[src];
        v_cache[dst] = v_new[src];
      }
    }
  }
  return ORACLE_OK;
}

/* KV append into q8_0 pages: the same scatter as oracle_kv_append, each
 * (token, head) row of D values quantized in groups of 32 on the way in. */
int oracle_kv_append_q8(const uint16_t* k_new, const uint16_t* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                        uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks, int block_size, int num_kv_heads,
                        int head_dim) {
  if (block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 32 || n_tokens < 0) return ORACLE_ERR_ARG;
  const size_t slab = q8_slab_bytes(block_size, head_dim);
  for (int64_t i = 0; i < n_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    int64_t block = slot / block_size;
    int off = (int)(slot % block_size);
    if (block >= num_blocks) return ORACLE_ERR_INDEX;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int which = 0; which < 2; ++which) {
        const uint16_t* row = (which ? v_new : k_new) + ((size_t)i * num_kv_heads + h) * head_dim;
        uint8_t* s = (which ? v_cache : k_cache) + ((size_t)block * num_kv_heads + h) * slab;
        for (int g = 0; g < head_dim / 32; ++g) {
          int8_t codes[32];
          uint16_t scale;
          quantize_group_q8(row + 32 * g, codes, &scale);
          memcpy(s + (size_t)off * head_dim + 32 * g, codes, 32);
          uint8_t* sc = s + (size_t)block_size * head_dim + 2 * ((size_t)off * (head_dim / 32) + g);
          sc[0] = (uint8_t)(scale & 0xff);
          sc[1] = (uint8_t)(scale >> 8);
        }
      }
    }
  }
  return ORACLE_OK;
}

/*
 * Block copy (copy-on-write): before a branch writes into a block it shares
 * with another request, it gets its own copy of that block; the filled
 * read-only blocks stay shared ("Inference optimisation", AI-infra book
 * ch. 8, §8.3.2 and Fig. 8-15: the shared tail block holding a, b, c is
 * copied, then each branch appends its own token).  For pair i the whole
 * block src[i] (every kv head, every token slot, K and V) is written into
 * block dst[i]; pairs are applied in order.  A pair with an id outside the
 * pool is skipped; the return value is the number of skipped pairs.
 */
int64_t oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, int64_t num_blocks, int block_size,
                           int num_kv_heads, int head_dim, const int32_t* src, const int32_t* dst, int64_t n_pairs) {
  int64_t skipped = 0;
  for (int64_t i = 0; i < n_pairs; ++i) {
    if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
      ++skipped;
      continue;
    }
    for (int h = 0; h < num_kv_heads; ++h)
      for (int off = 0; off < block_size; ++off)
        for (int d = 0; d < head_dim; ++d) {
          size_t from = kv_offset(src[i], h, off, d, num_kv_heads, block_size, head_dim);
          size_t to = kv_offset(dst[i], h, off, d, num_kv_heads, block_size, head_dim);
          k_cache[to] = k_cache[from];
          v_cache[to] = v_cache[from];
        }
  }
  return skipped;
}

/* Shared argument bundle for the attention definition. */
typedef struct {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int max_blocks_per_req;
  const int32_t* seq_lens;
  const int32_t* qo_indptr;
  int num_reqs, Hq, Hkv, D, p;
  double sm_scale;
  const uint8_t* kq;  /* q8_0 pages instead of k_cache / v_cache, or NULL */
  const uint8_t* vq;
} attn_args;

/* Element d of token `off` of block `block`, kv head kvh, of the K
 * (which = 0) or V (which = 1) cache: a bf16 value, or a q8_0 code times
 * its group's scale. */
static double kv_elem(const attn_args* a, int which, int64_t block, int kvh, int off, int d) {
  if (a->kq) return q8_elem(which ? a->vq : a->kq, block, kvh, off, d, a->Hkv, a->p, a->D);
  const uint16_t* c = which ? a->v_cache : a->k_cache;
  return bf16_to_double(c[kv_offset(block, kvh, off, d, a->Hkv, a->p, a->D)]);
}

/*
 * One output element set: query token `tok` (global index into q) of
 * request r, query head h.  Writes o[0..D) and *lse.  `s` is scratch for
 * seq_len scores.  Returns ORACLE_ERR_INDEX on a block id outside the pool.
 */
static int attend_one(const attn_args* a, int r, int tok, int h, double* s, double* o, double* lse) {
  int qo_len = a->qo_indptr[r + 1] - a->qo_indptr[r];
  int seq_len = a->seq_lens[r];
  int j = tok - a->qo_indptr[r];
  int pos = seq_len - qo_len + j;    /* absolute position of this query */
  int n_keys = pos + 1;              /* causal: keys 0 .. pos */
  int G = a->Hq / a->Hkv;
  int kvh = h / G;                   /* contiguous GQA groups */
  const uint16_t* qv = a->q + ((size_t)tok * (size_t)a->Hq + (size_t)h) * (size_t)a->D;
  const int32_t* table = a->block_tables + (size_t)r * (size_t)a->max_blocks_per_req;

  /* scores s_t = scale * <q, K[t]> over the gathered keys */
  double m = -INFINITY;
  for (int t = 0; t < n_keys; ++t) {
    int64_t block = table[t / a->p];
    if (block < 0 || block >= a->num_blocks) return ORACLE_ERR_INDEX;
    double dot = 0.0;
    for (int d = 0; d < a->D; ++d)
      dot += bf16_to_double(qv[d]) * kv_elem(a, 0, block, kvh, t % a->p, d);
    s[t] = a->sm_scale * dot;
    if (s[t] > m) m = s[t];
  }
  /* softmax weights and the weighted sum of values */
  double l = 0.0;
  for (int d = 0; d < a->D; ++d) o[d] = 0.0;
  for (int t = 0; t < n_keys; ++t) {
    int64_t block = table[t / a->p];
    double w = exp(s[t] - m);
    l += w;
    for (int d = 0; d < a->D; ++d)
      o[d] += w * kv_elem(a, 1, block, kvh, t % a->p, d);
  }
  for (int d = 0; d < a->D; ++d) o[d] /= l;
  *lse = m + log(l);
  return ORACLE_OK;
}

static int check_args(const attn_args* a) {
  if (a->num_reqs < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->D <= 0 || a->p <= 0) return ORACLE_ERR_ARG;
  if (a->Hq % a->Hkv != 0) return ORACLE_ERR_ARG;
  if (a->num_reqs > 0 && a->qo_indptr[0] != 0) return ORACLE_ERR_ARG;
  for (int r = 0; r < a->num_reqs; ++r) {
    int qo_len = a->qo_indptr[r + 1] - a->qo_indptr[r];
    if (qo_len < 0 || qo_len > a->seq_lens[r]) return ORACLE_ERR_ARG;
    if ((a->seq_lens[r] + a->p - 1) / a->p > a->max_blocks_per_req) return ORACLE_ERR_ARG;
  }
  return ORACLE_OK;
}

static int request_of(const attn_args* a, int tok) {
  for (int r = 0; r < a->num_reqs; ++r)
    if (tok >= a->qo_indptr[r] && tok < a->qo_indptr[r + 1]) return r;
  return -1;
}

/*
 * Full attention over a varlen batch: out[total_q, Hq, D] and
 * lse[total_q, Hq] in fp64 (lse may be NULL).  `scratch` must hold
 * n_threads * max_seq_len doubles for the scores; the caller provides it so
 * this file allocates nothing.
 */
static int attention_all(const attn_args* a, double* out, double* lse, double* scratch, int max_seq_len,
                         int n_threads) {
  int rc = check_args(a);
  if (rc) return rc;
  for (int r = 0; r < a->num_reqs; ++r)
    if (a->seq_lens[r] > max_seq_len) return ORACLE_ERR_ARG;
  int total_q = a->num_reqs > 0 ? a->qo_indptr[a->num_reqs] : 0;
  long n_items = (long)total_q * a->Hq;
  int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 4) num_threads(n_threads)
  for (long it = 0; it < n_items; ++it) {
    int tok = (int)(it / a->Hq), h = (int)(it % a->Hq);
#ifdef _OPENMP
    double* s = scratch + (size_t)omp_get_thread_num() * (size_t)max_seq_len;
#else
    double* s = scratch;
#endif
    double l_out;
    int e = attend_one(a, request_of(a, tok), tok, h, s, out + (size_t)it * (size_t)a->D, &l_out);
    if (lse) lse[it] = l_out;
    if (e) {
#pragma omp atomic write
      err = e;
    }
  }
  return err;
}

int oracle_attention_varlen(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_blocks,
                            const int32_t* block_tables, int max_blocks_per_req, const int32_t* seq_lens,
                            const int32_t* qo_indptr, int num_reqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, double sm_scale, double* out, double* lse, double* scratch,
                            int max_seq_len, int n_threads) {
  attn_args a = {q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                 num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, sm_scale, NULL, NULL};
  return attention_all(&a, out, lse, scratch, max_seq_len, n_threads);
}

/* The same definition over q8_0 pages (each K and V element is its code
 * times its group's scale). */
int oracle_attention_varlen_q8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache, int64_t num_blocks,
                               const int32_t* block_tables, int max_blocks_per_req, const int32_t* seq_lens,
                               const int32_t* qo_indptr, int num_reqs, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, double sm_scale, double* out, double* lse,
                               double* scratch, int max_seq_len, int n_threads) {
  if (head_dim % 32) return ORACLE_ERR_ARG;
  attn_args a = {q, NULL, NULL, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                 num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, sm_scale, k_cache, v_cache};
  return attention_all(&a, out, lse, scratch, max_seq_len, n_threads);
}

/*
 * The same definition evaluated only at a list of (query token, head)
 * samples, so that full-size batches can be checked one output at a time.
 * out[n_samples, D], lse[n_samples].
 */
int oracle_attention_sampled(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_blocks,
                             const int32_t* block_tables, int max_blocks_per_req, const int32_t* seq_lens,
                             const int32_t* qo_indptr, int num_reqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, double sm_scale, int n_samples, const int32_t* sample_tok,
                             const int32_t* sample_head, double* out, double* lse, double* scratch, int max_seq_len,
                             int n_threads) {
  attn_args a = {q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                 num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, sm_scale, NULL, NULL};
  int rc = check_args(&a);
  if (rc) return rc;
  for (int r = 0; r < num_reqs; ++r)
    if (seq_lens[r] > max_seq_len) return ORACLE_ERR_ARG;
  int total_q = num_reqs > 0 ? qo_indptr[num_reqs] : 0;
  for (int i = 0; i < n_samples; ++i)
    if (sample_tok[i] < 0 || sample_tok[i] >= total_q || sample_head[i] < 0 || sample_head[i] >= num_q_heads)
      return ORACLE_ERR_ARG;
  int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
  for (int i = 0; i < n_samples; ++i) {
#ifdef _OPENMP
    double* s = scratch + (size_t)omp_get_thread_num() * (size_t)max_seq_len;
#else
    double* s = scratch;
#endif
    int e = attend_one(&a, request_of(&a, sample_tok[i]), sample_tok[i], sample_head[i], s,
                       out + (size_t)i * (size_t)head_dim, &lse[i]);
    if (e) {
#pragma omp atomic write
      err = e;
    }
  }
  return err;
}

/*
 * LSE merge of two partial attentions (o_a, lse_a) and (o_b, lse_b) over
 * disjoint key sets A and B of the same query:
 *   M = max(lse_a, lse_b), w_a = exp(lse_a - M), w_b = exp(lse_b - M),
 *   o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = M + log(w_a + w_b).
 * An empty part has lse = -inf and weight 0; if both are empty the result is
 * o = 0, lse = -inf.  Inputs o are bf16 patterns; outputs are fp64.
 */
int oracle_merge_lse(const uint16_t* o_a, const double* lse_a, const uint16_t* o_b, const double* lse_b,
                     double* o_out, double* lse_out, int64_t rows, int num_heads, int head_dim) {
  if (rows < 0 || num_heads <= 0 || head_dim <= 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < rows * num_heads; ++i) {
    double la = lse_a[i], lb = lse_b[i];
    double M = la > lb ? la : lb;
    if (M == -INFINITY) {
      for (int d = 0; d < head_dim; ++d) o_out[i * head_dim + d] = 0.0;
      lse_out[i] = -INFINITY;
      continue;
    }
    double wa = exp(la - M), wb = exp(lb - M);
    for (int d = 0; d < head_dim; ++d) {
      double va = bf16_to_double(o_a[i * head_dim + d]);
      double vb = bf16_to_double(o_b[i * head_dim + d]);
      /* a part with weight 0 contributes nothing, whatever its o holds */
      double ta = wa > 0.0 ? wa * va : 0.0, tb = wb > 0.0 ? wb * vb : 0.0;
      o_out[i * head_dim + d] = (ta + tb) / (wa + wb);
    }
    lse_out[i] = M + log(wa + wb);
  }
  return ORACLE_OK;
}
