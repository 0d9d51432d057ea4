"""Seeded synthetic batches for paged varlen attention.

This module only builds inputs: a KV pool with pages placed by a seeded
random permutation, block tables, sequence lengths, query offsets, query and
new-token tensors, and the slots the new tokens go to.  It holds none of the
attention arithmetic; both the CUDA path and the CPU oracle consume what it
produces.

Recipe (all values are exact bf16 bit patterns, numpy ``uint16``):

* q, k_new, v_new and every cached token before this step are i.i.d.
  N(0, 1), drawn in float32 from ``numpy.random.default_rng(seed)`` and
  rounded to bf16 (nearest even).
* Pool blocks are handed out in the order of one random permutation of the
  pool; shared-prefix blocks are taken first and referenced by every request
  that shares them, then each request takes its private blocks.
* Slots that hold no valid token (unused blocks, the tail of a request's last
  block, and the slots this step's new tokens will be written to) hold finite
  sentinels (K = 8.0, V = 512.0), so a read outside a request's keys or a
  missing append shows up as a large error.
* seq_lens[r] is the KV length after this step's append; the request's
  qo_len new tokens occupy positions seq_len - qo_len .. seq_len - 1, and
  slot_mapping gives each new token its (block, offset) slot as
  block * page_size + offset.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

K_SENTINEL = 0x4100   # bf16 8.0
V_SENTINEL = 0x4400   # bf16 512.0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def _to_bf16_bits_fast(x: np.ndarray) -> np.ndarray:
    """Same rounding as f32_to_bf16_bits (nearest even), via torch when it is
    importable (several times faster on large arrays)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        return f32_to_bf16_bits(x)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """i.i.d. N(0,1) rounded to bf16, generated in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = _to_bf16_bits_fast(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclass
class Batch:
    q: np.ndarray              # uint16 [total_q, Hq, D]
    k_cache: np.ndarray        # uint16 [num_blocks, Hkv, P, D]  (state before this step's append)
    v_cache: np.ndarray        # uint16 [num_blocks, Hkv, P, D]
    block_tables: np.ndarray   # int32 [num_reqs, max_blocks]; -1 past each request's pages
    seq_lens: np.ndarray       # int32 [num_reqs]
    qo_indptr: np.ndarray      # int32 [num_reqs + 1]
    k_new: np.ndarray          # uint16 [total_q, Hkv, D]
    v_new: np.ndarray          # uint16 [total_q, Hkv, D]
    slot_mapping: np.ndarray   # int64 [total_q]
    sm_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])


def make_batch(seq_lens, qo_lens, *, num_blocks: int, seed: int, num_q_heads: int = 32, num_kv_heads: int = 8,
               head_dim: int = 128, page_size: int = 16, shared_prefix_tokens: int = 0,
               sm_scale: float | None = None, fill_pool: bool = True) -> Batch:
    """Build one step's batch.

    seq_lens / qo_lens: per request; qo_len = 1 is a decode row, > 1 a
    chunked-prefill row, 0 a request with no query this step.
    shared_prefix_tokens: the first tokens of every request, a multiple of
    page_size, stored once in shared blocks (requests must be at least that
    long)."""
    seq_lens = np.asarray(seq_lens, np.int64)
    qo_lens = np.asarray(qo_lens, np.int64)
    R = seq_lens.shape[0]
    if qo_lens.shape[0] != R:
        raise ValueError("seq_lens and qo_lens differ in length")
    if np.any(qo_lens < 0) or np.any(qo_lens > seq_lens):
        raise ValueError("need 0 <= qo_len <= seq_len")
    if shared_prefix_tokens % page_size:
        raise ValueError("shared prefix must be whole pages")
    if R and shared_prefix_tokens and np.any(seq_lens - qo_lens < shared_prefix_tokens):
        raise ValueError("the shared prefix must be cached before this step")
    rng = np.random.default_rng(seed)
    Hkv, D, P = num_kv_heads, head_dim, page_size

    pages = [-(-int(L) // P) for L in seq_lens]
    n_shared = shared_prefix_tokens // P
    need = n_shared + sum(p - n_shared for p in pages) if R else 0
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need} pages")
    perm = rng.permutation(num_blocks).astype(np.int64)
    shared_ids = perm[:n_shared]
    nxt = n_shared
    max_blocks = max(pages) if R else 1
    tables = np.full((R, max(max_blocks, 1)), -1, np.int32)
    for r in range(R):
        own = pages[r] - n_shared
        tables[r, :n_shared] = shared_ids
        tables[r, n_shared:pages[r]] = perm[nxt:nxt + own]
        nxt += own

    k_cache = np.full((num_blocks, Hkv, P, D), K_SENTINEL, np.uint16)
    v_cache = np.full((num_blocks, Hkv, P, D), V_SENTINEL, np.uint16)
    if fill_pool:
        # cached tokens (positions before this step's new ones), page by page;
        # shared pages are written once, by the first request.
        written = set()
        full, partial = [], []
        for r in range(R):
            old = int(seq_lens[r] - qo_lens[r])
            for i in range(-(-old // P)):
                blk = int(tables[r, i])
                if blk in written and i < n_shared:
                    continue
                written.add(blk)
                n_tok = min(P, old - i * P)
                (full if n_tok == P else partial).append((blk, n_tok))
        ids = np.array([blk for blk, _ in full], np.int64)
        for s in range(0, len(ids), 4096):   # whole pages, in bounded batches
            part = ids[s:s + 4096]
            k_cache[part] = normal_bf16(rng, (len(part), Hkv, P, D))
            v_cache[part] = normal_bf16(rng, (len(part), Hkv, P, D))
        for blk, n_tok in partial:
            k_cache[blk, :, :n_tok, :] = normal_bf16(rng, (Hkv, n_tok, D))
            v_cache[blk, :, :n_tok, :] = normal_bf16(rng, (Hkv, n_tok, D))

    qo_indptr = np.zeros(R + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    total_q = int(qo_indptr[-1])
    q = normal_bf16(rng, (total_q, num_q_heads, D))
    k_new = normal_bf16(rng, (total_q, Hkv, D))
    v_new = normal_bf16(rng, (total_q, Hkv, D))
    slot_mapping = np.empty(total_q, np.int64)
    for r in range(R):
        for j in range(int(qo_lens[r])):
            pos = int(seq_lens[r] - qo_lens[r]) + j
            slot_mapping[qo_indptr[r] + j] = int(tables[r, pos // P]) * P + pos % P
    if sm_scale is None:
        sm_scale = 1.0 / float(np.sqrt(D))
    return Batch(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables, seq_lens=seq_lens.astype(np.int32),
                 qo_indptr=qo_indptr, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping, sm_scale=sm_scale,
                 meta=dict(seed=seed, num_blocks=num_blocks, shared_prefix_tokens=shared_prefix_tokens,
                           pages_used=need))


# ---------------------------------------------------------------------------
# The five workloads (one layer each; the 36-layer sweep repeats a layer).
# Pool sizes: 12 GiB over 36 layers is 5461 blocks of 64 KiB per layer; the
# short-dialogue batch needs ~8.7k pages, so its pool is doubled to 10,922,
# and the mixed batch gets 24,576 blocks.
# ---------------------------------------------------------------------------
SEED0 = 20261202
POOL_12GIB_PER_LAYER = 5461
_WL_SEED = {"tiny": 1, "short": 2, "shared": 3, "mixed": 4, "verify": 6}


def workload(name: str, *, scale: float = 1.0, seed_offset: int = 0) -> dict:
    """Length recipe of a named workload.  `scale` < 1 shrinks request
    counts for quick parity runs while keeping the length mix."""
    rng = np.random.default_rng(SEED0 + _WL_SEED[name] + seed_offset)
    if name == "tiny":
        seq = [17, 100, 256, 513]
        return dict(seq_lens=seq, qo_lens=[1] * 4, num_blocks=64, shared_prefix_tokens=0)
    if name == "short":
        n = max(1, int(round(64 * scale)))
        seq = rng.integers(2048, 2303 + 1, n).tolist()
        return dict(seq_lens=seq, qo_lens=[1] * n, num_blocks=2 * POOL_12GIB_PER_LAYER, shared_prefix_tokens=0)
    if name == "shared":
        n = max(1, int(round(16 * scale)))
        seq = rng.integers(8192, 8447 + 1, n).tolist()
        return dict(seq_lens=seq, qo_lens=[1] * n, num_blocks=POOL_12GIB_PER_LAYER, shared_prefix_tokens=6144)
    if name == "mixed":
        n = max(1, int(round(63 * scale)))
        seq = [2048] + rng.integers(2048, 8192 + 1, n).tolist()
        return dict(seq_lens=seq, qo_lens=[512] + [1] * n, num_blocks=24576, shared_prefix_tokens=0)
    if name == "verify":
        # speculative verification ("Inference optimisation" §8.5.1): each of
        # the short-dialogue requests checks a 4-token draft, i.e. 5 query
        # tokens (the 4 drafts and the token after them) over its context
        n = max(1, int(round(64 * scale)))
        seq = rng.integers(2048, 2303 + 1, n).tolist()
        return dict(seq_lens=seq, qo_lens=[5] * n, num_blocks=2 * POOL_12GIB_PER_LAYER, shared_prefix_tokens=0)
    raise KeyError(name)


def workload_batch(name: str, *, scale: float = 1.0, seed_offset: int = 0, **kw) -> Batch:
    spec = workload(name, scale=scale, seed_offset=seed_offset)
    seed = SEED0 + 100 + _WL_SEED[name] + seed_offset
    return make_batch(spec["seq_lens"], spec["qo_lens"], num_blocks=spec["num_blocks"], seed=seed,
                      shared_prefix_tokens=spec["shared_prefix_tokens"], **kw)


def sweep_point(batch: int, context: int, *, seed: int = SEED0 + 5) -> dict:
    """One point of the 36-layer decode sweep: `batch` decode rows at
    `context` tokens; 8192-token rows share a 6144-token prefix.  The pool is
    what the batch needs plus 10 % (the 12 GiB budget is exceeded at the
    larger points)."""
    shared = 6144 if context == 8192 else 0
    pages = -(-context // 16)
    need = shared // 16 + batch * (pages - shared // 16)
    return dict(seq_lens=[context] * batch, qo_lens=[1] * batch, num_blocks=int(need * 1.1) + 1,
                shared_prefix_tokens=shared, seed=seed)


# ---------------------------------------------------------------------------
# Byte accounting of one step (per layer), for throughput figures.
#   KV: 2 (K, V) x kv heads x head_dim x 2 B = 4096 B per token per layer
#   (for 8 kv heads, 128 dims).  Unique bytes count each physical page once
#   (whole pages of shared prefixes, exact tokens of private tails); logical
#   bytes count every request's keys.  q and out: total_q x Hq x D x 2 B each.
#   Block table: 4 B per page read.  Append: k_new + v_new read and written
#   (4 x Hkv x D x 2 B... i.e. 2 x 4096 B per token) plus the 8-byte slot.
# Split-KV partial results are implementation overhead and are not counted.
# With prefix_pages > 0 (the shared-prefix call) the decode kernel reads only
# the pages after the prefix, and the prefix pass reads the prefix pages once
# plus every query.
# ---------------------------------------------------------------------------
def step_bytes(b: Batch, prefix_pages: int = 0, kv: str = "bf16") -> dict:
    """kv = "q8": the pools hold q8_0 pages ("Inference optimisation"
    §8.4.2): 34 bytes per 32 values instead of 64."""
    total_q, Hq, D = b.q.shape
    _, Hkv, P, _ = b.k_cache.shape
    per_tok = 2 * Hkv * D * 2 if kv == "bf16" else 2 * Hkv * (D + D // 32 * 2)
    new_tok = 2 * Hkv * D * 2           # the step's new K/V arrive as bf16
    qo = np.diff(b.qo_indptr)
    active = qo > 0
    seq = b.seq_lens.astype(np.int64)
    logical_kv = int((seq[active] * per_tok).sum())
    # unique: tokens held by distinct physical pages that active rows read
    seen = {}
    for r in np.nonzero(active)[0]:
        L = int(seq[r])
        for i in range(-(-L // P)):
            blk = int(b.block_tables[r, i])
            seen[blk] = max(seen.get(blk, 0), min(P, L - i * P))
    unique_kv = sum(seen.values()) * per_tok
    decode = active & (qo == 1)
    qo_bytes = 2 * total_q * Hq * D * 2
    table_bytes = int(sum(4 * (-(-int(L) // P)) for L in seq[active]))
    meta_bytes = 8 * len(seq) + 4
    append_bytes = int((b.slot_mapping >= 0).sum()) * (new_tok + per_tok + 8)
    dec_seen = {}
    for r in np.nonzero(decode)[0]:
        L = int(seq[r])
        for i in range(prefix_pages, -(-L // P)):
            blk = int(b.block_tables[r, i])
            dec_seen[blk] = max(dec_seen.get(blk, 0), min(P, L - i * P))
    decode_kv_unique = sum(dec_seen.values()) * per_tok
    n_dec = int(decode.sum())
    # per decode row: its K/V pages, q read and out written (Hq x D bf16
    # each), one 4-byte block-table entry per page; split partials are
    # implementation overhead and not counted
    decode_kernel = decode_kv_unique + 2 * n_dec * Hq * D * 2 + int(
        sum(4 * (-(-int(L) // P) - prefix_pages) for L in seq[decode]))
    prefix_kernel = prefix_pages * P * per_tok + total_q * Hq * D * 2 + 4 * prefix_pages if prefix_pages else 0
    # tensor-core tile kernel (rows with qo_len > 1): the keys each row reads
    # once per kv head (after the prefix), its q, its table entries; flops
    # of the causal QK^T and PV products (2 x 2 flop per pair, head and dim)
    pre_kv, pre_q, pre_tab, pre_flops = 0, 0, 0, 0
    for r in np.nonzero(qo > 1)[0]:
        L, c = int(seq[r]), int(qo[r])
        h = L - c
        pre_kv += (L - prefix_pages * P) * per_tok
        pre_q += 2 * c * Hq * D * 2          # q read, out written
        pre_tab += 4 * (-(-L // P) - prefix_pages)
        pre_flops += (c * h + c * (c + 1) // 2) * Hq * D * 4
    prefill_kernel = pre_kv + pre_q + pre_tab
    # the decode step's one kernel (pa_decode_step): the decode kernel's
    # bytes plus the append of every row's new token (read as bf16, written
    # into its page) and the seq_lens it plans from
    step_kernel = decode_kernel + n_dec * (new_tok + per_tok) + 4 * len(seq)
    return dict(unique=unique_kv + qo_bytes + table_bytes + meta_bytes + append_bytes,
                logical=logical_kv + qo_bytes + table_bytes + meta_bytes + append_bytes,
                unique_kv=unique_kv, logical_kv=logical_kv, decode_kernel=decode_kernel,
                prefix_kernel=prefix_kernel, prefill_kernel=prefill_kernel, prefill_flops=pre_flops,
                step_kernel=step_kernel,
                query_tokens=int(total_q))
