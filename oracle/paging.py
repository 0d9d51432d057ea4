"""Page and byte arithmetic of a paged KV cache -- TEST INFRASTRUCTURE ONLY.

Each function states the rule it follows and where it is given:

* "Inference optimisation" (AI-infra book ch. 8), §8.1.2: KV bytes per token
  k = 2 (K and V) x layers x kv heads x head_dim x bytes per element, and the
  reservation of ceil-to-block token counts.
* same, §8.2.1: bytes read per decode round D(b, L) = D_w + b L k and the
  batch size at which KV reads reach the shared weight reads,
  b_KV = ceil(D_w / (L k)).
* same, §8.3.1: a length-L sequence needs ceil(L / p) blocks and wastes
  p ceil(L / p) - L <= p - 1 slots; shared prefix blocks are stored once.
* same, §8.3.2: physical blocks are the distinct block ids that block tables
  reference; references are all entries.
* same, §8.2.3: N_pair = c h + c (c + 1) / 2 query-key pairs for a chunk of c
  new tokens over h old ones.  The oracle's attention is pinned to this count
  through its causal mask (tests), not through this function alone.
"""
from __future__ import annotations

from typing import Iterable, Sequence

MIB = 1 << 20


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """k = 2 x layers x kv heads x head_dim x bytes per element (K and V)."""
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def blocks_needed(seq_len: int, block_size: int) -> int:
    """ceil(L / p): blocks a length-L sequence occupies."""
    return -(-seq_len // block_size)


def reserved_tokens(seq_len: int, block_size: int) -> int:
    """Token slots reserved by whole blocks: p ceil(L / p)."""
    return blocks_needed(seq_len, block_size) * block_size


def block_waste(seq_len: int, block_size: int) -> int:
    """Unused slots at the end of the last block: p ceil(L / p) - L."""
    return reserved_tokens(seq_len, block_size) - seq_len


def physical_blocks(block_tables: Iterable[Sequence[int]]) -> int:
    """Distinct physical blocks referenced by a set of block tables."""
    seen = set()
    for table in block_tables:
        seen.update(int(b) for b in table)
    return len(seen)


def references(block_tables: Iterable[Sequence[int]]) -> int:
    """Block-table entries (references), shared blocks counted once per table."""
    return sum(len(t) for t in block_tables)


def capacity(budget_bytes: int, per_request_bytes: int, shared_bytes: int = 0) -> int:
    """Requests of a given footprint that fit a budget after a shared part."""
    return (budget_bytes - shared_bytes) // per_request_bytes


def round_read_bytes(weight_bytes: int, batch: int, context_len: int, k: int) -> int:
    """D(b, L) = D_w + b L k: bytes read per decode round with no shared KV."""
    return weight_bytes + batch * context_len * k


def batch_where_kv_reaches_weights(weight_bytes: int, context_len: int, k: int) -> int:
    """b_KV = ceil(D_w / (L k))."""
    return -(-weight_bytes // (context_len * k))


def pair_count(c: int, h: int) -> int:
    """N_pair = c h + c (c + 1) / 2 for c new tokens over h old ones."""
    return c * h + c * (c + 1) // 2
