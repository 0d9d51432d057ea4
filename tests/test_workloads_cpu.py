"""The seeded synthetic workloads the parity tests and bench.py run: their
shapes and length mixes as the bench lines describe them, the pool sized from
the pages' 12 GiB budget, shared prefixes stored once, and slots that follow
the block table.  Runs without a GPU."""
import functools

import numpy as np
import pytest

from paged_kv_decode_varlen_gb300 import workloads as W


@functools.lru_cache(maxsize=None)
def _batch(name):
    return W.workload_batch(name)


@pytest.fixture(scope="module", autouse=True)
def _free_batches():
    yield
    _batch.cache_clear()  # the full-size pools (~1.7 GB) are not kept for later modules


def _rows(b):
    seq = b.seq_lens.astype(np.int64)
    qo = np.diff(b.qo_indptr)
    return seq, qo


def test_pool_from_the_12_gib_budget():
    # 147,456 B per token over 36 layers ("Inference optimisation" §8.3.1):
    # 12 GiB holds 87,381 tokens, i.e. 5,461 sixteen-token blocks per layer
    assert W.POOL_12GIB_PER_LAYER == (12 << 30) // 147456 // 16 == 5461


def test_short_dialogue():
    b = _batch("short")
    seq, qo = _rows(b)
    assert len(seq) == 64 and np.all(qo == 1)
    assert seq.min() >= 2048 and seq.max() <= 2303
    assert b.k_cache.shape == (10922, 8, 16, 128) and b.q.shape == (64, 32, 128)


def test_shared_prefix_long_context():
    b = _batch("shared")
    seq, qo = _rows(b)
    assert len(seq) == 16 and np.all(qo == 1) and seq.min() >= 8192 and seq.max() <= 8447
    # the 6,144-token prefix (384 pages) is one set of physical blocks, the
    # tails are private
    assert np.all(b.block_tables[:, :384] == b.block_tables[0, :384])
    tails = [set(b.block_tables[r, 384:-(-int(seq[r]) // 16)].tolist()) for r in range(16)]
    assert all(not (tails[i] & tails[j]) for i in range(16) for j in range(i))
    assert not (set(b.block_tables[0, :384].tolist()) & set().union(*tails))


def test_mixed_chunked_prefill():
    b = _batch("mixed")
    seq, qo = _rows(b)
    assert len(seq) == 64 and qo[0] == 512 and seq[0] == 2048 and np.all(qo[1:] == 1)
    assert seq[1:].min() >= 2048 and seq[1:].max() <= 8192
    assert b.k_cache.shape[0] == 24576


def test_verify_rows():
    b = _batch("verify")
    seq, qo = _rows(b)
    assert len(seq) == 64 and np.all(qo == 5) and seq.min() >= 2048 and seq.max() <= 2303


def test_tiny_and_scaled():
    assert _rows(_batch("tiny"))[0].tolist() == [17, 100, 256, 513]
    seq, qo = _rows(W.workload_batch("short", scale=0.25))
    assert len(seq) == 16 and seq.min() >= 2048 and seq.max() <= 2303


def test_slots_follow_the_block_table():
    for name in ("short", "mixed", "verify", "shared"):
        b = _batch(name)
        seq, qo = _rows(b)
        i = 0
        for r in range(len(seq)):
            for pos in range(int(seq[r] - qo[r]), int(seq[r])):
                assert b.slot_mapping[i] == b.block_tables[r, pos // 16] * 16 + pos % 16, (name, r, pos)
                i += 1
        assert i == len(b.slot_mapping) == b.k_new.shape[0]


def test_seeded_and_repeatable():
    a, c = W.workload_batch("mixed", scale=0.25), W.workload_batch("mixed", scale=0.25)
    for x, y in ((a.q, c.q), (a.k_cache, c.k_cache), (a.block_tables, c.block_tables), (a.seq_lens, c.seq_lens)):
        assert np.array_equal(x, y)
    d = W.workload_batch("mixed", scale=0.25, seed_offset=1)
    assert not np.array_equal(a.q, d.q)
