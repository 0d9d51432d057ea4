"""Pins for the CPU oracle: checks against what the pages and mathematics
fix, never against the oracle's own formula retyped.

Each pin is a function taking an ``oracle.Oracle`` and raising
AssertionError on failure, so the same pins can be run against deliberately
mutated copies of the oracle (tests/test_oracle_mutations.py) to show that a
plausible mistake anywhere in it fails at least one of them.

Run as a script (``python -m tests.oracle_pins LIB``) it loads LIB, runs every
pin and exits with the number of pins that failed.
"""
from __future__ import annotations

import json
import math
import os
import sys

import numpy as np
from scipy import special

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from oracle import paging  # noqa: E402
from paged_kv_decode_varlen_gb300 import workloads  # noqa: E402

GOLDEN = json.load(open(os.path.join(HERE, "golden", "page_arithmetic.json")))
f64 = oracle.bf16_to_f64


def bits(x) -> int:
    """bf16 bit pattern of one value (round to nearest even)."""
    return int(workloads.f32_to_bf16_bits(np.array([x], np.float32))[0])


def _pool(num_blocks, Hkv, P, D, rng):
    k = workloads.normal_bf16(rng, (num_blocks, Hkv, P, D))
    v = workloads.normal_bf16(rng, (num_blocks, Hkv, P, D))
    return k, v


def _tables(rng, num_blocks, seq_lens, P):
    perm = rng.permutation(num_blocks)
    pages = [-(-L // P) for L in seq_lens]
    t = np.full((len(seq_lens), max(pages)), -1, np.int32)
    nxt = 0
    for r, n in enumerate(pages):
        t[r, :n] = perm[nxt:nxt + n]
        nxt += n
    return t


def _indptr(qo_lens):
    return np.concatenate([[0], np.cumsum(qo_lens)]).astype(np.int32)


def _gather(cache, table, kvh, n, P):
    """Logical rows 0..n-1 of one kv head, gathered through a block table
    (numpy fancy indexing; independent of the oracle's loops)."""
    t = np.arange(n)
    return cache[np.asarray(table)[t // P], kvh, t % P, :]


# ---------------------------------------------------------------- page maths
def pin_page_arithmetic(o=None):
    g = GOLDEN["kv_bytes_per_token"]
    k = paging.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["elem_bytes"])
    assert k == g["value"] == 144 * 1024
    for tokens, mib in GOLDEN["kv_after_prefill_mib"]["cases"]:
        assert tokens * k == mib * paging.MIB
    g = GOLDEN["reserved_after_256_outputs"]
    for c in g["cases"]:
        assert paging.reserved_tokens(c["tokens"], g["block_size"]) == c["reserved_tokens"]
        assert c["reserved_tokens"] * k == c["mib"] * paging.MIB
        assert paging.capacity(g["budget_mib"], c["mib"]) == c["capacity"]
    assert paging.capacity(g["budget_mib"], 288) == g["prefill_only_capacity_short"]
    assert g["prefill_only_capacity_short"] * 324 == g["prefill_only_short_total_after_output_mib"]
    g = GOLDEN["paged_allocation_example"]
    each = [paging.reserved_tokens(L, g["block_size"]) for L in g["lengths"]]
    assert each == g["paged_reserved_each"] and sum(each) == g["paged_reserved_total"]
    assert len(g["lengths"]) * g["max_len"] == g["contiguous_reserved"]
    assert g["contiguous_reserved"] - sum(g["lengths"]) == g["unused_contiguous"]
    assert sum(paging.block_waste(L, g["block_size"]) for L in g["lengths"]) == g["unused_paged"]
    for L in range(1, 200):
        assert 0 <= paging.block_waste(L, 16) <= 15
    # A and B share their first two 4-token blocks: build the tables and count
    p = g["block_size"]
    shared = [0, 1]
    nxt = iter(range(2, 100))
    tabs = []
    for i, L in enumerate(g["lengths"]):
        n = paging.blocks_needed(L, p)
        if i < 2:
            tabs.append(shared + [next(nxt) for _ in range(n - 2)])
        else:
            tabs.append([next(nxt) for _ in range(n)])
    assert paging.physical_blocks(tabs) * p == g["paged_reserved_with_sharing"]
    g = GOLDEN["branch_sharing"]
    tabs = [list(range(g["shared_blocks"])) + [1000 + 100 * b + i for i in range(g["private_blocks_each"])]
            for b in range(g["branches"])]
    assert paging.references(tabs) == g["references"]
    assert paging.physical_blocks(tabs) == g["physical"]
    g = GOLDEN["shared_prefix_group"]
    assert g["prefix_tokens"] * k == g["prefix_mib"] * paging.MIB
    assert paging.reserved_tokens(g["private_tokens"], 16) * k == g["private_reserved_mib"] * paging.MIB
    assert g["prefix_mib"] + g["requests"] * g["private_reserved_mib"] == g["total_mib"]
    assert g["requests"] * 1188 == g["unshared_total_mib"]
    assert paging.capacity(g["budget_mib"], 1188) == g["capacity_unshared"]
    assert paging.capacity(g["budget_mib"], g["private_reserved_mib"], g["prefix_mib"]) == g["capacity_shared"]
    for c in GOLDEN["chunk_pair_counts"]["cases"]:
        assert paging.pair_count(c["c"], c["h"]) == c["pairs"]
    g = GOLDEN["decode_round_bytes"]
    for b, gb in g["gb_by_batch"]:
        assert round(paging.round_read_bytes(g["weight_bytes"], b, g["context"], g["k"]) / 1e9, 2) == gb
    for L, b in g["b_kv"]:
        assert paging.batch_where_kv_reaches_weights(g["weight_bytes"], L, g["k"]) == b


# ------------------------------------------------------------- bf16 rounding
def pin_round_bf16(o):
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.0, 0.0, 1.0 + 2 ** -8 + 2 ** -30, 3.0e38 * 1.2])
    want = np.array([0x3F80, 0x3F80, 0x3F82, 0xC000, 0x0000, 0x3F81, 0x7F80], np.uint16)
    assert np.array_equal(o.round_bf16(x), want), o.round_bf16(x)
    # every bf16 value in [1, 2) rounds to itself; the midpoints go to even
    m = np.arange(128)
    vals = 1.0 + m / 128.0
    assert np.array_equal(o.round_bf16(vals), (0x3F80 + m).astype(np.uint16))
    mids = 1.0 + (m[:-1] + 0.5) / 128.0
    assert np.array_equal(o.round_bf16(mids), (0x3F80 + m[:-1] + (m[:-1] & 1)).astype(np.uint16))


# ------------------------------------------------------ attention: closed forms
def pin_single_key(o):
    """seq_len = 1: softmax over one key is 1, so out is V[0] exactly and
    lse is the one score."""
    rng = np.random.default_rng(1)
    Hq, Hkv, P, D = 32, 8, 16, 128
    k, v = _pool(8, Hkv, P, D, rng)
    q = np.zeros((1, Hq, D), np.uint16)
    q[0, :, 5] = bits(2.0)
    tab = np.array([[6]], np.int32)
    out, lse = o.attention_varlen(q, k, v, tab, np.array([1], np.int32), _indptr([1]), 0.125)
    for h in range(Hq):
        assert np.array_equal(o.round_bf16(out[0, h]), v[6, h // 4, 0]), h
        assert lse[0, h] == 0.125 * 2.0 * f64(k[6, h // 4, 0, 5])


def pin_one_hot_score(o):
    """One key's score far above the rest: out equals that key's V row."""
    rng = np.random.default_rng(2)
    Hq, Hkv, P, D = 8, 2, 16, 128
    L = 45
    k, v = _pool(12, Hkv, P, D, rng)
    tab = _tables(rng, 12, [L], P)
    tstar = 29
    for t in range(L):           # key t is the unit vector e_(t mod D)
        blk = tab[0, t // P]
        k[blk, :, t % P, :] = 0
        k[blk, :, t % P, t % D] = bits(1.0)
    q = np.zeros((1, Hq, D), np.uint16)
    q[0, :, tstar] = bits(4000.0)
    out, lse = o.attention_varlen(q, k, v, tab, np.array([L], np.int32), _indptr([1]), 1 / math.sqrt(D))
    blk = tab[0, tstar // P]
    for h in range(Hq):
        assert np.array_equal(o.round_bf16(out[0, h]), v[blk, h // 4, tstar % P]), h
        assert abs(lse[0, h] - 4000.0 / math.sqrt(D)) < 1e-9


def pin_two_key_sigmoid(o):
    """Two keys: out = (1 - s) V0 + s V1 with s = expit(scale q.(k1 - k0)),
    lse = logaddexp of the two scores (scipy routines)."""
    rng = np.random.default_rng(3)
    Hq, Hkv, P, D = 4, 1, 16, 8
    k, v = _pool(3, Hkv, P, D, rng)
    a, b0, b1, scale = 1.5, 0.75, -1.25, 0.3
    k[2, 0, 0, :] = 0
    k[2, 0, 1, :] = 0
    k[2, 0, 0, 0] = bits(b0)
    k[2, 0, 1, 0] = bits(b1)
    q = np.zeros((1, Hq, D), np.uint16)
    q[0, :, 0] = bits(a)
    out, lse = o.attention_varlen(q, k, v, np.array([[2]], np.int32), np.array([2], np.int32), _indptr([1]), scale)
    s = special.expit(scale * a * (b1 - b0))
    want = (1 - s) * f64(v[2, 0, 0]) + s * f64(v[2, 0, 1])
    for h in range(Hq):
        assert np.allclose(out[0, h], want, rtol=1e-13, atol=1e-13)
        assert abs(lse[0, h] - np.logaddexp(scale * a * b0, scale * a * b1)) < 1e-13


def pin_uniform_scores(o):
    """q = 0 makes every visible score 0: out is the plain mean of the visible
    V rows (gathered here with numpy) and lse = ln(number visible), so
    sum_j exp(lse_j) over a chunk is the page's N_pair."""
    rng = np.random.default_rng(4)
    Hq, Hkv, P, D = 4, 2, 16, 16
    seq, qo = [37, 64, 20], [5, 16, 1]
    k, v = _pool(16, Hkv, P, D, rng)
    tab = _tables(rng, 16, seq, P)
    ind = _indptr(qo)
    q = np.zeros((ind[-1], Hq, D), np.uint16)
    out, lse = o.attention_varlen(q, k, v, tab, np.array(seq, np.int32), ind, 0.2)
    for r in range(3):
        for j in range(qo[r]):
            n = seq[r] - qo[r] + j + 1
            for h in range(Hq):
                rows = f64(_gather(v, tab[r], h // 2, n, P))
                assert np.allclose(out[ind[r] + j, h], rows.mean(axis=0), rtol=1e-12, atol=1e-12)
                assert abs(lse[ind[r] + j, h] - math.log(n)) < 1e-12
    for c in GOLDEN["chunk_pair_counts"]["cases"]:
        cc, hh = c["c"], c["h"]
        L = hh + cc
        nb = -(-L // P)
        k1 = np.zeros((nb, 1, P, 2), np.uint16)
        v1 = np.zeros((nb, 1, P, 2), np.uint16)
        q1 = np.zeros((cc, 1, 2), np.uint16)
        _, l1 = o.attention_varlen(q1, k1, v1, np.arange(nb, dtype=np.int32)[None], np.array([L], np.int32),
                                   _indptr([cc]), 1.0)
        assert round(float(np.exp(l1).sum())) == c["pairs"], (c, float(np.exp(l1).sum()))


def pin_gqa_grouping(o):
    """Query head h reads kv head h // (Hq / Hkv): with V of kv head g set to
    the constant g + 1, every output of head h is h // 4 + 1."""
    rng = np.random.default_rng(5)
    Hq, Hkv, P, D = 32, 8, 16, 16
    k, v = _pool(6, Hkv, P, D, rng)
    for g in range(Hkv):
        v[:, g] = bits(g + 1)
    tab = _tables(rng, 6, [70], P)
    q = workloads.normal_bf16(rng, (1, Hq, D))
    out, _ = o.attention_varlen(q, k, v, tab, np.array([70], np.int32), _indptr([1]), 0.25)
    for h in range(Hq):
        assert np.allclose(out[0, h], h // 4 + 1, rtol=1e-13), h


def pin_scipy_dense(o):
    """Contiguous single request: the result equals a dense causal softmax
    attention written with scipy.special.softmax / logsumexp."""
    rng = np.random.default_rng(6)
    Hq, Hkv, P, D = 4, 1, 16, 32
    L, c = 37, 5
    nb = 3
    k, v = _pool(nb, Hkv, P, D, rng)
    q = workloads.normal_bf16(rng, (c, Hq, D))
    tab = np.arange(nb, dtype=np.int32)[None]
    out, lse = o.attention_varlen(q, k, v, tab, np.array([L], np.int32), _indptr([c]), 0.17)
    K = f64(k[:, 0].reshape(-1, D))[:L]
    V = f64(v[:, 0].reshape(-1, D))[:L]
    mask = np.arange(L)[None, :] <= (L - c + np.arange(c))[:, None]
    for h in range(Hq):
        S = 0.17 * f64(q[:, h]) @ K.T
        S = np.where(mask, S, -np.inf)
        assert np.allclose(out[:, h], special.softmax(S, axis=1) @ V, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[:, h], special.logsumexp(S, axis=1), rtol=1e-13, atol=1e-13)


# ------------------------------------------------------ attention: invariances
def _random_batch(seed, seq, qo, nblocks, Hq=8, Hkv=2, D=32, shared=0):
    b = workloads.make_batch(seq, qo, num_blocks=nblocks, seed=seed, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D, shared_prefix_tokens=shared)
    rng = np.random.default_rng(seed + 7)
    # make the new-token slots hold real values too (as after the append)
    for i, s in enumerate(b.slot_mapping):
        b.k_cache[s // 16, :, s % 16] = workloads.normal_bf16(rng, (Hkv, D))
        b.v_cache[s // 16, :, s % 16] = workloads.normal_bf16(rng, (Hkv, D))
    return b


def pin_page_permutation(o):
    """Moving pages to other physical blocks (and updating the block tables)
    changes nothing, bit for bit."""
    b = _random_batch(11, [40, 17, 66], [1, 9, 1], 20)
    base = o.attention_varlen(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    perm = np.random.default_rng(12).permutation(20)
    k2 = np.empty_like(b.k_cache)
    v2 = np.empty_like(b.v_cache)
    k2[perm] = b.k_cache
    v2[perm] = b.v_cache
    t2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    moved = o.attention_varlen(b.q, k2, v2, t2, b.seq_lens, b.qo_indptr, b.sm_scale)
    assert np.array_equal(base[0], moved[0]) and np.array_equal(base[1], moved[1])


def pin_shared_equals_duplicated(o):
    """Requests whose prefix blocks are shared give the same result as the
    same requests with private copies of those blocks."""
    b = _random_batch(13, [70, 55, 90], [1, 1, 4], 40, shared=48)
    assert b.block_tables[0, 0] == b.block_tables[1, 0] == b.block_tables[2, 0]
    base = o.attention_varlen(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    k2, v2, t2 = b.k_cache.copy(), b.v_cache.copy(), b.block_tables.copy()
    used = set(int(x) for x in b.block_tables.ravel() if x >= 0)
    free = [i for i in range(40) if i not in used]
    for r in (1, 2):
        for i in range(3):
            nb = free.pop()
            k2[nb], v2[nb] = b.k_cache[t2[r, i]], b.v_cache[t2[r, i]]
            t2[r, i] = nb
    assert paging.physical_blocks([t[t >= 0] for t in t2]) == paging.physical_blocks(
        [t[t >= 0] for t in b.block_tables]) + 6
    dup = o.attention_varlen(b.q, k2, v2, t2, b.seq_lens, b.qo_indptr, b.sm_scale)
    assert np.array_equal(base[0], dup[0]) and np.array_equal(base[1], dup[1])


def pin_chunked_equals_oneshot(o):
    """A prefill done as chunks at increasing offsets equals the one-shot
    prefill, row by row (bit for bit)."""
    rng = np.random.default_rng(14)
    Hq, Hkv, P, D = 8, 2, 16, 32
    L = 96
    k, v = _pool(8, Hkv, P, D, rng)
    tab = _tables(rng, 8, [L], P)
    q = workloads.normal_bf16(rng, (L, Hq, D))
    full, full_lse = o.attention_varlen(q, k, v, tab, np.array([L], np.int32), _indptr([L]), 0.2)
    for off, c in [(0, 32), (32, 16), (48, 40), (88, 8)]:
        part, part_lse = o.attention_varlen(q[off:off + c], k, v, tab, np.array([off + c], np.int32), _indptr([c]),
                                            0.2)
        assert np.array_equal(part, full[off:off + c]) and np.array_equal(part_lse, full_lse[off:off + c])


def pin_merge_identity(o):
    """Attention over keys [0, a) and [a, L) separately, merged by LSE, equals
    attention over all L keys (the log-sum-exp identity).  Merge inputs are
    bf16, so o agrees to bf16 rounding; lse agrees to fp64 rounding."""
    rng = np.random.default_rng(15)
    Hq, Hkv, P, D = 8, 2, 16, 64
    L, a = 80, 48
    k, v = _pool(10, Hkv, P, D, rng)
    tab = _tables(rng, 10, [L], P)
    q = workloads.normal_bf16(rng, (1, Hq, D))
    full, full_lse = o.attention_varlen(q, k, v, tab, np.array([L], np.int32), _indptr([1]), 0.2)
    o1, l1 = o.attention_varlen(q, k, v, tab, np.array([a], np.int32), _indptr([1]), 0.2)
    o2, l2 = o.attention_varlen(q, k, v, tab[:, a // P:], np.array([L - a], np.int32), _indptr([1]), 0.2)
    m, ml = o.merge_lse(o.round_bf16(o1), l1, o.round_bf16(o2), l2)
    assert np.allclose(ml, full_lse, rtol=1e-13, atol=1e-13)
    assert np.max(np.abs(m - full)) <= 2 ** -8 * max(np.abs(o1).max(), np.abs(o2).max())
    # an empty part (lse = -inf) has weight zero, whatever its o holds
    junk = np.full_like(o.round_bf16(o1), 0x7FC0)
    m2, l2b = o.merge_lse(o.round_bf16(o1), l1, junk, np.full_like(l1, -np.inf))
    assert np.array_equal(m2, f64(o.round_bf16(o1))) and np.array_equal(l2b, l1)
    m3, l3 = o.merge_lse(junk, np.full_like(l1, -np.inf), junk, np.full_like(l1, -np.inf))
    assert np.all(m3 == 0) and np.all(l3 == -np.inf)


def pin_append_then_read(o):
    """kv_append writes each new token where attention later reads it: after
    the append, a query aimed at that token's key returns that token's V;
    negative slots write nothing; a slot beyond the pool is an error."""
    Hq, Hkv, P, D = 8, 2, 16, 128
    b = workloads.make_batch([20, 33, 16], [1, 3, 1], num_blocks=12, seed=16, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D)
    k, v = b.k_cache.copy(), b.v_cache.copy()
    k[:] = 0                       # cached keys score 0 against the probes below
    k_before = k.copy()
    slots = b.slot_mapping.copy()
    slots_skip = slots.copy()
    slots_skip[2] = -1
    k_new = b.k_new.copy()
    for i in range(len(slots)):       # key i is 4 e_(i), others never look like it
        k_new[i] = 0
        k_new[i, :, i] = bits(1.0)
    o.kv_append(k_new, b.v_new, slots_skip, k, v)
    changed = np.argwhere((k != k_before).any(axis=-1))
    assert len(changed) == (len(slots) - 1) * Hkv          # one (block, head, offset) row per token and head
    q = np.zeros((b.total_q, Hq, D), np.uint16)
    for i in range(b.total_q):
        q[i, :, i] = bits(4000.0)
    out, _ = o.attention_varlen(q, k, v, b.block_tables, b.seq_lens, b.qo_indptr, 1 / math.sqrt(D))
    for i in range(b.total_q):
        if i == 2:
            continue
        for h in range(Hq):
            assert np.array_equal(o.round_bf16(out[i, h]), b.v_new[i, h // 4]), (i, h)
    # a token whose slot is negative alone: the pool is left as it was (no
    # other token's write could hide a stray one)
    k_alone, v_alone = k.copy(), v.copy()
    o.kv_append(k_new[2:3], b.v_new[2:3], np.array([-1], np.int64), k_alone, v_alone)
    assert np.array_equal(k_alone, k) and np.array_equal(v_alone, v)
    bad = slots.copy()
    bad[0] = 12 * P
    try:
        o.kv_append(k_new, b.v_new, bad, k, v)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("slot beyond the pool was accepted")


def pin_copy_on_write(o):
    """Copy-on-write of a shared tail block ("Inference optimisation"
    §8.3.2, Fig. 8-15): two branches share every block, the last one only
    partly filled; branch B copies that tail block, then each branch appends
    its own next token.  Each branch must then attend exactly as if it had
    private copies of every block, and the shared blocks are untouched.
    Pairs naming a block outside the pool are skipped and counted."""
    Hq, Hkv, P, D = 8, 2, 16, 32
    rng = np.random.default_rng(19)
    nb = 12
    k = workloads.normal_bf16(rng, (nb, Hkv, P, D))
    v = workloads.normal_bf16(rng, (nb, Hkv, P, D))
    shared = np.array([3, 7, 1, 9], np.int32)          # 3 full pages + a tail page holding 2 tokens
    L0 = 3 * P + 2
    k_ref, v_ref = k.copy(), v.copy()
    # B gets its own tail: copy block 9 into free block 5
    assert o.copy_blocks(k, v, np.array([9, 9], np.int32), np.array([5, nb + 3], np.int32)) == 1
    assert np.array_equal(k[5], k[9]) and np.array_equal(v[5], v[9])
    assert np.array_equal(np.delete(k, 5, 0), np.delete(k_ref, 5, 0))
    ta = shared.copy()
    tb = shared.copy()
    tb[3] = 5
    new_a = workloads.normal_bf16(rng, (2, Hkv, D))       # (K, V) of A's token, then B's
    new_b = workloads.normal_bf16(rng, (2, Hkv, D))
    o.kv_append(new_a[:1], new_a[1:], np.array([9 * P + 2], np.int64), k, v)
    o.kv_append(new_b[:1], new_b[1:], np.array([5 * P + 2], np.int64), k, v)
    q = workloads.normal_bf16(rng, (2, Hq, D))
    tables = np.stack([ta, tb]).astype(np.int32)
    seq = np.array([L0 + 1, L0 + 1], np.int32)
    ind = np.array([0, 1, 2], np.int32)
    out, lse = o.attention_varlen(q, k, v, tables, seq, ind, 1 / math.sqrt(D))
    for r, new in ((0, new_a), (1, new_b)):
        # private copies: blocks 0..3 of a fresh pool, the appended token at L0
        kp = np.zeros((4, Hkv, P, D), np.uint16)
        vp = np.zeros((4, Hkv, P, D), np.uint16)
        kp[:] = k_ref[shared]
        vp[:] = v_ref[shared]
        kp[3, :, 2] = new[0]
        vp[3, :, 2] = new[1]
        po, pl = o.attention_varlen(q[r:r + 1], kp, vp, np.arange(4, dtype=np.int32)[None], seq[r:r + 1],
                                    np.array([0, 1], np.int32), 1 / math.sqrt(D))
        assert np.array_equal(out[r], po[0]) and np.array_equal(lse[r], pl[0]), r
    assert not np.array_equal(out[0], out[1])


def pin_decode_step(o):
    """A decode step ("Inference optimisation" §8.3.1 and Fig. 8-10) puts
    each row's new token at the end of its sequence, position seq_len - 1,
    in the block the table gives for it, and the row then attends over its
    old keys followed by that token.  Checked against the cache bytes and a
    dense softmax over [old keys gathered by numpy; the new token appended
    by hand].  Padding rows (seq_len 0) write nothing and give out 0, lse
    -inf; rows past max_seq_len are counted and treated as padding."""
    rng = np.random.default_rng(23)
    Hq, Hkv, P, D = 8, 2, 16, 32
    nb = 24
    lens = [1, 16, 17, 40, 0, 33]
    k, v = _pool(nb, Hkv, P, D, rng)
    tab = _tables(rng, nb, [max(L, 1) for L in lens], P)
    R = len(lens)
    q = workloads.normal_bf16(rng, (R, Hq, D))
    kn = workloads.normal_bf16(rng, (R, Hkv, D))
    vn = workloads.normal_bf16(rng, (R, Hkv, D))
    k2, v2 = k.copy(), v.copy()
    seq = np.array(lens, np.int32)
    out, lse, bad = o.decode_step(q, kn, vn, k2, v2, tab, seq, 0.21, 64)
    assert bad == 0
    expect = set()
    for r, L in enumerate(lens):
        if L == 0:
            continue
        blk, off = int(tab[r, (L - 1) // P]), (L - 1) % P
        for h in range(Hkv):
            expect.add((blk, h, off))
            assert np.array_equal(k2[blk, h, off], kn[r, h]) and np.array_equal(v2[blk, h, off], vn[r, h]), (r, h)
    changed = set(tuple(x) for x in np.argwhere((k2 != k).any(axis=-1) | (v2 != v).any(axis=-1)).tolist())
    assert changed == expect, (sorted(changed - expect), sorted(expect - changed))
    G = Hq // Hkv
    for r, L in enumerate(lens):
        if L == 0:
            assert np.all(out[r] == 0) and np.all(lse[r] == -np.inf)
            continue
        for h in range(Hq):
            g = h // G
            K = np.concatenate([f64(_gather(k, tab[r], g, L - 1, P)), f64(kn[r, g])[None]])
            V = np.concatenate([f64(_gather(v, tab[r], g, L - 1, P)), f64(vn[r, g])[None]])
            S = 0.21 * (K @ f64(q[r, h]))
            assert np.allclose(out[r, h], special.softmax(S) @ V, rtol=1e-12, atol=1e-12), (r, h)
            assert abs(lse[r, h] - special.logsumexp(S)) <= 1e-12, (r, h)
    # a row longer than the call's bound is counted and left as padding
    k3, v3 = k.copy(), v.copy()
    out3, lse3, bad3 = o.decode_step(q, kn, vn, k3, v3, tab, seq, 0.21, 39)
    assert bad3 == 1 and np.all(out3[3] == 0) and np.all(lse3[3] == -np.inf)
    assert not np.array_equal(out3[5], np.zeros_like(out3[5]))


def pin_f16_conversion(o):
    """The oracle's binary32 -> binary16 rounding (used for the q8_0 scales)
    agrees with numpy's IEEE conversion on random values across the range
    and on the edge cases (ties, subnormals, the largest finite, overflow)."""
    rng = np.random.default_rng(21)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(2.0) ** rng.integers(-30, 17, 4000),
        np.array([0.0, -0.0, 1.0, 65504.0, 65519.0, 65520.0, 1e30, 2 ** -24, 2 ** -25, 3 * 2 ** -26,
                  2 ** -14, 2 ** -14 * 0.9995, 1 + 2 ** -11, 1 + 3 * 2 ** -11, -2.5e-6], np.float32)])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([o.f32_to_f16(v) for v in x], np.uint16)
    assert np.array_equal(got, ref), x[got != ref][:5]
    for h in (0x0001, 0x03ff, 0x0400, 0x3c00, 0x7bff, 0xc248):
        assert o.f16_value(h) == float(np.array([h], np.uint16).view(np.float16)[0])


def pin_q8_layout_arithmetic(o=None):
    """The q8_0 page layout reproduces the pages' byte counts: 34 bytes per
    32 values (8.5 bits), so one 8K context drops from 1152 MiB to 612 MiB,
    the 1188 MiB block-allocated long request to 631.125 MiB, and 16 such
    requests need 9.86 GiB of the 12 GiB reserve."""
    g = json.load(open(os.path.join(HERE, "golden", "q8_arithmetic.json")))
    D, P = 128, 16
    slab = oracle.q8_slab_bytes(P, D)
    bf16_slab = P * D * 2
    assert slab * 64 == bf16_slab * g["group"]["q8_bytes"]
    assert slab * 8 / (P * D) == g["group"]["q8_bits_per_value"]
    assert (P * D // 2 + P * (D // 32) * 2) * 8 / (P * D) == g["group"]["q4_bits_per_value"]
    per_tok_bf16 = paging.kv_bytes_per_token(36, 8, 128, 2)
    per_tok_q8 = 2 * 36 * 8 * (slab // P)
    c = g["context_8k_mib"]
    assert per_tok_bf16 * 8192 / 2 ** 20 == c["bf16"]
    assert per_tok_q8 * 8192 / 2 ** 20 == c["q8"]
    assert c["bf16"] - c["q8"] == c["q8_saved"] and c["bf16"] - c["q4"] == c["q8_saved"] + 288
    lr = g["long_request_after_generation"]
    assert per_tok_q8 * paging.reserved_tokens(8447, 16) / 2 ** 20 == lr["q8_mib"]
    assert round(lr["requests"] * lr["q8_mib"] / 1024, 2) == lr["total_gib"] <= lr["reserve_gib"]


def pin_q8_quantization(o):
    """q8_0 codes and scales by their closed forms: the scale is the
    binary16 of max|x| / 127 (numpy's conversion), the largest element of a
    group gets code +-127, every value is within half a scale step of its
    dequantized code, codes stay in [-127, 127], an all-zero group is zero."""
    rng = np.random.default_rng(22)
    x = workloads.normal_bf16(rng, (64, 128))
    x[3, 32:64] = 0                                        # an all-zero group
    x[5, :32] = bits(0.0)
    x[5, 7] = bits(-3.0)                                    # one nonzero element
    codes, scales = o.quantize_q8(x)
    xv = oracle.bf16_to_f64(x).reshape(64, 4, 32)
    cg = codes.astype(np.float64).reshape(64, 4, 32)
    amax = np.abs(xv).max(axis=2)
    ref_scale = (amax.astype(np.float32) / np.float32(127)).astype(np.float16)
    assert np.array_equal(scales, ref_scale.view(np.uint16))
    d16 = ref_scale.astype(np.float64)
    assert np.all(np.abs(codes.astype(np.int32)) <= 127)
    assert np.all(np.abs(xv - cg * d16[..., None]) <= d16[..., None] * (0.5 + 2 ** -20))
    top = np.abs(xv).argmax(axis=2)
    for i in range(64):
        for gi in range(4):
            if amax[i, gi] > 0:
                assert cg[i, gi, top[i, gi]] == 127 * np.sign(xv[i, gi, top[i, gi]])
    assert scales[3, 1] == 0 and not codes[3, 32:64].any()
    assert codes[5, 7] == -127 and np.count_nonzero(codes[5, :32]) == 1
    # groups whose scale is a binary16 subnormal (max|x| / 127 near 1.1-1.5 x
    # 2^-24): the scale rounds down by up to a third, |x| / d16 passes 127.5
    # and the clamp acts.  Both the rounding and the clamp are odd functions,
    # so a negated group gets the same scale and negated codes, all in
    # [-127, 127]; the largest element's code is the clamp itself.
    tiny = np.zeros((8, 32))
    for gi in range(8):
        amax = 127 * (1.1 + 0.05 * gi) * 2.0 ** -24
        tiny[gi] = rng.uniform(-amax, amax, 32)
        tiny[gi, gi] = -amax if gi % 2 == 0 else amax
    xt = o.round_bf16(tiny)
    ct, st = o.quantize_q8(xt)
    cn, sn = o.quantize_q8(xt ^ np.uint16(0x8000))
    assert np.array_equal(st, sn) and np.array_equal(cn.astype(np.int32), -ct.astype(np.int32))
    assert np.all(np.abs(ct.astype(np.int32)) <= 127)
    d16 = st.view(np.float16).astype(np.float64)
    at = np.abs(oracle.bf16_to_f64(xt).reshape(8, 32))
    assert np.any(at.max(axis=1) / d16 > 127.5)             # the clamp is exercised
    for gi in range(8):
        assert abs(int(ct.reshape(8, 32)[gi, gi])) == 127


def _q8_values(cache, P, D):
    """Dequantized values [nb, Hkv, P, D] of q8_0 pages, decoded here from
    the slab bytes (codes, then little-endian binary16 scales)."""
    nb, Hkv, slab = cache.shape
    codes = cache[:, :, :P * D].view(np.int8).reshape(nb, Hkv, P, D // 32, 32).astype(np.float64)
    sc = cache[:, :, P * D:].copy().view(np.float16).reshape(nb, Hkv, P, D // 32).astype(np.float64)
    with np.errstate(invalid="ignore"):  # never-written slots may hold NaN scales; they are not read
        return (codes * sc[..., None]).reshape(nb, Hkv, P, D)


def pin_q8_attention(o):
    """q8_0 pages: kv_append_q8 stores what quantize_q8 gives, and attention
    over q8_0 pages equals a numpy fp64 softmax attention over the values
    decoded from the slab bytes (gathered through the block tables)."""
    Hq, Hkv, P, D = 8, 2, 16, 64
    b = workloads.make_batch([40, 17, 70], [1, 5, 1], num_blocks=16, seed=23, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D)
    slab = oracle.q8_slab_bytes(P, D)
    rng = np.random.default_rng(24)
    kq = rng.integers(0, 256, (16, Hkv, slab)).astype(np.uint8)   # junk, then fill every token used
    vq = kq.copy()
    for r in range(b.num_reqs):
        toks = workloads.normal_bf16(rng, (int(b.seq_lens[r]), 2, Hkv, D))
        slots = np.array([b.block_tables[r, t // P] * P + t % P for t in range(int(b.seq_lens[r]))], np.int64)
        o.kv_append_q8(toks[:, 0], toks[:, 1], slots, kq, vq)
    one = workloads.normal_bf16(rng, (1, Hkv, D))
    ck, sk = o.quantize_q8(one)
    s0 = int(b.block_tables[0, 0]) * P
    o.kv_append_q8(one, one, np.array([s0], np.int64), kq, vq)
    got_codes = kq[s0 // P, :, :P * D].view(np.int8).reshape(Hkv, P, D)[:, 0]
    got_scales = kq[s0 // P, :, P * D:].copy().view(np.uint16).reshape(Hkv, P, D // 32)[:, 0]
    assert np.array_equal(got_codes, ck[0]) and np.array_equal(got_scales, sk[0])
    out, lse = o.attention_varlen_q8(b.q, kq, vq, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    Kv, Vv = _q8_values(kq, P, D), _q8_values(vq, P, D)
    qv = oracle.bf16_to_f64(b.q)
    for r in range(b.num_reqs):
        L = int(b.seq_lens[r])
        c = int(b.qo_indptr[r + 1] - b.qo_indptr[r])
        Kr = np.stack([Kv[b.block_tables[r, t // P], :, t % P] for t in range(L)])   # [L, Hkv, D]
        Vr = np.stack([Vv[b.block_tables[r, t // P], :, t % P] for t in range(L)])
        for j in range(c):
            tok = int(b.qo_indptr[r]) + j
            n = L - c + j + 1
            for h in range(Hq):
                sc = b.sm_scale * Kr[:n, h // (Hq // Hkv)] @ qv[tok, h]
                w = np.exp(sc - sc.max())
                ref = w @ Vr[:n, h // (Hq // Hkv)] / w.sum()
                assert np.allclose(out[tok, h], ref, rtol=1e-10, atol=1e-12), (r, j, h)
                assert abs(lse[tok, h] - (sc.max() + np.log(w.sum()))) < 1e-10


def pin_brute_force(o):
    """Cross-check against the pure-Python fp64 restatement (oracle/brute.py)
    on a tiny mixed batch (decode rows and a chunk)."""
    from oracle import brute
    b = _random_batch(17, [23, 40], [1, 6], 6, Hq=4, Hkv=2, D=16)
    out, lse = o.attention_varlen(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    bo, bl = brute.attention(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    assert np.allclose(out, np.array(bo), rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, np.array(bl), rtol=1e-12, atol=1e-12)


def pin_sampled_matches_full(o):
    """The sampled entry point is the same definition at chosen outputs."""
    b = _random_batch(18, [50, 31, 64], [1, 7, 1], 16)
    out, lse = o.attention_varlen(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    tok = np.array([0, 1, 4, 7, 8, 8], np.int32)
    head = np.array([0, 3, 7, 2, 5, 0], np.int32)
    so, sl = o.attention_sampled(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale,
                                 tok, head)
    assert np.array_equal(so, out[tok, head]) and np.array_equal(sl, lse[tok, head])


ALL_PINS = [pin_page_arithmetic, pin_round_bf16, pin_single_key, pin_one_hot_score, pin_two_key_sigmoid,
            pin_uniform_scores, pin_gqa_grouping, pin_scipy_dense, pin_page_permutation,
            pin_shared_equals_duplicated, pin_chunked_equals_oneshot, pin_merge_identity, pin_append_then_read,
            pin_copy_on_write, pin_f16_conversion, pin_q8_layout_arithmetic, pin_q8_quantization, pin_q8_attention,
            pin_brute_force, pin_sampled_matches_full, pin_decode_step]


def run_all(o) -> list:
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception as e:  # noqa: BLE001 - a mutant may fail in any way
            failed.append((pin.__name__, f"{type(e).__name__}: {e}"[:200]))
    return failed


if __name__ == "__main__":
    failed = run_all(oracle.Oracle(sys.argv[1]))
    for name, why in failed:
        print(f"FAILED {name}: {why}")
    sys.exit(min(len(failed), 100))
