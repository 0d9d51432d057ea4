"""The algorithmic bytes and flops that every reported rate divides by
(`workloads.step_bytes`), checked against closed forms and the pages' own
figures.  Runs without a GPU."""
import json
import os

import numpy as np

from paged_kv_decode_varlen_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.json")
HQ, HKV, D, P = 32, 8, 128, 16
PER_TOK = 2 * HKV * D * 2  # K and V of one token over the kv heads, bf16


def _batch(seq, qo, **kw):
    need = sum(-(-L // P) for L in seq)
    return W.make_batch(seq, qo, num_blocks=need + 3, seed=kw.pop("seed", 5), **kw)


def test_prefill_flops_follow_the_pages_pair_counts():
    # "Inference optimisation" §8.2.3, the N_pair equation and Fig. 8-8 / 8-9:
    # a chunk of c tokens after h cached ones forms h c + c (c + 1) / 2
    # (query, key) pairs; each pair costs 2 x 2 flop per head and dim (QK^T, PV)
    cases = json.load(open(GOLDEN))["chunk_pair_counts"]["cases"]
    for case in cases:
        c, h, pairs = case["c"], case["h"], case["pairs"]
        got = W.step_bytes(_batch([h + c], [c]))["prefill_flops"]
        assert got == pairs * HQ * D * 4, case


def test_mixed_chunk_flops():
    # the mixed batch's 512-token chunk after 1,536 cached tokens: 917,760
    # pairs per head, 15.04 GFLOP over 32 heads
    got = W.step_bytes(_batch([2048], [512]))["prefill_flops"]
    assert got == (512 * 1536 + 512 * 513 // 2) * HQ * D * 4 == 15_036_579_840


def test_decode_bytes_closed_form():
    rng = np.random.default_rng(3)
    seq = [int(x) for x in rng.integers(1, 3000, 40)]
    sb = W.step_bytes(_batch(seq, [1] * 40))
    n = len(seq)
    pages = sum(-(-L // P) for L in seq)
    # every key read once per kv head, q read and out written, one table
    # entry per page
    assert sb["decode_kernel"] == PER_TOK * sum(seq) + 2 * n * HQ * D * 2 + 4 * pages
    assert sb["unique_kv"] == sb["logical_kv"] == PER_TOK * sum(seq)
    # the whole step adds the seq_lens / qo_indptr words and the append of
    # each new token (read as bf16, written into its page, its 8-byte slot)
    assert sb["unique"] == (PER_TOK * sum(seq) + 2 * n * HQ * D * 2 + 4 * pages + 8 * n + 4
                            + n * (PER_TOK + PER_TOK + 8))
    # the decode step's one kernel: the decode bytes, the append, the seq_lens
    assert sb["step_kernel"] == sb["decode_kernel"] + n * 2 * PER_TOK + 4 * n
    assert sb["prefill_flops"] == 0 and sb["prefill_kernel"] == 0


def test_shared_prefix_pages_counted_once():
    seq = [6144 + 100, 6144 + 2048, 6144 + 37]
    S = 6144
    b = _batch(seq, [1, 1, 1], shared_prefix_tokens=S)
    sb = W.step_bytes(b, prefix_pages=S // P)
    assert sb["unique_kv"] == PER_TOK * (S + sum(L - S for L in seq))
    assert sb["logical_kv"] == PER_TOK * sum(seq)
    # the decode kernel reads only the rows' own pages after the prefix; the
    # prefix pass reads the prefix once
    own_pages = sum(-(-L // P) - S // P for L in seq)
    assert sb["decode_kernel"] == PER_TOK * sum(L - S for L in seq) + 2 * 3 * HQ * D * 2 + 4 * own_pages
    assert sb["prefix_kernel"] == S * PER_TOK + 3 * HQ * D * 2 + 4 * (S // P)


def test_q8_pages_hold_34_of_64_bytes():
    # "Inference optimisation" §8.4.2: 32 values share a 2-byte scale next to
    # their 8-bit codes, 34 bytes instead of 64
    seq = [2048, 777, 1500]
    b = _batch(seq, [1, 1, 1])
    bf, q8 = W.step_bytes(b), W.step_bytes(b, kv="q8")
    assert q8["unique_kv"] * 64 == bf["unique_kv"] * 34
