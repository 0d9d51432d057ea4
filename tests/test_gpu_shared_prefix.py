"""Shared-prefix (cascade) attention through the C ABI against the CPU oracle.

pa_attention_varlen_shared_prefix computes the same attention as
pa_attention_varlen; the oracle knows nothing of the split (it attends every
query to all of its keys through the block table), so every case here is
checked against the plain definition at the stated tolerance."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import DevBatch, compare, oracle_step

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


def _append(d):
    ws = B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    return ws


def _shared(d, pages, workspace=None):
    return B.pa_attention_varlen_shared_prefix(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                               d.b.sm_scale, pages, seq_lens_host=d.seq_lens_host,
                                               qo_indptr_host=d.qo_indptr_host, workspace=workspace,
                                               return_lse=True)


def _plain(d):
    return B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr, d.b.sm_scale,
                                 seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host, return_lse=True)


def _check_against_oracle(b, pages, what):
    d = DevBatch(b)
    ws_a = _append(d)
    out, lse = _shared(d, pages)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws_a) == 0
    ref, ref_lse, _, _ = oracle_step(b)
    return d, out, lse, compare(out, ref, lse, ref_lse, what=what)


def test_shared_workload():
    """16 long requests sharing a 6144-token prefix (384 pages), decode rows:
    many key chunks merged by the last CTA of each (query tile, kv head)."""
    b = W.workload_batch("shared")
    _check_against_oracle(b, 384, "shared workload")


# (seq_lens, qo_lens, shared prefix tokens)
CASES = {
    # decode rows with a prefix that is not a whole number of 64-key tiles
    "decode_prefix_5_pages": ([300, 120, 81, 1000], [1, 1, 1, 1], 80),
    # the own part of a row is a single token (seq_len = prefix + 1)
    "own_part_one_token": ([257, 300, 256 + 16], [1, 1, 1], 256),
    # prefill rows whose chunk starts right after the prefix and later
    "prefill_after_prefix": ([800, 900, 700, 1000, 560], [1, 48, 1, 1, 48], 512),
    # rows without queries, the first of them before the first active row
    "empty_rows": ([600, 700, 650, 900], [0, 1, 0, 33], 320),
    # a chunk whose 16-token tiles end ragged, next to decode rows
    "ragged_chunk": ([1110, 1300, 1200], [77, 1, 1], 1024),
    # enough query tiles that the prefix is one chunk written directly
    "single_chunk_many_queries": ([2600, 2700, 2100, 2000], [640, 1, 1, 100], 1536),
    # a prefix of one page
    "one_page_prefix": ([40, 17, 33], [1, 1, 1], 16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_cases(case):
    seq, qo, prefix = CASES[case]
    need = prefix // 16 + sum(-(-L // 16) - prefix // 16 for L in seq)
    b = W.make_batch(seq, qo, num_blocks=need + 9, seed=zlib.crc32(case.encode()) % 1000,
                     shared_prefix_tokens=prefix)
    _check_against_oracle(b, prefix // 16, case)


def test_sweep_point_128x8192_sampled():
    """The largest sweep point (128 requests of 8192 tokens sharing 6144)
    at the size the 36-layer sweep runs, one layer, checked on sampled
    (token, head) outputs."""
    spec = W.sweep_point(128, 8192)
    b = W.make_batch(spec["seq_lens"], spec["qo_lens"], num_blocks=spec["num_blocks"], seed=spec["seed"],
                     shared_prefix_tokens=spec["shared_prefix_tokens"])
    d = DevBatch(b)
    ws_a = _append(d)
    out, lse = _shared(d, spec["shared_prefix_tokens"] // 16)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws_a) == 0
    k, v = b.k_cache.copy(), b.v_cache.copy()
    oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, k, v)
    rng = np.random.default_rng(77)
    tok = rng.integers(0, b.total_q, 256).astype(np.int32)
    head = rng.integers(0, b.q.shape[1], 256).astype(np.int32)
    ref, ref_lse = oracle.attention_sampled(b.q, k, v, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale, tok,
                                            head)
    got = out[torch.from_numpy(tok).long().cuda(), torch.from_numpy(head).long().cuda()]
    got_lse = lse[torch.from_numpy(tok).long().cuda(), torch.from_numpy(head).long().cuda()]
    compare(got, ref, got_lse, ref_lse, what="sweep 128x8192 shared prefix")


def test_matches_plain_entry_point():
    """Both entry points compute the same attention: outputs within the
    bf16 rounding of each other."""
    b = W.make_batch([900, 1000, 1100, 950], [1, 1, 1, 1], num_blocks=300, seed=41, shared_prefix_tokens=768)
    d = DevBatch(b)
    _append(d)
    out_s, lse_s = _shared(d, 48)
    out_p, lse_p = _plain(d)
    torch.cuda.synchronize()
    diff = (out_s.float() - out_p.float()).abs()
    assert float(diff.max()) <= 1.6e-2  # at most an ulp or two of bf16 near |x| ~ 1
    assert float((lse_s - lse_p).abs().max()) <= 1e-4


def test_one_active_request_runs_the_plain_path():
    """With a single request that has queries there is nothing to share: the
    call runs the plain path and its output is bit-identical to it."""
    b = W.make_batch([700, 500], [1, 0], num_blocks=80, seed=43, shared_prefix_tokens=256)
    d = DevBatch(b)
    _append(d)
    out_s, lse_s = _shared(d, 16)
    out_p, lse_p = _plain(d)
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), out_p.view(torch.int16))
    assert torch.equal(lse_s, lse_p)


def test_zero_prefix_pages_is_plain():
    b = W.make_batch([300, 200, 100], [1, 1, 5], num_blocks=60, seed=45)
    d = DevBatch(b)
    _append(d)
    out_s, lse_s = _shared(d, 0)
    out_p, lse_p = _plain(d)
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), out_p.view(torch.int16))


def test_workspace_reused():
    """Consecutive calls on one workspace (decode counters left at zero,
    prefix partials overwritten) give the same result."""
    b = W.make_batch([1200, 1300, 1250, 1400, 1500], [1, 1, 20, 1, 1], num_blocks=500, seed=47,
                     shared_prefix_tokens=1024)
    d = DevBatch(b)
    _append(d)
    ref, ref_lse, _, _ = oracle_step(b)
    ws = B.new_workspace(B.pa_shared_prefix_workspace_size(5, b.total_q, 32, 128, 1500, 64), "cuda")
    outs = []
    for _ in range(3):
        out, lse = _shared(d, 64, workspace=ws)
        torch.cuda.synchronize()
        compare(out, ref, lse, ref_lse, what="reuse")
        outs.append(out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
    assert B.pa_get_device_error(ws) == 0


def test_prefix_must_precede_queries():
    b = W.make_batch([300, 200], [1, 60], num_blocks=40, seed=49, shared_prefix_tokens=128)
    d = DevBatch(b)
    with pytest.raises(B.PAError) as e:
        _shared(d, 9)  # 200 - 60 = 140 < 144 keys of prefix
    assert e.value.status == B.PA_ERR_INVALID_ARG


def _kinds(d, pages):
    B.pa_trace_enable(1)
    B.pa_trace_read()
    _shared(d, pages)
    torch.cuda.synchronize()
    kinds = [k for k, _ in B.pa_trace_read()]
    B.pa_trace_enable(0)
    return kinds


def test_launches_prefix_pass():
    """Decode rows only: the decode kernel folds the prefix pass's key-chunk
    partials itself; with a prefill row the chunks are merged first and both
    kernels fold the merged partial."""
    b = W.make_batch([600, 700, 650], [1, 1, 1], num_blocks=200, seed=51, shared_prefix_tokens=512)
    d = DevBatch(b)
    _append(d)
    torch.cuda.synchronize()
    assert _kinds(d, 32) == ["prefix", "decode"]
    b = W.make_batch([600, 700, 650], [1, 40, 1], num_blocks=200, seed=52, shared_prefix_tokens=512)
    d = DevBatch(b)
    _append(d)
    torch.cuda.synchronize()
    assert _kinds(d, 32) == ["prefix", "prefix_merge", "prefill", "decode"]
