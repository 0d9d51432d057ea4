"""pa_attention_varlen_noalloc: the attention call for callers that cannot
allocate device memory (a serving loop that must stay out of the allocator,
a host framework that owns all device memory, a plugin handed only its
input and output pointers).  It takes no workspace; its scratch is one fixed
array inside the library that every call on a device shares and reuses.

Its results are checked against the oracle and against pa_attention_varlen
(bit for bit: both run the same kernels on the same launch plan), on calls
made back to back, so that state left in the shared array by one call (the
cut-row counters, the error word) would show up in the next.

Kept in a file of its own that is collected last, and independent of the
other tests' state, so it passes both alone and after the whole suite."""
import numpy as np
import pytest
import torch

from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import DevBatch, compare, oracle_step

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


def _prepared(name, scale):
    """A workload batch on the GPU with this step's tokens appended, and the
    oracle's result for it."""
    b = W.workload_batch(name, scale=scale)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    ref_out, ref_lse, _, _ = oracle_step(b)
    args = (d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr, b.sm_scale)
    kw = dict(seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host, return_lse=True)
    return args, kw, ref_out, ref_lse


def test_noalloc_matches_oracle_and_workspace_call_on_calls_in_a_row():
    B.pa_set_decode_ctas(0)
    # mixed: decode rows cut between CTAs (partials + counters) and one
    # chunked-prefill row; short: decode rows only, every one cut between
    # CTAs, run after the mixed batch has left its state in the array
    mixed = _prepared("mixed", 0.25)
    short = _prepared("short", 0.5)
    refs = {}
    for name, (args, kw, _, _) in (("mixed", mixed), ("short", short)):
        refs[name] = B.pa_attention_varlen(*args, **kw)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, (name, (args, kw, ref_out, ref_lse)) in enumerate(
            (("mixed", mixed), ("mixed", mixed), ("short", short), ("mixed", mixed))):
        out, lse = B.pa_attention_varlen_noalloc(*args, device_error=err, **kw)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call} ({name}): device error {int(err.item())}"
        compare(out, ref_out, lse, ref_lse, what=f"noalloc call {call} ({name}) vs oracle")
        ws_out, ws_lse = refs[name]
        assert torch.equal(out, ws_out), f"call {call} ({name}): differs from pa_attention_varlen"
        assert torch.equal(lse, ws_lse), f"call {call} ({name}): lse differs from pa_attention_varlen"


def test_noalloc_reports_a_bad_block_id_and_then_recovers():
    b = W.make_batch([100, 200, 300], [1, 1, 1], num_blocks=40, seed=W.SEED0 + 71)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    bad = b.block_tables.copy()
    bad[1, 3] = 10_000                # outside the 40-block pool: masked and recorded
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.pa_attention_varlen_noalloc(d.q, d.k_cache, d.v_cache, torch.from_numpy(bad).cuda(), d.seq_lens,
                                  d.qo_indptr, b.sm_scale, seq_lens_host=d.seq_lens_host,
                                  qo_indptr_host=d.qo_indptr_host, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PA_ERR_DEVICE_INDEX
    # the next call starts from a clear error word and clean counters
    out, lse = B.pa_attention_varlen_noalloc(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                             b.sm_scale, seq_lens_host=d.seq_lens_host,
                                             qo_indptr_host=d.qo_indptr_host, device_error=err, return_lse=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_out, ref_lse, _, _ = oracle_step(b)
    compare(out, ref_out, lse, ref_lse, what="noalloc after a recorded error")


def test_noalloc_scratch_bounds():
    scratch = 24 << 20
    # every batch of the pages' head shape (8 kv heads, 32 q heads) fits the
    # fixed scratch: at most 65,535 requests and a decode grid of at most
    # 1,024 CTAs (4 warp segments each)
    assert 0 < B.pa_attention_workspace_size(65535, 65535, 32, 128, 1 << 20) <= scratch
    # more requests than pa_attention_varlen accepts: rejected as an invalid
    # argument before any host array is read
    n = 65536
    seq = torch.full((n,), 16, dtype=torch.int32)
    ind = torch.zeros(n + 1, dtype=torch.int32)
    q = torch.zeros((0, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PAError) as e:
        B.pa_attention_varlen_noalloc(q, kc, kc, torch.zeros((n, 1), dtype=torch.int32, device="cuda"),
                                      seq.cuda(), ind.cuda(), 0.088, seq_lens_host=seq, qo_indptr_host=ind)
    assert e.value.status == B.PA_ERR_INVALID_ARG
    # a valid batch whose workspace exceeds the scratch (64 kv heads: the
    # per-(request, kv head) counters alone take 16 MiB) is refused on the
    # host with PA_ERR_UNSUPPORTED; nothing is launched
    n = 65535
    assert B.pa_attention_workspace_size(n, 0, 256, 128, 16) > scratch
    seq = torch.full((n,), 16, dtype=torch.int32)
    ind = torch.zeros(n + 1, dtype=torch.int32)
    q = torch.zeros((0, 256, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 64, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PAError) as e:
        B.pa_attention_varlen_noalloc(q, kc, kc, torch.zeros((n, 1), dtype=torch.int32, device="cuda"),
                                      seq.cuda(), ind.cuda(), 0.088, seq_lens_host=seq, qo_indptr_host=ind)
    assert e.value.status == B.PA_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)


def test_noalloc_in_a_captured_graph_replays_exactly():
    # the first call on a device looks up the scratch array (before any
    # capture); a call captured into a CUDA graph then replays with the same
    # results as the workspace call, replay after replay
    B.pa_set_decode_ctas(0)
    args, kw, ref_out, ref_lse = _prepared("short", 0.25)
    ws_out, ws_lse = B.pa_attention_varlen(*args, **kw)
    B.pa_attention_varlen_noalloc(*args, **kw)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out, lse = B.pa_attention_varlen_noalloc(*args, **kw)
    for replay in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ws_out), f"replay {replay}: differs from pa_attention_varlen"
        assert torch.equal(lse, ws_lse), f"replay {replay}: lse differs from pa_attention_varlen"
    compare(out, ref_out, lse, ref_lse, what="noalloc graph replay vs oracle")
