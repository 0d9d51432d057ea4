"""CUDA path (through the C ABI) against the CPU oracle on the same seeded
inputs.  Append and indexing are bit-exact; attention outputs meet max-abs
1.5e-2 and mean-abs 2e-3 against the fp64 oracle."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import DevBatch, bf16_host, compare, oracle_step

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


@pytest.fixture(autouse=True)
def _reset_splits():
    yield
    if torch.cuda.is_available():
        B.pa_set_decode_ctas(0)


def run_step(d: DevBatch, return_lse=True):
    """One step through the C ABI: append, then attention.  Returns (out, lse, ws)."""
    ws_a = B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    out, lse = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                     d.b.sm_scale, seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host,
                                     return_lse=True)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws_a) == 0
    return out, lse


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("name", ["tiny", "mixed"])
def test_kv_append_bit_exact(name):
    b = W.workload_batch(name)
    d = DevBatch(b)
    ws = B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    k, v = b.k_cache.copy(), b.v_cache.copy()
    oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, k, v)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == 0
    assert np.array_equal(bf16_host(d.k_cache), k)
    assert np.array_equal(bf16_host(d.v_cache), v)


def test_kv_append_skip_and_out_of_range():
    b = W.make_batch([20, 40, 33], [1, 1, 8], num_blocks=12, seed=5)
    d = DevBatch(b)
    slots = b.slot_mapping.copy()
    slots[0] = -1                    # padding: skipped
    slots[5] = 12 * 16 + 3           # beyond the pool: skipped, recorded
    d.slot_mapping = torch.from_numpy(slots).cuda()
    ws = B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_INDEX
    k, v = b.k_cache.copy(), b.v_cache.copy()
    keep = slots.copy()
    keep[5] = -1
    oracle.kv_append(b.k_new, b.v_new, keep, k, v)
    assert np.array_equal(bf16_host(d.k_cache), k) and np.array_equal(bf16_host(d.v_cache), v)
    B.pa_clear_device_error(ws)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == 0


# ------------------------------------------------------- attention: workloads
@pytest.mark.parametrize("name,scale", [("tiny", 1.0), ("short", 1.0), ("shared", 1.0), ("mixed", 0.25),
                                        ("mixed", 1.0), ("verify", 0.25), ("verify", 1.0)])
def test_workload_parity(name, scale):
    b = W.workload_batch(name, scale=scale)
    d = DevBatch(b)
    out, lse = run_step(d)
    ref, ref_lse, k, v = oracle_step(b)
    assert np.array_equal(bf16_host(d.k_cache), k)
    compare(out, ref, lse, ref_lse, what=f"{name}x{scale}")


@pytest.mark.parametrize("batch,context", [(1, 2048), (128, 2048), (8, 8192)])
def test_sweep_point_parity(batch, context):
    """Points of the 36-layer decode sweep, one layer each (layers are
    independent calls over their own pools)."""
    spec = W.sweep_point(batch, context)
    b = W.make_batch(spec["seq_lens"], spec["qo_lens"], num_blocks=spec["num_blocks"], seed=spec["seed"],
                     shared_prefix_tokens=spec["shared_prefix_tokens"])
    d = DevBatch(b)
    out, lse = run_step(d)
    ref, ref_lse, _, _ = oracle_step(b)
    compare(out, ref, lse, ref_lse, what=f"sweep b={batch} L={context}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 456, 1024])
def test_forced_decode_grid(ctas):
    """Every persistent grid size -- one CTA for all key ranges, ranges cut
    across many CTAs, more CTAs than pages -- gives the same attention."""
    b = W.make_batch([2100, 37, 16, 1, 700, 129], [1] * 6, num_blocks=400, seed=20 + ctas)
    d = DevBatch(b)
    B.pa_set_decode_ctas(ctas)
    out, lse = run_step(d)
    ref, ref_lse, _, _ = oracle_step(b)
    compare(out, ref, lse, ref_lse, what=f"ctas={ctas}")


@pytest.mark.parametrize("ctas", [8, 16])
def test_many_rows_per_cta(ctas):
    """64 short rows on one or two segments per kv head: a CTA walks up to
    64 rows, each with its q staged in shared memory while the previous row
    ends (the longest chain of the per-row q copies), next to rows cut
    between the two segments."""
    seq = [int(x) for x in np.random.default_rng(41).integers(1, 200, 64)]
    need = sum(-(-L // 16) for L in seq)
    b = W.make_batch(seq, [1] * 64, num_blocks=need + 5, seed=40 + ctas)
    d = DevBatch(b)
    B.pa_set_decode_ctas(ctas)
    out, lse = run_step(d)
    ref, ref_lse, _, _ = oracle_step(b)
    compare(out, ref, lse, ref_lse, what=f"64 rows on ctas={ctas}")


@pytest.mark.parametrize("scale", [0.0, -0.0883883])
def test_nonpositive_sm_scale(scale):
    """sm_scale may be any finite value: zero weighs every key alike and a
    negative scale turns the softmax around.  Decode rows (cut between CTAs)
    and chunked-prefill rows (tensor-core tiles) both follow the oracle."""
    seq, qo = [1500, 300, 2000, 77], [1, 40, 1, 9]
    need = sum(-(-L // 16) for L in seq)
    b = W.make_batch(seq, qo, num_blocks=need + 5, seed=51, sm_scale=scale)
    d = DevBatch(b)
    out, lse = run_step(d)
    ref, ref_lse, _, _ = oracle_step(b)
    compare(out, ref, lse, ref_lse, what=f"sm_scale={scale}")


def test_workspace_reused_across_grid_sizes():
    """The item counters in the workspace return to zero after every call,
    so one workspace serves consecutive calls with different grid sizes."""
    b = W.make_batch([1500, 700, 33, 2000], [1] * 4, num_blocks=300, seed=29)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    ref, ref_lse, _, _ = oracle_step(b)
    ws = B.new_workspace(B.pa_attention_workspace_size(4, 4, 32, 128, 2000), "cuda")
    for splits in (7, 3, 64, 1, 5, 5, 300):
        B.pa_set_decode_ctas(splits)
        out, lse = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                         b.sm_scale, workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        compare(out, ref, lse, ref_lse, what=f"reuse splits={splits}")
    counters = ws[256:256 + 4 * 8 * 4].view(torch.int32)
    assert int(counters.abs().sum()) == 0


# ----------------------------------------------------------------- edge cases
EDGE = {
    "single_token_context": ([1], [1]),
    "exact_page_multiple": ([16, 32, 256], [1, 1, 1]),
    "empty_rows_mixed_in": ([50, 30, 70, 9], [1, 0, 5, 0]),
    "prefill_from_zero": ([40], [40]),
    "prefill_ragged_tiles": ([100, 77, 19], [17, 2, 19]),
    "prefill_one_page_chunk": ([64], [16]),
    "many_small_rows": ([int(x) for x in np.random.default_rng(3).integers(1, 90, 300)], [1] * 300),
    "mixed_prefill_decode": ([300, 2000, 1500, 17], [33, 1, 64, 1]),
    "long_prefill_chunk": ([2048], [512]),
    "all_empty": ([10, 20], [0, 0]),
    # more decode rows than one launch's plan carries (1024): two launches
    "decode_rows_over_one_launch": ([int(x) for x in np.random.default_rng(5).integers(1, 60, 1100)], [1] * 1100),
    # one 128K-token row: 8192 pages cut over every segment of each kv head
    "one_long_row_128k": ([131072], [1]),
    # more query tiles than one tile launch carries (1536): two launches
    "prefill_items_over_one_launch": ([int(x) for x in np.random.default_rng(7).integers(2, 40, 1600)], [2] * 1600),
    # verify rows of unequal lengths, enough jobs for the persistent tile grid
    "verify_rows_persistent_grid": ([int(x) for x in np.random.default_rng(9).integers(6, 300, 400)], [5] * 400),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_cases(case):
    seq, qo = EDGE[case]
    need = sum(-(-L // 16) for L in seq)
    b = W.make_batch(seq, qo, num_blocks=need + 7, seed=zlib.crc32(case.encode()) % 1000)
    d = DevBatch(b)
    if b.total_q == 0:
        out = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                    b.sm_scale)
        torch.cuda.synchronize()
        assert out.shape[0] == 0
        return
    out, lse = run_step(d)
    ref, ref_lse, _, _ = oracle_step(b)
    compare(out, ref, lse, ref_lse, what=case)


@pytest.mark.parametrize("ctas", [1, 3, 7, 16, -1])
def test_prefill_jobs_beside_the_decode_launch(ctas):
    """The tensor-core jobs of the qo_len > 1 rows on `ctas` persistent CTAs
    beside the decode launch (each CTA runs several jobs in turn: its rings,
    barrier phases and tensor-memory buffers continue from job to job), or
    first and one CTA per job (-1): the same results as the oracle, no device
    error, the row counters back at zero."""
    seq, qo = [300, 2000, 1500, 17, 900, 1200], [33, 1, 64, 1, 1, 40]
    need = sum(-(-L // 16) for L in seq)
    b = W.make_batch(seq, qo, num_blocks=need + 7, seed=W.SEED0 + 81)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    ws = B.new_workspace(B.pa_attention_workspace_size(b.num_reqs, b.total_q, 32, 128, max(seq)), "cuda")
    B.pa_set_prefill_ctas(ctas)
    try:
        outs = [B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                      b.sm_scale, seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host,
                                      workspace=ws, return_lse=True) for _ in range(2)]
        torch.cuda.synchronize()
    finally:
        B.pa_set_prefill_ctas(0)
    assert B.pa_get_device_error(ws) == 0
    ref, ref_lse, _, _ = oracle_step(b)
    for i, (out, lse) in enumerate(outs):
        compare(out, ref, lse, ref_lse, what=f"prefill jobs on {ctas} CTAs, call {i}")
    assert torch.equal(outs[0][0], outs[1][0])


@pytest.mark.parametrize("ctas", [1, 5, 37])
def test_prefill_only_batch_on_persistent_ctas(ctas):
    """A batch of rows with qo_len > 1 only (chunks, verify rows, a ragged
    tail) forced onto `ctas` persistent CTAs: each runs its jobs in turn with
    no CTA barrier between them (the next job's copies and first products
    overlap this one's end); the same results as the oracle on two calls, no
    device error."""
    seq, qo = [300, 2000, 1500, 900, 1200, 64, 2048], [33, 5, 64, 5, 40, 64, 512]
    need = sum(-(-L // 16) for L in seq)
    b = W.make_batch(seq, qo, num_blocks=need + 7, seed=W.SEED0 + 83)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    ws = B.new_workspace(B.pa_attention_workspace_size(b.num_reqs, b.total_q, 32, 128, max(seq)), "cuda")
    B.pa_set_prefill_ctas(ctas)
    try:
        outs = [B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                      b.sm_scale, seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host,
                                      workspace=ws, return_lse=True) for _ in range(2)]
        torch.cuda.synchronize()
    finally:
        B.pa_set_prefill_ctas(0)
    assert B.pa_get_device_error(ws) == 0
    ref, ref_lse, _, _ = oracle_step(b)
    for i, (out, lse) in enumerate(outs):
        compare(out, ref, lse, ref_lse, what=f"prefill-only jobs on {ctas} CTAs, call {i}")
    assert torch.equal(outs[0][0], outs[1][0])


def test_shared_prefix_mixed_with_prefill():
    b = W.make_batch([800, 900, 700, 1000], [1, 48, 1, 1], num_blocks=300, seed=33, shared_prefix_tokens=512)
    d = DevBatch(b)
    out, lse = run_step(d)
    ref, ref_lse, _, _ = oracle_step(b)
    compare(out, ref, lse, ref_lse, what="shared+prefill")


# ------------------------------------------------------------- invariances
def _attn(d, k=None, v=None, tables=None):
    return B.pa_attention_varlen(d.q, d.k_cache if k is None else k, d.v_cache if v is None else v,
                                 d.block_tables if tables is None else tables, d.seq_lens, d.qo_indptr,
                                 d.b.sm_scale, seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host)


def test_page_permutation_bit_identical():
    b = W.make_batch([300, 41, 1000, 77], [1, 1, 20, 1], num_blocks=120, seed=41)
    d = DevBatch(b)
    base = _attn(d).clone()
    perm = torch.from_numpy(np.random.default_rng(42).permutation(120)).cuda()
    k2 = torch.empty_like(d.k_cache)
    v2 = torch.empty_like(d.v_cache)
    k2[perm] = d.k_cache
    v2[perm] = d.v_cache
    t2 = torch.where(d.block_tables >= 0, perm[d.block_tables.clamp(min=0).long()].int(), d.block_tables)
    moved = _attn(d, k2, v2, t2)
    torch.cuda.synchronize()
    assert torch.equal(base.view(torch.int16), moved.view(torch.int16))


def test_shared_equals_duplicated_bit_identical():
    b = W.make_batch([900, 700, 1200], [1, 1, 1], num_blocks=200, seed=43, shared_prefix_tokens=512)
    d = DevBatch(b)
    base = _attn(d).clone()
    t2 = b.block_tables.copy()
    k2, v2 = d.k_cache.clone(), d.v_cache.clone()
    used = set(int(x) for x in t2.ravel() if x >= 0)
    free = [i for i in range(200) if i not in used]
    for r in (1, 2):
        for i in range(32):
            nb = free.pop()
            k2[nb] = d.k_cache[int(t2[r, i])]
            v2[nb] = d.v_cache[int(t2[r, i])]
            t2[r, i] = nb
    dup = _attn(d, k2, v2, torch.from_numpy(t2).cuda())
    torch.cuda.synchronize()
    assert torch.equal(base.view(torch.int16), dup.view(torch.int16))


def test_chunked_prefill_matches_one_shot():
    """A 2048-token prompt as four 512-token chunks gives the rows of the
    one-shot prefill (within tolerance of the oracle, and of each other)."""
    b = W.make_batch([2048], [2048], num_blocks=140, seed=44)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    one = _attn(d)
    parts = []
    for off in range(0, 2048, 512):
        q = d.q[off:off + 512].contiguous()
        sl = torch.tensor([off + 512], dtype=torch.int32)
        qi = torch.tensor([0, 512], dtype=torch.int32)
        parts.append(B.pa_attention_varlen(q, d.k_cache, d.v_cache, d.block_tables, sl.cuda(), qi.cuda(),
                                           b.sm_scale, seq_lens_host=sl, qo_indptr_host=qi))
    torch.cuda.synchronize()
    chunked = torch.cat(parts)
    ref, _, _, _ = oracle_step(b)
    compare(one, ref, what="one-shot")
    compare(chunked, ref, what="chunked")
    assert (one.float() - chunked.float()).abs().max().item() <= 1.5e-2


# ------------------------------------------------------------- error word
def test_bad_block_id_sets_error_word_without_fault():
    b = W.make_batch([100, 200], [1, 4], num_blocks=30, seed=45)
    d = DevBatch(b)
    t = b.block_tables.copy()
    t[0, 2] = 10_000                  # outside the pool
    t[1, 5] = -7
    ws = B.new_workspace(B.pa_attention_workspace_size(2, b.total_q, 32, 128, 200), "cuda")
    B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, torch.from_numpy(t).cuda(), d.seq_lens, d.qo_indptr,
                          b.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_INDEX
    # the context is still usable
    out = _attn(d)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------------- merge
def test_merge_lse_parity_and_identity():
    rng = np.random.default_rng(46)
    rows, H, D = 37, 32, 128
    o_a = W.normal_bf16(rng, (rows, H, D))
    o_b = W.normal_bf16(rng, (rows, H, D))
    la = rng.normal(0, 3, (rows, H)).astype(np.float32)
    lb = rng.normal(0, 3, (rows, H)).astype(np.float32)
    la[0, :5] = -np.inf
    lb[1, :5] = -np.inf
    la[2, :3] = lb[2, :3] = -np.inf
    from tests.util import bf16_dev
    go, gl = B.pa_merge_lse(bf16_dev(o_a), torch.from_numpy(la).cuda(), bf16_dev(o_b), torch.from_numpy(lb).cuda())
    ro, rl = oracle.merge_lse(o_a, la.astype(np.float64), o_b, lb.astype(np.float64))
    got = oracle.bf16_to_f64(bf16_host(go))
    assert np.max(np.abs(got - ro)) <= 2 ** -8 * np.max(np.abs(ro)) + 1e-6
    glh = gl.cpu().double().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(glh))
    assert np.max(np.abs(glh[fin] - rl[fin])) < 1e-5
    # in place into o_a
    oa_dev = bf16_dev(o_a)
    B.pa_merge_lse(oa_dev, torch.from_numpy(la).cuda(), bf16_dev(o_b), torch.from_numpy(lb).cuda(), o_out=oa_dev)
    torch.cuda.synchronize()
    assert torch.equal(oa_dev.view(torch.int16), go.view(torch.int16))


def test_merge_of_split_attention_equals_full():
    """Attention over keys [0, a) and [a, L) by two calls, merged by
    pa_merge_lse, equals attention over all L keys."""
    b = W.make_batch([1000] * 4, [1] * 4, num_blocks=300, seed=47)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    full, full_lse = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                           b.sm_scale, return_lse=True)
    a = 384
    sl1 = torch.full((4,), a, dtype=torch.int32)
    sl2 = torch.full((4,), 1000 - a, dtype=torch.int32)
    o1, l1 = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, sl1.cuda(), d.qo_indptr, b.sm_scale,
                                   seq_lens_host=sl1, return_lse=True)
    t2 = d.block_tables[:, a // 16:].contiguous()
    o2, l2 = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, t2, sl2.cuda(), d.qo_indptr, b.sm_scale,
                                   seq_lens_host=sl2, return_lse=True)
    m, ml = B.pa_merge_lse(o1, l1, o2, l2)
    torch.cuda.synchronize()
    assert (m.float() - full.float()).abs().max().item() < 1.5e-2
    assert (ml - full_lse).abs().max().item() < 1e-3


def test_launch_count_and_trace():
    b = W.workload_batch("tiny")
    d = DevBatch(b)
    n0 = B.pa_launch_count()
    B.pa_trace_enable(True)
    run_step(d)
    B.pa_trace_enable(False)
    rec = B.pa_trace_read()
    assert B.pa_launch_count() - n0 == len(rec) >= 2
    names = [k for k, _ in rec]
    assert names[0] == "kv_append" and "decode" in names
    assert all(ms > 0 for _, ms in rec)


# ------------------------------------------------ bounded waits (timeout path)
def test_decode_wait_timeout_is_recorded_and_the_context_stays_usable():
    # Rows long enough that every CTA's segment holds several pages; the
    # diagnostic decode kernel arms CTA 0's second page without copying it,
    # so that wait runs out after 1 ms: no fault, no hang.
    b = W.make_batch([700, 900, 1200, 1500], [1, 1, 1, 1], num_blocks=300, seed=W.SEED0 + 72)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    ws = B.new_workspace(B.pa_attention_workspace_size(4, 4, 32, 128, 1500), "cuda")
    B.pa_set_decode_fault_injection(True)
    try:
        B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr, b.sm_scale,
                              seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host, workspace=ws)
        torch.cuda.synchronize()
    finally:
        B.pa_set_decode_fault_injection(False)
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_TIMEOUT
    # a timed-out call leaves counters of the rows it cut; after zeroing the
    # workspace the next call is exact again
    ws.zero_()
    out, lse = B.pa_attention_varlen(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr,
                                     b.sm_scale, seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host,
                                     workspace=ws, return_lse=True)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == 0
    ref_out, ref_lse, _, _ = oracle_step(b)
    compare(out, ref_out, lse, ref_lse, what="after a timed-out call")
