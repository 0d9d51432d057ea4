"""The C-ABI library loads and exports what include/pa.h declares, and its
host-side validation rejects bad arguments before launching anything.
Runs without a GPU: no call here reaches a kernel."""
import ctypes
import subprocess

import numpy as np

import pytest

from paged_kv_decode_varlen_gb300 import binding as b

lib = b._lib
FAKE = ctypes.c_void_p(1 << 20)  # non-null, aligned; never dereferenced on these paths


def test_header_symbols_exported():
    names = b.header_functions()
    assert len(names) >= 13
    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared in pa.h but not exported: {missing}"
    for n in names:
        assert getattr(lib, n) is not None


def test_abi_version_and_status_strings():
    assert b.pa_abi_version() == 1
    assert b.status_string(0) == "PA_OK"
    assert b.status_string(5) == "PA_ERR_DEVICE_INDEX"
    assert b.status_string(99) == "PA_ERR_UNKNOWN"


def test_workspace_size_query():
    small = b.pa_attention_workspace_size(4, 4, 32, 128, 513)
    big = b.pa_attention_workspace_size(64, 64, 32, 128, 2303)
    assert small >= b.PA_ERROR_WORD_BYTES and big >= small and big % 256 == 0 and small % 256 == 0
    # error word + counters (num_reqs x 8 int32) + two partial slots of 4 heads x 129 fp32 per warp
    # segment (4 per CTA) for a 480-CTA bound
    slots = 2 * 480 * 4 * 4
    assert b.pa_attention_workspace_size(1, 1, 32, 128, 16) == 256 + 256 + slots * 512 + slots * 4
    assert b.pa_attention_workspace_size(100, 100, 32, 128, 16) == 256 + 3328 + slots * 512 + slots * 4
    # very long rows raise the grid bound (1024 pages per CTA at most)
    assert b.pa_attention_workspace_size(1024, 1024, 32, 128, 1 << 20) > big


def _attn(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, nb=64, bt=FAKE, mb=40, sl=FAKE, qi=FAKE, slh=None, qih=None, R=2, tq=2, Hq=32,
                Hkv=8, D=128, P=16, scale=0.088, out=FAKE, lse=None, ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    slh = (ctypes.c_int32 * 2)(*kw.get("seq", (17, 100)))
    qih = (ctypes.c_int32 * 3)(*kw.get("ind", (0, 1, 2)))
    return lib.pa_attention_varlen(args["q"], args["k"], args["v"], args["nb"], args["bt"], args["mb"], args["sl"],
                                   args["qi"], slh, qih, args["R"], args["tq"], args["Hq"], args["Hkv"], args["D"],
                                   args["P"], args["scale"], args["out"], args["lse"], args["ws"], args["wsb"],
                                   args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), b.PA_ERR_UNSUPPORTED),
    (dict(P=32), b.PA_ERR_UNSUPPORTED),
    (dict(Hq=16), b.PA_ERR_UNSUPPORTED),
    (dict(Hkv=0), b.PA_ERR_INVALID_ARG),
    (dict(q=None), b.PA_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((1 << 20) + 2)), b.PA_ERR_INVALID_ARG),
    (dict(ws=ctypes.c_void_p((1 << 20) + 16)), b.PA_ERR_INVALID_ARG),
    (dict(ind=(0, 1, 3)), b.PA_ERR_INVALID_ARG),          # qo_indptr[R] != total_q
    (dict(ind=(1, 1, 2)), b.PA_ERR_INVALID_ARG),          # qo_indptr[0] != 0
    (dict(ind=(0, 2, 1), tq=1), b.PA_ERR_INVALID_ARG),    # decreasing
    (dict(seq=(0, 100)), b.PA_ERR_INVALID_ARG),           # qo_len 1 > seq_len 0
    (dict(seq=(17, 1000)), b.PA_ERR_INVALID_ARG),         # 63 pages > max_blocks_per_req 40
    (dict(seq=(17, (1 << 20) + 1)), b.PA_ERR_UNSUPPORTED),
    (dict(wsb=1024, seq=(17, 600)), b.PA_ERR_WORKSPACE_TOO_SMALL),
    (dict(nb=0), b.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), b.PA_ERR_INVALID_ARG),
])
def test_attention_validation(kw, status):
    assert _attn(**kw) == status
    assert lib.pa_last_error_message().decode() != ""


def test_append_validation():
    ws = FAKE
    assert lib.pa_kv_append(FAKE, FAKE, FAKE, -1, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_kv_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 16, 8, 64, ws, 256, None) == b.PA_ERR_UNSUPPORTED
    assert lib.pa_kv_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 8, 8, 128, ws, 256, None) == b.PA_ERR_UNSUPPORTED
    assert lib.pa_kv_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 16, 8, 128, ws, 64, None) == \
        b.PA_ERR_WORKSPACE_TOO_SMALL
    assert lib.pa_kv_append(None, FAKE, FAKE, 4, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_kv_append(ctypes.c_void_p((1 << 20) + 8), FAKE, FAKE, 4, FAKE, FAKE, 64, 16, 8, 128, ws, 256,
                            None) == b.PA_ERR_INVALID_ARG
    # zero tokens: valid, launches nothing
    n0 = lib.pa_launch_count()
    assert lib.pa_kv_append(None, None, None, 0, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == b.PA_OK
    assert lib.pa_launch_count() == n0


def test_merge_validation():
    assert lib.pa_merge_lse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 32, 100, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_merge_lse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 32, 128, None) == b.PA_ERR_INVALID_ARG
    # lse_out overlapping lse_a is refused
    assert lib.pa_merge_lse(FAKE, ctypes.c_void_p(1 << 24), FAKE, ctypes.c_void_p(1 << 25), FAKE,
                            ctypes.c_void_p((1 << 24) + 8), 4, 32, 128, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_merge_lse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 32, 128, None) == b.PA_OK


def test_grid_override_bounds():
    assert lib.pa_set_decode_ctas(1025) == b.PA_ERR_INVALID_ARG
    assert lib.pa_set_decode_ctas(-1) == b.PA_ERR_INVALID_ARG
    assert lib.pa_set_decode_ctas(0) == b.PA_OK
    assert lib.pa_set_prefill_ctas(-2) == b.PA_ERR_INVALID_ARG
    assert lib.pa_set_prefill_ctas(1025) == b.PA_ERR_INVALID_ARG
    assert lib.pa_set_prefill_ctas(-1) == b.PA_OK
    assert lib.pa_set_prefill_ctas(16) == b.PA_OK
    assert lib.pa_set_prefill_ctas(0) == b.PA_OK


def test_fault_injection_switch_bounds():
    assert lib.pa_set_decode_fault_injection(2) == b.PA_ERR_INVALID_ARG
    assert lib.pa_set_decode_fault_injection(-1) == b.PA_ERR_INVALID_ARG
    assert lib.pa_set_decode_fault_injection(0) == b.PA_OK


def test_shared_prefix_workspace_size():
    base = b.pa_attention_workspace_size(16, 16, 32, 128, 8447)
    assert b.pa_shared_prefix_workspace_size(16, 16, 32, 128, 8447, 0) == base
    # + prefix partial (16 x 32 rows of 128 fp32) + its lse
    # + 48 key-chunk partials (one per 128-key tile; the 512-CTA bound / 8 kv heads is larger)
    # + two int32 counters per (query tile, kv head), in 256-byte units
    rows = 16 * 32
    flags = lambda qtiles: (2 * qtiles * 8 * 4 + 255) // 256 * 256
    assert b.pa_shared_prefix_workspace_size(16, 16, 32, 128, 8447, 384) == \
        base + rows * 512 + rows * 4 + 48 * rows * 512 + 48 * rows * 4 + flags(1)
    # a 5-page prefix is one 128-key tile: one chunk, no chunk partials
    assert b.pa_shared_prefix_workspace_size(16, 16, 32, 128, 8447, 5) == base + rows * 512 + rows * 4 + flags(1)
    # 64 query tiles of 32 tokens x 8 kv heads reach the CTA bound: one chunk
    base2 = b.pa_attention_workspace_size(4, 2048, 32, 128, 3000)
    assert b.pa_shared_prefix_workspace_size(4, 2048, 32, 128, 3000, 96) == \
        base2 + 2048 * 32 * 512 + 2048 * 32 * 4 + flags(64)
    # 32 query tiles x 8 kv heads: two chunks
    base3 = b.pa_attention_workspace_size(4, 1024, 32, 128, 3000)
    assert b.pa_shared_prefix_workspace_size(4, 1024, 32, 128, 3000, 96) == \
        base3 + 3 * (1024 * 32 * 512 + 1024 * 32 * 4) + flags(32)
    assert b.pa_shared_prefix_workspace_size(4, 4, 32, 128, 100, -1) == 0


def _attn_prefix(pages, seq=(40, 100), ind=(0, 1, 2), wsb=1 << 30, mb=40):
    slh = (ctypes.c_int32 * 2)(*seq)
    qih = (ctypes.c_int32 * 3)(*ind)
    return lib.pa_attention_varlen_shared_prefix(FAKE, FAKE, FAKE, 64, FAKE, mb, FAKE, FAKE, slh, qih, 2, ind[2],
                                                 32, 8, 128, 16, pages, 0.088, FAKE, None, FAKE, wsb, None)


def test_shared_prefix_validation():
    assert _attn_prefix(-1) == b.PA_ERR_INVALID_ARG
    assert _attn_prefix(41) == b.PA_ERR_INVALID_ARG                      # beyond max_blocks_per_req
    assert _attn_prefix(3) == b.PA_ERR_INVALID_ARG                       # 40 - 1 = 39 cached keys < 48
    assert _attn_prefix(2, seq=(40, 40), ind=(0, 1, 11)) == b.PA_ERR_INVALID_ARG  # 40 - 10 = 30 < 32
    # the base workspace is not enough once the prefix pass runs
    need = b.pa_shared_prefix_workspace_size(2, 2, 32, 128, 100, 2)
    assert _attn_prefix(2, wsb=need - 256) == b.PA_ERR_WORKSPACE_TOO_SMALL
    assert "workspace" in lib.pa_last_error_message().decode()


def test_copy_blocks_validation():
    ws = FAKE
    assert lib.pa_copy_blocks(FAKE, FAKE, -1, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(None, FAKE, 2, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(FAKE, FAKE, 2, FAKE, FAKE, 0, 16, 8, 128, ws, 256, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(FAKE, FAKE, 2, FAKE, FAKE, 64, 8, 8, 128, ws, 256, None) == b.PA_ERR_UNSUPPORTED
    assert lib.pa_copy_blocks(FAKE, FAKE, 2, FAKE, FAKE, 64, 16, 8, 128, ws, 64, None) == \
        b.PA_ERR_WORKSPACE_TOO_SMALL
    assert lib.pa_copy_blocks(FAKE, FAKE, 2, ctypes.c_void_p((1 << 20) + 8), FAKE, 64, 16, 8, 128, ws, 256,
                              None) == b.PA_ERR_INVALID_ARG
    n0 = lib.pa_launch_count()
    assert lib.pa_copy_blocks(None, None, 0, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == b.PA_OK
    assert lib.pa_launch_count() == n0


def test_q8_validation():
    ws = FAKE
    assert lib.pa_kv_append_q8(FAKE, FAKE, FAKE, -1, FAKE, FAKE, 64, 16, 8, 128, ws, 256, None) == \
        b.PA_ERR_INVALID_ARG
    assert lib.pa_kv_append_q8(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 16, 8, 64, ws, 256, None) == \
        b.PA_ERR_UNSUPPORTED
    slh = (ctypes.c_int32 * 2)(40, 100)
    qih = (ctypes.c_int32 * 3)(0, 1, 5)      # request 1 has 4 queries: not a decode row
    assert lib.pa_attention_varlen_q8(FAKE, FAKE, FAKE, 64, FAKE, 40, FAKE, FAKE, slh, qih, 2, 5, 32, 8, 128, 16,
                                      0.088, FAKE, None, FAKE, 1 << 30, None) == b.PA_ERR_UNSUPPORTED
    assert "q8_0" in lib.pa_last_error_message().decode()


def test_decode_step_sizes_and_buckets():
    assert [b.pa_decode_step_bucket(n) for n in (0, 1, 2, 3, 5, 64, 65, 1024)] == [1, 1, 2, 4, 8, 64, 128, 1024]
    assert b.pa_decode_step_bucket(1025) == -1 and b.pa_decode_step_bucket(-1) == -1
    small = b.pa_decode_step_workspace_size(8, 32, 128, 4096)
    assert small > b.PA_ERROR_WORD_BYTES and small % 256 == 0
    # the size depends only on the scalars; more rows or longer rows never shrink it
    assert b.pa_decode_step_workspace_size(8, 32, 128, 4096) == small
    assert b.pa_decode_step_workspace_size(64, 32, 128, 4096) >= small
    assert b.pa_decode_step_workspace_size(8, 32, 128, 1 << 16) >= small
    for bad in [(1025, 32, 128, 4096), (8, 32, 128, 0), (8, 32, 128, (1 << 20) + 1), (-1, 32, 128, 16),
                (8, 2, 128, 16), (1024, 32, 128, 1 << 20)]:
        assert b.pa_decode_step_workspace_size(*bad) == 0, bad


def _step(**kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, k=FAKE, v=FAKE, nb=64, bt=FAKE, mb=40, sl=FAKE, R=4, maxlen=600, Hq=32,
             Hkv=8, D=128, P=16, scale=0.088, out=FAKE, lse=None, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.pa_decode_step(a["q"], a["kn"], a["vn"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"], a["R"],
                              a["maxlen"], a["Hq"], a["Hkv"], a["D"], a["P"], a["scale"], a["out"], a["lse"], a["ws"],
                              a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), b.PA_ERR_INVALID_ARG),
    (dict(kn=None), b.PA_ERR_INVALID_ARG),
    (dict(sl=None), b.PA_ERR_INVALID_ARG),
    (dict(ws=None), b.PA_ERR_INVALID_ARG),
    (dict(vn=ctypes.c_void_p((1 << 20) + 8)), b.PA_ERR_INVALID_ARG),
    (dict(maxlen=0), b.PA_ERR_INVALID_ARG),
    (dict(maxlen=(1 << 20) + 1), b.PA_ERR_INVALID_ARG),
    (dict(nb=0), b.PA_ERR_INVALID_ARG),
    (dict(mb=0), b.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), b.PA_ERR_INVALID_ARG),
    (dict(R=1025), b.PA_ERR_UNSUPPORTED),
    (dict(Hkv=4), b.PA_ERR_UNSUPPORTED),
    (dict(D=64), b.PA_ERR_UNSUPPORTED),
    (dict(wsb=1024), b.PA_ERR_WORKSPACE_TOO_SMALL),
    (dict(R=1024, maxlen=1 << 20), b.PA_ERR_UNSUPPORTED),
])
def test_decode_step_validation(kw, status):
    n0 = lib.pa_launch_count()
    assert _step(**kw) == status, lib.pa_last_error_message().decode()
    assert lib.pa_launch_count() == n0


def test_decode_step_empty_batch_launches_nothing():
    n0 = lib.pa_launch_count()
    assert _step(R=0, q=None, kn=None, vn=None, bt=None, sl=None, out=None) == b.PA_OK
    assert lib.pa_launch_count() == n0


# ------------------------------------------------- tile-job grid (host model)
def _tile_jobs(batch, kv_heads=8):
    """Key tiles of each tensor-core job in the kernel's order (for each kv
    head, the 32-query tiles by decreasing key extent) and the decode rows'
    (page, kv head) slab count, from a batch's metadata."""
    seq = [int(x) for x in batch.seq_lens]
    qoi = [int(x) for x in batch.qo_indptr]
    qo = [qoi[i + 1] - qoi[i] for i in range(len(seq))]
    ext = sorted((L - q + min(q, j0 + 32) for L, q in zip(seq, qo) if q > 1 for j0 in range(0, q, 32)), reverse=True)
    slabs = sum(-(-L // 16) for L, q in zip(seq, qo) if q == 1) * kv_heads
    return [-(-e // 128) for e in ext] * kv_heads, slabs


def test_tile_grid_model_picks_the_measured_grids():
    from paged_kv_decode_varlen_gb300 import workloads as W
    # mixed batch: the 512-token chunk's 128 jobs beside the decode launch on
    # 16 CTAs (step 215.5 us; 8 / 12 / 24 CTAs measured 359 / 253 / 220 us)
    jobs, slabs = _tile_jobs(W.workload_batch("mixed", scale=1.0))
    assert len(jobs) == 128 and slabs > 0
    assert b.pa_plan_tile_grid(jobs, slabs, 152) == 16
    # verify rows: 512 jobs of 17-18 tiles alone on 128 CTAs, four full
    # rounds (measured 106.6 us against 114.1 us on 152 and 115.3 us on 104)
    jobs, slabs = _tile_jobs(W.workload_batch("verify", scale=1.0))
    assert len(jobs) == 512 and slabs == 0 and set(jobs) <= {17, 18}
    assert b.pa_plan_tile_grid(jobs, 0, 152) == 128


def test_tile_grid_model_rounds_and_fallbacks():
    # equal jobs alone: the smallest grid for the fewest rounds (320 jobs: 3
    # rounds of 107, not 152 + 152 + 16)
    assert b.pa_plan_tile_grid([16] * 320, 0, 152) == 107
    # 1024 jobs: 7 rounds either way, every SM busy
    assert b.pa_plan_tile_grid([16] * 1024, 0, 152) == 152
    # fewer than two jobs per SM alone, or no jobs: one CTA per job
    assert b.pa_plan_tile_grid([16] * 303, 0, 152) == 0
    assert b.pa_plan_tile_grid([], 0, 152) == 0
    # beside a decode stream: fewer CTAs than jobs, at most half the SMs
    g = b.pa_plan_tile_grid([16] * 40, 10 ** 6, 152)
    assert 0 <= g < 40 and g <= 76
    # a decode stream too short to hide the jobs behind: the jobs first
    assert b.pa_plan_tile_grid([16] * 128, 8, 152) == 0


def test_tile_grid_model_rejects_bad_arguments():
    arr = (ctypes.c_int32 * 2)(16, 16)
    out = ctypes.c_int32(7)
    assert lib.pa_plan_tile_grid(arr, 2, 0, 152, None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_tile_grid(None, 2, 0, 152, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG and out.value == 0
    assert lib.pa_plan_tile_grid(arr, -1, 0, 152, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_tile_grid(arr, 393217, 0, 152, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_tile_grid(arr, 2, 0, 0, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_tile_grid(arr, 2, 0, 1025, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_tile_grid(arr, 2, -1, 152, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG
    bad = (ctypes.c_int32 * 2)(16, 0)
    assert lib.pa_plan_tile_grid(bad, 2, 0, 152, ctypes.byref(out)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_tile_grid(arr, 2, 0, 152, ctypes.byref(out)) == b.PA_OK and out.value == 0


# ------------------------------------------------------- decode plan (host)
def test_decode_plan_picks_the_measured_kernels():
    from paged_kv_decode_varlen_gb300 import workloads as W
    # short dialogue: the warp-granular kernel, one 12-warp CTA per SM
    seq = [int(x) for x in W.workload_batch("short", scale=1.0).seq_lens]
    assert b.pa_plan_decode_grid(seq, 8, 152) == (152, True)
    # 36-layer sweep at 2048 tokens: short segments at b = 1 and 8 keep the
    # CTA-granular kernel (the warp-granular one measured 28.6 and 23.9 us
    # per layer there against 10.5 and 22.2); from b = 32 the warp-granular
    for bsz, wg in [(1, False), (8, False), (32, True), (64, True), (128, True)]:
        grid, got = b.pa_plan_decode_grid([2048] * bsz, 8, 152)
        assert got == wg and grid % 8 == 0, (bsz, grid, got)
        if wg:
            assert grid == 152
        else:
            assert grid <= 3 * 152
    # a single 128K-token row: every SM, warp segments of whole pages
    assert b.pa_plan_decode_grid([131072], 8, 152) == (152, True)


@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
@pytest.mark.parametrize("rows", [1, 64, 1024])
def test_decode_plan_size_limit(hkv, rows):
    # one launch's decode rows hold at most 1,048,576 / num_kv_heads pages
    per_row = (1048576 // hkv) // rows
    grid, _ = b.pa_plan_decode_grid([per_row * 16] * rows, hkv, 152)
    assert grid == 1024
    with pytest.raises(b.PAError) as e:
        b.pa_plan_decode_grid([(per_row + 1) * 16] * rows, hkv, 152)
    assert e.value.status == b.PA_ERR_UNSUPPORTED


def test_decode_plan_grids_are_whole_kv_heads():
    rng = np.random.default_rng(11)
    for _ in range(40):
        n = int(rng.integers(1, 1025))
        hkv = int(rng.choice([1, 2, 4, 8]))
        # lengths within the size limit (at most 1,048,576 / hkv pages)
        cap = max(1, min(20000, (1048576 // hkv) // n * 16))
        seq = [int(x) for x in rng.integers(1, cap + 1, n)]
        grid, wg = b.pa_plan_decode_grid(seq, hkv, 152)
        assert 0 < grid <= 1024 and grid % hkv == 0
        # the warp-granular kernel fills one wave of one CTA per SM before it
        # takes more (segments capped at 3,072 pages or 192 rows)
        pages = sum(-(-L // 16) for L in seq)
        if wg and grid > 152:
            assert pages > (152 // hkv) * 3072 or n > (152 // hkv) * 192 or grid // hkv > 152 // hkv
    assert b.pa_plan_decode_grid([], 8, 152) == (0, False)


def test_decode_plan_follows_a_forced_grid():
    b.pa_set_decode_ctas(64)
    try:
        grid, _ = b.pa_plan_decode_grid([2048] * 64, 8, 152)
    finally:
        b.pa_set_decode_ctas(0)
    assert grid == 64


def test_decode_plan_rejects_bad_arguments():
    arr = (ctypes.c_int32 * 2)(100, 200)
    g, w = ctypes.c_int32(5), ctypes.c_int32(5)
    ok_args = (arr, 2, 8, 152, ctypes.byref(g), ctypes.byref(w))
    assert lib.pa_plan_decode_grid(*ok_args) == b.PA_OK and g.value > 0
    assert lib.pa_plan_decode_grid(arr, 2, 8, 152, None, ctypes.byref(w)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_decode_grid(arr, 2, 8, 152, ctypes.byref(g), None) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_decode_grid(None, 2, 8, 152, ctypes.byref(g), ctypes.byref(w)) == b.PA_ERR_INVALID_ARG
    assert g.value == 0 and w.value == 0
    assert lib.pa_plan_decode_grid(arr, 1025, 8, 152, ctypes.byref(g), ctypes.byref(w)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_decode_grid(arr, 2, 0, 152, ctypes.byref(g), ctypes.byref(w)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_decode_grid(arr, 2, 257, 152, ctypes.byref(g), ctypes.byref(w)) == b.PA_ERR_INVALID_ARG
    assert lib.pa_plan_decode_grid(arr, 2, 8, 0, ctypes.byref(g), ctypes.byref(w)) == b.PA_ERR_INVALID_ARG
    bad = (ctypes.c_int32 * 2)(100, 0)
    assert lib.pa_plan_decode_grid(bad, 2, 8, 152, ctypes.byref(g), ctypes.byref(w)) == b.PA_ERR_INVALID_ARG


def test_binding_signatures_match_the_header():
    """Every prototype in include/pa.h has a ctypes signature in the binding
    with the same number of arguments and matching C types, so no argument
    crosses the C ABI in the wrong width."""
    import re
    src = re.sub(r"/\*.*?\*/", "", open(b.HEADER).read(), flags=re.S)
    protos = dict(re.findall(r"\b(pa_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S))
    rets = dict((n, t.strip()) for t, n in re.findall(r"^\s*([\w\s\*]+?)\s*\b(pa_\w+)\s*\(", src, flags=re.M))
    assert set(protos) == set(b._SIGS) and len(protos) >= 26

    def ctype_of(decl):
        decl = decl.strip()
        if "*" in decl or decl.split()[0] == "pa_stream_t":
            return "ptr"
        base = decl.replace("const ", "").split()[0]
        return {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
                "float": ctypes.c_float, "pa_status": ctypes.c_int32}[base]

    for name, (res, args) in b._SIGS.items():
        params = [p for p in (x.strip() for x in protos[name].split(",")) if p and p != "void"]
        assert len(params) == len(args), name
        for p, a in zip(params, args):
            want = ctype_of(p)
            if want == "ptr":
                assert a in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(a, "_type_") and a.__name__.startswith("LP_"), \
                    (name, p, a)
            else:
                assert a is want, (name, p, a)
        ret = rets[name]
        want = ctypes.c_char_p if "char" in ret and "*" in ret else ctype_of(ret)
        assert res is want, (name, ret, res)
