"""pa_decode_step -- KV append and decode attention in one self-planned
launch ("Inference optimisation" §8.2.4 and "Continuous batching
architecture", section "CUDA graphs": a launch captured once for a padded
batch shape and replayed) -- through the C ABI against the oracle's decode
step: outputs within the bf16 tolerance, the pools bit-exact after the
append, padding rows zero, and one captured CUDA graph replayed over batches
with other lengths, tables and tokens."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import bf16_dev, bf16_host, compare

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


def step_inputs(seq_lens, *, num_blocks, seed, max_blocks=None, Hq=32, Hkv=8, D=128):
    """A padded decode batch: rows with seq_len 0 are padding (block-table
    row -1); every other row's blocks are private and randomly placed, its
    first seq_len - 1 tokens already in the pool."""
    rng = np.random.default_rng(seed)
    R = len(seq_lens)
    pages = [-(-int(L) // 16) for L in seq_lens]
    mb = max_blocks or max(max(pages), 1)
    assert sum(pages) <= num_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    tab = np.full((R, mb), -1, np.int32)
    nxt = 0
    for r, n in enumerate(pages):
        tab[r, :n] = perm[nxt:nxt + n]
        nxt += n
    k_cache = W.normal_bf16(rng, (num_blocks, Hkv, 16, D))
    v_cache = W.normal_bf16(rng, (num_blocks, Hkv, 16, D))
    # the new tokens' slots hold the workload sentinels until the append, so
    # a step that reads them instead of the new token is far off
    for r, L in enumerate(seq_lens):
        if 0 < L <= 16 * mb:
            blk, off = tab[r, (L - 1) // 16], (L - 1) % 16
            k_cache[blk, :, off] = W.K_SENTINEL
            v_cache[blk, :, off] = W.V_SENTINEL
    return dict(
        q=W.normal_bf16(rng, (R, Hq, D)),
        k_new=W.normal_bf16(rng, (R, Hkv, D)),
        v_new=W.normal_bf16(rng, (R, Hkv, D)),
        k_cache=k_cache,
        v_cache=v_cache,
        block_tables=tab,
        seq_lens=np.asarray(seq_lens, np.int32),
        sm_scale=1.0 / np.sqrt(D),
    )


class DevStep:
    """Device copies of a step's inputs (static buffers for graph capture)."""

    def __init__(self, h):
        self.q = bf16_dev(h["q"])
        self.k_new = bf16_dev(h["k_new"])
        self.v_new = bf16_dev(h["v_new"])
        self.k_cache = bf16_dev(h["k_cache"])
        self.v_cache = bf16_dev(h["v_cache"])
        self.block_tables = torch.from_numpy(h["block_tables"]).cuda()
        self.seq_lens = torch.from_numpy(h["seq_lens"]).cuda()

    def load(self, h):
        """Rewrite the buffers in place with another batch of the same shape."""
        for name in ("q", "k_new", "v_new", "k_cache", "v_cache"):
            getattr(self, name).copy_(bf16_dev(h[name]))
        self.block_tables.copy_(torch.from_numpy(h["block_tables"]))
        self.seq_lens.copy_(torch.from_numpy(h["seq_lens"]))


def run_step(d, h, max_seq_len, ws=None):
    out, lse = B.pa_decode_step(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                                h["sm_scale"], max_seq_len, workspace=ws, return_lse=True)
    return out, lse


def oracle_step(h, max_seq_len):
    k, v = h["k_cache"].copy(), h["v_cache"].copy()
    out, lse, bad = oracle.decode_step(h["q"], h["k_new"], h["v_new"], k, v, h["block_tables"], h["seq_lens"],
                                       h["sm_scale"], max_seq_len)
    return out, lse, k, v, bad


def check(d, out, lse, h, max_seq_len, what, ws=None):
    ref, ref_lse, k, v, bad = oracle_step(h, max_seq_len)
    torch.cuda.synchronize()
    pad = h["seq_lens"] == 0
    got_lse = lse.detach().cpu().double().numpy()
    assert np.all(np.isneginf(got_lse[pad])), f"{what}: padding lse"
    assert not np.any(bf16_host(out)[pad]), f"{what}: padding out"
    live = ~pad
    compare(out[torch.from_numpy(live).cuda()], ref[live], lse[torch.from_numpy(live).cuda()], ref_lse[live],
            what=what)
    assert np.array_equal(bf16_host(d.k_cache), k) and np.array_equal(bf16_host(d.v_cache), v), f"{what}: pools"
    if ws is not None:
        assert B.pa_get_device_error(ws) == 0, what
    return bad


@pytest.mark.parametrize("name,lens", [
    ("tiny", [17, 100, 256, 513]),
    ("one_token", [1]),
    ("page_edges", [16, 17, 32, 33, 15, 1, 48, 49]),
    ("ragged", [2100, 37, 16, 1, 700, 129, 4097, 300]),
])
def test_step_parity(name, lens):
    h = step_inputs(lens, num_blocks=sum(-(-L // 16) for L in lens) + 7, seed=310 + len(lens))
    d = DevStep(h)
    ws = B.new_workspace(B.pa_decode_step_workspace_size(len(lens), 32, 128, max(lens)), "cuda")
    out, lse = run_step(d, h, max(lens), ws)
    check(d, out, lse, h, max(lens), name, ws)


def test_step_short_dialogue():
    """The short-dialogue step: 64 rows of 2048..2303 tokens in a 5461-block pool."""
    b = W.workload_batch("short")
    assert np.all(np.diff(b.qo_indptr) == 1)
    h = dict(q=b.q, k_new=b.k_new, v_new=b.v_new, k_cache=b.k_cache, v_cache=b.v_cache,
             block_tables=b.block_tables, seq_lens=b.seq_lens.astype(np.int32), sm_scale=b.sm_scale)
    # the step's slots are the workload's own slot_mapping
    slots, bad = oracle.decode_step_slots(h["block_tables"], h["seq_lens"], 16, 4096)
    assert bad == 0 and np.array_equal(slots, b.slot_mapping)
    d = DevStep(h)
    out, lse = run_step(d, h, 4096)
    check(d, out, lse, h, 4096, "short")


def test_step_padding_rows():
    """A batch padded to its bucket: padding rows anywhere in the batch write
    nothing and give out 0, lse -inf."""
    lens = [300, 0, 17, 0, 0, 1000, 64, 0]
    assert B.pa_decode_step_bucket(4) == 4 and B.pa_decode_step_bucket(5) == 8
    h = step_inputs(lens, num_blocks=120, seed=321)
    d = DevStep(h)
    out, lse = run_step(d, h, 2048)
    check(d, out, lse, h, 2048, "padding")


def test_step_graph_replay():
    """One CUDA graph captured for an 8-row bucket (max_seq_len 4096) and
    replayed over three batches with other lengths, tables, padding, tokens
    and pool contents, each matching the oracle."""
    R, maxlen, nb = 8, 4096, 900
    batches = [
        step_inputs([2048, 2049, 17, 1, 4096, 333, 0, 0], num_blocks=nb, seed=331, max_blocks=256),
        step_inputs([5, 0, 0, 0, 0, 0, 0, 0], num_blocks=nb, seed=332, max_blocks=256),
        step_inputs([1000, 1001, 1002, 1003, 3000, 16, 32, 4095], num_blocks=nb, seed=333, max_blocks=256),
    ]
    d = DevStep(batches[0])
    ws = B.new_workspace(B.pa_decode_step_workspace_size(R, 32, 128, maxlen), "cuda")
    out = torch.empty_like(d.q)
    lse = torch.empty((R, 32), dtype=torch.float32, device="cuda")
    args = (d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, batches[0]["sm_scale"], maxlen)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.pa_decode_step(*args, out=out, lse=lse, workspace=ws, stream=s)  # warm-up (attributes set)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.pa_decode_step(*args, out=out, lse=lse, workspace=ws)
    launches = B.pa_launch_count()
    for i, h in enumerate(batches):
        d.load(h)
        g.replay()
        check(d, out, lse, h, maxlen, f"replay {i}", ws)
    assert B.pa_launch_count() == launches  # replays launch through the graph only


@pytest.mark.parametrize("ctas", [8, 16, 24])
def test_step_item_windows(ctas):
    """Segments holding more than 64 rows are walked in windows of 64 items:
    200 one- or two-page rows on 1 to 3 segments per kv head."""
    rng = np.random.default_rng(340 + ctas)
    lens = list(rng.integers(1, 33, size=200))
    B.pa_set_decode_ctas(ctas)
    try:
        h = step_inputs(lens, num_blocks=420, seed=341 + ctas)
        d = DevStep(h)
        ws = B.new_workspace(B.pa_decode_step_workspace_size(len(lens), 32, 128, 32), "cuda")
        out, lse = run_step(d, h, 32, ws)
        torch.cuda.synchronize()
    finally:
        B.pa_set_decode_ctas(0)
    check(d, out, lse, h, 32, f"windows {ctas}", ws)


@pytest.mark.parametrize("ctas", [1, 7, 456, 1024])
def test_step_forced_grid(ctas):
    lens = [2100, 37, 16, 1, 700, 129, 0, 513]
    B.pa_set_decode_ctas(ctas)
    try:
        h = step_inputs(lens, num_blocks=260, seed=350 + ctas)
        d = DevStep(h)
        ws = B.new_workspace(B.pa_decode_step_workspace_size(len(lens), 32, 128, 2200), "cuda")
        out, lse = run_step(d, h, 2200, ws)
        torch.cuda.synchronize()
    finally:
        B.pa_set_decode_ctas(0)
    check(d, out, lse, h, 2200, f"grid {ctas}", ws)


def test_step_errors_recorded_without_fault():
    """A block id outside the pool and a row longer than max_seq_len are
    recorded in the error word; the row past the bound gives zero output,
    the other rows are unaffected, and the context stays usable."""
    lens = [100, 50, 900]
    h = step_inputs(lens, num_blocks=80, seed=361)
    d = DevStep(h)
    ws = B.new_workspace(max(B.pa_decode_step_workspace_size(3, 32, 128, 512),
                             B.pa_decode_step_workspace_size(3, 32, 128, 1024)), "cuda")
    out, lse = run_step(d, h, 512, ws)           # row 2 is longer than 512
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_INDEX
    assert not np.any(bf16_host(out)[2]) and torch.all(torch.isneginf(lse[2]))
    ref, ref_lse, _, _, bad = oracle_step(h, 512)
    assert bad == 1
    compare(out[:2], ref[:2], lse[:2], ref_lse[:2], what="rows within the bound")
    ws.zero_()
    bad_tab = h["block_tables"].copy()
    bad_tab[0, 2] = 10 ** 6
    d.block_tables.copy_(torch.from_numpy(bad_tab))
    run_step(d, h, 1024, ws)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_INDEX
    torch.zeros(1, device="cuda").sum().item()  # the context still works


def test_step_sweep_point_b128_2048():
    """The largest 2048-token sweep point (128 rows) through pa_decode_step,
    against the oracle on every output."""
    lens = [2048] * 128
    h = step_inputs(lens, num_blocks=128 * 128 + 50, seed=371)
    d = DevStep(h)
    out, lse = run_step(d, h, 2048)
    check(d, out, lse, h, 2048, "b128 x 2048")


def test_step_graph_of_layers():
    """A CUDA graph of 4 layers (one pa_decode_step each, own pools, one
    shared workspace), as the 36-layer sweep captures it; every layer's
    output and pools match the oracle after a replay with new lengths."""
    R, maxlen, nb, layers = 8, 1024, 600, 4
    lens0 = [1024, 700, 33, 1, 512, 0, 64, 999]
    lens1 = [17, 1000, 256, 0, 0, 640, 1, 1024]
    hs = [step_inputs(lens0, num_blocks=nb, seed=380 + l, max_blocks=64) for l in range(layers)]
    ds = [DevStep(h) for h in hs]
    ws = B.new_workspace(B.pa_decode_step_workspace_size(R, 32, 128, maxlen), "cuda")
    outs = [torch.empty_like(d.q) for d in ds]
    lses = [torch.empty((R, 32), dtype=torch.float32, device="cuda") for _ in ds]

    def step():
        for d, o, l_ in zip(ds, outs, lses):
            B.pa_decode_step(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                             hs[0]["sm_scale"], maxlen, out=o, lse=l_, workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for lens, seed in ((lens0, 390), (lens1, 395)):
        hs = [step_inputs(lens, num_blocks=nb, seed=seed + l, max_blocks=64) for l in range(layers)]
        for d, h in zip(ds, hs):
            d.load(h)
        g.replay()
        for l, (d, h) in enumerate(zip(ds, hs)):
            check(d, outs[l], lses[l], h, maxlen, f"layer {l} lens {lens[:3]}", ws)


def test_step_long_row_over_many_segments():
    """One 150,000-token row among short ones: its pages span dozens of CTAs
    (each segment at most 1,024 pages), its pieces are merged by the last."""
    lens = [150_000, 40, 2, 5000]
    h = step_inputs(lens, num_blocks=sum(-(-L // 16) for L in lens) + 10, seed=401)
    d = DevStep(h)
    ws = B.new_workspace(B.pa_decode_step_workspace_size(len(lens), 32, 128, 150_000), "cuda")
    out, lse = run_step(d, h, 150_000, ws)
    check(d, out, lse, h, 150_000, "long row", ws)
