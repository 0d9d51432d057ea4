#!/usr/bin/env python
"""Benchmark of the paged varlen attention hot path on GB300.

One step = pa_kv_append of the step's new tokens + pa_attention_varlen over
one layer of a continuous batch, both through the C ABI (libpa).  Default
workload: the short-dialogue decode step -- 64 decode rows with contexts
uniform in [2048, 2303], 16-token pages placed at random in a 10,922-block
pool, 32 q heads / 8 kv heads, head_dim 128, bf16, N(0,1) data.

Metric: achieved HBM GB/s of the step's algorithmic bytes (unique KV pages
+ q + out + block table + append), also reported as tokens per layer-step
per second.  Between timed steps a 256 MiB buffer is read to flush the
129 MB L2 (a read leaves no dirty lines to write back), outside the timed
events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

With N > 1 (launched by torch.distributed.run) every rank runs an
independent replica on its own GPU (the path has no exchange step); value is
the sum of all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_decode_varlen_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention achieved HBM GB/s (% of GB300 peak); tokens/layer-step/s"
L2_FLUSH_BYTES = 256 << 20
WORKLOADS = {
    "short": "short-dialogue decode step: 64 decode rows, seq_len U[2048,2303], 16-token pages in a 10,922-block "
             "pool, GQA 32/8 heads, head_dim 128, bf16, 1 layer, kv_append of 64 tokens",
    "shared": "shared-prefix long-context decode: 16 rows, seq_len U[8192,8447], first 6144 tokens (384 pages) "
              "shared, 5461-block pool, GQA 32/8, head_dim 128, bf16, 1 layer, kv_append of 16 tokens",
    "mixed": "mixed chunked-prefill batch: one 512-token chunk at offset 1536 + 63 decode rows seq_len "
             "U[2048,8192], 24,576-block pool, GQA 32/8, head_dim 128, bf16, 1 layer, kv_append of 575 tokens",
    "tiny": "tiny decode: 4 decode rows seq_len {17,100,256,513}, 64-block pool, GQA 32/8, head_dim 128, bf16",
    "verify": "speculative-verify step: 64 rows of 5 query tokens (4-token drafts) over seq_len U[2048,2303], "
              "10,922-block pool, GQA 32/8, head_dim 128, bf16, 1 layer, kv_append of 320 tokens",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_tflops_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["bf16_tflops"])
    return 1900.0


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("decode.cu", "common.cuh"):
        h.update(open(os.path.join(ROOT, "paged_kv_decode_varlen_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel="decode"):
    """DRAM bytes per launch of the decode kernel (kernel = "decode") or of
    the decode step ("decode_step") from the committed ncu summary, if it was
    taken on the current decode kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------ host inputs
def stage_layout(tensors, align=256):
    """Byte layout that lays the step's input tensors end to end in one
    buffer, each at an `align`-byte boundary, so the host->device transfer
    of a step is one copy.  Returns ({name: (offset, dtype, shape)}, nbytes)."""
    layout, off = {}, 0
    for name, t in tensors.items():
        off = (off + align - 1) // align * align
        layout[name] = (off, t.dtype, tuple(t.shape))
        off += t.numel() * t.element_size()
    return layout, off


def stage_views(buf, layout):
    """Typed views of one uint8 buffer laid out by stage_layout."""
    import torch
    views = {}
    for name, (off, dtype, shape) in layout.items():
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        views[name] = buf[off:off + n].view(dtype).view(shape)
    return views


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over the ranks of the default
    process group (the slowest rank's times); the input on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_gbs(bytes_per_rank, world, ms):
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        self.gpu_index = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.rows:
            if self.t0 is None or not (self.t0 - 0.05 <= t <= (self.t1 or t) + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_median": statistics.median(power)}


# --------------------------------------------------------------- CPU oracle
def oracle_step_time(batch, rows=None):
    """Wall time of the oracle doing one step (append on a copy of the pool,
    then attention) over `rows` (default all) of the batch."""
    import oracle
    b = batch if rows is None else subset(batch, rows)
    k, v = b.k_cache, b.v_cache
    t0 = time.perf_counter()
    oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, k, v)
    oracle.attention_varlen(b.q, k, v, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    return time.perf_counter() - t0, b


def subset(b, rows):
    """The sub-batch of the given requests (sharing the same pool arrays)."""
    rows = np.asarray(rows)
    qo = np.diff(b.qo_indptr)[rows]
    ind = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    toks = np.concatenate([np.arange(b.qo_indptr[r], b.qo_indptr[r + 1]) for r in rows]) if len(rows) else \
        np.zeros(0, np.int64)
    return W.Batch(q=b.q[toks], k_cache=b.k_cache, v_cache=b.v_cache, block_tables=b.block_tables[rows],
                   seq_lens=b.seq_lens[rows], qo_indptr=ind, k_new=b.k_new[toks], v_new=b.v_new[toks],
                   slot_mapping=b.slot_mapping[toks], sm_scale=b.sm_scale, meta=b.meta)


def cpu_baseline(batch, min_seconds=10.0, max_seconds=30.0):
    import oracle
    cores = oracle.host_threads()
    bytes_full = W.step_bytes(batch)["unique"]
    times = []
    while len(times) < 3 or (sum(times) < min_seconds and sum(times) + sum(times) / len(times) <= max_seconds):
        t, _ = oracle_step_time(batch)
        times.append(t)
        if len(times) >= 3 and sum(times) > max_seconds:
            break
    value = bytes_full / statistics.median(times) / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"median of {len(times)} full steps of the same workload (append + attention, all "
                      f"rows), {sum(times):.1f} s of CPU time, fp64 C oracle, {cores} threads"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    batch = W.workload_batch(args.workload)
    n_req = batch.num_reqs
    # size each step so that warm-up + timed steps take about 90 s
    t_row, _ = oracle_step_time(batch, rows=[0])
    budget = 90.0 / max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(n_req, budget // max(t_row, 1e-6))))
    cursor = 0

    def step():
        nonlocal cursor
        rows = [(cursor + i) % n_req for i in range(rows_per_step)]
        cursor = (cursor + rows_per_step) % n_req
        t, sb = oracle_step_time(batch, rows=rows)
        return t, W.step_bytes(sb)["unique"], sb.total_q

    for _ in range(args.warmup):
        step()
    tot_t, tot_b, tot_q = 0.0, 0, 0
    for _ in range(args.steps):
        t, nb, nq = step()
        tot_t += t
        tot_b += nb
        tot_q += nq
    value = tot_b / tot_t / 1e9
    cores = oracle.host_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "l2": "n/a (CPU)"},
        "tokens_per_layer_step_per_s": round(tot_q / tot_t, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {rows_per_step} of {n_req} requests (rotating), append + "
                                   f"attention, fp64 C oracle, {cores} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- 36-layer sweep
def device_batch(spec, device, layers):
    """One sweep point on the device: block tables, lengths and one K/V pool
    per layer, filled with seeded N(0,1) bf16 from a CUDA generator (the
    largest points hold ~40 GB, too much to generate on the host)."""
    import torch
    b = W.make_batch(spec["seq_lens"], spec["qo_lens"], num_blocks=spec["num_blocks"], seed=spec["seed"],
                     shared_prefix_tokens=spec["shared_prefix_tokens"], fill_pool=False)
    g = torch.Generator(device=device)
    g.manual_seed(spec["seed"])
    nb = spec["num_blocks"]
    pools = []
    for _ in range(layers):
        kc = torch.randn((nb, 8, 16, 128), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        vc = torch.randn((nb, 8, 16, 128), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        pools.append((kc, vc))
    return b, pools


def attention(B, prefix_pages, q, k_cache, v_cache, tables, seq, ind, scale, seq_h, ind_h, out, ws):
    """The step's attention call: the shared-prefix entry point when the
    batch's requests share leading pages, else pa_attention_varlen."""
    if prefix_pages:
        B.pa_attention_varlen_shared_prefix(q, k_cache, v_cache, tables, seq, ind, scale, prefix_pages,
                                            seq_lens_host=seq_h, qo_indptr_host=ind_h, out=out, workspace=ws)
    else:
        B.pa_attention_varlen(q, k_cache, v_cache, tables, seq, ind, scale, seq_lens_host=seq_h,
                              qo_indptr_host=ind_h, out=out, workspace=ws)


def call_name(prefix_pages):
    return (f"pa_attention_varlen_shared_prefix ({prefix_pages} shared pages)" if prefix_pages
            else "pa_attention_varlen")


def run_sweep(args):
    """Per-layer step time of append + attention for 36 layers captured in one
    CUDA graph, at each decode batch size and context of the sweep."""
    import torch
    from paged_kv_decode_varlen_gb300 import build as pa_build
    pa_build.build()
    from paged_kv_decode_varlen_gb300 import binding as B
    B.pa_set_decode_ctas(args.decode_ctas)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers = args.layers
    peak, _ = load_peaks()
    for context in [int(c) for c in args.contexts.split(",")]:
        for batch in [int(x) for x in args.batches.split(",")]:
            spec = W.sweep_point(batch, context)
            b, pools = device_batch(spec, dev, layers)
            # the decode step has no shared-prefix pass: points whose rows share
            # a prefix keep the cascade call
            use_step = args.api == "step" and (args.no_cascade or spec["shared_prefix_tokens"] == 0)
            ppages = 0 if (args.no_cascade or use_step) else spec["shared_prefix_tokens"] // 16
            sb = W.step_bytes(b, ppages)

            def bf(a):
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
            q, k_new, v_new = bf(b.q), bf(b.k_new), bf(b.v_new)
            tables = torch.from_numpy(b.block_tables).to(dev)
            seq = torch.from_numpy(b.seq_lens).to(dev)
            ind = torch.from_numpy(b.qo_indptr).to(dev)
            slots = torch.from_numpy(b.slot_mapping).to(dev)
            out = torch.empty_like(q)
            ws = B.new_workspace(B.pa_shared_prefix_workspace_size(b.num_reqs, b.total_q, 32, 128,
                                                                   int(b.seq_lens.max()), ppages), dev)
            ws_app = B.new_workspace(B.PA_ERROR_WORD_BYTES, dev)
            if use_step:
                ws = B.new_workspace(B.pa_decode_step_workspace_size(batch, 32, 128, context), dev)

            def step():
                if use_step:
                    for kc, vc in pools:
                        B.pa_decode_step(q, k_new, v_new, kc, vc, tables, seq, b.sm_scale, context, out=out,
                                         workspace=ws)
                    return
                for kc, vc in pools:
                    B.pa_kv_append(k_new, v_new, slots, kc, vc, workspace=ws_app)
                    attention(B, ppages, q, kc, vc, tables, seq, ind, b.sm_scale, b.seq_lens, b.qo_indptr, out, ws)
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for _ in range(2):
                    step()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            if B.pa_get_device_error(ws) or B.pa_get_device_error(ws_app):
                raise RuntimeError("device error word set in the sweep")
            ms_step = e0.elapsed_time(e1) / args.steps
            per_layer = ms_step / layers
            line = {"mode": "sweep", "context": context, "batch": batch, "layers": layers,
                    "ms_per_step": round(ms_step, 4), "us_per_layer": round(per_layer * 1e3, 3),
                    "unique_gbs": round(sb["unique"] / (per_layer * 1e-3) / 1e9, 1),
                    "logical_gbs": round(sb["logical"] / (per_layer * 1e-3) / 1e9, 1),
                    "frac_of_measured_hbm": round(sb["unique"] / (per_layer * 1e-3) / 1e9 / peak, 4),
                    "tokens_per_layer_step_per_s": round(batch / (per_layer * 1e-3), 1),
                    "bytes_per_layer": sb["unique"], "pool_blocks": spec["num_blocks"],
                    "attention_call": ("pa_decode_step (append + attention in one launch, max_seq_len %d)" % context
                                       if use_step else call_name(ppages)),
                    "l2": "not flushed (36 layers x distinct pools stream %.1f GB per step)" %
                          (sb["unique"] * layers / 1e9),
                    "graph": ("36 x pa_decode_step" if use_step else "36 x (kv_append + attention)")
                    + " in one CUDA graph", "decode_ctas": args.decode_ctas or "automatic"}
            print(json.dumps(line), flush=True)
            del pools, graph
            torch.cuda.empty_cache()
    return 0


# ------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="short")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-ctas", type=int, default=0, help="force the persistent decode grid size (0 = automatic)")
    ap.add_argument("--prefill-ctas", type=int, default=0,
                    help="CTAs of the prefill jobs beside the decode launch (0 = automatic, -1 = the jobs first)")
    ap.add_argument("--sweep", action="store_true",
                    help="36-layer decode sweep (b in 1..128 at 2048 and 8192-with-shared-prefix), one JSON line "
                         "per point, 36 x (append + attention) captured in a CUDA graph")
    ap.add_argument("--layers", type=int, default=36)
    ap.add_argument("--contexts", default="2048,8192", help="sweep contexts")
    ap.add_argument("--batches", default="1,8,32,64,128", help="sweep decode batch sizes")
    ap.add_argument("--kv", choices=["bf16", "q8"], default="bf16",
                    help="KV page format: bf16, or q8_0 (decode workloads only)")
    ap.add_argument("--api", choices=["varlen", "step"], default="varlen",
                    help="varlen: pa_kv_append + the attention call; step: pa_decode_step (append and attention in "
                         "one self-planned launch; decode-only bf16 batches)")
    ap.add_argument("--no-cascade", action="store_true",
                    help="run shared-prefix batches through pa_attention_varlen instead of the shared-prefix call")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        return run_sweep(args)

    import torch
    import torch.distributed as dist
    from paged_kv_decode_varlen_gb300 import build as pa_build
    pa_build.build()
    from paged_kv_decode_varlen_gb300 import binding as B

    B.pa_set_decode_ctas(args.decode_ctas)
    B.pa_set_prefill_ctas(args.prefill_ctas)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    batch = W.workload_batch(args.workload, seed_offset=rank)
    q8 = args.kv == "q8"
    if q8 and np.any(np.diff(batch.qo_indptr) > 1):
        raise SystemExit("--kv q8 serves decode rows only; this workload has rows with qo_len > 1")
    use_step = args.api == "step"
    if use_step and (q8 or np.any(np.diff(batch.qo_indptr) != 1)):
        raise SystemExit("--api step serves bf16 batches of decode rows only")
    ppages = 0 if (args.no_cascade or q8 or use_step) else batch.meta["shared_prefix_tokens"] // 16
    sb = W.step_bytes(batch, ppages, kv=args.kv)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    inputs = {
        "q": bf(batch.q), "k_new": bf(batch.k_new), "v_new": bf(batch.v_new),
        "slot_mapping": torch.from_numpy(batch.slot_mapping),
        "block_tables": torch.from_numpy(batch.block_tables),
        "seq_lens": torch.from_numpy(batch.seq_lens),
        "qo_indptr": torch.from_numpy(batch.qo_indptr),
    }
    if use_step:  # the step plans on the device: no slot_mapping, no qo_indptr
        del inputs["slot_mapping"], inputs["qo_indptr"]
    # the step's inputs live in one pinned host buffer and one device buffer
    # with the same layout, so the end-to-end leg moves them with one copy
    layout, stage_bytes = stage_layout(inputs)
    host_buf = torch.zeros(stage_bytes, dtype=torch.uint8).pin_memory()
    host = stage_views(host_buf, layout)
    for k_, t in inputs.items():
        host[k_].copy_(t)
    dev_buf = host_buf.to(dev)
    d = stage_views(dev_buf, layout)
    if q8:
        # q8_0 pools: every cached token quantized into its slot once, on the GPU
        nb, Hkv = batch.k_cache.shape[:2]
        k_cache = B.new_q8_pool(nb, Hkv, dev)
        v_cache = B.new_q8_pool(nb, Hkv, dev)
        for r in range(batch.num_reqs):
            L = int(batch.seq_lens[r]) - int(batch.qo_indptr[r + 1] - batch.qo_indptr[r])
            t = np.arange(L)
            blk = batch.block_tables[r, t // 16].astype(np.int64)
            B.pa_kv_append_q8(bf(batch.k_cache[blk, :, t % 16]).to(dev), bf(batch.v_cache[blk, :, t % 16]).to(dev),
                              torch.from_numpy(blk * 16 + t % 16).to(dev), k_cache, v_cache)
        torch.cuda.synchronize()
    else:
        k_cache = bf(batch.k_cache).to(dev)
        v_cache = bf(batch.v_cache).to(dev)
    out = torch.empty_like(d["q"])
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    R, total_q = batch.num_reqs, batch.total_q
    max_len = int(batch.seq_lens.max())
    if use_step:
        ws = B.new_workspace(B.pa_decode_step_workspace_size(R, 32, 128, max_len), dev)
    else:
        ws = B.new_workspace(B.pa_shared_prefix_workspace_size(R, total_q, 32, 128, max_len, ppages), dev)
    ws_app = B.new_workspace(B.PA_ERROR_WORD_BYTES, dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        torch.sum(flush, dim=0, out=flush_sink)
    seq_h = host["seq_lens"]
    ind_h = host.get("qo_indptr")
    stream = torch.cuda.current_stream()

    def step(src, dst=None):
        dst = out if dst is None else dst
        if use_step:
            B.pa_decode_step(src["q"], src["k_new"], src["v_new"], k_cache, v_cache, src["block_tables"],
                             src["seq_lens"], batch.sm_scale, max_len, out=dst, workspace=ws)
            return
        if q8:
            B.pa_kv_append_q8(src["k_new"], src["v_new"], src["slot_mapping"], k_cache, v_cache, workspace=ws_app)
            B.pa_attention_varlen_q8(src["q"], k_cache, v_cache, src["block_tables"], src["seq_lens"],
                                     src["qo_indptr"], batch.sm_scale, seq_lens_host=seq_h, qo_indptr_host=ind_h,
                                     out=dst, workspace=ws)
            return
        B.pa_kv_append(src["k_new"], src["v_new"], src["slot_mapping"], k_cache, v_cache, workspace=ws_app)
        attention(B, ppages, src["q"], k_cache, v_cache, src["block_tables"], src["seq_lens"], src["qo_indptr"],
                  batch.sm_scale, seq_h, ind_h, dst, ws)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush_l2()
        step(d)
    torch.cuda.synchronize()
    if B.pa_get_device_error(ws) or B.pa_get_device_error(ws_app):
        raise RuntimeError("device error word set during warm-up")

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except AttributeError:
        gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[local_rank]
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    n0 = B.pa_launch_count()
    clocks.mark(True)
    for i in range(args.steps):
        flush_l2()
        evs[i][0].record(stream)
        step(d)
        evs[i][1].record(stream)
    barrier()
    clocks.mark(False)
    launches = B.pa_launch_count() - n0
    step_ms = [a.elapsed_time(b) for a, b in evs]
    # per-kernel durations: the same steps again with the library's events
    # around every launch (kept out of the pass above: an event between two
    # kernels cuts their programmatic launch overlap)
    trace_steps = min(args.steps, 2000)
    barrier()
    B.pa_trace_enable(True)
    for i in range(trace_steps):
        flush_l2()
        step(d)
    barrier()
    B.pa_trace_enable(False)
    trace = B.pa_trace_read(1 << 15)
    clk = clocks.stop()

    # end to end through the C ABI with host buffers: H2D of the step's
    # inputs from pinned memory, the step, D2H of the output
    h2d = host_buf.numel()
    d2h = out.numel() * out.element_size()
    e2e_steps = min(args.steps, 1000)
    eevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    barrier()
    for i in range(e2e_steps):
        flush_l2()
        eevs[i][0].record(stream)
        dev_buf.copy_(host_buf, non_blocking=True)
        step(d)
        out_host.copy_(out, non_blocking=True)
        eevs[i][1].record(stream)
    barrier()
    e2e_ms = [a.elapsed_time(b) for a, b in eevs]

    # the same end-to-end steps as a serving loop runs them: double-buffered,
    # the host->device copy of step i + 1's inputs on a copy stream while step
    # i runs (step i + 1 waits for it), the device->host copy of step i's
    # output on the copy stream after step i, while step i + 1 runs.  Every
    # step's copies are inside the timed region; the inputs (the KV pool
    # above all) exceed L2, so no flush runs between these steps.
    copy_stream = torch.cuda.Stream(device=dev)
    dev_bufs = [dev_buf, torch.empty_like(dev_buf)]
    srcs = [d, stage_views(dev_bufs[1], layout)]
    outs = [out, torch.empty_like(out)]
    outs_host = [out_host, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    step_done = [torch.cuda.Event(), torch.cuda.Event()]
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    p0.record(stream)
    copy_stream.wait_stream(stream)
    with torch.cuda.stream(copy_stream):
        dev_bufs[0].copy_(host_buf, non_blocking=True)
    in_ready[0].record(copy_stream)
    for i in range(e2e_steps):
        bi = i & 1
        stream.wait_event(in_ready[bi])
        step(srcs[bi], outs[bi])
        step_done[bi].record(stream)
        with torch.cuda.stream(copy_stream):
            if i + 1 < e2e_steps:
                if i >= 1:  # the other buffer's inputs were last read by step i - 1
                    copy_stream.wait_event(step_done[bi ^ 1])
                dev_bufs[bi ^ 1].copy_(host_buf, non_blocking=True)
                in_ready[bi ^ 1].record(copy_stream)
            copy_stream.wait_event(step_done[bi])
            outs_host[bi].copy_(outs[bi], non_blocking=True)
    stream.wait_stream(copy_stream)
    p1.record(stream)
    barrier()
    t_e2e_pipe = p0.elapsed_time(p1) / e2e_steps
    if B.pa_get_device_error(ws) or B.pa_get_device_error(ws_app):
        raise RuntimeError("device error word set during the timed steps")

    # the median step (the mean is reported beside it)
    t_step = statistics.median(step_ms)
    t_e2e = statistics.median(e2e_ms)
    t_step_mean = sum(step_ms) / len(step_ms)
    t_step, t_e2e, t_e2e_pipe = max_over_ranks([t_step, t_e2e, t_e2e_pipe], dev)
    value = whole_job_gbs(sb["unique"], world, t_step)
    e2e_value = whole_job_gbs(sb["unique"], world, t_e2e)
    e2e_pipe_value = whole_job_gbs(sb["unique"], world, t_e2e_pipe)

    peak, peak_kind = load_peaks()
    tflops_peak = load_tflops_peak()
    pre = [ms for k_, ms in trace if k_ == "prefix"]
    pre_ms = sum(pre) / len(pre) if pre else None
    kernel_share = {}
    for k_, ms in trace:
        kernel_share[k_] = kernel_share.get(k_, 0.0) + ms
    # roofline of the kernel with the largest share of the step: the decode
    # kernel (HBM-bound), or the tensor-core tile kernel of rows with
    # qo_len > 1, bound by HBM or by the tensor pipe by its arithmetic intensity
    dom = max(("decode", "prefill", "decode_step"), key=lambda k_: kernel_share.get(k_, 0.0))
    dom_ms_list = [ms for k_, ms in trace if k_ == dom]
    dom_ms = sum(dom_ms_list) / len(dom_ms_list) if dom_ms_list else None
    if dom == "decode":
        bound, dom_bytes, dom_flops = "hbm", sb["decode_kernel"], None
    elif dom == "decode_step":
        bound, dom_bytes, dom_flops = "hbm", sb["step_kernel"], None
    else:
        dom_bytes, dom_flops = sb["prefill_kernel"], sb["prefill_flops"]
        bound = "tensor" if dom_flops / max(dom_bytes, 1) > tflops_peak * 1e12 / (peak * 1e9) else "hbm"
    if bound == "hbm":
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9 if dom_ms else None
        r_peak, r_unit = peak, "GB/s"
        r_source = f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s"
    else:
        achieved = dom_flops / (dom_ms * 1e-3) / 1e12 if dom_ms else None
        r_peak, r_unit = tflops_peak, "TFLOP/s"
        r_source = "measured (MEASURED_PEAKS.json bf16_tflops)"
    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step, 5), "ms_per_step_mean": round(t_step_mean, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "parallelism": f"replicas x{world}",
                   "kv_format": "q8_0 (34 of 64 bytes per 32 values)" if q8 else "bf16",
                   "l2": "flushed between timed steps (256 MiB read outside the events)",
                   "attention_call": ("pa_decode_step (append + attention in one launch)" if use_step
                                      else call_name(ppages)),
                   "bytes_per_step": sb["unique"], "logical_bytes_per_step": sb["logical"],
                   "query_tokens_per_step": sb["query_tokens"],
                   **({"prefill_ctas": args.prefill_ctas} if args.prefill_ctas else {})},
        "tokens_per_layer_step_per_s": round(sb["query_tokens"] * world / (t_step * 1e-3), 1),
        "frac_of_nominal_8tbs": round(value / world / 8000.0, 4),
        "roofline": {"bound": bound, "kernel": dom, "achieved": round(achieved, 2) if achieved else None,
                     "peak": r_peak, "peak_source": r_source, "unit": r_unit,
                     "frac": round(achieved / r_peak, 4) if achieved else None,
                     **({"frac_of_nominal_8tbs": round(achieved / 8000.0, 4)} if bound == "hbm" and achieved else {}),
                     "traffic": (profiled_traffic(args.workload, dom)
                                 if dom in ("decode", "decode_step") and not q8 else None),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     **({"algorithmic_flops_per_launch": dom_flops} if dom_flops else {}),
                     "avg_launch_ms": round(dom_ms, 5) if dom_ms else None,
                     "timing": f"CUDA events around each {dom} launch, {trace_steps} steps after the timed pass",
                     "kernel_time_share": {k_: round(v / sum(kernel_share.values()), 4)
                                           for k_, v in kernel_share.items()}},
        **({"prefix_pass": {"algorithmic_bytes_per_launch": sb["prefix_kernel"],
                            "avg_launch_ms": round(pre_ms, 5),
                            "achieved_gbs": round(sb["prefix_kernel"] / (pre_ms * 1e-3) / 1e9, 2)}}
           if pre_ms else {}),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(t_e2e, 5), "steps": e2e_steps,
                "copies": "on the step's stream before and after it, L2 flushed between steps (outside the "
                          "events), median step",
                "pipelined": {"value": round(e2e_pipe_value, 2), "ms_per_step": round(t_e2e_pipe, 5),
                              "copies": "double-buffered: step i+1's inputs host->device on a copy stream while "
                                        "step i runs, step i's output device->host while step i+1 runs; whole "
                                        "loop timed, no L2 flush (inputs > L2); eager launches, so a step whose "
                                        "host calls take longer than its kernels is host-bound here"}},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batch)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
