"""Shared test helpers: move a workloads.Batch to the GPU and compare the
CUDA path's output with the oracle's."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# The tolerance the attention outputs must meet (bf16 outputs vs the fp64
# oracle): max-abs 1.5e-2 and mean-abs 2e-3 over all elements.
MAX_ABS = 1.5e-2
MEAN_ABS = 2e-3
# lse is fp32 throughout; scores of 128 bf16 products carry ~1e-6 relative
# error, so 1e-3 absolute on lse is generous.
LSE_ABS = 1e-3


def bf16_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class DevBatch:
    def __init__(self, b, device="cuda"):
        self.b = b
        self.q = bf16_dev(b.q, device)
        self.k_cache = bf16_dev(b.k_cache, device)
        self.v_cache = bf16_dev(b.v_cache, device)
        self.block_tables = torch.from_numpy(b.block_tables).to(device)
        self.seq_lens = torch.from_numpy(b.seq_lens).to(device)
        self.qo_indptr = torch.from_numpy(b.qo_indptr).to(device)
        self.k_new = bf16_dev(b.k_new, device)
        self.v_new = bf16_dev(b.v_new, device)
        self.slot_mapping = torch.from_numpy(b.slot_mapping).to(device)
        self.seq_lens_host = torch.from_numpy(b.seq_lens)
        self.qo_indptr_host = torch.from_numpy(b.qo_indptr)


def oracle_step(b):
    """Oracle of one step: append on a CPU copy of the pool, then attention.
    Returns (out fp64, lse fp64, k_pool, v_pool)."""
    k, v = b.k_cache.copy(), b.v_cache.copy()
    oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, k, v)
    out, lse = oracle.attention_varlen(b.q, k, v, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    return out, lse, k, v


def compare(out_gpu: torch.Tensor, out_ref: np.ndarray, lse_gpu=None, lse_ref=None, what=""):
    got = oracle.bf16_to_f64(bf16_host(out_gpu))
    err = np.abs(got - out_ref)
    if not np.all(np.isfinite(got)):
        bad = np.argwhere(~np.isfinite(got).all(axis=-1))
        raise AssertionError(f"{what}: non-finite outputs at {len(bad)} (row, head) pairs, first {bad[:12].tolist()}")
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if mx > MAX_ABS:
        bad = np.argwhere((err > MAX_ABS).any(axis=-1))
        raise AssertionError(f"{what}: max abs err {mx:.3e} > {MAX_ABS} at {len(bad)} (row, head) pairs, "
                             f"first {bad[:12].tolist()}")
    assert mean <= MEAN_ABS, f"{what}: mean abs err {mean:.3e} > {MEAN_ABS}"
    if lse_gpu is not None:
        le = np.abs(lse_gpu.detach().cpu().double().numpy() - lse_ref)
        assert float(le.max()) <= LSE_ABS, f"{what}: lse err {float(le.max()):.3e}"
    return mx, mean
