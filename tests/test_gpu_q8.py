"""q8_0 KV pages ("Inference optimisation" §8.4.2) through the C ABI against
the oracle: the quantizing append is bit-exact (codes and scales), decode
attention over q8_0 pages meets the bf16-output tolerance against the
oracle's q8_0 definition."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import bf16_dev, bf16_host, compare

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


def _cached_tokens(b):
    """K, V rows and slots of every token already in the pool (before the
    step's append), request by request."""
    ks, vs, slots = [], [], []
    for r in range(b.num_reqs):
        L = int(b.seq_lens[r]) - int(b.qo_indptr[r + 1] - b.qo_indptr[r])
        t = np.arange(L)
        blk = b.block_tables[r, t // 16].astype(np.int64)
        ks.append(b.k_cache[blk, :, t % 16])
        vs.append(b.v_cache[blk, :, t % 16])
        slots.append(blk * 16 + t % 16)
    return np.concatenate(ks), np.concatenate(vs), np.concatenate(slots)


def build_q8(b):
    """q8_0 pools holding the batch's cached tokens and the step's new ones,
    made on the GPU and by the oracle.  Returns (kq, vq device, kq, vq host,
    the append workspace)."""
    nb, Hkv = b.k_cache.shape[:2]
    kq, vq = B.new_q8_pool(nb, Hkv, "cuda"), B.new_q8_pool(nb, Hkv, "cuda")
    hk = np.zeros((nb, Hkv, B.PA_Q8_SLAB_BYTES), np.uint8)
    hv = np.zeros_like(hk)
    ck, cv, cs = _cached_tokens(b)
    ws = B.pa_kv_append_q8(bf16_dev(ck), bf16_dev(cv), torch.from_numpy(cs).cuda(), kq, vq)
    oracle.kv_append_q8(ck, cv, cs, hk, hv)
    B.pa_kv_append_q8(bf16_dev(b.k_new), bf16_dev(b.v_new), torch.from_numpy(b.slot_mapping).cuda(), kq, vq,
                      workspace=ws)
    oracle.kv_append_q8(b.k_new, b.v_new, b.slot_mapping, hk, hv)
    torch.cuda.synchronize()
    return kq, vq, hk, hv, ws


def _attn_q8(b, kq, vq, **kw):
    return B.pa_attention_varlen_q8(bf16_dev(b.q), kq, vq, torch.from_numpy(b.block_tables).cuda(),
                                    torch.from_numpy(b.seq_lens).cuda(), torch.from_numpy(b.qo_indptr).cuda(),
                                    b.sm_scale, seq_lens_host=torch.from_numpy(b.seq_lens),
                                    qo_indptr_host=torch.from_numpy(b.qo_indptr), return_lse=True, **kw)


@pytest.mark.parametrize("name", ["tiny", "short"])
def test_append_q8_bit_exact_and_attention(name):
    b = W.workload_batch(name)
    kq, vq, hk, hv, ws = build_q8(b)
    assert B.pa_get_device_error(ws) == 0
    assert np.array_equal(kq.cpu().numpy(), hk) and np.array_equal(vq.cpu().numpy(), hv)
    out, lse = _attn_q8(b, kq, vq)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_varlen_q8(b.q, hk, hv, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    compare(out, ref, lse, ref_lse, what=f"q8 {name}")


@pytest.mark.parametrize("ctas", [1, 7, 456, 1024])
def test_q8_forced_decode_grid(ctas):
    b = W.make_batch([2100, 37, 16, 1, 700, 129], [1] * 6, num_blocks=400, seed=70 + ctas)
    kq, vq, hk, hv, _ = build_q8(b)
    B.pa_set_decode_ctas(ctas)
    try:
        out, lse = _attn_q8(b, kq, vq)
        torch.cuda.synchronize()
    finally:
        B.pa_set_decode_ctas(0)
    ref, ref_lse = oracle.attention_varlen_q8(b.q, hk, hv, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    compare(out, ref, lse, ref_lse, what=f"q8 ctas={ctas}")


EDGE = {
    "single_token_context": ([1], [1]),
    "exact_page_multiple": ([16, 32, 256], [1, 1, 1]),
    "empty_rows_mixed_in": ([50, 30, 70, 9], [1, 0, 1, 0]),
    "many_small_rows": ([int(x) for x in np.random.default_rng(5).integers(1, 90, 200)], [1] * 200),
    "shared_prefix_pages": ([700, 900, 650], [1, 1, 1]),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_q8_edge_cases(case):
    seq, qo = EDGE[case]
    shared = 512 if case == "shared_prefix_pages" else 0
    need = sum(-(-L // 16) for L in seq)
    b = W.make_batch(seq, qo, num_blocks=need + 7, seed=zlib.crc32(case.encode()) % 1000,
                     shared_prefix_tokens=shared)
    kq, vq, hk, hv, _ = build_q8(b)
    out, lse = _attn_q8(b, kq, vq)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_varlen_q8(b.q, hk, hv, b.block_tables, b.seq_lens, b.qo_indptr, b.sm_scale)
    compare(out, ref, lse, ref_lse, what=f"q8 {case}")


def test_q8_rejects_prefill_rows_and_records_bad_slots():
    b = W.make_batch([300, 200], [1, 9], num_blocks=40, seed=77)
    kq, vq, _, _, _ = build_q8(W.make_batch([300, 200], [1, 1], num_blocks=40, seed=77))
    with pytest.raises(B.PAError) as e:
        _attn_q8(b, kq, vq)
    assert e.value.status == B.PA_ERR_UNSUPPORTED
    k_new = np.zeros((2, 8, 128), np.uint16)
    ws = B.pa_kv_append_q8(bf16_dev(k_new), bf16_dev(k_new), torch.tensor([5, 40 * 16 + 1]).cuda(), kq, vq)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_INDEX
