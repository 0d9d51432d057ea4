"""pa_copy_blocks (copy-on-write block copy) through the C ABI against the
oracle: bit-exact, out-of-pool ids skipped and recorded, and the
copy-on-write sequence of "Inference optimisation" §8.3.2 (Fig. 8-15) end
to end with pa_kv_append and attention."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import bf16_dev, bf16_host, compare

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


def _pool(nb, seed):
    rng = np.random.default_rng(seed)
    return W.normal_bf16(rng, (nb, 8, 16, 128)), W.normal_bf16(rng, (nb, 8, 16, 128))


@pytest.mark.parametrize("n_pairs", [1, 7, 300])
def test_copy_blocks_bit_exact(n_pairs):
    nb = 2 * n_pairs + 11
    k, v = _pool(nb, 60 + n_pairs)
    perm = np.random.default_rng(61).permutation(nb).astype(np.int32)
    src, dst = perm[:n_pairs], perm[n_pairs:2 * n_pairs]
    kd, vd = bf16_dev(k), bf16_dev(v)
    ws = B.pa_copy_blocks(torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), kd, vd)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == 0
    assert oracle.copy_blocks(k, v, src, dst) == 0
    assert np.array_equal(bf16_host(kd), k) and np.array_equal(bf16_host(vd), v)


def test_copy_blocks_out_of_pool_skipped():
    nb = 20
    k, v = _pool(nb, 62)
    src = np.array([3, 4, 5, -1], np.int32)
    dst = np.array([10, nb, 11, 12], np.int32)
    kd, vd = bf16_dev(k), bf16_dev(v)
    ws = B.pa_copy_blocks(torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), kd, vd)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == B.PA_ERR_DEVICE_INDEX
    assert oracle.copy_blocks(k, v, src, dst) == 2
    assert np.array_equal(bf16_host(kd), k) and np.array_equal(bf16_host(vd), v)


def test_copy_on_write_branches():
    """Four branches share a 2055-token context whose last block holds 7
    tokens.  Branches 1-3 copy that tail block, then every branch appends
    its own next token.  Each branch's attention matches the oracle on the
    same pool, and the shared blocks are untouched."""
    P, L0 = 16, 2055
    pages = -(-L0 // P)
    nb = pages + 3 + 5
    k, v = _pool(nb, 63)
    rng = np.random.default_rng(64)
    shared = rng.permutation(nb)[:pages].astype(np.int32)
    free = [i for i in range(nb) if i not in set(shared.tolist())]
    src = np.full(3, shared[-1], np.int32)
    dst = np.array(free[:3], np.int32)
    tables = np.tile(shared, (4, 1))
    tables[1:, -1] = dst
    kd, vd = bf16_dev(k), bf16_dev(v)
    ws = B.pa_copy_blocks(torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), kd, vd)
    oracle.copy_blocks(k, v, src, dst)
    k_new = W.normal_bf16(rng, (4, 8, 128))
    v_new = W.normal_bf16(rng, (4, 8, 128))
    slots = (tables[:, -1].astype(np.int64) * P + (L0 % P))
    B.pa_kv_append(bf16_dev(k_new), bf16_dev(v_new), torch.from_numpy(slots).cuda(), kd, vd, workspace=ws)
    oracle.kv_append(k_new, v_new, slots, k, v)
    q = W.normal_bf16(rng, (4, 32, 128))
    seq = np.full(4, L0 + 1, np.int32)
    ind = np.arange(5, dtype=np.int32)
    out, lse = B.pa_attention_varlen(bf16_dev(q), kd, vd, torch.from_numpy(tables).cuda(),
                                     torch.from_numpy(seq).cuda(), torch.from_numpy(ind).cuda(), 1 / math.sqrt(128),
                                     return_lse=True)
    torch.cuda.synchronize()
    assert B.pa_get_device_error(ws) == 0
    assert np.array_equal(bf16_host(kd), k) and np.array_equal(bf16_host(vd), v)
    ref, ref_lse = oracle.attention_varlen(q, k, v, tables, seq, ind, 1 / math.sqrt(128))
    compare(out, ref, lse, ref_lse, what="copy-on-write branches")
    # the branches differ only in their last token, so their outputs differ
    assert not np.array_equal(bf16_host(out[0]), bf16_host(out[1]))
