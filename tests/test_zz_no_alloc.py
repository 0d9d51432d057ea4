"""pa_attention_varlen_noalloc: the attention call for callers that cannot
allocate device memory (no workspace argument; the scratch is a fixed array
inside the library).  Its results must match pa_attention_varlen's, call
after call, because every call shares and reuses that array.

Kept in a file of its own that is collected last, and independent of the
other tests' state, so it passes both alone and after the whole suite."""
import numpy as np
import pytest
import torch

from paged_kv_decode_varlen_gb300 import workloads as W
from tests.util import LSE_ABS, MAX_ABS, MEAN_ABS, DevBatch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from paged_kv_decode_varlen_gb300 import binding as B


def _diff(a, b):
    d = (a.float() - b.float()).abs()
    return d.max().item(), d.mean().item()


def test_noalloc_matches_workspace_call_twice_in_a_row():
    B.pa_set_decode_ctas(0)
    # decode rows whose key ranges are cut between CTAs (partials + counters)
    # and one chunked-prefill row
    b = W.workload_batch("mixed", scale=0.25)
    d = DevBatch(b)
    B.pa_kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
    args = (d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.qo_indptr, b.sm_scale)
    kw = dict(seq_lens_host=d.seq_lens_host, qo_indptr_host=d.qo_indptr_host, return_lse=True)
    ref_out, ref_lse = B.pa_attention_varlen(*args, **kw)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out, lse = B.pa_attention_varlen_noalloc(*args, device_error=err, **kw)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        mx, mean = _diff(out, ref_out)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, f"call {call}: max {mx:.3e} mean {mean:.3e}"
        assert (lse - ref_lse).abs().max().item() <= LSE_ABS
        assert torch.isfinite(out.float()).all()


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    # more rows than the fixed scratch has room for (229,376 rows x 8 kv
    # heads x 4-byte counters is 7 MiB, plus the split partials); the call
    # is refused on the host before anything is launched
    n = 229376
    assert B.pa_attention_workspace_size(n, n, 32, 128, 16) > (8 << 20)
    seq = torch.full((n,), 16, dtype=torch.int32)
    ind = torch.arange(n + 1, dtype=torch.int32)
    q = torch.zeros((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((n, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(B.PAError) as e:
        B.pa_attention_varlen_noalloc(q, kc, kc, bt, seq.cuda(), ind.cuda(), 0.088, seq_lens_host=seq,
                                      qo_indptr_host=ind)
    assert e.value.status == B.PA_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
