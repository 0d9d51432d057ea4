"""Pure-Python fp64 restatement of paged varlen attention for tiny inputs --
TEST INFRASTRUCTURE ONLY.

A second, independent transcription of the same definition as pa_oracle.c
(different language, different loop structure: the key set is first
gathered into a contiguous list, as the block-table description in
"Inference optimisation" §8.3.1 / Fig. 8-10 recovers the logical order),
used to cross-check the C oracle's marshalling and indexing on inputs of a
few dozen tokens.  It is a cross-check, not a pin: the pins are the closed
forms and invariants in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np


def _val(bits) -> float:
    return float((np.uint32(bits) << np.uint32(16)).view(np.float32))


def attention(q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale):
    """Same argument conventions as oracle.attention_varlen (uint16 bf16
    patterns).  Returns (out, lse) as nested Python lists of floats."""
    total_q, Hq, D = q.shape
    _, Hkv, P, _ = k_cache.shape
    G = Hq // Hkv
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(total_q)]
    lse = [[0.0] * Hq for _ in range(total_q)]
    for r in range(len(seq_lens)):
        L = int(seq_lens[r])
        start, end = int(qo_indptr[r]), int(qo_indptr[r + 1])
        c = end - start
        for kvh in range(Hkv):
            # gather the request's keys and values in logical order
            keys, vals = [], []
            for t in range(L):
                blk = int(block_tables[r][t // P])
                keys.append([_val(x) for x in k_cache[blk, kvh, t % P]])
                vals.append([_val(x) for x in v_cache[blk, kvh, t % P]])
            for g in range(G):
                h = kvh * G + g
                for j in range(c):
                    visible = L - c + j + 1
                    qv = [_val(x) for x in q[start + j, h]]
                    scores = [sm_scale * sum(a * b for a, b in zip(qv, keys[t])) for t in range(visible)]
                    m = max(scores)
                    w = [math.exp(s - m) for s in scores]
                    z = sum(w)
                    out[start + j][h] = [sum(w[t] * vals[t][d] for t in range(visible)) / z for d in range(D)]
                    lse[start + j][h] = m + math.log(z)
    return out, lse
