"""The tensor-core tile's FMA-pipe exponential (`exp2_fma2` in csrc/prefill.cu),
replayed step by step in float32 on the host: range reduction by a
round-toward--inf add of 1.5 * 2^23, a cubic for 2^f on [0, 1), and the integer
add of floor(d) into the exponent field.  Its constants are read from the
kernel source, so a change there is checked here.  Runs without a GPU."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "paged_kv_decode_varlen_gb300", "csrc", "prefill.cu")


def _constants():
    s = open(SRC).read()
    m = re.search(r"constexpr float kC1 = ([0-9.e+-]+)f, kC2 = ([0-9.e+-]+)f, kC3 = ([0-9.e+-]+)f;", s)
    assert m, "exp2_fma2 constants not found"
    return tuple(np.float32(float(v)) for v in m.groups())


def _exp2_fma2(d):
    """The kernel's steps on a float32 array (each op rounded to float32)."""
    c1, c2, c3 = _constants()
    shift = np.float32(12582912.0)
    d = np.maximum(d.astype(np.float32), np.float32(-127.0))
    # add.rm: the exact sum lies in [shift + floor(d), shift + floor(d) + 1)
    t = (np.floor(d.astype(np.float64)) + 12582912.0).astype(np.float32)
    j = (t - shift).astype(np.float32)
    f = (d - j).astype(np.float32)
    q = (c3 * f + c2).astype(np.float32)
    q = (q * f + c1).astype(np.float32)
    q = (q * f + np.float32(1.0)).astype(np.float32)
    bits = (q.view(np.uint32).astype(np.uint64) + ((t.view(np.uint32).astype(np.uint64) << 23) & 0xFFFFFFFF))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_cubic_meets_two_at_one_and_one_at_zero():
    c1, c2, c3 = (float(c) for c in _constants())
    # p(0) = 1 by construction; p(1) = 2 keeps 2^d continuous across integers
    assert abs(1.0 + c1 + c2 + c3 - 2.0) < 1e-6


def test_relative_error_over_the_softmax_range():
    # d = score * scale - running max lies in [-inf, 8] (8 = the rescale slack)
    d = np.concatenate([np.linspace(-126.0, 8.0, 1_000_001, dtype=np.float32),
                        np.float32([-1.0, -2.0, -0.5, 0.0, -0.0, 1e-30, -1e-30, 8.0, 7.9999995])])
    got = _exp2_fma2(d).astype(np.float64)
    want = np.exp2(d.astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1.1e-4, rel.max()
    # well inside half an ulp of bf16 (P is rounded to bf16 for the PV product)
    assert rel.max() < 2.0 ** -9 / 10
    # exact powers of two come out exact
    ints = np.arange(-126, 9, dtype=np.float32)
    assert np.array_equal(_exp2_fma2(ints).astype(np.float64), np.exp2(ints.astype(np.float64)))


def test_masked_and_far_below_give_zero_or_subnormal():
    assert np.all(_exp2_fma2(np.float32([-np.inf, -127.0, -1000.0, -3.0e38])) == 0.0)
    sub = _exp2_fma2(np.float32([-126.5, -126.01])).astype(np.float64)
    assert np.all((sub >= 0.0) & (sub < 2.0 ** -126))
    # monotone over a fine grid (the sum l and the bf16 P see no reversals)
    d = np.linspace(-20.0, 8.0, 200_001, dtype=np.float32)
    assert np.all(np.diff(_exp2_fma2(d).astype(np.float64)) >= 0.0)
