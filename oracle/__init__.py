"""CPU oracle for paged varlen attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA product path never
imports it, and it never imports the product path.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64; its header names the
passages each function follows).  This module compiles it with gcc and
marshals numpy arrays into it.  ``paging.py`` holds the page and byte
arithmetic, ``brute.py`` a pure-Python fp64 restatement for tiny cases.

bf16 tensors are passed as numpy ``uint16`` bit patterns (exact bf16 values);
outputs are fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")


class OracleError(RuntimeError):
    pass


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 -fopenmp; -ffp-contract=off keeps every multiply and add a
    separate IEEE operation, so x86 and Arm hosts give the same bits."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", "-std=c11",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into liboracle.so next to it when stale."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _check(rc: int, what: str):
    if rc == 1:
        raise OracleError(f"{what}: invalid argument")
    if rc == 2:
        raise OracleError(f"{what}: block id or slot outside the pool")
    if rc != 0:
        raise OracleError(f"{what}: status {rc}")


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test's
    deliberately mutated copy)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_round_bf16_array.restype = None
        lib.oracle_round_bf16_array.argtypes = [P, P, i64]
        lib.oracle_kv_append.restype = i32
        lib.oracle_kv_append.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32]
        lib.oracle_attention_varlen.restype = i32
        lib.oracle_attention_varlen.argtypes = [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, f64,
                                                P, P, P, i32, i32]
        lib.oracle_attention_sampled.restype = i32
        lib.oracle_attention_sampled.argtypes = [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, f64,
                                                 i32, P, P, P, P, P, i32, i32]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f16_value.restype = f64
        lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_quantize_q8.restype = None
        lib.oracle_quantize_q8.argtypes = [P, i64, P, P]
        lib.oracle_kv_append_q8.restype = i32
        lib.oracle_kv_append_q8.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32]
        lib.oracle_attention_varlen_q8.restype = i32
        lib.oracle_attention_varlen_q8.argtypes = [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, f64,
                                                   P, P, P, i32, i32]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_copy_blocks.argtypes = [P, P, i64, i32, i32, i32, P, P, i64]
        lib.oracle_decode_step_slots.restype = i32
        lib.oracle_decode_step_slots.argtypes = [P, i32, P, i32, i32, i32, P]
        lib.oracle_merge_lse.restype = i32
        lib.oracle_merge_lse.argtypes = [P, P, P, P, P, P, i64, i32, i32]
        self.lib = lib
        self.path = lib_path

    def round_bf16(self, x) -> np.ndarray:
        """fp64 -> bf16 bit patterns, round to nearest even."""
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.zeros(x.shape, np.uint16)
        self.lib.oracle_round_bf16_array(_ptr(x), _ptr(out), x.size)
        return out

    def kv_append(self, k_new, v_new, slot_mapping, k_cache, v_cache):
        """Scatter new K/V rows into the HND pools, in place.

        k_new, v_new: uint16 [N, Hkv, D]; slot_mapping int64 [N] (negative =
        skip); k_cache, v_cache: uint16 [num_blocks, Hkv, P, D]."""
        k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
        slot_mapping = _c(slot_mapping, np.int64)
        for c in (k_cache, v_cache):
            if not (c.flags.c_contiguous and c.dtype == np.uint16):
                raise TypeError("caches must be C-contiguous uint16")
        N, Hkv, D = k_new.shape
        nb, _, P, _ = k_cache.shape
        _check(self.lib.oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_cache),
                                         _ptr(v_cache), nb, P, Hkv, D), "kv_append")

    def decode_step_slots(self, block_tables, seq_lens, block_size, max_seq_len):
        """Slot of each decode row's new token (position seq_len - 1), -1 for
        padding and invalid rows.  Returns (slots int64 [R], invalid rows)."""
        block_tables = _c(block_tables, np.int32)
        seq_lens = _c(seq_lens, np.int32)
        R = seq_lens.shape[0]
        slots = np.full(R, -1, np.int64)
        bad = self.lib.oracle_decode_step_slots(_ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), R,
                                                block_size, max_seq_len, _ptr(slots))
        return slots, int(bad)

    def decode_step(self, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, sm_scale, max_seq_len,
                    n_threads=None):
        """One decode step of a padded batch: row r's new token is appended
        at position seq_lens[r] - 1 (slots from decode_step_slots; the
        caches change in place), then every valid row attends over its
        seq_len keys.  Padding and invalid rows get out = 0, lse = -inf.
        Returns (out fp64 [R, Hq, D], lse fp64 [R, Hq], invalid rows)."""
        q = _c(q, np.uint16)
        R, Hq, D = q.shape
        P = k_cache.shape[2]
        slots, bad = self.decode_step_slots(block_tables, seq_lens, P, max_seq_len)
        self.kv_append(k_new, v_new, slots, k_cache, v_cache)
        out = np.zeros((R, Hq, D), np.float64)
        lse = np.full((R, Hq), -np.inf, np.float64)
        rows = np.flatnonzero(slots >= 0)
        if len(rows):
            o, l = self.attention_varlen(q[rows], k_cache, v_cache, _c(block_tables, np.int32)[rows],
                                         _c(seq_lens, np.int32)[rows], np.arange(len(rows) + 1, dtype=np.int32),
                                         sm_scale, n_threads=n_threads)
            out[rows], lse[rows] = o, l
        return out, lse, bad

    def copy_blocks(self, k_cache, v_cache, src, dst):
        """Copy whole blocks src[i] -> dst[i] (K and V, every kv head), in
        order, in place.  Returns the number of pairs skipped for an id
        outside the pool."""
        for c in (k_cache, v_cache):
            if not (c.flags.c_contiguous and c.dtype == np.uint16):
                raise TypeError("caches must be C-contiguous uint16")
        src, dst = _c(src, np.int32), _c(dst, np.int32)
        if src.shape != dst.shape or src.ndim != 1:
            raise ValueError("src and dst must be 1-D and of equal length")
        nb, Hkv, P, D = k_cache.shape
        return int(self.lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), nb, P, Hkv, D, _ptr(src), _ptr(dst),
                                               src.shape[0]))

    def _common(self, q, k_cache, v_cache, block_tables, seq_lens, qo_indptr):
        q = _c(q, np.uint16)
        k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        block_tables = _c(block_tables, np.int32)
        if block_tables.ndim != 2:
            raise TypeError("block_tables must be 2-D")
        seq_lens, qo_indptr = _c(seq_lens, np.int32), _c(qo_indptr, np.int32)
        return q, k_cache, v_cache, block_tables, seq_lens, qo_indptr

    def attention_varlen(self, q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale, n_threads=None):
        """Exact paged varlen attention.

        q uint16 [total_q, Hq, D]; caches uint16 [num_blocks, Hkv, P, D];
        block_tables int32 [num_reqs, max_blocks]; seq_lens int32 [num_reqs]
        (KV length after this step's append); qo_indptr int32 [num_reqs + 1].
        Returns (out fp64 [total_q, Hq, D], lse fp64 [total_q, Hq])."""
        q, k_cache, v_cache, block_tables, seq_lens, qo_indptr = self._common(
            q, k_cache, v_cache, block_tables, seq_lens, qo_indptr)
        total_q, Hq, D = q.shape
        nb, Hkv, P, _ = k_cache.shape
        R = seq_lens.shape[0]
        nt = n_threads or host_threads()
        max_len = max(int(seq_lens.max()) if R else 1, 1)
        out = np.zeros((total_q, Hq, D), np.float64)
        lse = np.zeros((total_q, Hq), np.float64)
        scratch = np.zeros(nt * max_len, np.float64)
        _check(self.lib.oracle_attention_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                                block_tables.shape[1], _ptr(seq_lens), _ptr(qo_indptr), R, Hq, Hkv,
                                                D, P, float(sm_scale), _ptr(out), _ptr(lse), _ptr(scratch), max_len,
                                                nt), "attention_varlen")
        return out, lse

    # ---------------------------------------------------------------- q8_0
    def f32_to_f16(self, x: float) -> int:
        """binary16 bits of a binary32 value (round to nearest even)."""
        return int(self.lib.oracle_f32_to_f16(float(x)))

    def f16_value(self, h: int) -> float:
        return float(self.lib.oracle_f16_value(int(h)))

    def quantize_q8(self, x):
        """q8_0 of bf16 values x (uint16 [..., 32 k]): int8 codes of x's shape
        and uint16 binary16 scales [..., k]."""
        x = _c(x, np.uint16)
        if x.shape[-1] % 32:
            raise ValueError("the last dimension must be a multiple of 32")
        codes = np.zeros(x.shape, np.int8)
        scales = np.zeros(x.shape[:-1] + (x.shape[-1] // 32,), np.uint16)
        self.lib.oracle_quantize_q8(_ptr(x), x.size // 32, _ptr(codes), _ptr(scales))
        return codes, scales

    def kv_append_q8(self, k_new, v_new, slot_mapping, k_cache, v_cache):
        """kv_append into q8_0 pages, in place: caches uint8
        [num_blocks, Hkv, q8_slab_bytes(P, D)]."""
        k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
        slot_mapping = _c(slot_mapping, np.int64)
        for c in (k_cache, v_cache):
            if not (c.flags.c_contiguous and c.dtype == np.uint8):
                raise TypeError("q8 caches must be C-contiguous uint8")
        N, Hkv, D = k_new.shape
        nb = k_cache.shape[0]
        P = q8_page_tokens(k_cache.shape[2], D)
        _check(self.lib.oracle_kv_append_q8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_cache),
                                            _ptr(v_cache), nb, P, Hkv, D), "kv_append_q8")

    def attention_varlen_q8(self, q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale, n_threads=None):
        """attention_varlen over q8_0 pages (uint8 [num_blocks, Hkv, slab])."""
        q = _c(q, np.uint16)
        k_cache, v_cache = _c(k_cache, np.uint8), _c(v_cache, np.uint8)
        block_tables = _c(block_tables, np.int32)
        seq_lens, qo_indptr = _c(seq_lens, np.int32), _c(qo_indptr, np.int32)
        total_q, Hq, D = q.shape
        nb, Hkv, slab = k_cache.shape
        P = q8_page_tokens(slab, D)
        R = seq_lens.shape[0]
        nt = n_threads or host_threads()
        max_len = max(int(seq_lens.max()) if R else 1, 1)
        out = np.zeros((total_q, Hq, D), np.float64)
        lse = np.zeros((total_q, Hq), np.float64)
        scratch = np.zeros(nt * max_len, np.float64)
        _check(self.lib.oracle_attention_varlen_q8(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                                   block_tables.shape[1], _ptr(seq_lens), _ptr(qo_indptr), R, Hq,
                                                   Hkv, D, P, float(sm_scale), _ptr(out), _ptr(lse), _ptr(scratch),
                                                   max_len, nt), "attention_varlen_q8")
        return out, lse

    def attention_sampled(self, q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale, sample_tok,
                          sample_head, n_threads=None):
        """The same definition at a list of (query token, q head) samples.
        Returns (out fp64 [n, D], lse fp64 [n])."""
        q, k_cache, v_cache, block_tables, seq_lens, qo_indptr = self._common(
            q, k_cache, v_cache, block_tables, seq_lens, qo_indptr)
        st, sh = _c(sample_tok, np.int32), _c(sample_head, np.int32)
        total_q, Hq, D = q.shape
        nb, Hkv, P, _ = k_cache.shape
        R = seq_lens.shape[0]
        nt = n_threads or host_threads()
        max_len = max(int(seq_lens.max()) if R else 1, 1)
        n = st.shape[0]
        out = np.zeros((n, D), np.float64)
        lse = np.zeros((n,), np.float64)
        scratch = np.zeros(nt * max_len, np.float64)
        _check(self.lib.oracle_attention_sampled(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                                 block_tables.shape[1], _ptr(seq_lens), _ptr(qo_indptr), R, Hq, Hkv,
                                                 D, P, float(sm_scale), n, _ptr(st), _ptr(sh), _ptr(out), _ptr(lse),
                                                 _ptr(scratch), max_len, nt), "attention_sampled")
        return out, lse

    def merge_lse(self, o_a, lse_a, o_b, lse_b):
        """LSE merge of two partial attentions.  o_* uint16 [rows, H, D]
        (bf16 bits), lse_* [rows, H].  Returns (o fp64, lse fp64)."""
        o_a, o_b = _c(o_a, np.uint16), _c(o_b, np.uint16)
        lse_a = np.ascontiguousarray(np.asarray(lse_a, np.float64))
        lse_b = np.ascontiguousarray(np.asarray(lse_b, np.float64))
        rows, H, D = o_a.shape
        o = np.zeros((rows, H, D), np.float64)
        lse = np.zeros((rows, H), np.float64)
        _check(self.lib.oracle_merge_lse(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o), _ptr(lse), rows,
                                         H, D), "merge_lse")
        return o, lse


_default = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def round_bf16(x):
    return default().round_bf16(x)


def kv_append(*a, **kw):
    return default().kv_append(*a, **kw)


def copy_blocks(*a, **kw):
    return default().copy_blocks(*a, **kw)


def decode_step_slots(*a, **kw):
    return default().decode_step_slots(*a, **kw)


def decode_step(*a, **kw):
    return default().decode_step(*a, **kw)


def q8_slab_bytes(page_tokens: int, head_dim: int) -> int:
    """Bytes of one (block, kv head) q8_0 slab: codes, then binary16 scales."""
    return page_tokens * head_dim + page_tokens * (head_dim // 32) * 2


def q8_page_tokens(slab_bytes: int, head_dim: int) -> int:
    per_token = head_dim + (head_dim // 32) * 2
    if slab_bytes % per_token:
        raise ValueError("slab size does not match the head dimension")
    return slab_bytes // per_token


def quantize_q8(*a, **kw):
    return default().quantize_q8(*a, **kw)


def kv_append_q8(*a, **kw):
    return default().kv_append_q8(*a, **kw)


def attention_varlen_q8(*a, **kw):
    return default().attention_varlen_q8(*a, **kw)


def attention_varlen(*a, **kw):
    return default().attention_varlen(*a, **kw)


def attention_sampled(*a, **kw):
    return default().attention_sampled(*a, **kw)


def merge_lse(*a, **kw):
    return default().merge_lse(*a, **kw)
