"""Python binding of libpa (include/pa.h): argument marshalling only.

Every function has the name of the C entry point it calls.  torch tensors
supply device memory and the current CUDA stream; every step of the
computation runs in libpa's kernels.  A non-PA_OK status raises PAError.

The library is loaded on import; if libpa.so has not been built this
module raises ImportError (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pa.h")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE_TOO_SMALL = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_INDEX = 5
PA_ERR_DEVICE_TIMEOUT = 6
PA_ERROR_WORD_BYTES = 256
KERNEL_KINDS = {1: "kv_append", 2: "decode", 3: "combine", 4: "prefill", 5: "merge", 6: "prefix", 7: "prefix_merge", 8: "copy_blocks",
                9: "decode_step"}


class PAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with paged_kv_decode_varlen_gb300/build.py "
                      "(or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_i32, _i64, _f32, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "pa_abi_version": (_i32, []),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_last_error_message": (ctypes.c_char_p, []),
    "pa_kv_append": (_i32, [_P, _P, _P, _i64, _P, _P, _i64, _i32, _i32, _i32, _P, _sz, _P]),
    "pa_copy_blocks": (_i32, [_P, _P, _i64, _P, _P, _i64, _i32, _i32, _i32, _P, _sz, _P]),
    "pa_kv_append_q8": (_i32, [_P, _P, _P, _i64, _P, _P, _i64, _i32, _i32, _i32, _P, _sz, _P]),
    "pa_attention_varlen_q8": (_i32, [_P, _P, _P, _i64, _P, _i32, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32,
                                      _i32, _f32, _P, _P, _P, _sz, _P]),
    "pa_attention_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "pa_attention_varlen": (_i32, [_P, _P, _P, _i64, _P, _i32, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32, _i32,
                                   _f32, _P, _P, _P, _sz, _P]),
    "pa_decode_step": (_i32, [_P, _P, _P, _P, _P, _i64, _P, _i32, _P, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _P,
                              _P, _P, _sz, _P]),
    "pa_decode_step_workspace_size": (_sz, [_i32, _i32, _i32, _i32]),
    "pa_decode_step_bucket": (_i32, [_i32]),
    "pa_shared_prefix_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_attention_varlen_shared_prefix": (_i32, [_P, _P, _P, _i64, _P, _i32, _P, _P, _P, _P, _i32, _i32, _i32, _i32,
                                                 _i32, _i32, _i32, _f32, _P, _P, _P, _sz, _P]),
    "pa_attention_varlen_noalloc": (_i32, [_P, _P, _P, _i64, _P, _i32, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32,
                                           _i32, _f32, _P, _P, _P, _P]),
    "pa_merge_lse": (_i32, [_P, _P, _P, _P, _P, _P, _i64, _i32, _i32, _P]),
    "pa_get_device_error": (_i32, [_P, ctypes.POINTER(_i32)]),
    "pa_clear_device_error": (_i32, [_P, _P]),
    "pa_set_decode_ctas": (_i32, [_i32]),
    "pa_set_prefill_ctas": (_i32, [_i32]),
    "pa_plan_tile_grid": (_i32, [ctypes.POINTER(_i32), _i32, _i64, _i32, ctypes.POINTER(_i32)]),
    "pa_plan_decode_grid": (_i32, [ctypes.POINTER(_i32), _i32, _i32, _i32, ctypes.POINTER(_i32),
                                   ctypes.POINTER(_i32)]),
    "pa_set_decode_fault_injection": (_i32, [_i32]),
    "pa_launch_count": (_i64, []),
    "pa_trace_enable": (_i32, [_i32]),
    "pa_trace_read": (_i32, [ctypes.POINTER(_i32), ctypes.POINTER(_f32), _i32, ctypes.POINTER(_i32)]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def header_functions() -> list:
    """Names of the functions include/pa.h declares."""
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(pa_\w+)\s*\(", src, flags=re.M)))


def status_string(status: int) -> str:
    return _lib.pa_status_string(status).decode()


def _check(status: int):
    if status != PA_OK:
        raise PAError(status, _lib.pa_last_error_message().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed device workspace of at least nbytes (256-byte aligned)."""
    return torch.zeros(max(int(nbytes), PA_ERROR_WORD_BYTES), dtype=torch.uint8, device=device)


def pa_abi_version() -> int:
    return int(_lib.pa_abi_version())


def pa_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, workspace=None, stream=None):
    """Scatter k_new/v_new [N, Hkv, D] bf16 into the HND pools by slot_mapping
    (int64 [N], negative = skip)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(slot_mapping, torch.int64, "slot_mapping")
    N, Hkv, D = k_new.shape
    nb, Hkv2, P, D2 = k_cache.shape
    if v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or Hkv2 != Hkv or D2 != D \
            or slot_mapping.shape != (N,):
        raise ValueError("inconsistent shapes")
    if workspace is None:
        workspace = new_workspace(PA_ERROR_WORD_BYTES, k_cache.device)
    _check(_lib.pa_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_cache), _ptr(v_cache), nb, P,
                             Hkv, D, _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


PA_Q8_SLAB_BYTES = 16 * 128 + 16 * (128 // 32) * 2


def new_q8_pool(num_blocks, num_kv_heads, device):
    """An empty q8_0 pool [num_blocks, Hkv, PA_Q8_SLAB_BYTES] (uint8)."""
    return torch.zeros((num_blocks, num_kv_heads, PA_Q8_SLAB_BYTES), dtype=torch.uint8, device=device)


def pa_kv_append_q8(k_new, v_new, slot_mapping, k_cache, v_cache, workspace=None, stream=None):
    """Quantize k_new / v_new [N, Hkv, D] bf16 into q8_0 pools (uint8
    [num_blocks, Hkv, PA_Q8_SLAB_BYTES]) at slot_mapping (int64 [N])."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(k_cache, torch.uint8, "k_cache")
    _need(v_cache, torch.uint8, "v_cache")
    _need(slot_mapping, torch.int64, "slot_mapping")
    N, Hkv, D = k_new.shape
    nb = k_cache.shape[0]
    if v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or k_cache.shape[1:] != (Hkv, PA_Q8_SLAB_BYTES) \
            or slot_mapping.shape != (N,):
        raise ValueError("inconsistent shapes")
    if workspace is None:
        workspace = new_workspace(PA_ERROR_WORD_BYTES, k_cache.device)
    _check(_lib.pa_kv_append_q8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_cache), _ptr(v_cache), nb,
                                16, Hkv, D, _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def pa_attention_varlen_q8(q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale, *, seq_lens_host=None,
                           qo_indptr_host=None, out=None, lse=None, workspace=None, stream=None, return_lse=False):
    """pa_attention_varlen over q8_0 pools (decode rows)."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.uint8, "k_cache")
    _need(v_cache, torch.uint8, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(qo_indptr, torch.int32, "qo_indptr")
    total_q, Hq, D = q.shape
    nb, Hkv, slab = k_cache.shape
    R = seq_lens.shape[0]
    if v_cache.shape != k_cache.shape or slab != PA_Q8_SLAB_BYTES or qo_indptr.shape != (R + 1,) \
            or block_tables.dim() != 2 or block_tables.shape[0] != R:
        raise ValueError("inconsistent shapes")
    slh = _host_i32(seq_lens if seq_lens_host is None else seq_lens_host)
    qih = _host_i32(qo_indptr if qo_indptr_host is None else qo_indptr_host)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if workspace is None:
        max_len = int(slh.max()) if R else 1
        workspace = new_workspace(pa_attention_workspace_size(R, total_q, Hq, D, max_len), q.device)
    _check(_lib.pa_attention_varlen_q8(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                       block_tables.shape[1], _ptr(seq_lens), _ptr(qo_indptr),
                                       ctypes.c_void_p(slh.data_ptr()), ctypes.c_void_p(qih.data_ptr()), R, total_q,
                                       Hq, Hkv, D, 16, float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                       workspace.numel(), _stream(stream)))
    return (out, lse) if (return_lse or lse is not None) else out


def pa_copy_blocks(src_blocks, dst_blocks, k_cache, v_cache, workspace=None, stream=None):
    """Copy whole blocks src_blocks[i] -> dst_blocks[i] of both HND pools
    (int32 [n] device ids; copy-on-write of shared blocks)."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(src_blocks, torch.int32, "src_blocks")
    _need(dst_blocks, torch.int32, "dst_blocks")
    if src_blocks.shape != dst_blocks.shape or src_blocks.dim() != 1 or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    nb, Hkv, P, D = k_cache.shape
    if workspace is None:
        workspace = new_workspace(PA_ERROR_WORD_BYTES, k_cache.device)
    _check(_lib.pa_copy_blocks(_ptr(src_blocks), _ptr(dst_blocks), src_blocks.shape[0], _ptr(k_cache),
                               _ptr(v_cache), nb, P, Hkv, D, _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def pa_attention_workspace_size(num_reqs, total_q, num_q_heads, head_dim, max_seq_len) -> int:
    return int(_lib.pa_attention_workspace_size(num_reqs, total_q, num_q_heads, head_dim, max_seq_len))


def _host_i32(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu", torch.int32).contiguous()
    else:
        t = torch.tensor(list(t), dtype=torch.int32)
    return t


def pa_attention_varlen(q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale, *, seq_lens_host=None,
                        qo_indptr_host=None, out=None, lse=None, workspace=None, stream=None, return_lse=False):
    """Paged varlen attention (see include/pa.h).  q [total_q, Hq, D] bf16;
    caches [num_blocks, Hkv, 16, D] bf16; block_tables int32 [R, max_blocks];
    seq_lens int32 [R]; qo_indptr int32 [R+1].  Host copies of seq_lens and
    qo_indptr are read back from the device when not given.  Returns out (and
    lse when return_lse or lse is given)."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(qo_indptr, torch.int32, "qo_indptr")
    total_q, Hq, D = q.shape
    nb, Hkv, P, D2 = k_cache.shape
    R = seq_lens.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or qo_indptr.shape != (R + 1,) or block_tables.dim() != 2 \
            or block_tables.shape[0] != R:
        raise ValueError("inconsistent shapes")
    slh = _host_i32(seq_lens if seq_lens_host is None else seq_lens_host)
    qih = _host_i32(qo_indptr if qo_indptr_host is None else qo_indptr_host)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if workspace is None:
        max_len = int(slh.max()) if R else 1
        workspace = new_workspace(pa_attention_workspace_size(R, total_q, Hq, D, max_len), q.device)
    _check(_lib.pa_attention_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                    block_tables.shape[1], _ptr(seq_lens), _ptr(qo_indptr),
                                    ctypes.c_void_p(slh.data_ptr()), ctypes.c_void_p(qih.data_ptr()), R, total_q, Hq,
                                    Hkv, D, P, float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                    workspace.numel(), _stream(stream)))
    return (out, lse) if (return_lse or lse is not None) else out


def pa_decode_step_workspace_size(num_reqs, num_q_heads, head_dim, max_seq_len) -> int:
    return int(_lib.pa_decode_step_workspace_size(num_reqs, num_q_heads, head_dim, max_seq_len))


def pa_decode_step_bucket(num_reqs) -> int:
    return int(_lib.pa_decode_step_bucket(num_reqs))


def pa_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, sm_scale, max_seq_len, *, out=None,
                   lse=None, workspace=None, stream=None, return_lse=False):
    """KV append + attention of a padded decode-only batch in one launch (see
    include/pa.h).  q [R, Hq, D] bf16; k_new / v_new [R, Hkv, D] bf16; caches
    [num_blocks, Hkv, 16, D] bf16 (the new tokens are written into them);
    block_tables int32 [R, max_blocks]; seq_lens int32 [R] on the device (0 =
    padding row).  Nothing is read back to the host, so the call can be
    captured in a CUDA graph and replayed with new contents of the same
    tensors.  Returns out (and lse when return_lse or lse is given)."""
    _need(q, torch.bfloat16, "q")
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    R, Hq, D = q.shape
    nb, Hkv, P, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or k_new.shape != (R, Hkv, D) or v_new.shape != (R, Hkv, D) \
            or seq_lens.shape != (R,) or block_tables.dim() != 2 or block_tables.shape[0] != R:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if lse is None and return_lse:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if workspace is None:
        workspace = new_workspace(pa_decode_step_workspace_size(R, Hq, D, max_seq_len), q.device)
    _check(_lib.pa_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), nb,
                               _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), R, int(max_seq_len), Hq,
                               Hkv, D, P, float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                               _stream(stream)))
    return (out, lse) if (return_lse or lse is not None) else out


def pa_shared_prefix_workspace_size(num_reqs, total_q, num_q_heads, head_dim, max_seq_len,
                                    shared_prefix_pages) -> int:
    return int(_lib.pa_shared_prefix_workspace_size(num_reqs, total_q, num_q_heads, head_dim, max_seq_len,
                                                    shared_prefix_pages))


def pa_attention_varlen_shared_prefix(q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale,
                                      shared_prefix_pages, *, seq_lens_host=None, qo_indptr_host=None, out=None,
                                      lse=None, workspace=None, stream=None, return_lse=False):
    """pa_attention_varlen for a batch whose block tables all begin with the
    same shared_prefix_pages blocks (see include/pa.h): the prefix is
    attended once for every query and merged into each row by log-sum-exp."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(qo_indptr, torch.int32, "qo_indptr")
    total_q, Hq, D = q.shape
    nb, Hkv, P, D2 = k_cache.shape
    R = seq_lens.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or qo_indptr.shape != (R + 1,) or block_tables.dim() != 2 \
            or block_tables.shape[0] != R:
        raise ValueError("inconsistent shapes")
    slh = _host_i32(seq_lens if seq_lens_host is None else seq_lens_host)
    qih = _host_i32(qo_indptr if qo_indptr_host is None else qo_indptr_host)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if workspace is None:
        max_len = int(slh.max()) if R else 1
        workspace = new_workspace(pa_shared_prefix_workspace_size(R, total_q, Hq, D, max_len, shared_prefix_pages),
                                  q.device)
    _check(_lib.pa_attention_varlen_shared_prefix(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        _ptr(qo_indptr), ctypes.c_void_p(slh.data_ptr()), ctypes.c_void_p(qih.data_ptr()), R, total_q, Hq, Hkv, D,
        P, int(shared_prefix_pages), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return (out, lse) if (return_lse or lse is not None) else out


def pa_attention_varlen_noalloc(q, k_cache, v_cache, block_tables, seq_lens, qo_indptr, sm_scale, *,
                                seq_lens_host=None, qo_indptr_host=None, out=None, lse=None, device_error=None,
                                stream=None, return_lse=False):
    """pa_attention_varlen for callers that cannot allocate device memory:
    the scratch is a fixed array inside libpa (see include/pa.h), so no
    workspace is passed.  `out`, `lse` and `device_error` (int32 [1]) are the
    caller's; this function allocates them only when they are not given."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(qo_indptr, torch.int32, "qo_indptr")
    total_q, Hq, D = q.shape
    nb, Hkv, P, D2 = k_cache.shape
    R = seq_lens.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or qo_indptr.shape != (R + 1,) or block_tables.dim() != 2 \
            or block_tables.shape[0] != R:
        raise ValueError("inconsistent shapes")
    slh = _host_i32(seq_lens if seq_lens_host is None else seq_lens_host)
    qih = _host_i32(qo_indptr if qo_indptr_host is None else qo_indptr_host)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if device_error is not None:
        _need(device_error, torch.int32, "device_error")
    _check(_lib.pa_attention_varlen_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                            block_tables.shape[1], _ptr(seq_lens), _ptr(qo_indptr),
                                            ctypes.c_void_p(slh.data_ptr()), ctypes.c_void_p(qih.data_ptr()), R,
                                            total_q, Hq, Hkv, D, P, float(sm_scale), _ptr(out), _ptr(lse),
                                            _ptr(device_error), _stream(stream)))
    return (out, lse) if (return_lse or lse is not None) else out


def pa_merge_lse(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """LSE merge of two partial attentions; o_* [rows, H, D] bf16, lse_*
    [rows, H] float32.  o_out may be o_a or o_b."""
    for t, n in ((o_a, "o_a"), (o_b, "o_b")):
        _need(t, torch.bfloat16, n)
    for t, n in ((lse_a, "lse_a"), (lse_b, "lse_b")):
        _need(t, torch.float32, n)
    rows, H, D = o_a.shape
    if o_b.shape != o_a.shape or lse_a.shape != (rows, H) or lse_b.shape != (rows, H):
        raise ValueError("inconsistent shapes")
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    _check(_lib.pa_merge_lse(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out), _ptr(lse_out), rows, H, D,
                             _stream(stream)))
    return o_out, lse_out


def pa_get_device_error(workspace) -> int:
    v = _i32(0)
    _check(_lib.pa_get_device_error(_ptr(workspace), ctypes.byref(v)))
    return int(v.value)


def pa_clear_device_error(workspace, stream=None):
    _check(_lib.pa_clear_device_error(_ptr(workspace), _stream(stream)))


def pa_set_decode_ctas(n: int):
    _check(_lib.pa_set_decode_ctas(int(n)))


def pa_set_prefill_ctas(n: int):
    """Prefill jobs beside the decode launch: n > 0 CTAs, -1 never, 0
    automatic (see include/pa.h)."""
    _check(_lib.pa_set_prefill_ctas(int(n)))


def pa_plan_tile_grid(job_tiles, decode_slabs: int, sms: int) -> int:
    """The persistent CTA count the library picks for tensor-core jobs of
    job_tiles[i] 128-key tiles (kernel order), beside decode_slabs (page, kv
    head) slabs of decode rows (0: the jobs alone), on sms SMs; 0 = one CTA
    per job (see include/pa.h).  Host only."""
    n = len(job_tiles)
    arr = (_i32 * max(n, 1))(*[int(t) for t in job_tiles])
    out = _i32(0)
    _check(_lib.pa_plan_tile_grid(arr if n else None, n, int(decode_slabs), int(sms), ctypes.byref(out)))
    return out.value


def pa_plan_decode_grid(seq_lens, num_kv_heads: int, sms: int):
    """(grid, warp_granular) of the decode launch planned for decode rows
    of these seq_lens on sms SMs (see include/pa.h).  Host only."""
    n = len(seq_lens)
    arr = (_i32 * max(n, 1))(*[int(x) for x in seq_lens])
    grid, wg = _i32(0), _i32(0)
    _check(_lib.pa_plan_decode_grid(arr if n else None, n, int(num_kv_heads), int(sms), ctypes.byref(grid),
                                    ctypes.byref(wg)))
    return grid.value, bool(wg.value)


def pa_set_decode_fault_injection(on: bool):
    """Test switch of the bounded-wait path (see include/pa.h): with on, the
    decode kernel's CTA 0 lets one wait run out (1 ms) and the call records
    PA_ERR_DEVICE_TIMEOUT."""
    _check(_lib.pa_set_decode_fault_injection(1 if on else 0))


def pa_launch_count() -> int:
    return int(_lib.pa_launch_count())


def pa_trace_enable(on: bool):
    _check(_lib.pa_trace_enable(1 if on else 0))


def pa_trace_read(capacity: int = 4096):
    """[(kernel name, ms)] for the launches recorded since the last read."""
    kinds = (_i32 * capacity)()
    ms = (_f32 * capacity)()
    n = _i32(0)
    _check(_lib.pa_trace_read(kinds, ms, capacity, ctypes.byref(n)))
    return [(KERNEL_KINDS.get(kinds[i], str(kinds[i])), float(ms[i])) for i in range(n.value)]
