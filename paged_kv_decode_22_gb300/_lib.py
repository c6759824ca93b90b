"""ctypes binding of libpkd.so (C ABI in include/pkd.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors are torch CUDA tensors; their device pointers and the
current CUDA stream are passed through.  If the library has not been built
this module raises on first use: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkd.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pkd.h")

FP16, BF16 = 0, 1
PATH_SIMT, PATH_TC, PATH_TC_CLUSTER, PATH_TC_STREAM = 0, 1, 2, 3
PARTITION_STREAM = -1   # partition_size that asks for the stream form
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_LEN, DEV_TIMEOUT = 1, 2, 4, 8

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

_SIGS = {
    "pkd_decode_plan": (_c_int, [_c_int] * 7 + [ctypes.POINTER(_c_int)] * 3 +
                        [ctypes.POINTER(_c_size)]),
    "pkd_decode_workspace_bytes": (_c_size, [_c_int] * 4),
    "pkd_paged_decode_attention": (_c_int, [_vp] * 5 + [_c_int, _vp] + [_c_int] * 7 +
                                   [_c_float, _c_int, _c_int, _vp, _c_size, _vp, _vp]),
    "pkd_paged_decode_attention_ex": (_c_int, [_vp] * 5 + [_c_int, _vp] + [_c_int] * 7 +
                                      [_c_float, _vp, _c_int, _c_int, _vp, _c_size, _vp, _vp]),
    "pkd_paged_decode_attention_static_ws": (_c_int, [_vp] * 5 + [_c_int, _vp] + [_c_int] * 7 +
                                             [_c_float, _c_int, _c_int, _vp, _vp]),
    "pkd_paged_prefill_attention": (_c_int, [_vp] * 5 + [_c_int, _vp, _vp] + [_c_int] * 9 +
                                    [_c_float, _vp, _c_int, _vp, _vp]),
    "pkd_gather_cached_kv": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_vp, _vp]),
    "pkd_reshape_and_cache": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_vp, _vp]),
    "pkd_selftest_bounded_wait": (_c_int, [_vp, ctypes.c_longlong, _vp]),
    "pkd_status_string": (ctypes.c_char_p, [_c_int]),
    "pkd_last_error": (ctypes.c_char_p, []),
    "pkd_version": (_c_int, []),
}

_lib = None


class PkdError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed with status {status}: {text}")
        self.status = status


def exported_names():
    """Function names the public header declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"PKD_API\s+[\w\s\*]+?\b(pkd_\w+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """Load libpkd.so once; raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run paged_kv_decode_22_gb300.build.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        text = lib().pkd_status_string(status).decode()
        detail = lib().pkd_last_error().decode()
        raise PkdError(fn, status, text + (f" [{detail}]" if detail and status == 6 else ""))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FP16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dense(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def decode_plan(num_seqs, num_heads, num_kv_heads, head_size, block_size, max_context_len,
                partition_size=0):
    """(partition_size, num_partitions, path, workspace_bytes) the library will use."""
    ps, npart, path = _c_int(), _c_int(), _c_int()
    ws = _c_size()
    st = lib().pkd_decode_plan(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                               max_context_len, partition_size, ctypes.byref(ps),
                               ctypes.byref(npart), ctypes.byref(path), ctypes.byref(ws))
    _check("pkd_decode_plan", st)
    return ps.value, npart.value, path.value, ws.value


def decode_workspace_bytes(num_seqs, num_heads, head_size, max_context_len):
    """Workspace bytes that serve paged_decode_attention with partition_size 0
    for any KV-head count and block size with these sizes (0: none needed)."""
    return lib().pkd_decode_workspace_bytes(num_seqs, num_heads, head_size, max_context_len)


def paged_decode_attention(out, q, key_cache, value_cache, block_tables, context_lens,
                           max_context_len, scale, partition_size=0, workspace=None,
                           device_status=None, stream=None, alibi_slopes=None):
    """out[s, h] = softmax(scale * q[s, h] . K_s^T [+ ALiBi]) V_s through the block table.

    q/out [S, H, D]; key_cache/value_cache [NB, B, Hk, D]; block_tables int32
    [S, MB]; context_lens int32 [S]; alibi_slopes: None or float32 [H].
    ``workspace`` (uint8 CUDA tensor) is allocated here through torch when the
    plan needs one and none is given.
    """
    _dense(out, q, key_cache, value_cache, block_tables, context_lens, workspace, device_status,
           alibi_slopes)
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or
                                     alibi_slopes.numel() != q.shape[1]):
        raise TypeError("alibi_slopes must be float32 [num_heads]")
    S, H, D = q.shape
    NB, B, Hk, _ = key_cache.shape
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    ps, npart, _, ws_bytes = decode_plan(S, H, Hk, D, B, max_context_len, partition_size)
    if ws_bytes > 0 and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = lib().pkd_paged_decode_attention_ex(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), max_context_len, S, H, Hk, D, B, NB,
        float(scale), _ptr(alibi_slopes), _dtype_code(q), partition_size, _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(device_status), _stream(stream))
    _check("pkd_paged_decode_attention_ex", st)
    return out


def paged_decode_attention_static_ws(out, q, key_cache, value_cache, block_tables, context_lens,
                                     max_context_len, scale, partition_size=0,
                                     device_status=None, stream=None):
    """paged_decode_attention without a workspace argument, for callers that
    cannot allocate device memory: the library's built-in scratch array is
    used (see pkd_paged_decode_attention_static_ws in include/pkd.h)."""
    _dense(out, q, key_cache, value_cache, block_tables, context_lens, device_status)
    S, H, D = q.shape
    NB, B, Hk, _ = key_cache.shape
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    st = lib().pkd_paged_decode_attention_static_ws(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), max_context_len, S, H, Hk, D, B, NB,
        float(scale), _dtype_code(q), partition_size, _ptr(device_status), _stream(stream))
    _check("pkd_paged_decode_attention_static_ws", st)
    return out


def paged_prefill_attention(out, q, key_cache, value_cache, block_tables, context_lens,
                            query_start, max_query_len, max_context_len, scale,
                            device_status=None, stream=None, alibi_slopes=None):
    """Chunk queries attending causally over the paged cache.

    q/out [T, H, D] (T packed query tokens); query_start int32 [S + 1];
    key_cache/value_cache [NB, B, Hk, D]; block_tables int32 [S, MB];
    context_lens int32 [S] (counting each chunk); alibi_slopes: None or
    float32 [H].  Query i of sequence s sits at position
    context_lens[s] - n_s + i and sees the cache up to that position.
    """
    _dense(out, q, key_cache, value_cache, block_tables, context_lens, query_start,
           device_status, alibi_slopes)
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or
                                     alibi_slopes.numel() != q.shape[1]):
        raise TypeError("alibi_slopes must be float32 [num_heads]")
    T, H, D = q.shape
    NB, B, Hk, _ = key_cache.shape
    S = context_lens.numel()
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or
            query_start.dtype != torch.int32 or query_start.numel() != S + 1):
        raise TypeError("block_tables, context_lens and query_start [S + 1] must be int32")
    st = lib().pkd_paged_prefill_attention(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), _ptr(query_start), T, max_query_len,
        max_context_len, S, H, Hk, D, B, NB, float(scale), _ptr(alibi_slopes), _dtype_code(q),
        _ptr(device_status), _stream(stream))
    _check("pkd_paged_prefill_attention", st)
    return out


def gather_cached_kv(key_out, value_out, key_cache, value_cache, slot_mapping,
                     device_status=None, stream=None):
    """key_out[t] = key_cache[slot // B, slot % B] (and V), slot = slot_mapping[t]."""
    _dense(key_out, value_out, key_cache, value_cache, slot_mapping, device_status)
    NB, B, H, D = key_cache.shape
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    st = lib().pkd_gather_cached_kv(
        _ptr(key_out), _ptr(value_out), _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping),
        slot_mapping.numel(), H, D, B, NB, _dtype_code(key_cache), _ptr(device_status),
        _stream(stream))
    _check("pkd_gather_cached_kv", st)
    return key_out, value_out


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, device_status=None,
                      stream=None):
    """key_cache[slot // B, slot % B] = key[t] (and V); negative slots are skipped."""
    _dense(key, value, key_cache, value_cache, slot_mapping, device_status)
    NB, B, H, D = key_cache.shape
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    st = lib().pkd_reshape_and_cache(
        _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping),
        slot_mapping.numel(), H, D, B, NB, _dtype_code(key_cache), _ptr(device_status),
        _stream(stream))
    _check("pkd_reshape_and_cache", st)


def version() -> int:
    return lib().pkd_version()
