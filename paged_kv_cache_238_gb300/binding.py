"""Thin Python binding over libpa's C ABI (``include/pa.h``): argument marshalling only.

Every function takes torch tensors that already live on the GPU, derives the sizes the C
call needs from their shapes, and passes raw device pointers plus the current CUDA stream.
All computation happens in the library's sm_103a kernels; there is no other code path. If
the library cannot be built or loaded, the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional

from . import _build

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = 0, 1, 2, 3
PA_F32, PA_BF16 = 0, 1
PA_DEVERR_SLOT_RANGE, PA_DEVERR_BLOCK_RANGE, PA_DEVERR_LEN_RANGE, PA_DEVERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
BLOCK_SIZE = 16

#: every symbol that include/pa.h declares
EXPORTED = ("pa_reshape_and_cache", "pa_decode_workspace_size", "pa_decode", "pa_prefill_chunk",
            "pa_decode_noalloc", "pa_get_device_errors", "pa_status_string")
#: size of the library's fixed scratch used by pa_decode_noalloc
PA_DECODE_NOALLOC_MAX_BYTES = 16 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class PaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


def load(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load libpa.so (compiling it first when its sources changed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_needed else _build.LIB
            lib = ctypes.CDLL(path)
            vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            lib.pa_status_string.restype = ctypes.c_char_p
            lib.pa_status_string.argtypes = [ctypes.c_int]
            lib.pa_reshape_and_cache.restype = ctypes.c_int
            lib.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int, vp]
            lib.pa_decode_workspace_size.restype = sz
            lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, ctypes.c_int]
            lib.pa_decode.restype = ctypes.c_int
            lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, f32,
                                      ctypes.c_int, vp, sz, vp]
            lib.pa_prefill_chunk.restype = ctypes.c_int
            lib.pa_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                             i32, f32, ctypes.c_int, vp]
            lib.pa_decode_noalloc.restype = ctypes.c_int
            lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, f32,
                                              ctypes.c_int, vp]
            lib.pa_get_device_errors.restype = ctypes.c_int
            lib.pa_get_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


pa_status_string = status_string


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PaError(fn, status)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need_cuda(*ts) -> None:
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("libpa takes contiguous CUDA tensors")


def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """k, v: [T, H_kv, D]; k_cache, v_cache: [NB, H_kv, 16, D]; slot_mapping: [T] int64."""
    _need_cuda(k, v, k_cache, v_cache, slot_mapping)
    T, H_kv, D = k.shape
    _check("pa_reshape_and_cache", load().pa_reshape_and_cache(
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, H_kv, D, k_cache.shape[0],
        _dtype_code(k), _stream(stream)))


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                             max_seq_len: int, dtype) -> int:
    import torch
    code = dtype if isinstance(dtype, int) else (PA_F32 if dtype == torch.float32 else PA_BF16)
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, code))


def pa_decode(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
              workspace=None, stream=None) -> None:
    """out, q: [S, H_q, D]; block_table: [S, max_blocks] int32; seq_lens: [S] int32;
    workspace: uint8 CUDA tensor of at least pa_decode_workspace_size(...) bytes (or None
    when that size is 0)."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens, workspace)
    S, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode", load().pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, float(scale), _dtype_code(q), _ptr(workspace),
        ws_bytes, _stream(stream)))


def pa_decode_noalloc(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
                      stream=None) -> None:
    """pa_decode without a workspace argument, for callers that cannot allocate device
    memory: the library's fixed device scratch (PA_DECODE_NOALLOC_MAX_BYTES) is used instead.
    Calls share that scratch, so they must not overlap on the GPU."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens)
    S, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    _check("pa_decode_noalloc", load().pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, float(scale), _dtype_code(q), _stream(stream)))


def pa_prefill_chunk(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, max_chunk_len: int,
                     max_seq_len: int, scale: float, stream=None) -> None:
    """out, q: [T_q, H_q, D]; block_table: [S, max_blocks] int32; seq_lens: [S] int32;
    query_start_loc: [S + 1] int32."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc)
    _, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    S = seq_lens.shape[0]
    _check("pa_prefill_chunk", load().pa_prefill_chunk(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(query_start_loc), S, int(max_chunk_len), int(max_seq_len), H_q, H_kv, D, NB,
        float(scale), _dtype_code(q), _stream(stream)))


def pa_get_device_errors(clear: bool = True) -> int:
    """PA_DEVERR_* bits raised by kernels on the current device since the last clear (syncs)."""
    v = ctypes.c_uint32(0)
    _check("pa_get_device_errors", load().pa_get_device_errors(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)
