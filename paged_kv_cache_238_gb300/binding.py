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

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_NO_SPACE = 0, 1, 2, 3, 4
PA_F32, PA_BF16 = 0, 1
PA_DEVERR_SLOT_RANGE, PA_DEVERR_BLOCK_RANGE, PA_DEVERR_LEN_RANGE, PA_DEVERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
PA_DEVERR_APPEND_SLOT = 0x10
PA_DEVERR_PREFIX_MISMATCH = 0x20
PA_DECODE_TABLES_READY = 0x1
PA_DECODE_POOL_READY = 0x2
PA_DRILL_OFF, PA_DRILL_DECODE_STAGE, PA_DRILL_PREFILL_K_TILE = 0, 1, 2
BLOCK_SIZE = 16

#: every symbol that include/pa.h declares
EXPORTED = ("pa_reshape_and_cache", "pa_decode_workspace_size", "pa_decode", "pa_prefill_chunk",
            "pa_decode_noalloc", "pa_get_device_errors", "pa_status_string",
            "pa_bm_create", "pa_bm_destroy", "pa_bm_num_free_blocks", "pa_bm_add_request", "pa_bm_append_tokens",
            "pa_bm_commit", "pa_bm_fork", "pa_bm_free_request", "pa_bm_get_blocks", "pa_bm_slot_mapping",
            "pa_bm_take_copies", "pa_bm_free_queue", "pa_bm_block_info", "pa_bm_num_blocks_for_memory", "pa_sha256",
            "pa_copy_blocks", "pa_reshape_and_cache_bs", "pa_decode_bs", "pa_prefill_chunk_bs",
            "pa_copy_blocks_bs", "pa_step", "pa_decode_append", "pa_bm_create_bs",
            "pa_bm_num_blocks_for_memory_bs", "pa_debug_set_wait_drill", "pa_decode_shared_prefix_workspace_size",
            "pa_decode_shared_prefix", "pa_debug_decode_slices")
#: block sizes the *_bs entry points accept
BLOCK_SIZES = (16, 32, 64, 128)
#: size of the library's fixed scratch used by pa_decode_noalloc
PA_DECODE_NOALLOC_MAX_BYTES = 16 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class StepDesc(ctypes.Structure):
    """Mirror of pa_step_desc in include/pa.h (same fields, same order, C layout)."""
    _fields_ = [
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("scale", ctypes.c_float), ("dtype", ctypes.c_int),
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p),
        ("num_new_tokens", ctypes.c_int32),
        ("prefill_out", ctypes.c_void_p), ("prefill_q", ctypes.c_void_p), ("prefill_block_table", ctypes.c_void_p),
        ("prefill_max_blocks_per_seq", ctypes.c_int32), ("prefill_seq_lens", ctypes.c_void_p),
        ("query_start_loc", ctypes.c_void_p),
        ("num_prefill_seqs", ctypes.c_int32), ("max_chunk_len", ctypes.c_int32),
        ("prefill_max_seq_len", ctypes.c_int32),
        ("decode_out", ctypes.c_void_p), ("decode_q", ctypes.c_void_p), ("decode_block_table", ctypes.c_void_p),
        ("decode_max_blocks_per_seq", ctypes.c_int32), ("decode_seq_lens", ctypes.c_void_p),
        ("num_decode_seqs", ctypes.c_int32), ("decode_max_seq_len", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("decode_sms", ctypes.c_int32), ("timing_events", ctypes.c_void_p),
    ]


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
            lib.pa_decode_shared_prefix_workspace_size.restype = sz
            lib.pa_decode_shared_prefix_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
            lib.pa_decode_shared_prefix.restype = ctypes.c_int
            lib.pa_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                                    vp, sz, ctypes.c_uint32, vp]
            lib.pa_debug_set_wait_drill.restype = ctypes.c_int
            lib.pa_debug_set_wait_drill.argtypes = [i32, ctypes.c_uint64]
            lib.pa_debug_decode_slices.restype = ctypes.c_int
            lib.pa_debug_decode_slices.argtypes = [ctypes.c_int64, i32, i32, i32, vp, vp]
            i64, pi32, pi64, pu8 = (ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_uint8))
            for name, res, args in (
                    ("pa_bm_create", ctypes.c_int, [i32, i32, ctypes.c_char_p, ctypes.POINTER(vp)]),
                    ("pa_bm_destroy", None, [vp]),
                    ("pa_bm_num_free_blocks", i32, [vp]),
                    ("pa_bm_add_request", ctypes.c_int, [vp, i64, pi32, i32, pu8, i32, pi32]),
                    ("pa_bm_append_tokens", ctypes.c_int, [vp, i64, pi32, i32]),
                    ("pa_bm_commit", ctypes.c_int, [vp, i64, i32]),
                    ("pa_bm_fork", ctypes.c_int, [vp, i64, i64]),
                    ("pa_bm_free_request", ctypes.c_int, [vp, i64]),
                    ("pa_bm_get_blocks", ctypes.c_int, [vp, i64, pi32, i32, pi32]),
                    ("pa_bm_slot_mapping", ctypes.c_int, [vp, i64, i32, i32, pi64]),
                    ("pa_bm_take_copies", ctypes.c_int, [vp, pi32, pi32, i32, pi32]),
                    ("pa_bm_free_queue", ctypes.c_int, [vp, pi32, i32, pi32]),
                    ("pa_bm_block_info", ctypes.c_int, [vp, i32, pi32, pu8, pi32]),
                    ("pa_bm_num_blocks_for_memory", i64, [sz, ctypes.c_double, i32, i32, i32, ctypes.c_int]),
                    ("pa_sha256", ctypes.c_int, [vp, sz, pu8]),
                    ("pa_copy_blocks", ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, ctypes.c_int, vp]),
                    ("pa_reshape_and_cache_bs", ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                               ctypes.c_int, vp]),
                    ("pa_decode_bs", ctypes.c_int, [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                                    f32, ctypes.c_int, vp, sz, vp]),
                    ("pa_prefill_chunk_bs", ctypes.c_int, [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                                           i32, i32, i32, f32, ctypes.c_int, vp]),
                    ("pa_copy_blocks_bs", ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int, vp]),
                    ("pa_step", ctypes.c_int, [ctypes.POINTER(StepDesc), vp]),
                    ("pa_bm_create_bs", ctypes.c_int, [i32, i32, i32, ctypes.c_char_p, ctypes.POINTER(vp)]),
                    ("pa_bm_num_blocks_for_memory_bs", i64, [sz, ctypes.c_double, i32, i32, i32, i32, ctypes.c_int]),
                    ("pa_decode_append", ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                        i32, i32, i32, f32, ctypes.c_int, vp, sz, ctypes.c_uint32,
                                                        vp])):
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
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


def _use_bs(k_cache, force: bool) -> bool:
    """The block size is the pool's third dimension; 16 goes through the plain entry point
    unless the *_bs one is asked for."""
    return force or int(k_cache.shape[2]) != BLOCK_SIZE


def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None, _bs: bool = False) -> None:
    """k, v: [T, H_kv, D]; k_cache, v_cache: [NB, H_kv, BS, D] (BS = block size: 16, 32, 64
    or 128); slot_mapping: [T] int64."""
    _need_cuda(k, v, k_cache, v_cache, slot_mapping)
    T, H_kv, D = k.shape
    lib = load()
    if _use_bs(k_cache, _bs):
        _check("pa_reshape_and_cache_bs", lib.pa_reshape_and_cache_bs(
            _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, H_kv, D, k_cache.shape[0],
            int(k_cache.shape[2]), _dtype_code(k), _stream(stream)))
        return
    _check("pa_reshape_and_cache", lib.pa_reshape_and_cache(
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, H_kv, D, k_cache.shape[0],
        _dtype_code(k), _stream(stream)))


def pa_reshape_and_cache_bs(k, v, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """pa_reshape_and_cache through the block-size entry point (block size = k_cache.shape[2])."""
    pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream, _bs=True)


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                             max_seq_len: int, dtype) -> int:
    import torch
    code = dtype if isinstance(dtype, int) else (PA_F32 if dtype == torch.float32 else PA_BF16)
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, code))


def pa_decode(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
              workspace=None, stream=None, _bs: bool = False) -> None:
    """out, q: [S, H_q, D]; block_table: [S, max_blocks] int32; seq_lens: [S] int32;
    k_cache, v_cache: [NB, H_kv, BS, D]; workspace: uint8 CUDA tensor of at least
    pa_decode_workspace_size(...) bytes (or None when that size is 0)."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens, workspace)
    S, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load()
    if _use_bs(k_cache, _bs):
        _check("pa_decode_bs", lib.pa_decode_bs(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
            _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, int(k_cache.shape[2]), float(scale),
            _dtype_code(q), _ptr(workspace), ws_bytes, _stream(stream)))
        return
    _check("pa_decode", lib.pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, float(scale), _dtype_code(q), _ptr(workspace),
        ws_bytes, _stream(stream)))


def pa_decode_shared_prefix_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                           max_seq_len: int, prefix_tokens: int) -> int:
    return int(load().pa_decode_shared_prefix_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                             max_seq_len, prefix_tokens))


def pa_decode_shared_prefix(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
                            prefix_tokens: int, workspace, stream=None, tables_ready: bool = False,
                            pool_ready: bool = False) -> None:
    """pa_decode for a batch whose table rows all start with the same prefix_tokens / 16 block
    ids (C ABI pa_decode_shared_prefix): the prefix is attended once per kv head; bf16.
    tables_ready / pool_ready: the promises PA_DECODE_TABLES_READY / PA_DECODE_POOL_READY about
    the kernel launched just before the call (see pa_decode_append)."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens, workspace)
    S, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pa_decode_shared_prefix", load().pa_decode_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, float(scale), int(prefix_tokens), _ptr(workspace),
        ws_bytes, (PA_DECODE_TABLES_READY if tables_ready else 0) | (PA_DECODE_POOL_READY if pool_ready else 0),
        _stream(stream)))


def pa_decode_bs(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
                 workspace=None, stream=None) -> None:
    """pa_decode through the block-size entry point (block size = k_cache.shape[2])."""
    pa_decode(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len, scale, workspace, stream, _bs=True)


def pa_decode_append(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, seq_lens,
                     max_seq_len: int, scale: float, workspace=None, stream=None, tables_ready: bool = False,
                     pool_ready: bool = False) -> None:
    """Decode step with its new tokens (C ABI pa_decode_append): k_new, v_new [S, H_kv, D] of
    sequence i's token at position seq_lens[i] - 1 are written to slot_mapping[i] ([S] int64)
    and attended to; one launch on the bf16 persistent path. tables_ready: the kernel launched
    just before on the stream writes neither seq_lens nor block_table (PA_DECODE_TABLES_READY);
    pool_ready: nor the pool rows this call reads (PA_DECODE_POOL_READY, implies tables_ready)."""
    _need_cuda(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, seq_lens, workspace)
    S, H_q, D = q.shape
    NB, H_kv, BS = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_append", load().pa_decode_append(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, int(BS),
        float(scale), _dtype_code(q), _ptr(workspace), ws_bytes,
        (PA_DECODE_TABLES_READY if tables_ready else 0) | (PA_DECODE_POOL_READY if pool_ready else 0),
        _stream(stream)))


def pa_decode_noalloc(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
                      stream=None) -> None:
    """pa_decode without a workspace argument, for callers that cannot allocate device
    memory: the library's fixed device scratch (PA_DECODE_NOALLOC_MAX_BYTES) is used instead.
    Calls share that scratch, so they must not overlap on the GPU. 16-token blocks only."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens)
    if int(k_cache.shape[2]) != BLOCK_SIZE:
        raise ValueError("pa_decode_noalloc takes 16-token blocks")
    S, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    _check("pa_decode_noalloc", load().pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), S, int(max_seq_len), H_q, H_kv, D, NB, float(scale), _dtype_code(q), _stream(stream)))


def pa_prefill_chunk(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, max_chunk_len: int,
                     max_seq_len: int, scale: float, stream=None, _bs: bool = False) -> None:
    """out, q: [T_q, H_q, D]; block_table: [S, max_blocks] int32; seq_lens: [S] int32;
    query_start_loc: [S + 1] int32; k_cache, v_cache: [NB, H_kv, BS, D]."""
    _need_cuda(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc)
    _, H_q, D = q.shape
    NB, H_kv = k_cache.shape[0], k_cache.shape[1]
    S = seq_lens.shape[0]
    lib = load()
    if _use_bs(k_cache, _bs):
        _check("pa_prefill_chunk_bs", lib.pa_prefill_chunk_bs(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
            _ptr(seq_lens), _ptr(query_start_loc), S, int(max_chunk_len), int(max_seq_len), H_q, H_kv, D, NB,
            int(k_cache.shape[2]), float(scale), _dtype_code(q), _stream(stream)))
        return
    _check("pa_prefill_chunk", lib.pa_prefill_chunk(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(query_start_loc), S, int(max_chunk_len), int(max_seq_len), H_q, H_kv, D, NB,
        float(scale), _dtype_code(q), _stream(stream)))


def pa_get_device_errors(clear: bool = True) -> int:
    """PA_DEVERR_* bits raised by kernels on the current device since the last clear (syncs)."""
    v = ctypes.c_uint32(0)
    _check("pa_get_device_errors", load().pa_get_device_errors(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def pa_debug_set_wait_drill(kind: int, limit_ns: int = 0) -> None:
    """Test hook: make one bounded wait of the named kernel run out (PA_DRILL_*), with
    limit_ns as those kernels' wait limit; PA_DRILL_OFF restores normal operation."""
    _check("pa_debug_set_wait_drill", load().pa_debug_set_wait_drill(int(kind), int(limit_ns)))


def pa_debug_decode_slices(units: int, ctas: int, light_ctas: int, light_units: int, owners: bool = True):
    """Test hook (host only): the bf16 grouped decode kernel's slices of `units` work units over
    `ctas` CTAs, the last `light_ctas` of them `light_units` units shorter. Returns (starts,
    owners): the first unit of each slice (ctas + 1 entries) and the slice of each unit (or
    None)."""
    starts = (ctypes.c_int64 * (int(ctas) + 1))()
    own = (ctypes.c_int32 * max(int(units), 1))() if owners else None
    _check("pa_debug_decode_slices",
           load().pa_debug_decode_slices(int(units), int(ctas), int(light_ctas), int(light_units),
                                         ctypes.cast(starts, ctypes.c_void_p),
                                         ctypes.cast(own, ctypes.c_void_p) if own is not None else None))
    return list(starts), (list(own)[:int(units)] if own is not None else None)


def pa_prefill_chunk_bs(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, max_chunk_len: int,
                        max_seq_len: int, scale: float, stream=None) -> None:
    """pa_prefill_chunk through the block-size entry point (block size = k_cache.shape[2])."""
    pa_prefill_chunk(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, max_chunk_len, max_seq_len,
                     scale, stream, _bs=True)


def pa_copy_blocks(k_cache, v_cache, block_pairs, stream=None, _bs: bool = False) -> None:
    """k_cache, v_cache: [NB, H_kv, BS, D]; block_pairs: int32 CUDA tensor [n, 2] of (src, dst)."""
    _need_cuda(k_cache, v_cache, block_pairs)
    NB, H_kv, BS, D = k_cache.shape
    lib = load()
    if _use_bs(k_cache, _bs):
        _check("pa_copy_blocks_bs", lib.pa_copy_blocks_bs(
            _ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), block_pairs.shape[0], H_kv, D, NB, int(BS),
            _dtype_code(k_cache), _stream(stream)))
        return
    _check("pa_copy_blocks", lib.pa_copy_blocks(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), block_pairs.shape[0], H_kv, D, NB, _dtype_code(k_cache),
        _stream(stream)))


def pa_copy_blocks_bs(k_cache, v_cache, block_pairs, stream=None) -> None:
    """pa_copy_blocks through the block-size entry point (block size = k_cache.shape[2])."""
    pa_copy_blocks(k_cache, v_cache, block_pairs, stream, _bs=True)


def pa_step(k_cache, v_cache, scale: float, k_new=None, v_new=None, slot_mapping=None,
            prefill_out=None, prefill_q=None, prefill_block_table=None, prefill_seq_lens=None, query_start_loc=None,
            max_chunk_len: int = 0, prefill_max_seq_len: int = 0,
            decode_out=None, decode_q=None, decode_block_table=None, decode_seq_lens=None,
            decode_max_seq_len: int = 0, workspace=None, decode_sms: int = 0, timing_events=None,
            stream=None) -> None:
    """One whole mixed step (C ABI pa_step): reshape_and_cache of the new tokens, then chunked
    prefill and decode attention side by side. A part whose tensors are None is skipped.
    k_cache, v_cache: [NB, H_kv, BS, D]; the other tensors as for the single-kernel calls.
    decode_sms: SMs held by the decode kernel while prefill runs (0 = 27/64 of them).
    timing_events: None or six torch.cuda.Event (or None) recorded before/after reshape,
    prefill and decode on the stream each kernel runs on."""
    _need_cuda(k_cache, v_cache, k_new, v_new, slot_mapping, prefill_out, prefill_q, prefill_block_table,
               prefill_seq_lens, query_start_loc, decode_out, decode_q, decode_block_table, decode_seq_lens,
               workspace)
    NB, H_kv, BS, D = k_cache.shape
    q_any = prefill_q if prefill_q is not None else decode_q
    d = StepDesc()
    d.k_cache, d.v_cache = _ptr(k_cache), _ptr(v_cache)
    d.num_blocks, d.block_size, d.num_kv_heads, d.head_dim = NB, BS, H_kv, D
    d.num_q_heads = q_any.shape[1] if q_any is not None else H_kv
    d.scale, d.dtype = float(scale), _dtype_code(k_cache)
    if slot_mapping is not None:
        d.k_new, d.v_new, d.slot_mapping = _ptr(k_new), _ptr(v_new), _ptr(slot_mapping)
        d.num_new_tokens = slot_mapping.shape[0]
    if prefill_q is not None:
        d.prefill_out, d.prefill_q = _ptr(prefill_out), _ptr(prefill_q)
        d.prefill_block_table, d.prefill_max_blocks_per_seq = _ptr(prefill_block_table), prefill_block_table.shape[1]
        d.prefill_seq_lens, d.query_start_loc = _ptr(prefill_seq_lens), _ptr(query_start_loc)
        d.num_prefill_seqs = prefill_seq_lens.shape[0]
        d.max_chunk_len, d.prefill_max_seq_len = int(max_chunk_len), int(prefill_max_seq_len)
    if decode_q is not None:
        d.decode_out, d.decode_q = _ptr(decode_out), _ptr(decode_q)
        d.decode_block_table, d.decode_max_blocks_per_seq = _ptr(decode_block_table), decode_block_table.shape[1]
        d.decode_seq_lens, d.num_decode_seqs = _ptr(decode_seq_lens), decode_seq_lens.shape[0]
        d.decode_max_seq_len = int(decode_max_seq_len)
    if workspace is not None:
        d.workspace, d.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    d.decode_sms = int(decode_sms)
    evs = None
    if timing_events is not None:
        if any(e is not None and not e.cuda_event for e in timing_events):
            raise ValueError("record each timing event once before passing it (torch creates events lazily)")
        evs = (ctypes.c_void_p * 6)(*[None if e is None else e.cuda_event for e in timing_events])
        d.timing_events = ctypes.cast(evs, ctypes.c_void_p)
    _check("pa_step", load().pa_step(ctypes.byref(d), _stream(stream)))


def pa_sha256(data: bytes) -> bytes:
    out = (ctypes.c_uint8 * 32)()
    buf = (ctypes.c_uint8 * max(1, len(data))).from_buffer_copy(data or b"\0")
    _check("pa_sha256", load().pa_sha256(ctypes.cast(buf, ctypes.c_void_p), len(data), out))
    return bytes(out)


def pa_bm_num_blocks_for_memory(free_bytes: int, utilization: float, num_layers: int, num_kv_heads: int,
                                head_dim: int, dtype, block_size: int = BLOCK_SIZE) -> int:
    import torch
    code = dtype if isinstance(dtype, int) else (PA_F32 if dtype == torch.float32 else PA_BF16)
    if block_size == BLOCK_SIZE:
        return int(load().pa_bm_num_blocks_for_memory(free_bytes, utilization, num_layers, num_kv_heads, head_dim,
                                                      code))
    return int(load().pa_bm_num_blocks_for_memory_bs(free_bytes, utilization, num_layers, num_kv_heads, head_dim,
                                                     int(block_size), code))


def _i32(xs):
    arr = (ctypes.c_int32 * max(1, len(xs)))(*xs)
    return arr


class BlockManager:
    """The library's host block manager (pa_bm_* in include/pa.h), one per KV pool."""

    def __init__(self, num_blocks: int, enable_caching: bool = True, hash_seed: Optional[str] = None,
                 block_size: int = BLOCK_SIZE):
        h = ctypes.c_void_p()
        seed = None if hash_seed is None else hash_seed.encode()
        if block_size == BLOCK_SIZE:
            _check("pa_bm_create", load().pa_bm_create(num_blocks, 1 if enable_caching else 0, seed, ctypes.byref(h)))
        else:
            _check("pa_bm_create_bs", load().pa_bm_create_bs(num_blocks, int(block_size), 1 if enable_caching else 0,
                                                             seed, ctypes.byref(h)))
        self.block_size = int(block_size)
        self._h = h
        self._lib = load()

    def close(self) -> None:
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(self._lib.pa_bm_num_free_blocks(self._h))

    def add_request(self, req_id: int, tokens, salt: bytes = b"") -> int:
        n = ctypes.c_int32(0)
        sb = (ctypes.c_uint8 * max(1, len(salt))).from_buffer_copy(salt or b"\0")
        _check("pa_bm_add_request", self._lib.pa_bm_add_request(self._h, req_id, _i32(list(tokens)), len(tokens), sb,
                                                                len(salt), ctypes.byref(n)))
        return int(n.value)

    def append_tokens(self, req_id: int, tokens) -> None:
        _check("pa_bm_append_tokens", self._lib.pa_bm_append_tokens(self._h, req_id, _i32(list(tokens)), len(tokens)))

    def commit(self, req_id: int, num_computed: int) -> None:
        _check("pa_bm_commit", self._lib.pa_bm_commit(self._h, req_id, num_computed))

    def fork(self, parent: int, child: int) -> None:
        _check("pa_bm_fork", self._lib.pa_bm_fork(self._h, parent, child))

    def free_request(self, req_id: int) -> None:
        _check("pa_bm_free_request", self._lib.pa_bm_free_request(self._h, req_id))

    def block_ids(self, req_id: int, capacity: Optional[int] = None):
        n = ctypes.c_int32(0)
        self._lib.pa_bm_get_blocks(self._h, req_id, None, 0, ctypes.byref(n))
        cap = n.value if capacity is None else capacity
        buf = (ctypes.c_int32 * max(1, cap))()
        st = self._lib.pa_bm_get_blocks(self._h, req_id, buf, cap, ctypes.byref(n))
        if st not in (PA_OK, PA_ERR_NO_SPACE):
            raise PaError("pa_bm_get_blocks", st)
        return list(buf[:cap])

    def slot_mapping(self, req_id: int, first: int, n: int):
        buf = (ctypes.c_int64 * max(1, n))()
        _check("pa_bm_slot_mapping", self._lib.pa_bm_slot_mapping(self._h, req_id, first, n, buf))
        return list(buf[:n])

    def take_copies(self, capacity: int = 4096):
        src, dst, n = (ctypes.c_int32 * capacity)(), (ctypes.c_int32 * capacity)(), ctypes.c_int32(0)
        _check("pa_bm_take_copies", self._lib.pa_bm_take_copies(self._h, src, dst, capacity, ctypes.byref(n)))
        return [(src[i], dst[i]) for i in range(n.value)]

    def free_queue(self):
        cap = max(1, self.num_free())
        buf, n = (ctypes.c_int32 * cap)(), ctypes.c_int32(0)
        _check("pa_bm_free_queue", self._lib.pa_bm_free_queue(self._h, buf, cap, ctypes.byref(n)))
        return list(buf[:n.value])

    def block_info(self, block_id: int):
        ref, has = ctypes.c_int32(0), ctypes.c_int32(0)
        h = (ctypes.c_uint8 * 32)()
        _check("pa_bm_block_info", self._lib.pa_bm_block_info(self._h, block_id, ctypes.byref(ref), h, ctypes.byref(has)))
        return int(ref.value), (bytes(h) if has.value else None)
