"""fp64 CPU oracle for paged-KV attention: TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never links, loads or
calls it, and it shares no code with the CUDA library: the C source here
(``pa_oracle.c``) is compiled with gcc into its own shared object.

Functions (numpy in, numpy out):

``reshape_and_cache``
    Bitwise scatter of new K/V rows into their slots: slot s lands in physical
    block s // 16 at offset s % 16 ("vLLM: what PagedAttention turned into",
    "The problem PagedAttention was actually solving": the int64
    slot_mapping; "My Understanding of vLLM and PagedAttention", "Logical
    Blocks").
``attention``
    Gathers each sequence's K/V from the block table into contiguous fp64
    arrays ("My Understanding...", "Block Table" and "Step 4 - Attention
    Computation") and evaluates softmax(scale * q K^T) V over the visible keys,
    all in fp64. Decode rows sit at position len - 1; prefill chunk rows are
    bottom-right aligned (row r of a chunk of C tokens sits at len - C + r).

bf16 arrays are passed as numpy ``uint16`` (or ``int16``) bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
# PA_SANITIZE=address,undefined: a sanitizer build (liboracle_san.so), as for libpa
_SANITIZE = os.environ.get("PA_SANITIZE", "").strip()
_LIB = os.path.join(_HERE, "liboracle_san.so" if _SANITIZE else "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
BLOCK_SIZE = 16


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` with gcc (OpenMP, no fast-math) into liboracle.so."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    san = [f"-fsanitize={_SANITIZE}", "-fno-omit-frame-pointer", "-g"] if _SANITIZE else []
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared"] + san + [_SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _declare(lib):
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.oracle_reshape_and_cache.restype = ctypes.c_int
    lib.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32,
                                     i32, i32, i32, i32, i32, ctypes.c_double, i32, i32]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype in (np.uint16, np.int16):
        return BF16
    raise TypeError(f"oracle supports float32 or bf16 bit patterns (uint16/int16), got {a.dtype}")


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype=None):
    a = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))
    return a


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, _lib_override=None) -> None:
    """In-place: k_cache[s // bs, :, s % bs, :] = k[t] (same for v), for s = slot_mapping[t] >= 0.

    k, v: [T, H_kv, D]; k_cache, v_cache: [num_blocks, H_kv, bs, D] (C-contiguous,
    modified in place; the block size bs is the pool's third dimension, 16 by default);
    slot_mapping: [T] int64.
    """
    k = _c(k)
    v = _c(v)
    slots = _c(slot_mapping, np.int64)
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    assert k.dtype == v.dtype == k_cache.dtype == v_cache.dtype
    T, H_kv, D = k.shape
    nb = k_cache.shape[0]
    bs = k_cache.shape[2]
    assert k_cache.shape == (nb, H_kv, bs, D) and v_cache.shape == k_cache.shape
    assert slots.shape == (T,)
    rc = (_lib_override or _load()).oracle_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slots),
                                          T, H_kv, D, nb, bs, k.dtype.itemsize)
    if rc != 0:
        raise ValueError("oracle_reshape_and_cache: slot outside the pool")


def attention(q, k_cache, v_cache, block_table, seq_lens, scale, query_start_loc=None,
              num_threads: int = 0, _lib_override=None) -> np.ndarray:
    """Exact fp64 paged attention. Returns float64 [T_q, H_q, D].

    q: [T_q, H_q, D] (T_q = S for decode); k_cache, v_cache: [NB, H_kv, bs, D] (bs, the
    block size, is the pool's third dimension);
    block_table: [S, max_blocks] int32; seq_lens: [S] int32 (keys incl. the current
    token); query_start_loc: None (decode) or [S + 1] int32 prefix sums of chunk lengths.
    num_threads: OpenMP threads (0 = runtime default).
    """
    q = _c(q)
    k_cache = _c(k_cache)
    v_cache = _c(v_cache)
    bt = _c(block_table, np.int32)
    lens = _c(seq_lens, np.int32)
    dt = _dtype_code(q)
    assert q.dtype == k_cache.dtype == v_cache.dtype
    T_q, H_q, D = q.shape
    nb, H_kv, bs, D2 = k_cache.shape
    assert bs > 0 and D2 == D and v_cache.shape == k_cache.shape
    S = lens.shape[0]
    if bt.ndim != 2 or bt.shape[0] != S:
        raise ValueError("block_table must be [S, max_blocks]")
    if query_start_loc is None:
        qsl_ptr = None
        if T_q != S:
            raise ValueError("decode expects one query row per sequence")
    else:
        qsl = _c(query_start_loc, np.int32)
        assert qsl.shape == (S + 1,) and qsl[-1] == T_q
        qsl_ptr = _ptr(qsl)
    out = np.empty((T_q, H_q, D), dtype=np.float64)
    rc = (_lib_override or _load()).oracle_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1],
                                  _ptr(lens), qsl_ptr, S, H_q, H_kv, D, nb, bs, float(scale), dt,
                                  int(num_threads))
    if rc != 0:
        raise ValueError("oracle_attention: invalid tables (block id, length or chunk out of range)")
    return out


def load_variant(so_path: str):
    """Load another build of the oracle source (used only to show that the pins catch
    a deliberately planted mistake); pass the result as ``_lib_override``."""
    return _declare(ctypes.CDLL(so_path))
