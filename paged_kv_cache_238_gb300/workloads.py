"""Seeded synthetic inputs for paged-KV attention (shared by the tests, the bench and the smoke check).

This module only draws inputs. It holds none of the attention arithmetic and
imports neither the CUDA binding nor the oracle.

Recipe (all values from ``numpy.random.default_rng(seed)``):
  * Q, K and V entries are drawn N(0, 1) in fp32; for bf16 workloads they are
    rounded to nearest-even bf16 and stored as uint16 bit patterns.
  * Physical block ids are a random permutation of 1..num_blocks-1, handed out
    in order: block 0 is the null block that "no block" points at ("vLLM: what
    PagedAttention turned into", "The block pool": the null block burned at
    construction). Unused block-table entries hold 0.
  * Every pool cell that no sequence owns (block 0, unused blocks and the
    unfilled tail of each last block) is poisoned with NaN, so a kernel that
    reads outside the visible keys produces NaN instead of a plausible number.
  * A decode sequence of length L stores keys 0..L-2 in the pool and brings
    key L-1 as a new token whose slot is block_table[L-1 // 16] * 16 + (L-1) % 16
    (slot = physical block * 16 + offset).
  * Context-length mixes follow the five workload descriptions: a tiny fp32
    case, lognormal lengths with mean about 195 tokens (the length implied by
    u = L / (L + 7.5) = 0.963, "Checking the 96.3%"), a 1024-token shared prefix
    aliased by 128 sequences, 8 x 32768-token sequences, and a mixed
    chunked-prefill + decode step.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

BLOCK = 16
BF16_NAN = np.uint16(0x7FC0)


# --------------------------------------------------------------------------------------
# bf16 helpers (bit patterns in uint16)
# --------------------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to nearest-even bf16; returns uint16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def _nan_like_pool(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return np.full(shape, BF16_NAN, dtype=np.uint16)
    return np.full(shape, np.nan, dtype=np.float32)


def as_f64(a: np.ndarray) -> np.ndarray:
    """Widen stored values (fp32 or bf16 bits) to fp64 exactly."""
    if a.dtype == np.float32:
        return a.astype(np.float64)
    return bf16_bits_to_f32(a).astype(np.float64)


# --------------------------------------------------------------------------------------
# Workload container
# --------------------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    dtype: str                      # "f32" or "bf16"
    H_q: int
    H_kv: int
    D: int
    num_blocks: int
    scale: float
    k_cache: np.ndarray             # [NB, H_kv, block_size, D]
    v_cache: np.ndarray
    # decode part
    q: Optional[np.ndarray] = None              # [S, H_q, D]
    block_table: Optional[np.ndarray] = None    # [S, max_blocks] int32
    seq_lens: Optional[np.ndarray] = None       # [S] int32
    # prefill part (chunked prefill sequences)
    q_prefill: Optional[np.ndarray] = None      # [T_p, H_q, D]
    block_table_prefill: Optional[np.ndarray] = None
    seq_lens_prefill: Optional[np.ndarray] = None
    query_start_loc: Optional[np.ndarray] = None  # [S_p + 1] int32
    # new tokens written by reshape_and_cache (all sequences, padding included)
    k_new: Optional[np.ndarray] = None          # [T, H_kv, D]
    v_new: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None   # [T] int64
    # contiguous per-sequence K/V (all keys incl. new tokens) for small cases only
    contiguous_k: Optional[List[np.ndarray]] = None   # each [len, H_kv, D]
    contiguous_v: Optional[List[np.ndarray]] = None
    contiguous_k_prefill: Optional[List[np.ndarray]] = None
    contiguous_v_prefill: Optional[List[np.ndarray]] = None
    info: Dict[str, object] = field(default_factory=dict)

    @property
    def S(self) -> int:
        return 0 if self.seq_lens is None else int(self.seq_lens.shape[0])


class _BlockAllocator:
    """Hands out physical ids 1..NB-1 in a seeded random order (0 stays the null block)."""

    def __init__(self, rng: np.random.Generator, num_blocks: int):
        self.ids = rng.permutation(np.arange(1, num_blocks, dtype=np.int64))
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        if self.next + n > self.ids.shape[0]:
            raise ValueError("pool too small for the requested workload")
        out = self.ids[self.next:self.next + n]
        self.next += n
        return out


def _table(ids_per_seq: List[np.ndarray], max_blocks: Optional[int] = None) -> np.ndarray:
    mb = max(1, max((len(x) for x in ids_per_seq), default=1))
    if max_blocks is not None:
        mb = max(mb, max_blocks)
    bt = np.zeros((len(ids_per_seq), mb), dtype=np.int32)
    for i, ids in enumerate(ids_per_seq):
        bt[i, :len(ids)] = ids
    return bt


def _store_tokens(pool: np.ndarray, ids: np.ndarray, first: int, vals: np.ndarray) -> None:
    """Place vals[j] (j = 0..n-1, [n, H_kv, D]) at logical positions first..first+n-1 of a
    sequence whose logical blocks are ``ids`` (block size = the pool's third dimension)."""
    n = vals.shape[0]
    if n == 0:
        return
    bs = pool.shape[2]
    pos = np.arange(first, first + n)
    pool[ids[pos // bs], :, pos % bs, :] = vals


# --------------------------------------------------------------------------------------
# Generic builders
# --------------------------------------------------------------------------------------

def build_decode(seed: int, lens, H_q: int, H_kv: int, D: int, num_blocks: int, dtype: str,
                 new_token: bool = True, shared_prefix_tokens: int = 0, keep_contiguous: bool = False,
                 name: str = "decode", max_blocks: Optional[int] = None, poison: bool = True,
                 block_size: int = BLOCK) -> Workload:
    """Decode batch: one query per sequence at position len-1.

    block_size: tokens per physical block (16 by default; 32, 64, 128 are the variants).
    shared_prefix_tokens: if > 0 (a multiple of the block size), every sequence's first
    shared_prefix_tokens keys alias the same physical blocks (same values).
    new_token: key len-1 of each sequence arrives through reshape_and_cache
    (its pool cell starts poisoned) instead of being in the pool already.
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    S = lens.shape[0]
    BS = int(block_size)
    if shared_prefix_tokens % BS:
        raise ValueError("shared prefix must be block aligned")
    if new_token and shared_prefix_tokens and np.any(lens <= shared_prefix_tokens):
        raise ValueError("a new token may not land in a shared block")
    alloc = _BlockAllocator(rng, num_blocks)
    pool_shape = (num_blocks, H_kv, BS, D)
    k_cache = _nan_like_pool(pool_shape, dtype) if poison else np.zeros(pool_shape, _np_dtype(dtype))
    v_cache = _nan_like_pool(pool_shape, dtype) if poison else np.zeros(pool_shape, _np_dtype(dtype))

    n_shared_blocks = shared_prefix_tokens // BS
    shared_ids = alloc.take(n_shared_blocks)
    shared_k = _draw(rng, (shared_prefix_tokens, H_kv, D), dtype)
    shared_v = _draw(rng, (shared_prefix_tokens, H_kv, D), dtype)
    _store_tokens(k_cache, shared_ids, 0, shared_k)
    _store_tokens(v_cache, shared_ids, 0, shared_v)

    ids_per_seq, ck, cv = [], [], []
    k_new = np.empty((S, H_kv, D), dtype=_np_dtype(dtype))
    v_new = np.empty_like(k_new)
    slots = np.empty((S,), dtype=np.int64)
    for i in range(S):
        L = int(lens[i])
        nblk = (L + BS - 1) // BS
        own = alloc.take(max(0, nblk - n_shared_blocks))
        ids = np.concatenate([shared_ids[:min(nblk, n_shared_blocks)], own]).astype(np.int64)
        ids_per_seq.append(ids)
        n_own_keys = max(0, L - shared_prefix_tokens)
        kk = _draw(rng, (n_own_keys, H_kv, D), dtype)
        vv = _draw(rng, (n_own_keys, H_kv, D), dtype)
        n_pool = n_own_keys - 1 if (new_token and L > 0) else n_own_keys
        _store_tokens(k_cache, ids, shared_prefix_tokens, kk[:n_pool])
        _store_tokens(v_cache, ids, shared_prefix_tokens, vv[:n_pool])
        if new_token and L > 0:
            k_new[i] = kk[-1]
            v_new[i] = vv[-1]
            slots[i] = int(ids[(L - 1) // BS]) * BS + (L - 1) % BS
        else:
            k_new[i] = 0
            v_new[i] = 0
            slots[i] = -1
        if keep_contiguous:
            pre = min(L, shared_prefix_tokens)
            ck.append(np.concatenate([shared_k[:pre], kk], axis=0))
            cv.append(np.concatenate([shared_v[:pre], vv], axis=0))
    q = _draw(rng, (S, H_q, D), dtype)
    wl = Workload(name=name, dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, num_blocks=num_blocks,
                  scale=1.0 / float(np.sqrt(D)), k_cache=k_cache, v_cache=v_cache, q=q,
                  block_table=_table(ids_per_seq, max_blocks), seq_lens=lens.astype(np.int32))
    if new_token:
        wl.k_new, wl.v_new, wl.slot_mapping = k_new, v_new, slots
    if keep_contiguous:
        wl.contiguous_k, wl.contiguous_v = ck, cv
    wl.info["blocks_used"] = int(alloc.next + 1)
    wl.info["shared_prefix_tokens"] = int(shared_prefix_tokens)
    return wl


def _np_dtype(dtype: str):
    return np.uint16 if dtype == "bf16" else np.float32


def build_mixed(seed: int, prior_lens, chunk_lens, decode_lens, H_q: int, H_kv: int, D: int,
                num_blocks: int, dtype: str = "bf16", pad_multiple: int = 256,
                keep_contiguous: bool = False, name: str = "mixed", block_size: int = BLOCK) -> Workload:
    """Mixed step: chunked-prefill sequences (prior context in the pool, a chunk of new
    tokens written by reshape_and_cache) plus decode sequences (one new token each).
    The new-token list is padded to a multiple of ``pad_multiple`` with padding slots
    that point into the null block 0 (slot i % block_size)."""
    BS = int(block_size)
    rng = np.random.default_rng(seed)
    prior_lens = np.asarray(prior_lens, dtype=np.int64)
    chunk_lens = np.asarray(chunk_lens, dtype=np.int64)
    decode_lens = np.asarray(decode_lens, dtype=np.int64)
    alloc = _BlockAllocator(rng, num_blocks)
    pool_shape = (num_blocks, H_kv, BS, D)
    k_cache = _nan_like_pool(pool_shape, dtype)
    v_cache = _nan_like_pool(pool_shape, dtype)

    new_k, new_v, new_slots = [], [], []
    ids_p, ck_p, cv_p = [], [], []
    for i in range(prior_lens.shape[0]):
        P, C = int(prior_lens[i]), int(chunk_lens[i])
        L = P + C
        ids = alloc.take((L + BS - 1) // BS)
        ids_p.append(ids)
        kk = _draw(rng, (L, H_kv, D), dtype)
        vv = _draw(rng, (L, H_kv, D), dtype)
        _store_tokens(k_cache, ids, 0, kk[:P])
        _store_tokens(v_cache, ids, 0, vv[:P])
        pos = np.arange(P, L)
        new_k.append(kk[P:])
        new_v.append(vv[P:])
        new_slots.append(ids[pos // BS] * BS + pos % BS)
        if keep_contiguous:
            ck_p.append(kk)
            cv_p.append(vv)
    ids_d, ck_d, cv_d = [], [], []
    for i in range(decode_lens.shape[0]):
        L = int(decode_lens[i])
        ids = alloc.take((L + BS - 1) // BS)
        ids_d.append(ids)
        kk = _draw(rng, (L, H_kv, D), dtype)
        vv = _draw(rng, (L, H_kv, D), dtype)
        _store_tokens(k_cache, ids, 0, kk[:L - 1])
        _store_tokens(v_cache, ids, 0, vv[:L - 1])
        new_k.append(kk[L - 1:])
        new_v.append(vv[L - 1:])
        new_slots.append(np.array([ids[(L - 1) // BS] * BS + (L - 1) % BS], dtype=np.int64))
        if keep_contiguous:
            ck_d.append(kk)
            cv_d.append(vv)
    k_new = np.concatenate(new_k, axis=0)
    v_new = np.concatenate(new_v, axis=0)
    slots = np.concatenate(new_slots).astype(np.int64)
    T = k_new.shape[0]
    T_pad = -(-T // pad_multiple) * pad_multiple if pad_multiple else T
    if T_pad > T:
        n_pad = T_pad - T
        k_new = np.concatenate([k_new, _draw(rng, (n_pad, H_kv, D), dtype)], axis=0)
        v_new = np.concatenate([v_new, _draw(rng, (n_pad, H_kv, D), dtype)], axis=0)
        slots = np.concatenate([slots, np.arange(n_pad, dtype=np.int64) % BS])  # block 0
    q_p = _draw(rng, (int(chunk_lens.sum()), H_q, D), dtype)
    q_d = _draw(rng, (decode_lens.shape[0], H_q, D), dtype)
    qsl = np.zeros((chunk_lens.shape[0] + 1,), dtype=np.int32)
    qsl[1:] = np.cumsum(chunk_lens)
    wl = Workload(name=name, dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, num_blocks=num_blocks,
                  scale=1.0 / float(np.sqrt(D)), k_cache=k_cache, v_cache=v_cache,
                  q=q_d, block_table=_table(ids_d), seq_lens=decode_lens.astype(np.int32),
                  q_prefill=q_p, block_table_prefill=_table(ids_p),
                  seq_lens_prefill=(prior_lens + chunk_lens).astype(np.int32), query_start_loc=qsl,
                  k_new=k_new, v_new=v_new, slot_mapping=slots)
    if keep_contiguous:
        wl.contiguous_k, wl.contiguous_v = ck_d, cv_d
        wl.contiguous_k_prefill, wl.contiguous_v_prefill = ck_p, cv_p
    wl.info["blocks_used"] = int(alloc.next + 1)
    wl.info["padding_tokens"] = int(T_pad - T)
    return wl


# --------------------------------------------------------------------------------------
# The five named workloads (seeds 1001 to 1005)
# --------------------------------------------------------------------------------------

def lognormal_lens(rng: np.random.Generator, n: int, mean: float = 195.0, sigma: float = 1.0,
                   lo: int = 16, hi: int = 2048) -> np.ndarray:
    """Lognormal lengths with the requested mean (mu = ln(mean) - sigma^2/2), clipped to [lo, hi].

    The n lengths sit at the stratified quantiles (i + 0.5) / n of the distribution and are
    then shuffled, so a batch of 64 has the stated mean instead of a +-30-token draw of it.
    """
    from statistics import NormalDist
    mu = np.log(mean) - 0.5 * sigma * sigma
    z = np.array([NormalDist().inv_cdf((i + 0.5) / n) for i in range(n)])
    x = np.exp(mu + sigma * z)
    return rng.permutation(np.clip(np.rint(x), lo, hi).astype(np.int64))


def tiny_fp32(seed: int = 1001, keep_contiguous: bool = True) -> Workload:
    """4 sequences, lengths {1, 15, 16, 33}, 4 q = 4 kv heads, D 64, 64-block pool, fp32."""
    return build_decode(seed, [1, 15, 16, 33], H_q=4, H_kv=4, D=64, num_blocks=64, dtype="f32",
                        keep_contiguous=keep_contiguous, name="tiny_fp32")


def gqa_decode(seed: int = 1002, S: int = 64, keep_contiguous: bool = False) -> Workload:
    """64 sequences, lognormal lengths (mean ~195, clipped 16..2048), 32 q / 8 kv heads,
    D 128, 4096-block pool, bf16; one new token per sequence written by reshape_and_cache."""
    rng = np.random.default_rng(seed)
    lens = lognormal_lens(rng, S)
    wl = build_decode(seed + 7919, lens, H_q=32, H_kv=8, D=128, num_blocks=4096, dtype="bf16",
                      keep_contiguous=keep_contiguous, name="gqa_decode_bs64")
    wl.info["mean_len"] = float(lens.mean())
    return wl


def prefix_sharing(seed: int = 1003, S: int = 128, keep_contiguous: bool = False) -> Workload:
    """128 sequences whose first 1024 tokens alias the same 64 physical blocks, plus a
    unique suffix of U{0..512} tokens; 32 q / 8 kv heads, D 128, 8192-block pool, bf16."""
    rng = np.random.default_rng(seed)
    lens = 1024 + rng.integers(0, 512, size=S, endpoint=True)
    return build_decode(seed + 7919, lens, H_q=32, H_kv=8, D=128, num_blocks=8192, dtype="bf16",
                        new_token=False, shared_prefix_tokens=1024, keep_contiguous=keep_contiguous,
                        name="prefix_sharing_bs128")


def long_split_kv(seed: int = 1004, S: int = 8, L: int = 32768) -> Workload:
    """8 sequences of 32768 tokens, 64 q / 8 kv heads, D 128, 20000-block pool, bf16."""
    return build_decode(seed, [L] * S, H_q=64, H_kv=8, D=128, num_blocks=20000, dtype="bf16",
                        name="long_split_kv")


def mixed_step(seed: int = 1005, n_prefill: int = 16, chunk: int = 512, n_decode: int = 240,
               num_blocks: int = 40000) -> Workload:
    """16 chunked-prefill sequences (512 new tokens on prior context U{0..4096}) plus 240
    decode sequences (context U{64..4096}); 32 q / 8 kv heads, D 128, bf16; new-token slots
    padded to a multiple of 256 with padding slots in the null block."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(0, 4096, size=n_prefill, endpoint=True)
    dec = rng.integers(64, 4096, size=n_decode, endpoint=True)
    need = int(np.sum(-(-(prior + chunk) // BLOCK)) + np.sum(-(-dec // BLOCK))) + 1
    nb = max(num_blocks, need)
    return build_mixed(seed + 7919, prior, np.full(n_prefill, chunk), dec, H_q=32, H_kv=8, D=128,
                       num_blocks=nb, dtype="bf16", name="mixed_step")


WORKLOADS = {"tiny_fp32": tiny_fp32, "gqa_decode": gqa_decode, "prefix_sharing": prefix_sharing,
             "long_split_kv": long_split_kv, "mixed_step": mixed_step}
