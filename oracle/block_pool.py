"""Reference model of the paged-KV block manager: plain Python, obviously correct, slow.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import or call this module; only
the tests do. It shares no code with the C++ block manager in the library.

What it models (the pages on vLLM's paged KV cache):
  * A pool of fixed-size physical blocks (16 tokens by default; "vLLM: what PagedAttention
    turned into" reports 16 to 128 performing alike, so 32, 64 and 128 are variants); a
    request reaches its blocks through a block list, and a slot is physical_block * size + offset ("My Understanding of vLLM and
    PagedAttention", "Logical Blocks", "Physical Blocks", "Block Table"; "vLLM: what
    PagedAttention turned into", "The problem PagedAttention was actually solving").
  * The null block: the first block of the free queue is taken at construction and never
    handed out, so "no block" is an ordinary id ("vLLM: what PagedAttention turned into",
    "The block pool, and the two tricks in it").
  * The free queue: one doubly linked eviction-ordered queue; a freed block without a hash
    goes to the front (reused first, LIFO), a freed block with a hash to the back (evicted
    last, FIFO); a request's blocks are freed tail first (same section).
  * Freed blocks keep their hash and stay findable; eviction happens lazily when the block
    is taken for new content (same section).
  * A block hash is the hash of (parent hash, the block's tokens, extra keys), chained from a
    fixed seed hash, SHA-256, with the group id appended to form the key; a per-request salt
    is folded in on the first block only ("What a block hash actually is"; "The environment
    variable that shouldn't have to exist").
  * Prefix lookup takes the longest run of cached full blocks from the start and stops at the
    first miss (same section).
  * Shared blocks are reference counted; a forked request (parallel sampling) shares every
    block, and appending into a shared, partly filled last block first copies it into a
    private block (copy-on-write) ("vLLM Internals", section 1.2; "vLLM: what PagedAttention
    turned into", "What a block hash actually is", last paragraph).
  * Pool sizing: a utilisation fraction of the free device memory divided by the per-block
    cost over all layers ("vLLM: what PagedAttention turned into", "Checking the 96.3%").

Readings where the pages are silent (the C++ manager follows the same ones):
  * Hash input: parent hash (32 bytes) || the block's token ids as int32 little-endian ||
    extra key bytes (the salt, first block only); the seed hash is SHA-256 of the seed string;
    the key is hash || group id (4 bytes, big-endian), group 0.
  * Within one free call the blocks are processed in the given order: each unhashed block is
    pushed to the front (so the last one pushed is reused first), each hashed block appended
    to the back.
  * A prompt never hits in full: at most (len - 1) // size blocks come from the cache, so at
    least one token is computed.
  * A full block is hashed and entered into the cache when the caller commits that its K/V has
    been computed; a hash already in the cache keeps its existing block and the new block
    stays unhashed.
  * Appending needs a new block only when the last block is full; a shared last block that
    is partly filled is first copied (copy-on-write).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

BLOCK = 16


def sha256(data: bytes) -> bytes:
    return hashlib.sha256(data).digest()


def none_hash(seed: str) -> bytes:
    return sha256(seed.encode())


def block_hash(parent: bytes, tokens: List[int], extra: bytes) -> bytes:
    """Hash of one full block: its tokens are all of the block (len(tokens) = block size)."""
    body = b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)
    return sha256(parent + body + extra)


def hash_key(h: bytes, group_id: int = 0) -> bytes:
    return h + group_id.to_bytes(4, "big", signed=False)


@dataclass
class Block:
    id: int
    ref: int = 0
    key: Optional[bytes] = None


@dataclass
class Request:
    tokens: List[int]
    blocks: List[int]
    salt: bytes
    computed: int = 0
    hashes: List[bytes] = field(default_factory=list)  # chained hashes of its full blocks


class BlockPool:
    def __init__(self, num_blocks: int, enable_caching: bool = True, seed: str = "paged-kv-none-hash",
                 block_size: int = BLOCK):
        assert num_blocks >= 2 and block_size > 0
        self.bs = block_size
        self.blocks = [Block(i) for i in range(num_blocks)]
        self.queue: List[int] = list(range(num_blocks))  # front = index 0
        self.null = self.queue.pop(0)
        self.caching = enable_caching
        self.cache: Dict[bytes, List[int]] = {}  # key -> blocks holding it, oldest first
        self.root = none_hash(seed)
        self.reqs: Dict[int, Request] = {}
        self.copies: List[Tuple[int, int]] = []

    # ---- pool ---------------------------------------------------------------------------
    def num_free(self) -> int:
        return len(self.queue)

    def _take(self, n: int) -> List[int]:
        if n > len(self.queue):
            raise MemoryError("out of blocks")
        out = []
        for _ in range(n):
            b = self.blocks[self.queue.pop(0)]
            if b.key is not None:  # lazy eviction
                lst = self.cache[b.key]
                lst.remove(b.id)
                if not lst:
                    del self.cache[b.key]
                b.key = None
            b.ref = 1
            out.append(b.id)
        return out

    def _touch(self, ids: List[int]) -> None:
        for i in ids:
            b = self.blocks[i]
            if b.ref == 0:
                self.queue.remove(i)
            b.ref += 1

    def _free(self, ids: List[int]) -> None:
        for i in ids:
            if i == self.null:
                continue
            b = self.blocks[i]
            b.ref -= 1
            assert b.ref >= 0
            if b.ref == 0:
                if b.key is None or not self.caching:
                    self.queue.insert(0, i)
                else:
                    self.queue.append(i)

    # ---- requests -----------------------------------------------------------------------
    def _hashes(self, tokens: List[int], salt: bytes, upto_blocks: int, prev: List[bytes]) -> List[bytes]:
        hs = list(prev)
        parent = hs[-1] if hs else self.root
        for k in range(len(hs), upto_blocks):
            extra = salt if k == 0 else b""
            parent = block_hash(parent, tokens[k * self.bs:(k + 1) * self.bs], extra)
            hs.append(parent)
        return hs

    def add_request(self, rid: int, tokens: List[int], salt: bytes = b"") -> int:
        assert rid not in self.reqs and len(tokens) > 0
        bs = self.bs
        n_full = len(tokens) // bs
        hs = self._hashes(tokens, salt, n_full, [])
        hits: List[int] = []
        if self.caching:
            for k in range(min(n_full, (len(tokens) - 1) // bs)):
                lst = self.cache.get(hash_key(hs[k]))
                if not lst:
                    break
                hits.append(lst[0])
        need = -(-len(tokens) // bs) - len(hits)
        if need > len(self.queue) - sum(1 for i in hits if self.blocks[i].ref == 0):
            raise MemoryError("out of blocks")
        self._touch(hits)
        new = self._take(need)
        r = Request(list(tokens), hits + new, salt, computed=len(hits) * bs, hashes=hs[:len(hits)])
        self.reqs[rid] = r
        return r.computed

    def append_tokens(self, rid: int, tokens: List[int]) -> None:
        r = self.reqs[rid]
        pos0 = len(r.tokens)
        bs = self.bs
        need = sum(1 for p in range(pos0, pos0 + len(tokens)) if p % bs == 0)
        cow = len(tokens) > 0 and pos0 % bs != 0 and self.blocks[r.blocks[-1]].ref > 1
        if need + int(cow) > len(self.queue):
            raise MemoryError("out of blocks")  # nothing changed
        for t in tokens:
            pos = len(r.tokens)
            if pos % bs == 0:
                r.blocks += self._take(1)
            else:
                last = self.blocks[r.blocks[-1]]
                if last.ref > 1:  # shared, partly filled: copy on write
                    (dst,) = self._take(1)
                    self.copies.append((last.id, dst))
                    self._free([last.id])
                    r.blocks[-1] = dst
            r.tokens.append(t)

    def commit(self, rid: int, num_computed: int) -> None:
        r = self.reqs[rid]
        assert num_computed <= len(r.tokens)
        r.computed = max(r.computed, num_computed)
        n_full = r.computed // self.bs
        r.hashes = self._hashes(r.tokens, r.salt, n_full, r.hashes)
        if not self.caching:
            return
        for k in range(n_full):
            b = self.blocks[r.blocks[k]]
            key = hash_key(r.hashes[k])
            if b.key is not None:
                continue
            if key in self.cache:
                continue  # another block already holds this content
            b.key = key
            self.cache[key] = [b.id]

    def fork(self, parent: int, child: int) -> None:
        p = self.reqs[parent]
        assert child not in self.reqs
        self._touch(list(p.blocks))
        self.reqs[child] = Request(list(p.tokens), list(p.blocks), p.salt, p.computed, list(p.hashes))

    def free_request(self, rid: int) -> None:
        r = self.reqs.pop(rid)
        self._free(list(reversed(r.blocks)))

    # ---- views --------------------------------------------------------------------------
    def block_ids(self, rid: int) -> List[int]:
        return list(self.reqs[rid].blocks)

    def slot_mapping(self, rid: int, first: int, n: int) -> List[int]:
        r = self.reqs[rid]
        bs = self.bs
        return [r.blocks[p // bs] * bs + p % bs for p in range(first, first + n)]

    def take_copies(self) -> List[Tuple[int, int]]:
        c, self.copies = self.copies, []
        return c


def num_blocks_for_memory(free_bytes: int, utilization: float, num_layers: int, num_kv_heads: int,
                          head_dim: int, elem_bytes: int, block_size: int = BLOCK) -> int:
    per_block = num_layers * 2 * num_kv_heads * block_size * head_dim * elem_bytes
    return int(int(free_bytes * utilization) // per_block)


def copy_blocks(k_cache, v_cache, pairs) -> None:
    """Copy each (src, dst) block of both pools, every kv head (numpy arrays [NB, H, BS, D])."""
    for s, d in pairs:
        k_cache[d] = k_cache[s]
        v_cache[d] = v_cache[s]
