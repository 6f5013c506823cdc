"""Pins for the block-manager reference model (oracle/block_pool.py) against what the pages
state about vLLM's block pool, block hashes and copy-on-write, plus closed forms."""
import hashlib

import numpy as np
import pytest

from oracle import block_pool as BP

BLOCK = BP.BLOCK


def toks(n, base=0):
    return [base + i for i in range(n)]


def test_null_block_is_burned_at_construction():
    # "vLLM: what PagedAttention turned into", block pool: the first block of the free queue
    # becomes the null block and is never handed out
    p = BP.BlockPool(8)
    assert p.null == 0 and p.num_free() == 7
    p.add_request(1, toks(7 * BLOCK))
    assert 0 not in p.block_ids(1) and p.num_free() == 0
    with pytest.raises(MemoryError):
        p.add_request(2, toks(1))


def test_fresh_pool_hands_out_blocks_in_queue_order():
    p = BP.BlockPool(10)
    p.add_request(1, toks(3 * BLOCK))
    assert p.block_ids(1) == [1, 2, 3]
    assert p.slot_mapping(1, 15, 3) == [1 * 16 + 15, 2 * 16 + 0, 2 * 16 + 1]


def test_unhashed_blocks_are_reused_first_lifo():
    # blocks without a hash go to the front of the free queue
    p = BP.BlockPool(10)
    p.add_request(1, toks(3 * BLOCK))      # blocks 1 2 3, never committed: no hashes
    p.free_request(1)                      # freed tail first: 3, 2, 1 each pushed to the front
    assert p.queue[:3] == [1, 2, 3]
    p.add_request(2, toks(BLOCK, 1000))
    assert p.block_ids(2) == [1]


def test_hashed_blocks_go_to_the_back_tail_first():
    # blocks with a hash go to the back; a request's last block is offered for eviction first
    p = BP.BlockPool(10)
    p.add_request(1, toks(3 * BLOCK + 1))  # blocks 1 2 3 4
    p.commit(1, 3 * BLOCK + 1)             # blocks 1 2 3 full and hashed, 4 partial
    p.free_request(1)
    assert p.queue[0] == 4                 # unhashed partial block: front
    assert p.queue[-3:] == [3, 2, 1]       # hashed: back, tail first


def test_freed_blocks_keep_their_hash_until_taken():
    # eviction is lazy: a freed, cached prefix is still a hit
    p = BP.BlockPool(12)
    prompt = toks(2 * BLOCK + 5)
    p.add_request(1, prompt)
    p.commit(1, len(prompt))
    p.free_request(1)
    assert p.add_request(2, prompt) == 2 * BLOCK
    assert p.block_ids(2)[:2] == [1, 2]
    p.free_request(2)
    # take every block in queue order: the cached ones (at the back) are evicted last
    n = p.num_free()
    p.add_request(3, toks(n * BLOCK, 5000))
    assert p.cache == {}
    p.free_request(3)
    assert p.add_request(4, prompt) == 0


def test_prefix_lookup_stops_at_first_miss_because_hashes_chain():
    p = BP.BlockPool(20)
    a = toks(4 * BLOCK + 1)
    p.add_request(1, a)
    p.commit(1, len(a))
    b = list(a)
    b[0] = -7                               # first block differs: every later block misses too
    assert p.add_request(2, b) == 0
    c = list(a)
    c[2 * BLOCK + 3] = -7                   # third block differs: two hits
    assert p.add_request(3, c) == 2 * BLOCK


def test_same_tokens_after_different_prefix_hash_differently():
    r = BP.none_hash("s")
    blk = toks(BLOCK, 100)
    h1 = BP.block_hash(BP.block_hash(r, toks(BLOCK, 0), b""), blk, b"")
    h2 = BP.block_hash(BP.block_hash(r, toks(BLOCK, 1), b""), blk, b"")
    assert h1 != h2


def test_salt_isolates_tenants_and_only_enters_the_first_block():
    p = BP.BlockPool(20)
    prompt = toks(3 * BLOCK + 1)
    p.add_request(1, prompt, salt=b"tenant-a")
    p.commit(1, len(prompt))
    assert p.add_request(2, prompt, salt=b"tenant-b") == 0
    assert p.add_request(3, prompt, salt=b"tenant-a") == 3 * BLOCK
    r = BP.none_hash("paged-kv-none-hash")
    h0 = BP.block_hash(r, prompt[:BLOCK], b"tenant-a")
    h1 = BP.block_hash(h0, prompt[BLOCK:2 * BLOCK], b"")
    assert p.reqs[1].hashes[:2] == [h0, h1]


def test_hash_is_sha256_of_parent_tokens_extra_and_key_appends_group():
    parent = bytes(range(32))
    t = toks(BLOCK, 3)
    want = hashlib.sha256(parent + np.array(t, dtype="<i4").tobytes() + b"x").digest()
    assert BP.block_hash(parent, t, b"x") == want
    assert BP.hash_key(want, 5) == want + b"\x00\x00\x00\x05"


def test_a_prompt_never_hits_in_full():
    p = BP.BlockPool(20)
    prompt = toks(2 * BLOCK)
    p.add_request(1, prompt)
    p.commit(1, len(prompt))
    assert p.add_request(2, prompt) == BLOCK   # at most (len - 1) // 16 blocks from the cache


def test_fork_shares_blocks_and_append_copies_the_shared_partial_block():
    p = BP.BlockPool(20)
    p.add_request(1, toks(BLOCK + 5))      # blocks 1 2, block 2 partial
    free0 = p.num_free()
    p.fork(1, 2)
    assert p.block_ids(2) == p.block_ids(1) and p.num_free() == free0
    p.append_tokens(2, [77])
    assert p.take_copies() == [(2, 3)]
    assert p.block_ids(2) == [1, 3] and p.block_ids(1) == [1, 2]
    p.append_tokens(1, [78])                # block 2 is now private to request 1: no copy
    assert p.take_copies() == []
    p.free_request(1)
    assert p.blocks[1].ref == 1             # still held by the child
    p.free_request(2)
    assert p.num_free() == 19


def test_pool_sizing_closed_form():
    # utilisation x free memory / (layers x K and V x heads x 16 x head_dim x elem)
    n = BP.num_blocks_for_memory(100 * 2**30, 0.92, 32, 8, 128, 2)
    assert n == int(int(100 * 2**30 * 0.92) // (32 * 2 * 8 * 16 * 128 * 2))


def test_copy_blocks_copies_both_pools():
    rng = np.random.default_rng(0)
    k = rng.standard_normal((6, 2, BLOCK, 8)).astype(np.float32)
    v = rng.standard_normal((6, 2, BLOCK, 8)).astype(np.float32)
    k0, v0 = k.copy(), v.copy()
    BP.copy_blocks(k, v, [(1, 4), (2, 5)])
    assert np.array_equal(k[4], k0[1]) and np.array_equal(v[5], v0[2])
    assert np.array_equal(k[:4], k0[:4])


def test_larger_blocks_hash_all_their_tokens_and_cap_hits_by_block():
    # "vLLM: what PagedAttention turned into": blocks of 16 to 128 tokens; a block hash covers
    # the whole block, slots are block * size + offset, and a prompt never hits in full
    bs = 32
    p = BP.BlockPool(12, block_size=bs)
    prompt = toks(2 * bs)
    p.add_request(1, prompt)
    assert p.block_ids(1) == [1, 2]
    assert p.slot_mapping(1, bs - 1, 2) == [1 * bs + bs - 1, 2 * bs]
    p.commit(1, len(prompt))
    r = BP.none_hash("paged-kv-none-hash")
    want = hashlib.sha256(r + np.array(prompt[:bs], dtype="<i4").tobytes()).digest()
    assert p.reqs[1].hashes[0] == want
    assert p.add_request(2, prompt) == bs            # (2 bs - 1) // bs = 1 block from the cache
    assert p.add_request(3, toks(2 * bs + 1)) == 2 * bs


def test_pool_sizing_scales_with_block_size():
    n16 = BP.num_blocks_for_memory(2**34, 0.9, 4, 8, 128, 2)
    n64 = BP.num_blocks_for_memory(2**34, 0.9, 4, 8, 128, 2, block_size=64)
    assert n64 == int(int(2**34 * 0.9) // (4 * 2 * 8 * 64 * 128 * 2)) and n16 // 4 - 1 <= n64 <= n16 // 4
