"""The library's C++ block manager (pa_bm_*) against the reference model (oracle/block_pool.py)
on seeded random request traffic, and its SHA-256 against hashlib. CPU only: no device calls."""
import hashlib
import os
import random
import shutil

import pytest

from oracle import block_pool as BP
from paged_kv_cache_238_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    os.path.join(ROOT, "paged_kv_cache_238_gb300", "libpa.so")), reason="needs nvcc to build libpa")


@pytest.mark.parametrize("n", [0, 1, 3, 55, 56, 63, 64, 65, 119, 1000])
def test_sha256_matches_hashlib(n):
    data = bytes((i * 37 + 11) % 256 for i in range(n))
    assert B.pa_sha256(data) == hashlib.sha256(data).digest()


def _state(ref: BP.BlockPool, bm: B.BlockManager):
    assert bm.num_free() == ref.num_free()
    assert bm.free_queue() == ref.queue
    for rid in ref.reqs:
        assert bm.block_ids(rid) == ref.block_ids(rid), rid
    for b in ref.blocks:
        if b.id == ref.null:
            continue
        cnt, h = bm.block_info(b.id)
        assert cnt == b.ref, b.id
        assert h == (None if b.key is None else b.key[:32]), b.id


def _run(seed: int, num_blocks: int, caching: bool, steps: int, block_size: int = 16):
    rng = random.Random(seed)
    ref = BP.BlockPool(num_blocks, enable_caching=caching, seed="s%d" % seed, block_size=block_size)
    bm = B.BlockManager(num_blocks, enable_caching=caching, hash_seed="s%d" % seed, block_size=block_size)
    scale = block_size // 16  # prompts and appends grow with the block size
    prefixes = [[rng.randrange(50) for _ in range(rng.randrange(1, 70 * scale))] for _ in range(4)]
    salts = [b"", b"", b"tenant-a", b"tenant-b"]
    next_id = 1
    for _ in range(steps):
        live = sorted(ref.reqs)
        op = rng.random()
        if op < 0.3 or not live:
            prompt = list(rng.choice(prefixes)) + [rng.randrange(50) for _ in range(rng.randrange(0, 40 * scale))]
            salt = rng.choice(salts)
            try:
                want = ref.add_request(next_id, prompt, salt)
            except MemoryError:
                with pytest.raises(B.PaError) as e:
                    bm.add_request(next_id, prompt, salt)
                assert e.value.status == B.PA_ERR_NO_SPACE
            else:
                assert bm.add_request(next_id, prompt, salt) == want
            next_id += 1
        elif op < 0.55:
            rid = rng.choice(live)
            toks = [rng.randrange(50) for _ in range(rng.randrange(1, 20 * scale))]
            try:
                ref.append_tokens(rid, toks)
            except MemoryError:
                with pytest.raises(B.PaError) as e:
                    bm.append_tokens(rid, toks)
                assert e.value.status == B.PA_ERR_NO_SPACE
            else:
                bm.append_tokens(rid, toks)
        elif op < 0.75:
            rid = rng.choice(live)
            n = rng.randrange(0, len(ref.reqs[rid].tokens) + 1)
            ref.commit(rid, n)
            bm.commit(rid, n)
        elif op < 0.85:
            rid = rng.choice(live)
            ref.fork(rid, next_id)
            bm.fork(rid, next_id)
            next_id += 1
        else:
            rid = rng.choice(live)
            ref.free_request(rid)
            bm.free_request(rid)
        assert bm.take_copies() == ref.take_copies()
        _state(ref, bm)
    for rid in sorted(ref.reqs):
        n = len(ref.reqs[rid].tokens)
        assert bm.slot_mapping(rid, 0, n) == ref.slot_mapping(rid, 0, n)


@pytest.mark.parametrize("seed", range(6))
def test_block_manager_matches_reference_model(seed):
    _run(seed, num_blocks=24 if seed % 2 else 64, caching=seed != 5, steps=400)


@pytest.mark.parametrize("block_size,seed", [(32, 10), (64, 11), (128, 12), (32, 13)])
def test_block_manager_matches_reference_model_larger_blocks(block_size, seed):
    _run(seed, num_blocks=24 if seed % 2 else 48, caching=seed != 13, steps=300, block_size=block_size)


def test_block_size_is_checked():
    with pytest.raises(B.PaError) as e:
        B.BlockManager(8, block_size=48)
    assert e.value.status == B.PA_ERR_UNSUPPORTED
    bm = B.BlockManager(8, block_size=64)
    assert bm.add_request(1, list(range(65))) == 0
    assert bm.block_ids(1) == [1, 2]
    assert bm.slot_mapping(1, 63, 2) == [1 * 64 + 63, 2 * 64]


def test_sha256_round_constants_are_the_cube_roots_of_the_first_primes():
    """FIPS 180-4: the 64 round constants are the first 32 bits of the fractional parts of
    the cube roots of the first 64 primes; the initial hash values likewise from the square
    roots of the first 8. Derived here with exact integer roots and compared with the table in
    the C++ source."""
    import re
    src = open(os.path.join(ROOT, "paged_kv_cache_238_gb300", "csrc", "block_manager.cpp")).read()
    table = [int(x, 16) for x in re.findall(r"0x([0-9a-f]{8})u", src)]
    primes = [p for p in range(2, 400) if all(p % d for d in range(2, int(p ** 0.5) + 1))]

    def frac_bits(p, k):  # floor(frac(p^(1/k)) * 2^32) via the integer k-th root of p * 2^(32k)
        x = p << (32 * k)
        r = int(round(x ** (1.0 / k)))
        while r ** k > x:
            r -= 1
        while (r + 1) ** k <= x:
            r += 1
        return r & 0xFFFFFFFF

    cube = [frac_bits(p, 3) for p in primes[:64]]
    square = [frac_bits(p, 2) for p in primes[:8]]
    i = table.index(cube[0])
    assert table[i:i + 64] == cube
    j = table.index(square[0])
    assert table[j:j + 8] == square


def test_bad_calls_change_nothing():
    bm = B.BlockManager(8)
    bm.add_request(1, list(range(20)))
    with pytest.raises(B.PaError):
        bm.add_request(1, [1])                  # known id
    with pytest.raises(B.PaError):
        bm.free_request(99)                     # unknown id
    with pytest.raises(B.PaError):
        bm.slot_mapping(1, 30, 5)               # beyond the request's blocks
    with pytest.raises(B.PaError) as e:
        bm.add_request(2, list(range(16 * 7)))  # more than the free blocks
    assert e.value.status == B.PA_ERR_NO_SPACE
    assert bm.num_free() == 5 and bm.block_ids(1) == [1, 2]


def test_pool_sizing_matches_reference():
    for args in [(80 * 2**30, 0.92, 32, 8, 128), (2**30, 0.5, 1, 4, 64)]:
        assert B.pa_bm_num_blocks_for_memory(*args, B.PA_BF16) == BP.num_blocks_for_memory(*args, 2)
        assert B.pa_bm_num_blocks_for_memory(*args, B.PA_F32) == BP.num_blocks_for_memory(*args, 4)
        for bs in (32, 128):
            assert (B.pa_bm_num_blocks_for_memory(*args, B.PA_BF16, block_size=bs) ==
                    BP.num_blocks_for_memory(*args, 2, block_size=bs))
    assert B.pa_bm_num_blocks_for_memory(1 << 30, 1.5, 1, 1, 64, B.PA_BF16) == -1
