"""GPU parity of copy_blocks (bit-exact against the reference copy) and of a full
parallel-sampling flow driven by the library's block manager: prompt K/V written through
reshape_and_cache, a fork, copy-on-write of the shared partial block, one new token per
branch, decode of both branches against the fp64 oracle on the same pool."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from oracle import block_pool as BP  # noqa: E402
from paged_kv_cache_238_gb300 import binding as B  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402

from helpers import assert_close, to_dev, to_f64, to_host_bits  # noqa: E402

pytestmark = pytest.mark.gpu


def _pool(rng, nb, H, D, dtype, bs=16):
    shape = (nb, H, bs, D)
    x = rng.standard_normal(shape).astype(np.float32)
    y = rng.standard_normal(shape).astype(np.float32)
    if dtype == "bf16":
        return W.f32_to_bf16_bits(x), W.f32_to_bf16_bits(y)
    return x, y


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 64)])
def test_copy_blocks_bit_exact(dtype, D):
    rng = np.random.default_rng(11)
    k, v = _pool(rng, 40, 4, D, dtype)
    pairs = np.array([[3, 17], [5, 5], [21, 2], [39, 0]], dtype=np.int32)  # incl. src == dst
    kd, vd = to_dev(k), to_dev(v)
    B.pa_get_device_errors(clear=True)
    B.pa_copy_blocks(kd, vd, to_dev(pairs))
    torch.cuda.synchronize()
    BP.copy_blocks(k, v, [tuple(p) for p in pairs])
    assert np.array_equal(to_host_bits(kd), k) and np.array_equal(to_host_bits(vd), v)
    assert B.pa_get_device_errors(clear=True) == 0


def test_copy_blocks_out_of_range_pair_is_skipped_and_flagged():
    rng = np.random.default_rng(12)
    k, v = _pool(rng, 8, 2, 64, "bf16")
    kd, vd = to_dev(k), to_dev(v)
    B.pa_get_device_errors(clear=True)
    B.pa_copy_blocks(kd, vd, to_dev(np.array([[1, 8], [2, 3]], dtype=np.int32)))
    torch.cuda.synchronize()
    k[3], v[3] = k[2], v[2]
    assert np.array_equal(to_host_bits(kd), k) and np.array_equal(to_host_bits(vd), v)
    assert B.pa_get_device_errors(clear=True) == B.PA_DEVERR_BLOCK_RANGE


@pytest.mark.parametrize("prompt_len,bs", [(37, 16), (48, 16), (100, 64), (128, 64), (70, 32)])
def test_fork_copy_on_write_decode_matches_oracle(prompt_len, bs):
    rng = np.random.default_rng(100 + prompt_len)
    NB, Hq, Hkv, D = 32, 8, 2, 128
    scale = 1.0 / np.sqrt(D)
    k_pool, v_pool = _pool(rng, NB, Hkv, D, "bf16", bs)  # unowned cells hold arbitrary values
    bm = B.BlockManager(NB, block_size=bs)
    kd, vd = to_dev(k_pool), to_dev(v_pool)

    def new_kv(n):
        return (W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D)).astype(np.float32)),
                W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D)).astype(np.float32)))

    def write(k_new, v_new, slots):
        B.pa_reshape_and_cache(to_dev(k_new), to_dev(v_new), kd, vd, to_dev(np.array(slots, dtype=np.int64)))
        oracle.reshape_and_cache(k_new, v_new, k_pool, v_pool, np.array(slots, dtype=np.int64))

    prompt = list(range(prompt_len))
    assert bm.add_request(1, prompt) == 0
    kp, vp = new_kv(prompt_len)
    write(kp, vp, bm.slot_mapping(1, 0, prompt_len))
    bm.commit(1, prompt_len)
    bm.fork(1, 2)
    for rid, tok in ((1, 1000), (2, 2000)):  # one sampled token per branch
        bm.append_tokens(rid, [tok])
    copies = bm.take_copies()
    if prompt_len % bs:
        assert len(copies) == 1  # the shared partial block was copied for the second branch
    if copies:
        pairs = np.array(copies, dtype=np.int32)
        B.pa_copy_blocks(kd, vd, to_dev(pairs))
        BP.copy_blocks(k_pool, v_pool, copies)
    kn, vn = new_kv(2)
    slots = [bm.slot_mapping(1, prompt_len, 1)[0], bm.slot_mapping(2, prompt_len, 1)[0]]
    assert slots[0] != slots[1]
    write(kn, vn, slots)
    max_blocks = 4
    bt = np.array([bm.block_ids(1, max_blocks), bm.block_ids(2, max_blocks)], dtype=np.int32)
    lens = np.array([prompt_len + 1] * 2, dtype=np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((2, Hq, D)).astype(np.float32))
    out = torch.empty((2, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(max(16, B.pa_decode_workspace_size(2, Hq, Hkv, D, prompt_len + 1, torch.bfloat16)),
                     dtype=torch.uint8, device="cuda")
    B.pa_decode(out, to_dev(q), kd, vd, to_dev(bt), to_dev(lens), prompt_len + 1, scale, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(kd)[1:], k_pool[1:])  # device pool == reference pool
    ref = oracle.attention(q, k_pool, v_pool, bt, lens, scale)
    assert_close(to_f64(out), ref, "bf16", "decode after fork + copy-on-write")
    # the two branches share the prompt but end differently
    assert not np.allclose(ref[0], ref[1])
    assert B.pa_get_device_errors(clear=True) == 0
