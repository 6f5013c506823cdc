"""Pins for the fp64 oracle: every check compares it with something other than itself.

* brute-force attention on contiguous K/V that never goes through the pool;
* torch's scaled_dot_product_attention (CPU, fp64) with an explicit causal mask;
* closed forms (one key, constant V, zero query, a hand-solved softmax);
* invariants the pages fix: physical placement is arbitrary ("vLLM Internals",
  section 1.1), identical prefixes share blocks ("vLLM Internals", section 1.2),
  the null block is an ordinary id ("vLLM: what PagedAttention turned into",
  "The block pool"), waste is at most 15 tokens per sequence (section 1.2);
* the page's worked block-table example ("My Understanding of vLLM and
  PagedAttention", "Logical Blocks" / "Physical Blocks" / "Block Table").
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_238_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _full_pool(wl):
    """Pool with the new tokens written (oracle scatter), as the kernels will see it."""
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    if wl.slot_mapping is not None:
        oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    return kc, vc


def brute_decode(q, ks, vs, scale, H_kv):
    """Contiguous attention, one query per sequence at its last key (numpy fp64)."""
    S, H_q, D = q.shape
    G = H_q // H_kv
    out = np.zeros((S, H_q, D))
    for i in range(S):
        K, V = W.as_f64(ks[i]), W.as_f64(vs[i])        # [L, H_kv, D]
        if K.shape[0] == 0:
            continue
        for h in range(H_q):
            z = scale * K[:, h // G, :] @ W.as_f64(q[i, h])
            p = np.exp(z - z.max())
            out[i, h] = (p / p.sum()) @ V[:, h // G, :]
    return out


# ----------------------------------------------------------------------------- reshape_and_cache

def test_reshape_roundtrip_and_untouched_cells():
    rng = np.random.default_rng(1)
    NB, H, D, T = 9, 3, 8, 40
    kc = rng.standard_normal((NB, H, 16, D)).astype(np.float32)
    vc = rng.standard_normal((NB, H, 16, D)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    k = rng.standard_normal((T, H, D)).astype(np.float32)
    v = rng.standard_normal((T, H, D)).astype(np.float32)
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int64)
    slots[5] = -1                                   # skipped
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    written = np.zeros((NB, 16), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), 16)
        written[b, o] = True
        assert np.array_equal(kc[b, :, o, :].view(np.uint32), k[t].view(np.uint32))
        assert np.array_equal(vc[b, :, o, :].view(np.uint32), v[t].view(np.uint32))
    for b in range(NB):
        for o in range(16):
            if not written[b, o]:
                assert np.array_equal(kc[b, :, o].view(np.uint32), k0[b, :, o].view(np.uint32))
                assert np.array_equal(vc[b, :, o].view(np.uint32), v0[b, :, o].view(np.uint32))


def test_reshape_bf16_bitwise_including_nan_payloads():
    rng = np.random.default_rng(2)
    NB, H, D, T = 4, 2, 16, 20
    kc = np.zeros((NB, H, 16, D), np.uint16)
    vc = np.zeros_like(kc)
    k = rng.integers(0, 65536, size=(T, H, D), dtype=np.uint16)   # arbitrary bit patterns
    v = rng.integers(0, 65536, size=(T, H, D), dtype=np.uint16)
    slots = np.arange(T, dtype=np.int64) + 16
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    assert np.array_equal(kc[1:3].transpose(0, 2, 1, 3).reshape(32, H, D)[:T], k)
    assert np.array_equal(vc[1:3].transpose(0, 2, 1, 3).reshape(32, H, D)[:T], v)
    assert not kc[0].any() and not kc[3].any()


def test_reshape_rejects_slot_beyond_pool():
    kc = np.zeros((2, 1, 16, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(np.ones((1, 1, 4), np.float32), np.ones((1, 1, 4), np.float32),
                                 kc, kc.copy(), np.array([32], np.int64))


def test_page_block_table_example():
    """Page tokens 1-16 -> logical block 0, 17-32 -> logical block 1; logical 0/1/2 -> physical
    7/21/3. Writing a 40-token sequence through its slots must land token n (1-based) in
    physical block table[(n-1)//16] at offset (n-1)%16, and attention through that table must
    equal attention over the contiguous sequence."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_example.json")))
    table = g["logical_to_physical"]
    bs = g["tokens_per_block"]
    for ex in g["page_examples"]:
        first, last = ex["page_tokens"]
        assert (first - 1) // bs == ex["logical_block"] == (last - 1) // bs
    rng = np.random.default_rng(3)
    H, D, L, NB = 2, 8, 40, 24
    k = rng.standard_normal((L, H, D)).astype(np.float32)
    v = rng.standard_normal((L, H, D)).astype(np.float32)
    slots = np.array([table[p // bs] * bs + p % bs for p in range(L)], np.int64)
    kc = np.full((NB, H, 16, D), np.nan, np.float32)
    vc = kc.copy()
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    for n in range(1, L + 1):
        phys = table[(n - 1) // bs]
        assert np.array_equal(kc[phys, :, (n - 1) % bs], k[n - 1])
    # every block other than 7, 21, 3 is untouched (still NaN); block 3 holds 8 tokens
    for b in range(NB):
        if b not in table:
            assert np.isnan(kc[b]).all()
    assert np.isnan(kc[3, :, 8:]).all() and not np.isnan(kc[3, :, :8]).any()
    q = rng.standard_normal((1, H, D)).astype(np.float32)
    bt = np.array([table], np.int32)
    out = oracle.attention(q, kc, vc, bt, np.array([L], np.int32), 0.3)
    ref = brute_decode(q, [k], [v], 0.3, H)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- attention: brute force

@pytest.mark.parametrize("lens,H_q,H_kv,D,dtype", [
    ([1, 15, 16, 33], 4, 4, 64, "f32"),            # the tiny fp32 workload's lengths
    ([17, 31, 32, 100, 5], 8, 2, 16, "bf16"),       # GQA 4
    ([64, 3, 48], 8, 1, 8, "bf16"),                 # MQA
    ([200, 1], 6, 3, 32, "f32"),                    # GQA 2
])
def test_decode_matches_bruteforce(lens, H_q, H_kv, D, dtype):
    wl = W.build_decode(11, lens, H_q=H_q, H_kv=H_kv, D=D, num_blocks=64, dtype=dtype,
                        keep_contiguous=True)
    kc, vc = _full_pool(wl)
    out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    ref = brute_decode(wl.q, wl.contiguous_k, wl.contiguous_v, wl.scale, H_kv)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.isfinite(out).all()


def test_tiny_fp32_workload_matches_bruteforce():
    wl = W.tiny_fp32()
    kc, vc = _full_pool(wl)
    out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    ref = brute_decode(wl.q, wl.contiguous_k, wl.contiguous_v, wl.scale, wl.H_kv)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_zero_length_sequence_gives_zero_row():
    wl = W.build_decode(12, [5, 9], H_q=2, H_kv=1, D=8, num_blocks=8, dtype="f32", new_token=False)
    lens = wl.seq_lens.copy()
    lens[1] = 0
    out = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, lens, wl.scale)
    assert not out[1].any()


# ----------------------------------------------------------------------------- attention: library routine

def test_prefill_matches_torch_sdpa_with_bottom_right_causal_mask():
    torch = pytest.importorskip("torch")
    wl = W.build_mixed(13, prior_lens=[0, 7, 40], chunk_lens=[5, 16, 9], decode_lens=[3],
                       H_q=4, H_kv=2, D=16, num_blocks=64, dtype="bf16", pad_multiple=8,
                       keep_contiguous=True)
    kc, vc = _full_pool(wl)
    out = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill,
                           wl.scale, query_start_loc=wl.query_start_loc)
    qsl = wl.query_start_loc
    G = wl.H_q // wl.H_kv
    for i in range(len(wl.seq_lens_prefill)):
        L = int(wl.seq_lens_prefill[i])
        C = int(qsl[i + 1] - qsl[i])
        qi = torch.from_numpy(W.as_f64(wl.q_prefill[qsl[i]:qsl[i + 1]])).transpose(0, 1)   # [H_q, C, D]
        K = torch.from_numpy(W.as_f64(wl.contiguous_k_prefill[i])).transpose(0, 1)        # [H_kv, L, D]
        V = torch.from_numpy(W.as_f64(wl.contiguous_v_prefill[i])).transpose(0, 1)
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        rows = torch.arange(C).unsqueeze(1) + (L - C)
        mask = torch.arange(L).unsqueeze(0) <= rows                                       # [C, L]
        ref = torch.nn.functional.scaled_dot_product_attention(qi, K, V, attn_mask=mask, scale=wl.scale)
        np.testing.assert_allclose(out[qsl[i]:qsl[i + 1]], ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_last_row_equals_decode_and_first_row_of_fresh_chunk_is_v0():
    wl = W.build_mixed(14, prior_lens=[0, 33], chunk_lens=[7, 20], decode_lens=[2],
                       H_q=4, H_kv=2, D=8, num_blocks=32, dtype="f32", pad_multiple=0,
                       keep_contiguous=True)
    kc, vc = _full_pool(wl)
    qsl = wl.query_start_loc
    out = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill,
                           wl.scale, query_start_loc=qsl)
    last_rows = wl.q_prefill[qsl[1:] - 1]
    dec = oracle.attention(last_rows, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale)
    assert np.array_equal(out[qsl[1:] - 1], dec)
    # sequence 0 has no prior context: its first chunk row sees only key 0
    v0 = W.as_f64(wl.contiguous_v_prefill[0][0])
    G = wl.H_q // wl.H_kv
    for h in range(wl.H_q):
        assert np.array_equal(out[0, h], v0[h // G])


# ----------------------------------------------------------------------------- closed forms

def test_single_key_returns_v0_exactly():
    wl = W.build_decode(15, [1, 1, 1], H_q=4, H_kv=2, D=16, num_blocks=8, dtype="bf16")
    kc, vc = _full_pool(wl)
    out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    for i in range(3):
        for h in range(4):
            assert np.array_equal(out[i, h], W.as_f64(wl.v_new[i, h // 2]))


def test_constant_v_and_zero_query_closed_forms():
    wl = W.build_decode(16, [37, 16, 50], H_q=2, H_kv=2, D=8, num_blocks=16, dtype="f32",
                        new_token=False, keep_contiguous=True)
    vc = wl.v_cache.copy()
    used = wl.block_table[wl.block_table > 0]
    vc[used] = 0.625                     # every visible value is 0.625 -> output 0.625
    out = oracle.attention(wl.q, wl.k_cache, vc, wl.block_table, wl.seq_lens, wl.scale)
    np.testing.assert_allclose(out, 0.625, rtol=0, atol=1e-15)
    q0 = np.zeros_like(wl.q)             # uniform weights -> mean of V over visible keys
    out = oracle.attention(q0, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    for i in range(3):
        np.testing.assert_allclose(out[i], W.as_f64(wl.contiguous_v[i]).mean(axis=0), rtol=1e-13, atol=1e-14)
    kc = wl.k_cache.copy()               # all keys equal -> also the mean of V
    kc[used] = 1.5
    out = oracle.attention(wl.q, kc, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    for i in range(3):
        np.testing.assert_allclose(out[i], W.as_f64(wl.contiguous_v[i]).mean(axis=0), rtol=1e-13, atol=1e-14)


def test_hand_solved_softmax():
    """Two keys, q.k = ln 3 and 0 -> weights 3/4 and 1/4; V rows (4, 0) and (0, 8) -> (3, 2)."""
    kc = np.full((2, 1, 16, 2), np.nan, np.float64).astype(np.float32)
    vc = kc.copy()
    kc[1, 0, 0] = [1.0, 0.0]
    kc[1, 0, 1] = [0.0, 0.0]
    vc[1, 0, 0] = [4.0, 0.0]
    vc[1, 0, 1] = [0.0, 8.0]
    q = np.array([[[math.log(3.0), 0.0]]], np.float32)
    out = oracle.attention(q, kc, vc, np.array([[1]], np.int32), np.array([2], np.int32), 1.0)
    # q was rounded to fp32: the exact weights follow from the stored value
    w = 1.0 / (1.0 + math.exp(-float(np.float32(math.log(3.0)))))
    np.testing.assert_allclose(out[0, 0], [4.0 * w, 8.0 * (1 - w)], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(out[0, 0], [3.0, 2.0], rtol=1e-7)


# ----------------------------------------------------------------------------- invariants

def test_permutation_of_physical_ids_is_bit_identical():
    wl = W.build_decode(17, [40, 3, 77, 16], H_q=8, H_kv=2, D=16, num_blocks=32, dtype="bf16")
    kc, vc = _full_pool(wl)
    base = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    rng = np.random.default_rng(5)
    perm = np.concatenate([[0], 1 + rng.permutation(31)])      # new id of old block b = perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    out = oracle.attention(wl.q, kc2, vc2, perm[wl.block_table].astype(np.int32), wl.seq_lens, wl.scale)
    assert np.array_equal(base, out)


def test_alias_versus_copy_of_shared_prefix_is_bit_identical():
    wl = W.build_decode(18, [70, 64, 90], H_q=4, H_kv=2, D=8, num_blocks=64, dtype="bf16",
                        new_token=False, shared_prefix_tokens=64)
    shared = wl.block_table[0, :4].copy()
    assert (wl.block_table[:, :4] == shared).all()
    base = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    kc, vc, bt = wl.k_cache.copy(), wl.v_cache.copy(), wl.block_table.copy()
    free = [b for b in range(1, 64) if b not in set(bt.ravel().tolist())]
    for i in range(1, 3):                 # give sequences 1 and 2 private copies
        for j in range(4):
            nb = free.pop()
            kc[nb], vc[nb] = kc[shared[j]], vc[shared[j]]
            bt[i, j] = nb
    out = oracle.attention(wl.q, kc, vc, bt, wl.seq_lens, wl.scale)
    assert np.array_equal(base, out)


def test_null_block_contents_do_not_matter():
    wl = W.build_decode(19, [5, 21, 16], H_q=2, H_kv=1, D=8, num_blocks=8, dtype="f32", new_token=False)
    assert np.isnan(wl.k_cache[0]).all()          # the generator poisons block 0
    a = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    kc[0], vc[0] = 7.0, -3.0
    b = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    assert np.isfinite(a).all() and np.array_equal(a, b)


def test_block_count_and_waste_bound():
    """A sequence of L tokens uses ceil(L/16) blocks and wastes at most 15 slots."""
    for L in [1, 15, 16, 17, 31, 32, 33, 195, 2048]:
        wl = W.build_decode(20, [L], H_q=1, H_kv=1, D=8, num_blocks=200, dtype="f32")
        nblk = int((wl.block_table[0] > 0).sum())
        assert nblk == -(-L // 16)
        assert 0 <= nblk * 16 - L <= 15


def test_lognormal_mix_has_the_length_implied_by_963_percent():
    """u = L / (L + 7.5) = 0.963 gives L ~ 195 ("Checking the 96.3%"); the decode batch
    generator targets that mean."""
    L = 7.5 * 0.963 / (1 - 0.963)
    assert abs(L - 195) < 1
    wl = W.gqa_decode()
    assert abs(float(wl.seq_lens.mean()) - L) / L < 0.05
    assert wl.seq_lens.min() >= 16 and wl.seq_lens.max() <= 2048


# ----------------------------------------------------------------------------- block-size variants

@pytest.mark.parametrize("bs", [32, 64, 128])
def test_decode_matches_bruteforce_for_larger_blocks(bs):
    # "vLLM: what PagedAttention turned into": block sizes 16 to 128 all work; the result is
    # still plain attention over the sequence's keys in logical order
    wl = W.build_decode(40 + bs, [1, bs - 1, bs, bs + 1, 3 * bs + 5], H_q=8, H_kv=2, D=16,
                        num_blocks=24, dtype="bf16", keep_contiguous=True, block_size=bs)
    assert wl.k_cache.shape[2] == bs
    kc, vc = _full_pool(wl)
    out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    ref = brute_decode(wl.q, wl.contiguous_k, wl.contiguous_v, wl.scale, wl.H_kv)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def _repack(kc, bt, lens, bs_new):
    """Move each sequence's keys, in logical order, into fresh blocks of size bs_new."""
    NB, H, bs, D = kc.shape
    per = [-(-int(L) // bs_new) for L in lens]
    out = np.zeros((1 + sum(per), H, bs_new, D), kc.dtype)
    bt2 = np.zeros((len(lens), max(per + [1])), np.int32)
    nxt = 1
    for i, L in enumerate(lens):
        for p in range(int(L)):
            if p % bs_new == 0:
                bt2[i, p // bs_new] = nxt
                nxt += 1
            out[bt2[i, p // bs_new], :, p % bs_new] = kc[bt[i, p // bs], :, p % bs]
    return out, bt2


@pytest.mark.parametrize("bs", [32, 128])
def test_reblocking_is_bit_identical(bs):
    """The same keys stored in 16-token blocks or in bs-token blocks give the same bits:
    the block size only changes where a key sits."""
    wl = W.build_decode(50 + bs, [7, 200, 129, 64], H_q=4, H_kv=2, D=8, num_blocks=16,
                        dtype="bf16", block_size=bs)
    kc, vc = _full_pool(wl)
    base = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    k16, bt16 = _repack(kc, wl.block_table, wl.seq_lens, 16)
    v16, _ = _repack(vc, wl.block_table, wl.seq_lens, 16)
    assert k16.shape[2] == 16
    out = oracle.attention(wl.q, k16, v16, bt16, wl.seq_lens, wl.scale)
    assert np.array_equal(base, out)


def test_reshape_with_64_token_blocks_places_slot_s_at_block_s_div_64():
    rng = np.random.default_rng(60)
    kc = np.zeros((4, 2, 64, 8), np.float32)
    vc = kc.copy()
    k = rng.standard_normal((3, 2, 8)).astype(np.float32)
    v = rng.standard_normal((3, 2, 8)).astype(np.float32)
    oracle.reshape_and_cache(k, v, kc, vc, np.array([0, 63, 64 * 3 + 17], np.int64))
    assert np.array_equal(kc[0, :, 0], k[0]) and np.array_equal(kc[0, :, 63], k[1])
    assert np.array_equal(kc[3, :, 17], k[2]) and np.array_equal(vc[3, :, 17], v[2])
    assert np.count_nonzero(kc) == 3 * 2 * 8


def test_prefill_with_64_token_blocks_matches_torch_sdpa():
    torch = pytest.importorskip("torch")
    wl = W.build_mixed(61, prior_lens=[0, 70], chunk_lens=[65, 30], decode_lens=[5], H_q=4, H_kv=2,
                       D=16, num_blocks=16, dtype="f32", pad_multiple=0, keep_contiguous=True,
                       block_size=64)
    kc, vc = _full_pool(wl)
    qsl = wl.query_start_loc
    out = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill,
                           wl.scale, query_start_loc=qsl)
    for i in range(2):
        L, C = int(wl.seq_lens_prefill[i]), int(qsl[i + 1] - qsl[i])
        qi = torch.from_numpy(W.as_f64(wl.q_prefill[qsl[i]:qsl[i + 1]])).transpose(0, 1)
        K = torch.from_numpy(W.as_f64(wl.contiguous_k_prefill[i])).transpose(0, 1).repeat_interleave(2, 0)
        V = torch.from_numpy(W.as_f64(wl.contiguous_v_prefill[i])).transpose(0, 1).repeat_interleave(2, 0)
        mask = torch.arange(L).unsqueeze(0) <= (torch.arange(C).unsqueeze(1) + L - C)
        ref = torch.nn.functional.scaled_dot_product_attention(qi, K, V, attn_mask=mask, scale=wl.scale)
        np.testing.assert_allclose(out[qsl[i]:qsl[i + 1]], ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)
