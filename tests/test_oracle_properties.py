"""Property tests of the oracle on random small cases (CPU): for any lengths, head layout,
block size, physical placement and chunking, paged attention equals plain attention on the
keys gathered in logical order, computed here by brute force in numpy."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402


def _brute(q_rows, K, V, scale, G, visible):
    """q_rows [R, H_q, D]; K, V [L, H_kv, D]; row r sees keys 0..visible[r]-1."""
    R, H_q, D = q_rows.shape
    out = np.zeros((R, H_q, D))
    for r in range(R):
        n = visible[r]
        for h in range(H_q):
            z = scale * K[:n, h // G] @ q_rows[r, h]
            p = np.exp(z - z.max())
            out[r, h] = (p / p.sum()) @ V[:n, h // G]
    return out


@settings(max_examples=40, deadline=None)
@given(lens=st.lists(st.integers(1, 90), min_size=1, max_size=5),
       h_kv=st.sampled_from([1, 2, 3]), group=st.sampled_from([1, 2, 4]),
       bs=st.sampled_from([16, 32, 64]), dtype=st.sampled_from(["f32", "bf16"]), seed=st.integers(0, 10_000))
def test_decode_equals_attention_on_gathered_keys(lens, h_kv, group, bs, dtype, seed):
    need = sum(-(-L // bs) for L in lens) + 2
    wl = W.build_decode(seed, lens, H_q=h_kv * group, H_kv=h_kv, D=8, num_blocks=need, dtype=dtype,
                        keep_contiguous=True, block_size=bs)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    for i, L in enumerate(lens):
        ref = _brute(W.as_f64(wl.q[i:i + 1]), W.as_f64(wl.contiguous_k[i]), W.as_f64(wl.contiguous_v[i]),
                     wl.scale, group, [L])
        np.testing.assert_allclose(out[i:i + 1], ref, rtol=1e-12, atol=1e-12)


@settings(max_examples=30, deadline=None)
@given(prior=st.lists(st.integers(0, 60), min_size=1, max_size=3), data=st.data(),
       bs=st.sampled_from([16, 32]), seed=st.integers(0, 10_000))
def test_chunked_prefill_equals_causal_attention_on_gathered_keys(prior, data, bs, seed):
    chunks = [data.draw(st.integers(0, 40)) for _ in prior]
    if sum(chunks) == 0:
        chunks[0] = 1
    lens = [p + c for p, c in zip(prior, chunks)]
    need = sum(-(-L // bs) for L in lens) + 4
    wl = W.build_mixed(seed, prior_lens=prior, chunk_lens=chunks, decode_lens=[], H_q=4, H_kv=2, D=8,
                       num_blocks=need, dtype="f32", pad_multiple=0, keep_contiguous=True, block_size=bs)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    qsl = wl.query_start_loc
    out = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                           query_start_loc=qsl)
    for i, (P, C) in enumerate(zip(prior, chunks)):
        if C == 0:
            continue
        rows = slice(qsl[i], qsl[i + 1])
        ref = _brute(W.as_f64(wl.q_prefill[rows]), W.as_f64(wl.contiguous_k_prefill[i]),
                     W.as_f64(wl.contiguous_v_prefill[i]), wl.scale, 2, [P + r + 1 for r in range(C)])
        np.testing.assert_allclose(out[rows], ref, rtol=1e-12, atol=1e-12)
