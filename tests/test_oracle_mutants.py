"""Plant plausible mistakes in a copy of the oracle's C source (CPU only) and check that the
pins catch each one: a pin that cannot tell a wrong oracle from the right one pins nothing."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from paged_kv_cache_238_gb300 import workloads as W

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

# (name, exact text in the source, replacement). Each keeps every memory access in bounds.
MUTANTS = [
    ("gqa_head_map", "const int32_t g = h / group;", "const int32_t g = h % H_kv;"),
    ("dropped_scale", "z[j] = scale * dot;", "z[j] = dot;"),
    ("softmax_sign", "z[j] = exp(z[j] - zmax);", "z[j] = exp(zmax - z[j]);"),
    ("v_replaced_by_k", "o[d] += w * Vg[(size_t)j * D + d];", "o[d] += w * Kg[(size_t)j * D + d];"),
    ("causal_one_short", "const int32_t pos = len - chunk + r;",
     "const int32_t pos = (len - chunk + r > 0) ? len - chunk + r - 1 : 0;"),
    ("top_left_causal", "const int32_t pos = len - chunk + r;", "const int32_t pos = (chunk > 1) ? r : len - 1;"),
    ("gather_offset", "(size_t)(j % block_size)) * D;", "(size_t)((j + 1) % block_size)) * D;"),
    ("gather_head_stride", "size_t src = (((size_t)phys * H_kv + g) * (size_t)block_size",
     "size_t src = (((size_t)phys * H_kv + (H_kv - 1 - g)) * (size_t)block_size"),
    ("pool_layout_swapped",
     "size_t dst = (((size_t)block * H_kv + h) * (size_t)block_size + (size_t)offset) * row;",
     "size_t dst = (((size_t)block * (size_t)block_size + (size_t)offset) * H_kv + h) * row;"),
    ("gather_block_size_fixed_16",
     "int32_t phys = block_table[(size_t)i * max_blocks_per_seq + j / block_size];",
     "int32_t phys = block_table[(size_t)i * max_blocks_per_seq + j / 16];"),
    ("reshape_block_size_fixed_16", "int64_t offset = slot % block_size;", "int64_t offset = slot % 16;"),
    ("bf16_widening", "<< 16;", "<< 15;"),
    ("negative_slot_written", "if (slot < 0) continue;", "if (slot < 0) slot = 0;"),
]


def _pins(lib):
    """A compact run of the pins; returns the names of the pins that failed."""
    failed = []

    def check(name, fn):
        try:
            fn()
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(name)

    def bf16_gqa_bruteforce():
        wl = W.build_decode(31, [17, 33, 5, 48], H_q=8, H_kv=2, D=16, num_blocks=32, dtype="bf16",
                            keep_contiguous=True)
        kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
        oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping, _lib_override=lib)
        out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale, _lib_override=lib)
        G = wl.H_q // wl.H_kv
        for i in range(wl.S):
            K, V = W.as_f64(wl.contiguous_k[i]), W.as_f64(wl.contiguous_v[i])
            for h in range(wl.H_q):
                z = wl.scale * K[:, h // G] @ W.as_f64(wl.q[i, h])
                p = np.exp(z - z.max())
                np.testing.assert_allclose(out[i, h], (p / p.sum()) @ V[:, h // G], rtol=1e-10, atol=1e-10)

    def prefill_sdpa():
        torch = pytest.importorskip("torch")
        wl = W.build_mixed(32, prior_lens=[3, 20], chunk_lens=[6, 9], decode_lens=[2], H_q=4, H_kv=2,
                           D=8, num_blocks=32, dtype="f32", pad_multiple=0, keep_contiguous=True)
        kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
        oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping, _lib_override=lib)
        qsl = wl.query_start_loc
        out = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill,
                               wl.scale, query_start_loc=qsl, _lib_override=lib)
        for i in range(2):
            L, C = int(wl.seq_lens_prefill[i]), int(qsl[i + 1] - qsl[i])
            qi = torch.from_numpy(W.as_f64(wl.q_prefill[qsl[i]:qsl[i + 1]])).transpose(0, 1)
            K = torch.from_numpy(W.as_f64(wl.contiguous_k_prefill[i])).transpose(0, 1).repeat_interleave(2, 0)
            V = torch.from_numpy(W.as_f64(wl.contiguous_v_prefill[i])).transpose(0, 1).repeat_interleave(2, 0)
            mask = torch.arange(L).unsqueeze(0) <= (torch.arange(C).unsqueeze(1) + L - C)
            ref = torch.nn.functional.scaled_dot_product_attention(qi, K, V, attn_mask=mask, scale=wl.scale)
            np.testing.assert_allclose(out[qsl[i]:qsl[i + 1]], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-10)

    def reshape_negative_slot_skipped():
        kc = np.full((2, 1, 16, 4), 9.0, np.float32)
        vc = kc.copy()
        oracle.reshape_and_cache(np.ones((2, 1, 4), np.float32), np.ones((2, 1, 4), np.float32), kc, vc,
                                 np.array([-1, 17], np.int64), _lib_override=lib)
        assert (kc[0] == 9.0).all() and (kc[1, 0, 1] == 1.0).all()

    def block_size_32_bruteforce():
        # 32-token blocks: the same brute force over a pool whose third dimension is 32
        wl = W.build_decode(35, [40, 64, 9], H_q=4, H_kv=2, D=8, num_blocks=12, dtype="f32",
                            keep_contiguous=True, block_size=32)
        kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
        oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping, _lib_override=lib)
        out = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale, _lib_override=lib)
        for i in range(wl.S):
            K, V = W.as_f64(wl.contiguous_k[i]), W.as_f64(wl.contiguous_v[i])
            for h in range(wl.H_q):
                z = wl.scale * K[:, h // 2] @ W.as_f64(wl.q[i, h])
                p = np.exp(z - z.max())
                np.testing.assert_allclose(out[i, h], (p / p.sum()) @ V[:, h // 2], rtol=1e-10, atol=1e-10)

    check("bf16_gqa_bruteforce", bf16_gqa_bruteforce)
    check("block_size_32_bruteforce", block_size_32_bruteforce)
    check("prefill_sdpa", prefill_sdpa)
    check("reshape_negative_slot_skipped", reshape_negative_slot_skipped)
    return failed


def _build_variant(tmp_path, text, repl, tag):
    src = open(SRC).read()
    assert src.count(text) >= 1, f"mutation anchor not found: {text}"
    path = tmp_path / f"mut_{tag}.c"
    path.write_text(src.replace(text, repl))
    so = tmp_path / f"libmut_{tag}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(path), "-o", str(so), "-lm"],
                   check=True)
    return oracle.load_variant(str(so))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = _build_variant(tmp_path, "#include <math.h>", "#include <math.h>", "identity")
    assert _pins(lib) == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,text,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, text, repl):
    lib = _build_variant(tmp_path, text, repl, name)
    with np.errstate(all="ignore"):
        failed = _pins(lib)
    assert failed, f"no pin caught the planted mistake {name}"
