"""GPU parity: the sm_103a kernels, called through the C ABI, against the fp64 oracle.

Every case draws seeded inputs from ``paged_kv_cache_238_gb300.workloads``; the oracle sees the
same bf16/fp32 values. Tolerances live in tests/helpers.py.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from paged_kv_cache_238_gb300 import binding as B  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402

from helpers import DeviceWorkload, assert_close, mixed_step_reference, to_f64, to_host_bits  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    B.pa_get_device_errors(clear=True)
    yield
    assert B.pa_get_device_errors(clear=True) == 0, "a kernel raised a device error"


def run_reshape(dw: DeviceWorkload):
    B.pa_reshape_and_cache(dw.k_new, dw.v_new, dw.k_cache, dw.v_cache, dw.slot_mapping)


def run_decode(dw: DeviceWorkload, max_seq_len=None):
    wl = dw.wl
    msl = int(wl.seq_lens.max()) if max_seq_len is None else max_seq_len
    ws_bytes = B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, dw.tdtype)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    B.pa_decode(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale, ws)
    torch.cuda.synchronize()
    return to_f64(dw.out)


def run_prefill(dw: DeviceWorkload):
    wl = dw.wl
    qsl = wl.query_start_loc
    max_chunk = int(np.max(np.diff(qsl))) if len(qsl) > 1 else 0
    B.pa_prefill_chunk(dw.out_prefill, dw.q_prefill, dw.k_cache, dw.v_cache, dw.block_table_prefill,
                       dw.seq_lens_prefill, dw.query_start_loc, max_chunk, int(wl.seq_lens_prefill.max()), wl.scale)
    torch.cuda.synchronize()
    return to_f64(dw.out_prefill)


def check_pool(dw: DeviceWorkload, kc_ref, vc_ref):
    kc, vc = to_host_bits(dw.k_cache), to_host_bits(dw.v_cache)
    raw = (lambda a: a.view(np.uint32)) if kc.dtype == np.float32 else (lambda a: a)
    # block 0 is the null block: padding writes land there, its contents are undefined
    assert np.array_equal(raw(kc[1:]), raw(kc_ref[1:])), "k_cache differs from the oracle"
    assert np.array_equal(raw(vc[1:]), raw(vc_ref[1:])), "v_cache differs from the oracle"


# ----------------------------------------------------------------------------- reshape_and_cache

@pytest.mark.parametrize("name", ["tiny_fp32", "gqa_decode", "mixed_step"])
def test_reshape_and_cache_bit_exact(name):
    dw = DeviceWorkload(W.WORKLOADS[name]())
    run_reshape(dw)
    torch.cuda.synchronize()
    kc_ref, vc_ref = dw.host_pool_after_writes()
    check_pool(dw, kc_ref, vc_ref)


def test_reshape_negative_slots_and_fp32_ragged():
    wl = W.build_decode(40, [3, 17, 33, 1, 64], H_q=4, H_kv=4, D=64, num_blocks=32, dtype="f32")
    wl.slot_mapping[1] = -1                    # skipped: the pool cell stays poisoned
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    torch.cuda.synchronize()
    kc_ref, vc_ref = dw.host_pool_after_writes()
    check_pool(dw, kc_ref, vc_ref)


# ----------------------------------------------------------------------------- decode: the five workloads

def _decode_vs_oracle(wl, rows=None, what=""):
    dw = DeviceWorkload(wl)
    if wl.slot_mapping is not None:
        run_reshape(dw)
    out = run_decode(dw)
    kc, vc = dw.host_pool_after_writes()
    idx = np.arange(wl.S) if rows is None else np.asarray(rows)
    ref = oracle.attention(wl.q[idx], kc, vc, wl.block_table[idx], wl.seq_lens[idx], wl.scale)
    assert_close(out[idx], ref, wl.dtype, what)
    return dw, out


def test_decode_tiny_fp32():
    _decode_vs_oracle(W.tiny_fp32(), what="tiny fp32")


def test_decode_gqa_bs64_bf16():
    _decode_vs_oracle(W.gqa_decode(), what="gqa decode bs64")


def test_decode_prefix_sharing_bs128():
    _decode_vs_oracle(W.prefix_sharing(), what="prefix sharing")


@pytest.mark.slow
def test_decode_long_split_kv():
    _decode_vs_oracle(W.long_split_kv(), what="long split-kv")


@pytest.mark.slow
def test_mixed_step_decode_all_rows():
    """All 240 decode rows of the mixed-step workload, element by element."""
    wl, kc, vc, ref_dec, _ = mixed_step_reference()
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    out = run_decode(dw)
    check_pool(dw, kc, vc)
    assert_close(out, ref_dec, "bf16", "mixed step, every decode row")


# ----------------------------------------------------------------------------- decode: edge cases

@pytest.mark.parametrize("lens", [[1, 15, 16, 17, 31, 32, 33], [16] * 9, [2048, 1, 700], [5] * 300])
@pytest.mark.parametrize("G", [1, 2, 4, 5, 6, 8, 16])
def test_decode_ragged_lengths_and_groups(lens, G):
    H_kv = 2 if G <= 8 else 1
    need = sum(-(-L // 16) for L in lens) + 2
    wl = W.build_decode(41 + G, lens, H_q=G * H_kv, H_kv=H_kv, D=128, num_blocks=need, dtype="bf16")
    _decode_vs_oracle(wl, what=f"lens {lens[:4]} G {G}")


@pytest.mark.parametrize("lens,H_kv", [([32768], 1), ([20000, 3, 9000], 2), ([700] * 3, 1)])
def test_decode_segments_cut_into_many_pieces(lens, H_kv):
    """One (sequence, kv head) spread over every streaming warp: the split reduce merges
    hundreds of pieces."""
    need = sum(-(-L // 16) for L in lens) + 2
    wl = W.build_decode(45, lens, H_q=4 * H_kv, H_kv=H_kv, D=128, num_blocks=need, dtype="bf16")
    _decode_vs_oracle(wl, what=f"long segments {lens}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_decode_head_dim_64(dtype, G):
    wl = W.build_decode(60 + G, [1, 9, 16, 100, 257], H_q=G * 2, H_kv=2, D=64, num_blocks=64, dtype=dtype)
    _decode_vs_oracle(wl, what=f"D64 {dtype} G{G}")


def test_decode_workspace_reuse_across_calls():
    """The split-merge counters return to zero after every call: reusing one workspace for
    many calls (and for different batches) gives bit-identical results."""
    wl = W.build_decode(46, [300, 17, 64, 1000, 5, 2048], H_q=32, H_kv=8, D=128, num_blocks=400, dtype="bf16",
                        new_token=False)
    dw = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    ws = torch.zeros(B.pa_decode_workspace_size(wl.S, 32, 8, 128, msl, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for _ in range(3):
        B.pa_decode(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale, ws)
        torch.cuda.synchronize()
        outs.append(to_host_bits(dw.out).copy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    ref = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(W.as_f64(outs[2]), ref, "bf16", "workspace reuse")


def test_decode_zero_length_rows_are_zero():
    wl = W.build_decode(70, [0, 40, 0, 3], H_q=8, H_kv=2, D=128, num_blocks=16, dtype="bf16", new_token=False)
    dw = DeviceWorkload(wl)
    out = run_decode(dw)
    assert not out[0].any() and not out[2].any()
    ref = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(out, ref, "bf16", "zero-length rows")


def test_decode_max_seq_len_above_actual():
    """The host bound may exceed every real length (more partitions than needed)."""
    wl = W.build_decode(71, [20, 3], H_q=2, H_kv=2, D=64, num_blocks=16, dtype="f32", max_blocks=64)
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    out = run_decode(dw, max_seq_len=1024)
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(out, ref, "f32", "max_seq_len above actual")


def test_decode_permuted_physical_ids_bit_identical():
    wl = W.build_decode(72, [300, 17, 64, 1000, 5], H_q=16, H_kv=4, D=128, num_blocks=160, dtype="bf16",
                        new_token=False)
    dw = DeviceWorkload(wl)
    run_decode(dw)
    a = to_host_bits(dw.out).copy()
    rng = np.random.default_rng(3)
    perm = np.concatenate([[0], 1 + rng.permutation(wl.num_blocks - 1)])
    kc, vc = np.empty_like(wl.k_cache), np.empty_like(wl.v_cache)
    kc[perm], vc[perm] = wl.k_cache, wl.v_cache
    wl2 = W.Workload(**{**wl.__dict__, "k_cache": kc, "v_cache": vc,
                        "block_table": perm[wl.block_table].astype(np.int32)})
    dw2 = DeviceWorkload(wl2)
    run_decode(dw2)
    assert np.array_equal(a, to_host_bits(dw2.out))


def test_decode_alias_versus_copy_bit_identical():
    wl = W.build_decode(73, [100, 64, 80, 200], H_q=32, H_kv=8, D=128, num_blocks=64, dtype="bf16",
                        new_token=False, shared_prefix_tokens=64)
    dw = DeviceWorkload(wl)
    run_decode(dw)
    a = to_host_bits(dw.out).copy()
    kc, vc, bt = wl.k_cache.copy(), wl.v_cache.copy(), wl.block_table.copy()
    used = set(bt.ravel().tolist())
    free = [b for b in range(1, wl.num_blocks) if b not in used]
    for i in range(1, wl.S):
        for j in range(4):
            nb = free.pop()
            kc[nb], vc[nb] = kc[bt[0, j]], vc[bt[0, j]]
            bt[i, j] = nb
    dw2 = DeviceWorkload(W.Workload(**{**wl.__dict__, "k_cache": kc, "v_cache": vc, "block_table": bt}))
    run_decode(dw2)
    assert np.array_equal(a, to_host_bits(dw2.out))


def test_decode_null_block_contents_do_not_matter():
    wl = W.build_decode(74, [33, 16, 7], H_q=8, H_kv=2, D=128, num_blocks=16, dtype="bf16", new_token=False)
    dw = DeviceWorkload(wl)
    run_decode(dw)
    a = to_host_bits(dw.out).copy()
    dw.k_cache[0] = 3.0
    dw.v_cache[0] = -2.0
    run_decode(dw)
    assert np.array_equal(a, to_host_bits(dw.out))


# ----------------------------------------------------------------------------- prefill

@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 64)])
def test_prefill_small_mixed(dtype, D):
    wl = W.build_mixed(80, prior_lens=[0, 5, 16, 100, 31], chunk_lens=[7, 16, 33, 1, 64],
                       decode_lens=[20, 1], H_q=8, H_kv=2, D=D, num_blocks=128, dtype=dtype, pad_multiple=32)
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    out = run_prefill(dw)
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                           query_start_loc=wl.query_start_loc)
    assert_close(out, ref, dtype, f"prefill {dtype} D{D}")


@pytest.mark.parametrize("G,H_kv", [(1, 2), (2, 2), (4, 2), (8, 1), (16, 1)])
def test_prefill_tensor_core_groups_and_ragged_tiles(G, H_kv):
    """bf16 / head_dim 128 runs the tcgen05 kernel: 128-row query tiles of 128/G tokens x G
    heads, 128-key tiles. Chunks that end mid-tile, prior context that ends mid-block and
    crosses several key tiles, and a chunk that starts at position 0."""
    wl = W.build_mixed(82 + G, prior_lens=[0, 1, 127, 300, 1000], chunk_lens=[200, 37, 129, 64, 300],
                       decode_lens=[9], H_q=G * H_kv, H_kv=H_kv, D=128, num_blocks=400, dtype="bf16",
                       pad_multiple=64)
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    out = run_prefill(dw)
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                           query_start_loc=wl.query_start_loc)
    assert_close(out, ref, "bf16", f"tensor-core prefill G{G}")


def test_prefill_empty_chunks_and_whole_prompt():
    wl = W.build_mixed(81, prior_lens=[10, 0, 3], chunk_lens=[0, 40, 0], decode_lens=[5], H_q=4, H_kv=1, D=128,
                       num_blocks=32, dtype="bf16", pad_multiple=0)
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    out = run_prefill(dw)
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                           query_start_loc=wl.query_start_loc)
    assert_close(out, ref, "bf16", "empty chunks")


@pytest.mark.slow
def test_mixed_step_prefill_all_rows():
    """Every row of all 16 prefill chunks of the mixed-step workload (8192 query rows over
    prior contexts of 0..4096 tokens), element by element, and the pool after the step's
    writes bit-exact."""
    wl, kc, vc, _, ref_pre = mixed_step_reference()
    dw = DeviceWorkload(wl)
    run_reshape(dw)
    out = run_prefill(dw)
    check_pool(dw, kc, vc)
    assert_close(out, ref_pre, "bf16", "mixed step, every prefill row")


# ----------------------------------------------------------------------------- maximum sizes

@pytest.mark.parametrize("S", [1024, 1025])
def test_decode_at_and_past_the_persistent_path_batch_limit(S):
    """1024 sequences is the largest batch whose tables the persistent kernel keeps in shared
    memory; 1025 takes the general path. Both against the oracle."""
    rng = np.random.default_rng(700 + S)
    lens = rng.integers(1, 40, size=S)
    wl = W.build_decode(700 + S, lens, H_q=8, H_kv=2, D=64, num_blocks=int(np.sum(-(-lens // 16))) + 2,
                        dtype="bf16")
    _decode_vs_oracle(wl, what=f"{S} sequences")


def test_decode_block_ids_at_the_top_of_a_large_pool():
    """A pool of 200 000 blocks whose tables name the highest ids (pool rows far past 2^24)."""
    NB, H_kv, D = 200_000, 1, 64
    lens = np.array([33, 700, 16, 1])
    wl = W.build_decode(710, lens, H_q=4, H_kv=H_kv, D=D, num_blocks=64, dtype="bf16", new_token=False,
                        poison=False)
    # move every used block to the top of a large pool
    used = sorted(set(wl.block_table[wl.block_table > 0].tolist()))
    remap = {b: NB - 1 - i for i, b in enumerate(used)}
    kc = np.zeros((NB, H_kv, 16, D), np.uint16)
    vc = np.zeros_like(kc)
    for b, nb in remap.items():
        kc[nb], vc[nb] = wl.k_cache[b], wl.v_cache[b]
    bt = np.vectorize(lambda x: remap.get(int(x), 0))(wl.block_table).astype(np.int32)
    wl2 = W.Workload(name="top", dtype="bf16", H_q=4, H_kv=H_kv, D=D, num_blocks=NB, scale=wl.scale, k_cache=kc,
                     v_cache=vc, q=wl.q, block_table=bt, seq_lens=wl.seq_lens)
    assert bt.max() == NB - 1
    _decode_vs_oracle(wl2, what="top of a large pool")
