"""GPU parity of the block-size variants (32, 64 and 128 tokens per block) against the fp64
oracle, which takes the block size from the pool's third dimension.

"vLLM: what PagedAttention turned into" gives 16 tokens as the block size and reports 16 to
128 performing alike. The kernels walk a block as block_size / 16 pages of 16 tokens, so on
top of oracle parity every kernel must give bit-identical results for the same keys stored in
16-token blocks (same pages, same order, same work split)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from paged_kv_cache_238_gb300 import binding as B  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402

from helpers import DeviceWorkload, assert_close, to_dev, to_f64, to_host_bits  # noqa: E402

pytestmark = pytest.mark.gpu
SIZES = [32, 64, 128]


@pytest.fixture(autouse=True)
def _clean_error_word():
    B.pa_get_device_errors(clear=True)
    yield
    assert B.pa_get_device_errors(clear=True) == 0, "a kernel raised a device error"


def _decode(dw, msl=None):
    wl = dw.wl
    msl = int(wl.seq_lens.max()) if msl is None else msl
    ws = torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, dw.tdtype)),
                     dtype=torch.uint8, device="cuda")
    B.pa_decode(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale, ws)
    torch.cuda.synchronize()
    return to_host_bits(dw.out)


def _prefill(dw):
    wl = dw.wl
    qsl = wl.query_start_loc
    B.pa_prefill_chunk(dw.out_prefill, dw.q_prefill, dw.k_cache, dw.v_cache, dw.block_table_prefill,
                       dw.seq_lens_prefill, dw.query_start_loc, int(np.max(np.diff(qsl))),
                       int(wl.seq_lens_prefill.max()), wl.scale)
    torch.cuda.synchronize()
    return to_host_bits(dw.out_prefill)


def _repack(pool, bt, lens, bs_new):
    """The same keys, in logical order, in fresh blocks of bs_new tokens (block 0 stays null)."""
    bs = pool.shape[2]
    per = [-(-int(L) // bs_new) for L in lens]
    out = np.zeros((1 + sum(per), pool.shape[1], bs_new, pool.shape[3]), pool.dtype)
    bt2 = np.zeros((len(lens), max(per + [1])), np.int32)
    nxt = 1
    for i, L in enumerate(lens):
        for b in range(per[i]):
            bt2[i, b] = nxt
            nxt += 1
        p = np.arange(int(L))
        out[bt2[i, p // bs_new], :, p % bs_new] = pool[bt[i, p // bs], :, p % bs]
    return out, bt2


# ----------------------------------------------------------------------------- reshape_and_cache

@pytest.mark.parametrize("bs", SIZES)
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_reshape_bit_exact(bs, dtype, D):
    wl = W.build_decode(300 + bs, [1, bs - 1, bs, bs + 1, 3 * bs + 7, 5], H_q=8, H_kv=2, D=D,
                        num_blocks=24, dtype=dtype, block_size=bs)
    wl.slot_mapping[5] = -1                      # padding: skipped
    dw = DeviceWorkload(wl)
    B.pa_reshape_and_cache(dw.k_new, dw.v_new, dw.k_cache, dw.v_cache, dw.slot_mapping)
    torch.cuda.synchronize()
    kc, vc = dw.host_pool_after_writes()
    raw = (lambda a: a.view(np.uint32)) if dtype == "f32" else (lambda a: a)
    assert np.array_equal(raw(to_host_bits(dw.k_cache)[1:]), raw(kc[1:]))
    assert np.array_equal(raw(to_host_bits(dw.v_cache)[1:]), raw(vc[1:]))


# ----------------------------------------------------------------------------- decode

@pytest.mark.parametrize("bs", SIZES)
@pytest.mark.parametrize("dtype,D,G", [("bf16", 128, 4), ("bf16", 128, 16), ("bf16", 64, 8), ("f32", 128, 1),
                                       ("bf16", 128, 2)])
def test_decode_matches_oracle(bs, dtype, D, G):
    """bf16 groups 4..16 run the balanced TMA kernel (3-D box for head_dim 128, 2-D for 64);
    fp32 and group 2 run the SIMT split-KV kernel."""
    H_kv = 2 if G <= 8 else 1
    lens = [1, 15, 16, 17, bs - 1, bs, bs + 1, 2 * bs + 3, 1000, 3000]
    need = sum(-(-L // bs) for L in lens) + 2
    wl = W.build_decode(310 + bs + G, lens, H_q=G * H_kv, H_kv=H_kv, D=D, num_blocks=need, dtype=dtype,
                        block_size=bs)
    dw = DeviceWorkload(wl)
    B.pa_reshape_and_cache(dw.k_new, dw.v_new, dw.k_cache, dw.v_cache, dw.slot_mapping)
    out = W.as_f64(_decode(dw))
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(out, ref, dtype, f"decode bs{bs} {dtype} D{D} G{G}")


@pytest.mark.parametrize("bs", SIZES)
@pytest.mark.parametrize("dtype,G", [("bf16", 4), ("f32", 1)])
def test_decode_reblocked_is_bit_identical(bs, dtype, G):
    lens = [3, bs + 9, 700, 4 * bs]
    wl = W.build_decode(320 + bs, lens, H_q=2 * G, H_kv=2, D=128, num_blocks=sum(-(-L // bs) for L in lens) + 1,
                        dtype=dtype, new_token=False, block_size=bs)
    a = _decode(DeviceWorkload(wl))
    k16, bt16 = _repack(wl.k_cache, wl.block_table, wl.seq_lens, 16)
    v16, _ = _repack(wl.v_cache, wl.block_table, wl.seq_lens, 16)
    wl16 = W.Workload(name="reblocked", dtype=dtype, H_q=wl.H_q, H_kv=2, D=128, num_blocks=k16.shape[0],
                      scale=wl.scale, k_cache=k16, v_cache=v16, q=wl.q, block_table=bt16, seq_lens=wl.seq_lens)
    b = _decode(DeviceWorkload(wl16))
    assert np.array_equal(a, b)


def test_decode_bs_entry_point_at_16_equals_plain_entry_point():
    wl = W.build_decode(330, [40, 1, 333, 16], H_q=8, H_kv=2, D=128, num_blocks=40, dtype="bf16", new_token=False)
    dw = DeviceWorkload(wl)
    a = _decode(dw)
    ws = torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, 8, 2, 128, 333, dw.tdtype)), dtype=torch.uint8,
                     device="cuda")
    B.pa_decode_bs(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, 333, wl.scale, ws)
    torch.cuda.synchronize()
    assert np.array_equal(a, to_host_bits(dw.out))


@pytest.mark.parametrize("bs", [32, 128])
def test_decode_length_beyond_table_is_flagged_and_clamped(bs):
    """A length past max_blocks * bs is clamped to what the table row addresses and flagged."""
    wl = W.build_decode(340 + bs, [2 * bs, 5], H_q=8, H_kv=2, D=128, num_blocks=8, dtype="bf16",
                        new_token=False, max_blocks=2, block_size=bs)
    dw = DeviceWorkload(wl)
    dw.seq_lens[0] = 2 * bs + 1
    out = W.as_f64(_decode(dw, msl=2 * bs))
    assert B.pa_get_device_errors(clear=True) == B.PA_DEVERR_LEN_RANGE
    ref = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(out, ref, "bf16", "clamped length")


# ----------------------------------------------------------------------------- prefill

@pytest.mark.parametrize("bs", SIZES)
@pytest.mark.parametrize("dtype,D,G", [("bf16", 128, 4), ("bf16", 128, 8), ("bf16", 64, 4), ("f32", 64, 2)])
def test_prefill_matches_oracle(bs, dtype, D, G):
    """bf16 head_dim 128 runs the tcgen05 kernel; the others run the SIMT path."""
    wl = W.build_mixed(350 + bs + G, prior_lens=[0, 1, bs - 1, 300, 1000], chunk_lens=[200, 37, bs + 1, 64, 300],
                       decode_lens=[9], H_q=G * 2, H_kv=2, D=D, num_blocks=2200 // bs + 16, dtype=dtype,
                       pad_multiple=64, block_size=bs)
    dw = DeviceWorkload(wl)
    B.pa_reshape_and_cache(dw.k_new, dw.v_new, dw.k_cache, dw.v_cache, dw.slot_mapping)
    out = W.as_f64(_prefill(dw))
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                           query_start_loc=wl.query_start_loc)
    assert_close(out, ref, dtype, f"prefill bs{bs} {dtype} D{D} G{G}")


@pytest.mark.parametrize("bs", SIZES)
def test_prefill_reblocked_is_bit_identical(bs):
    wl = W.build_mixed(360 + bs, prior_lens=[5, 250], chunk_lens=[300, 77], decode_lens=[3], H_q=8, H_kv=2, D=128,
                       num_blocks=700 // bs + 8, dtype="bf16", pad_multiple=0, block_size=bs)
    kc, vc = DeviceWorkload(wl).host_pool_after_writes()
    wl.k_cache, wl.v_cache, wl.slot_mapping = kc, vc, None
    a = _prefill(DeviceWorkload(wl))
    k16, bt16 = _repack(kc, wl.block_table_prefill, wl.seq_lens_prefill, 16)
    v16, _ = _repack(vc, wl.block_table_prefill, wl.seq_lens_prefill, 16)
    wl.k_cache, wl.v_cache, wl.block_table_prefill, wl.num_blocks = k16, v16, bt16, k16.shape[0]
    b = _prefill(DeviceWorkload(wl))
    assert np.array_equal(a, b)


# ----------------------------------------------------------------------------- copy_blocks

@pytest.mark.parametrize("bs", SIZES)
def test_copy_blocks_bit_exact(bs):
    rng = np.random.default_rng(370 + bs)
    shape = (12, 2, bs, 128)
    k = W.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    kd, vd = to_dev(k), to_dev(v)
    pairs = np.array([[3, 7], [5, 5], [11, 1]], dtype=np.int32)
    B.pa_copy_blocks(kd, vd, to_dev(pairs))
    torch.cuda.synchronize()
    for s, d in pairs:
        k[d], v[d] = k[s], v[s]
    assert np.array_equal(to_host_bits(kd), k) and np.array_equal(to_host_bits(vd), v)
    assert to_f64(kd).shape == shape
