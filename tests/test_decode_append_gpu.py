"""GPU parity of pa_decode_append (a decode step with its new tokens: the K/V write of each
sequence's token at position seq_lens[i] - 1 and decode attention, in one launch on the bf16
persistent path) against the fp64 oracle, which runs reshape_and_cache and then attention."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from paged_kv_cache_238_gb300 import binding as B  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402

from helpers import DeviceWorkload, assert_close, to_f64, to_host_bits  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    B.pa_get_device_errors(clear=True)
    yield
    assert B.pa_get_device_errors(clear=True) == 0, "a kernel raised a device error"


def _ws(wl, dw, msl):
    return torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, dw.tdtype)),
                       dtype=torch.uint8, device="cuda")


def _append(dw, msl=None):
    wl = dw.wl
    msl = int(wl.seq_lens.max()) if msl is None else msl
    B.pa_decode_append(dw.out, dw.q, dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache, dw.block_table,
                       dw.seq_lens, msl, wl.scale, _ws(wl, dw, msl))
    torch.cuda.synchronize()


def _check(dw, what):
    wl = dw.wl
    kc, vc = dw.host_pool_after_writes()
    raw = (lambda a: a.view(np.uint32)) if kc.dtype == np.float32 else (lambda a: a)
    assert np.array_equal(raw(to_host_bits(dw.k_cache)[1:]), raw(kc[1:])), f"{what}: k pool"
    assert np.array_equal(raw(to_host_bits(dw.v_cache)[1:]), raw(vc[1:])), f"{what}: v pool"
    ref = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(to_f64(dw.out), ref, wl.dtype, what)


LENS = [1, 2, 15, 16, 17, 31, 32, 33, 200, 1000, 2049]


@pytest.mark.parametrize("dtype,D,G,H_kv", [("bf16", 128, 4, 2), ("bf16", 128, 8, 2), ("bf16", 128, 16, 1),
                                            ("bf16", 64, 4, 2), ("bf16", 64, 12, 1), ("f32", 128, 4, 2),
                                            ("bf16", 128, 2, 4)])
@pytest.mark.parametrize("bs", [16, 32, 128])
def test_decode_append_matches_oracle(dtype, D, G, H_kv, bs):
    """bf16 groups 4..16 take the fused kernel (3-D boxes at head_dim 128, 2-D at 64); fp32 and
    group 2 launch reshape_and_cache and the SIMT decode."""
    need = sum(-(-L // bs) for L in LENS) + 2
    wl = W.build_decode(600 + G + bs, LENS, H_q=G * H_kv, H_kv=H_kv, D=D, num_blocks=need, dtype=dtype,
                        block_size=bs)
    dw = DeviceWorkload(wl)
    _append(dw)
    _check(dw, f"append {dtype} D{D} G{G} bs{bs}")


def test_decode_append_bit_identical_to_reshape_then_decode():
    wl = W.gqa_decode(seed=1002)
    a = DeviceWorkload(wl)
    _append(a)
    b = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    B.pa_reshape_and_cache(b.k_new, b.v_new, b.k_cache, b.v_cache, b.slot_mapping)
    B.pa_decode(b.out, b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, msl, wl.scale, _ws(wl, b, msl))
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(a.out), to_host_bits(b.out))
    assert np.array_equal(to_host_bits(a.k_cache)[1:], to_host_bits(b.k_cache)[1:])
    _check(a, "gqa decode batch")


def test_decode_append_many_sequences_and_repeated_calls():
    """300 sequences (several segments per warp, CTA-crossing segments) and the workspace reused
    across calls, each call appending the next token."""
    rng = np.random.default_rng(610)
    lens = rng.integers(1, 700, size=300)
    wl = W.build_decode(610, lens + 1, H_q=32, H_kv=8, D=128, num_blocks=int(np.sum(-(-(lens + 1) // 16))) + 2,
                        dtype="bf16", keep_contiguous=True)
    dw = DeviceWorkload(wl)
    _append(dw)
    _check(dw, "300 sequences")
    _append(dw)  # same token again: same pool, same result
    _check(dw, "second call")


def test_decode_append_slot_that_is_not_the_last_position_is_flagged():
    wl = W.build_decode(620, [20, 40, 7], H_q=8, H_kv=2, D=128, num_blocks=16, dtype="bf16")
    good = wl.slot_mapping.copy()
    dw = DeviceWorkload(wl)
    dw.slot_mapping[1] = -1                   # no write for sequence 1
    _append(dw)
    assert B.pa_get_device_errors(clear=True) == B.PA_DEVERR_APPEND_SLOT
    # attention still used the new rows at position len - 1: equal to the well-formed call
    ok = DeviceWorkload(wl)
    ok.slot_mapping.copy_(torch.from_numpy(good).cuda())
    _append(ok)
    assert np.array_equal(to_host_bits(dw.out), to_host_bits(ok.out))
    # and the pool cell of sequence 1's new token was not written
    b, o = int(good[1]) // 16, int(good[1]) % 16
    assert np.isnan(to_f64(dw.k_cache)[b, :, o]).all()


def test_decode_append_zero_sequences_is_a_no_op():
    wl = W.build_decode(630, [5], H_q=8, H_kv=2, D=128, num_blocks=4, dtype="bf16")
    dw = DeviceWorkload(wl)
    B.pa_decode_append(dw.out[:0], dw.q[:0], dw.k_new[:0], dw.v_new[:0], dw.slot_mapping[:0], dw.k_cache,
                       dw.v_cache, dw.block_table[:0], dw.seq_lens[:0], 0, wl.scale, None)
    torch.cuda.synchronize()


@pytest.mark.parametrize("pool_ready", [False, True])
@pytest.mark.parametrize("G,H_kv", [(4, 8), (16, 2)])
def test_decode_append_tables_ready_back_to_back(G, H_kv, pool_ready):
    """PA_DECODE_TABLES_READY: the lengths scan and the first block ids are read before the
    grid-dependency wait (with PA_DECODE_POOL_READY the first page copies too). Ten calls back
    to back on one stream (each a programmatic dependent of the one before, all rewriting the
    same new rows, which no call reads from the pool, and reading the same tables and keys)
    give the bits of one call without the flags."""
    wl = W.gqa_decode(seed=640)
    wl = W.build_decode(641, wl.seq_lens, H_q=G * H_kv, H_kv=H_kv, D=128,
                        num_blocks=int(np.sum(-(-wl.seq_lens.astype(np.int64) // 16))) + 2, dtype="bf16")
    a = DeviceWorkload(wl)
    _append(a)
    ref_bits = to_host_bits(a.out)
    b = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    ws = _ws(wl, b, msl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(10):
            B.pa_decode_append(b.out, b.q, b.k_new, b.v_new, b.slot_mapping, b.k_cache, b.v_cache, b.block_table,
                               b.seq_lens, msl, wl.scale, ws, stream=s, tables_ready=True, pool_ready=pool_ready)
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(b.out), ref_bits)
    _check(b, f"tables ready G{G}" + (" pool ready" if pool_ready else ""))


@pytest.mark.slow
def test_long_split_kv_through_decode_append_as_benchmarked():
    """The long split-KV workload (8 x 32 768 keys, 64 q / 8 kv heads) through pa_decode_append
    with PA_DECODE_TABLES_READY, as the benchmark launches it: every row against the oracle and
    the pool bit-exact."""
    wl = W.long_split_kv()
    dw = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    B.pa_decode_append(dw.out, dw.q, dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache, dw.block_table,
                       dw.seq_lens, msl, wl.scale, _ws(wl, dw, msl), tables_ready=True)
    torch.cuda.synchronize()
    _check(dw, "long split-KV through pa_decode_append")
