"""GPU parity of the whole-step entry point pa_step (reshape_and_cache, then chunked prefill
and decode side by side on an SM split) against the fp64 oracle, plus its scheduling cases:
SM shares from 1 to beyond the device, missing parts, the general (sequential) decode path,
graph capture and the timing events."""
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


def _mixed(seed, dtype="bf16", D=128, G=4, H_kv=2, bs=16, n_dec=40, n_pre=5):
    rng = np.random.default_rng(seed)
    prior = rng.integers(0, 600, size=n_pre)
    chunk = rng.integers(1, 300, size=n_pre)
    dec = rng.integers(1, 1500, size=n_dec)
    need = int(np.sum(-(-(prior + chunk) // bs)) + np.sum(-(-dec // bs))) + 2
    return W.build_mixed(seed, prior_lens=prior, chunk_lens=chunk, decode_lens=dec, H_q=G * H_kv, H_kv=H_kv, D=D,
                         num_blocks=need, dtype=dtype, pad_multiple=64, block_size=bs)


def _step(dw, decode=True, prefill=True, new=True, decode_sms=0, events=None, stream=None):
    wl = dw.wl
    kw = dict(decode_sms=decode_sms, timing_events=events, stream=stream)
    if new:
        kw.update(k_new=dw.k_new, v_new=dw.v_new, slot_mapping=dw.slot_mapping)
    if prefill:
        kw.update(prefill_out=dw.out_prefill, prefill_q=dw.q_prefill, prefill_block_table=dw.block_table_prefill,
                  prefill_seq_lens=dw.seq_lens_prefill, query_start_loc=dw.query_start_loc,
                  max_chunk_len=int(np.diff(wl.query_start_loc).max()),
                  prefill_max_seq_len=int(wl.seq_lens_prefill.max()))
    if decode:
        msl = int(wl.seq_lens.max())
        ws = torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, dw.tdtype)),
                         dtype=torch.uint8, device="cuda")
        dw.ws = ws
        kw.update(decode_out=dw.out, decode_q=dw.q, decode_block_table=dw.block_table, decode_seq_lens=dw.seq_lens,
                  decode_max_seq_len=msl, workspace=ws)
    B.pa_step(dw.k_cache, dw.v_cache, wl.scale, **kw)


def _check(dw, decode=True, prefill=True, what=""):
    wl = dw.wl
    torch.cuda.synchronize()
    kc, vc = dw.host_pool_after_writes()
    if prefill:
        ref = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                               query_start_loc=wl.query_start_loc)
        assert_close(to_f64(dw.out_prefill), ref, wl.dtype, f"{what} prefill")
    if decode:
        ref = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
        assert_close(to_f64(dw.out), ref, wl.dtype, f"{what} decode")


@pytest.mark.parametrize("decode_sms", [0, 1, 7, 76, 151, 152, 1000])
def test_step_side_by_side_matches_oracle(decode_sms):
    dw = DeviceWorkload(_mixed(500))
    _step(dw, decode_sms=decode_sms)
    _check(dw, what=f"decode_sms {decode_sms}")


def test_step_prefill_bit_identical_to_separate_calls():
    wl = _mixed(501)
    dw = DeviceWorkload(wl)
    _step(dw)
    torch.cuda.synchronize()
    a = to_host_bits(dw.out_prefill)
    B.pa_prefill_chunk(dw.out_prefill, dw.q_prefill, dw.k_cache, dw.v_cache, dw.block_table_prefill,
                       dw.seq_lens_prefill, dw.query_start_loc, int(np.diff(wl.query_start_loc).max()),
                       int(wl.seq_lens_prefill.max()), wl.scale)
    torch.cuda.synchronize()
    assert np.array_equal(a, to_host_bits(dw.out_prefill))
    _check(dw, what="bit identity")


@pytest.mark.parametrize("parts", [(True, False, True), (False, True, True), (True, True, False),
                                   (False, False, True), (True, False, False), (False, True, False)])
def test_step_with_missing_parts(parts):
    dec, pre, new = parts
    wl = _mixed(502)
    if not new:  # the pool already holds the new tokens
        kc, vc = DeviceWorkload(wl).host_pool_after_writes()
        wl.k_cache, wl.v_cache = kc, vc
    dw = DeviceWorkload(wl)
    _step(dw, decode=dec, prefill=pre, new=new)
    torch.cuda.synchronize()
    if new:
        kc, vc = dw.host_pool_after_writes()
        assert np.array_equal(to_host_bits(dw.k_cache)[1:], kc[1:])
    _check(dw, decode=dec, prefill=pre, what=f"parts {parts}")


@pytest.mark.parametrize("dtype,D,G", [("f32", 64, 4), ("bf16", 128, 2), ("bf16", 64, 8)])
def test_step_general_paths(dtype, D, G):
    """fp32 and group 2 decode take the SIMT path (sequential in the step); head_dim 64 prefill
    takes the SIMT prefill beside the balanced decode."""
    dw = DeviceWorkload(_mixed(503 + G, dtype=dtype, D=D, G=G, n_dec=12, n_pre=3))
    _step(dw)
    _check(dw, what=f"{dtype} D{D} G{G}")


@pytest.mark.parametrize("bs", [32, 128])
def test_step_block_sizes(bs):
    dw = DeviceWorkload(_mixed(510 + bs, bs=bs))
    _step(dw, decode_sms=40)
    _check(dw, what=f"bs {bs}")


def test_step_in_a_cuda_graph_and_timing_events():
    wl = _mixed(520)
    dw = DeviceWorkload(wl)
    s = torch.cuda.Stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record(s)
    with torch.cuda.stream(s):
        _step(dw, stream=s, events=evs)  # eager first call, with events
    torch.cuda.synchronize()
    times = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(3)]
    assert all(t > 0 for t in times), times
    eager_dec, eager_pre = to_host_bits(dw.out), to_host_bits(dw.out_prefill)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(dw, stream=s)
    dw.out.zero_()
    dw.out_prefill.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(dw.out_prefill), eager_pre)
    assert np.array_equal(to_host_bits(dw.out), eager_dec)  # same split, same bits
    _check(dw, what="graph replay")


@pytest.mark.slow
def test_full_mixed_step_through_pa_step_all_rows():
    """The mixed-step workload at full size, in the launch configuration the benchmark times
    (pa_step: the slot writes, then prefill beside decode on its default SM split, where decode
    runs on a capped grid): all 240 decode rows and all 8192 prefill rows against the oracle,
    element by element, and the pool bit-exact."""
    wl, kc, vc, ref_dec, ref_pre = mixed_step_reference()
    dw = DeviceWorkload(wl)
    _step(dw)
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(dw.k_cache)[1:], kc[1:])
    assert np.array_equal(to_host_bits(dw.v_cache)[1:], vc[1:])
    assert_close(to_f64(dw.out), ref_dec, "bf16", "pa_step, every decode row")
    assert_close(to_f64(dw.out_prefill), ref_pre, "bf16", "pa_step, every prefill row")
