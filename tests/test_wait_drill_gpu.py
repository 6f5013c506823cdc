"""The kernels' bounded waits, made to run out on purpose (pa_debug_set_wait_drill).

A drilled launch announces 16 bytes more on one barrier phase than its copies bring, so that
one wait can never be satisfied; nothing that the kernel would abandon is in flight. The wait
must give up after the (shortened) limit, raise PA_DEVERR_WAIT_TIMEOUT, let the issued copies
land and return, leaving the context usable: the same call without the drill, on the same
stream and buffers (the decode workspace zero-filled again, as pa.h asks), must then match the
oracle. No trap, fault or endless loop is involved."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from paged_kv_cache_238_gb300 import binding as B  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402

from helpers import DeviceWorkload, assert_close, to_f64  # noqa: E402

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # 2 ms instead of 1 s while a drill is on


@pytest.fixture(autouse=True)
def _drill_off_around_each_test():
    B.pa_debug_set_wait_drill(B.PA_DRILL_OFF)
    B.pa_get_device_errors(clear=True)
    yield
    B.pa_debug_set_wait_drill(B.PA_DRILL_OFF)
    B.pa_get_device_errors(clear=True)


def _drilled(kind, call):
    """Runs call() with the drill on; returns (device error bits, seconds until it finished)."""
    B.pa_debug_set_wait_drill(kind, LIMIT_NS)
    try:
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        B.pa_debug_set_wait_drill(B.PA_DRILL_OFF)
    return B.pa_get_device_errors(clear=True), dt


def _decode_setup(wl):
    dw = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    ws = torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, dw.tdtype)),
                     dtype=torch.uint8, device="cuda")
    return dw, msl, ws


def test_decode_wait_runs_out_and_the_next_call_matches_oracle():
    wl = W.build_decode(46, [300, 17, 64, 1000, 5, 2048], H_q=32, H_kv=8, D=128, num_blocks=400, dtype="bf16",
                        new_token=False)
    dw, msl, ws = _decode_setup(wl)

    def call():
        B.pa_decode(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale, ws)

    errs, dt = _drilled(B.PA_DRILL_DECODE_STAGE, call)
    assert errs & B.PA_DEVERR_WAIT_TIMEOUT, f"no timeout raised (errors {errs:#x})"
    assert dt < 0.5, f"the drilled call took {dt:.3f} s: the shortened limit was not used"
    ws.zero_()
    dw.out.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    assert B.pa_get_device_errors(clear=True) == 0
    ref = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(to_f64(dw.out), ref, "bf16", "decode after a drilled call")


@pytest.mark.parametrize("pool_ready", [False, True])
def test_decode_append_wait_runs_out_and_the_next_call_matches_oracle(pool_ready):
    """The benchmarked call: pa_decode_append on the GQA decode batch (64 sequences), with the
    first pages copied before the grid-dependency wait or after it."""
    wl = W.gqa_decode()
    dw, msl, ws = _decode_setup(wl)

    def call():
        B.pa_decode_append(dw.out, dw.q, dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache,
                           dw.block_table, dw.seq_lens, msl, wl.scale, ws, tables_ready=True,
                           pool_ready=pool_ready)

    errs, dt = _drilled(B.PA_DRILL_DECODE_STAGE, call)
    assert errs & B.PA_DEVERR_WAIT_TIMEOUT, f"no timeout raised (errors {errs:#x})"
    assert dt < 0.5
    ws.zero_()
    dw.out.fill_(float("nan"))
    call()  # writes the new tokens again (same values) and attends
    torch.cuda.synchronize()
    assert B.pa_get_device_errors(clear=True) == 0
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(to_f64(dw.out), ref, "bf16", "decode_append after a drilled call")


def test_prefill_wait_runs_out_and_the_next_call_matches_oracle():
    """Tensor-core prefill (G = 4, head_dim 128): the MMA warp's wait on the first K tile runs
    out; the CTA's warps wind down, free their tensor memory and return."""
    rng = np.random.default_rng(77)
    prior = rng.integers(0, 600, size=5)
    chunk = rng.integers(1, 300, size=5)
    need = int(np.sum(-(-(prior + chunk) // 16))) + 2
    wl = W.build_mixed(77, prior_lens=prior, chunk_lens=chunk, decode_lens=[], H_q=16, H_kv=4, D=128,
                       num_blocks=need, dtype="bf16", pad_multiple=64)
    dw = DeviceWorkload(wl)
    B.pa_reshape_and_cache(dw.k_new, dw.v_new, dw.k_cache, dw.v_cache, dw.slot_mapping)
    qsl = wl.query_start_loc
    max_chunk = int(np.max(np.diff(qsl)))

    def call():
        B.pa_prefill_chunk(dw.out_prefill, dw.q_prefill, dw.k_cache, dw.v_cache, dw.block_table_prefill,
                           dw.seq_lens_prefill, dw.query_start_loc, max_chunk, int(wl.seq_lens_prefill.max()),
                           wl.scale)

    errs, dt = _drilled(B.PA_DRILL_PREFILL_K_TILE, call)
    assert errs & B.PA_DEVERR_WAIT_TIMEOUT, f"no timeout raised (errors {errs:#x})"
    assert dt < 0.5
    dw.out_prefill.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    assert B.pa_get_device_errors(clear=True) == 0
    kc, vc = dw.host_pool_after_writes()
    ref = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                           query_start_loc=qsl)
    assert_close(to_f64(dw.out_prefill), ref, "bf16", "prefill after a drilled call")


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_shared_prefix_wait_runs_out_and_the_next_call_matches_oracle(kind):
    """pa_decode_shared_prefix runs both kernels: the drill stops one wait of the suffix decode
    or of the prefix kernel that runs beside it; the next call matches the oracle."""
    lens = 256 + np.array([0, 5, 40, 300, 17, 96])
    need = 16 + int(np.sum(-(-(lens - 256) // 16))) + 2
    wl = W.build_decode(670, lens, H_q=32, H_kv=8, D=128, num_blocks=need, dtype="bf16", new_token=False,
                        shared_prefix_tokens=256)
    dw = DeviceWorkload(wl)
    msl = int(lens.max())
    ws = torch.zeros(B.pa_decode_shared_prefix_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, 256),
                     dtype=torch.uint8, device="cuda")

    def call():
        B.pa_decode_shared_prefix(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale,
                                  256, ws)

    drill = B.PA_DRILL_DECODE_STAGE if kind == "decode" else B.PA_DRILL_PREFILL_K_TILE
    errs, dt = _drilled(drill, call)
    assert errs & B.PA_DEVERR_WAIT_TIMEOUT, f"no timeout raised (errors {errs:#x})"
    assert dt < 0.5
    ws.zero_()
    dw.out.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    assert B.pa_get_device_errors(clear=True) == 0
    ref = oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)
    assert_close(to_f64(dw.out), ref, "bf16", f"shared prefix after a drilled {kind} wait")
