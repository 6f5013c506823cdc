"""pa_decode_noalloc: the decode entry point for callers that cannot allocate device memory
(a host framework that owns the device-memory budget, a plug-in without an allocator, or a
path that must avoid cudaMalloc/cudaFree because they can synchronise the device). It uses
the library's fixed device scratch instead of a caller workspace.

Kept in its own file, collected last, so that a run stopping at the first failure has run
every other test first. Each case compares the no-allocation entry point with pa_decode on
the same inputs, on two calls in a row, within the parity tolerances of tests/helpers.py.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_cache_238_gb300 import binding as B  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402

from helpers import DeviceWorkload, assert_close, to_f64  # noqa: E402

pytestmark = pytest.mark.gpu


def _noalloc_call(dw, msl):
    """Through the C ABI directly: out, q, pool, tables, sizes, scale, dtype, stream."""
    wl = dw.wl
    lib = B.load()
    st = lib.pa_decode_noalloc(dw.out.data_ptr(), dw.q.data_ptr(), dw.k_cache.data_ptr(), dw.v_cache.data_ptr(),
                               dw.block_table.data_ptr(), dw.block_table.shape[1], dw.seq_lens.data_ptr(), wl.S,
                               msl, wl.H_q, wl.H_kv, wl.D, wl.num_blocks, ctypes.c_float(wl.scale),
                               B.PA_BF16 if wl.dtype == "bf16" else B.PA_F32,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.PA_OK, B.status_string(st)
    torch.cuda.synchronize()
    return to_f64(dw.out)


def _with_workspace(dw, msl):
    wl = dw.wl
    ws = torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, dw.tdtype)),
                     dtype=torch.uint8, device="cuda")
    B.pa_decode(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale, ws)
    torch.cuda.synchronize()
    return to_f64(dw.out)


@pytest.mark.parametrize("make", [
    lambda: W.gqa_decode(),                                                      # bf16, in-kernel split merge
    lambda: W.build_decode(90, [1, 15, 16, 33, 700], H_q=4, H_kv=4, D=64,
                           num_blocks=64, dtype="f32"),                          # fp32, separate reduce kernel
    lambda: W.build_decode(91, [4000, 3, 1200], H_q=64, H_kv=8, D=128,
                           num_blocks=400, dtype="bf16"),                        # long, many cut segments
], ids=["gqa_bs64_bf16", "tiny_fp32_split", "long_gqa8"])
def test_noalloc_matches_pa_decode_on_two_calls(make):
    wl = make()
    if wl.slot_mapping is not None:  # the new tokens are part of the keys
        import oracle
        oracle.reshape_and_cache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    dw = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    ref = _with_workspace(dw, msl)
    for _ in range(2):
        dw.out.fill_(float("nan"))
        got = _noalloc_call(dw, msl)
        assert_close(got, ref, wl.dtype, "pa_decode_noalloc vs pa_decode")
    assert B.pa_get_device_errors(clear=True) == 0


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch():
    # one merge counter per (sequence, kv head): 1024 x 8192 of them need 32 MiB of scratch
    S, H_kv, D, msl = 1024, 8192, 64, 256
    H_q = 4 * H_kv
    assert B.pa_decode_workspace_size(S, H_q, H_kv, D, msl, torch.bfloat16) > B.PA_DECODE_NOALLOC_MAX_BYTES
    lib = B.load()
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    st = lib.pa_decode_noalloc(p, p, p, p, p, msl // 16, p, S, msl, H_q, H_kv, D, 1024, ctypes.c_float(0.1),
                               B.PA_BF16, None)
    assert st == B.PA_ERR_UNSUPPORTED


def test_noalloc_general_path_then_grouped_path_matches_oracle():
    """The scratch keeps what the previous call left: an fp32 call (the general path writes
    plain partial results all over it) followed by a bf16 grouped call, whose cross-CTA merges
    count finished pieces in the scratch's leading words, must still give the oracle's result,
    because each call clears those counters before launching."""
    import oracle
    first = W.build_decode(92, [2048, 1500, 3000, 77], H_q=8, H_kv=8, D=128, num_blocks=500, dtype="f32",
                           new_token=False)
    d1 = DeviceWorkload(first)
    _noalloc_call(d1, int(first.seq_lens.max()))
    second = W.build_decode(93, [900, 1300, 40, 2600, 5, 610], H_q=32, H_kv=8, D=128, num_blocks=800,
                            dtype="bf16", new_token=False)
    d2 = DeviceWorkload(second)
    got = _noalloc_call(d2, int(second.seq_lens.max()))
    ref = oracle.attention(second.q, second.k_cache, second.v_cache, second.block_table, second.seq_lens,
                           second.scale)
    assert_close(got, ref, "bf16", "grouped call after a general-path call")
    assert B.pa_get_device_errors(clear=True) == 0
