"""GPU parity of pa_decode_shared_prefix (the prefix that every sequence aliases attended once per
kv head on the tensor cores, each suffix by the balanced decode kernel, the parts merged by the
log-sum-exp rule) against the fp64 oracle, which attends every sequence over all of its keys."""
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
    B.pa_get_device_errors(clear=True)


def _run(wl, prefix, ws=None):
    dw = DeviceWorkload(wl)
    msl = int(wl.seq_lens.max())
    if ws is None:
        n = B.pa_decode_shared_prefix_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, prefix)
        assert n > 0
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dw.out.fill_(float("nan"))
    B.pa_decode_shared_prefix(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale,
                              prefix, ws)
    torch.cuda.synchronize()
    return dw, ws


def _ref(wl):
    return oracle.attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.scale)


def test_prefix_sharing_workload_matches_oracle():
    """128 sequences whose first 1024 tokens alias the same 64 blocks, suffixes U{0..512}."""
    wl = W.prefix_sharing()
    dw, _ = _run(wl, 1024)
    assert B.pa_get_device_errors(clear=True) == 0
    assert_close(to_f64(dw.out), _ref(wl), "bf16", "shared-prefix decode, prefix-sharing batch")


@pytest.mark.parametrize("G", [4, 8, 16])
@pytest.mark.parametrize("prefix", [16, 272, 1024])
def test_ragged_suffixes_and_groups(G, prefix):
    """Suffixes of 0, 1, 15, 16, 17 and a few hundred keys (0: the output is the prefix part
    alone), prefixes that are one block, not a whole number of 128-key tiles, and eight tiles."""
    H_kv = 8 if G <= 8 else 2
    lens = prefix + np.array([0, 1, 15, 16, 17, 300, 2, 511, 0, 64])
    need = prefix // 16 + int(np.sum(-(-(lens - prefix) // 16))) + 2
    wl = W.build_decode(600 + G + prefix, lens, H_q=G * H_kv, H_kv=H_kv, D=128, num_blocks=need, dtype="bf16",
                        new_token=False, shared_prefix_tokens=prefix)
    dw, _ = _run(wl, prefix)
    assert B.pa_get_device_errors(clear=True) == 0
    assert_close(to_f64(dw.out), _ref(wl), "bf16", f"shared prefix {prefix}, G {G}")


def test_workspace_reuse_gives_identical_results():
    lens = 512 + np.arange(0, 40 * 37, 37) % 700
    need = 32 + int(np.sum(-(-(lens - 512) // 16))) + 2
    wl = W.build_decode(650, lens, H_q=32, H_kv=8, D=128, num_blocks=need, dtype="bf16", new_token=False,
                        shared_prefix_tokens=512)
    dw, ws = _run(wl, 512)
    first = to_host_bits(dw.out).copy()
    for _ in range(3):
        dw2, _ = _run(wl, 512, ws)
        assert np.array_equal(to_host_bits(dw2.out), first)
    assert B.pa_get_device_errors(clear=True) == 0
    assert_close(to_f64(dw.out), _ref(wl), "bf16", "workspace reuse")


def test_ready_flags_give_the_same_bits():
    """With PA_DECODE_TABLES_READY / PA_DECODE_POOL_READY (the kernel before each call is the
    previous call's prefix kernel, which writes neither the tables nor the pool) the suffix
    decode starts earlier; the results are bit for bit those of the call without flags."""
    wl = W.prefix_sharing()
    dw, ws = _run(wl, 1024)
    plain = to_host_bits(dw.out).copy()
    msl = int(wl.seq_lens.max())
    for tables_ready, pool_ready in ((True, False), (False, True), (True, True)):
        dw.out.fill_(float("nan"))
        for _ in range(3):  # back to back: each call's kernels follow the previous call's
            B.pa_decode_shared_prefix(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl,
                                      wl.scale, 1024, ws, tables_ready=tables_ready, pool_ready=pool_ready)
        torch.cuda.synchronize()
        assert B.pa_get_device_errors(clear=True) == 0
        assert np.array_equal(to_host_bits(dw.out), plain), (tables_ready, pool_ready)
    assert_close(to_f64(dw.out), _ref(wl), "bf16", "shared-prefix decode with ready flags")


def test_a_row_with_other_prefix_blocks_is_flagged():
    """Row 3's second prefix block is replaced by a copy of it in another physical block: the
    values are the same, so the output still matches, but the table breaks the call's contract
    and the merge kernel's check raises PA_DEVERR_PREFIX_MISMATCH."""
    lens = np.array([300, 290, 400, 350])
    need = 16 + int(np.sum(-(-(lens - 256) // 16))) + 3
    wl = W.build_decode(660, lens, H_q=32, H_kv=8, D=128, num_blocks=need, dtype="bf16", new_token=False,
                        shared_prefix_tokens=256)
    spare = min(set(range(1, need)) - set(wl.block_table.ravel().tolist()))
    old = int(wl.block_table[3, 1])
    wl.k_cache[spare] = wl.k_cache[old]
    wl.v_cache[spare] = wl.v_cache[old]
    wl.block_table[3, 1] = spare
    dw, _ = _run(wl, 256)
    assert B.pa_get_device_errors(clear=True) == B.PA_DEVERR_PREFIX_MISMATCH
    assert_close(to_f64(dw.out), _ref(wl), "bf16", "copied prefix block")


@pytest.mark.parametrize("S", [1, 3])
def test_every_suffix_empty(S):
    """Every sequence is exactly the shared prefix: the output is the prefix part alone."""
    lens = np.full(S, 384)
    wl = W.build_decode(680 + S, lens, H_q=32, H_kv=8, D=128, num_blocks=24 + 2, dtype="bf16", new_token=False,
                        shared_prefix_tokens=384)
    dw, _ = _run(wl, 384)
    assert B.pa_get_device_errors(clear=True) == 0
    assert_close(to_f64(dw.out), _ref(wl), "bf16", f"empty suffixes, S {S}")


def test_length_shorter_than_the_prefix_is_flagged():
    """A sequence shorter than prefix_tokens breaks the call's contract: PA_DEVERR_LEN_RANGE."""
    lens = np.array([300, 290, 400])
    need = 16 + int(np.sum(-(-(lens - 256) // 16))) + 2
    wl = W.build_decode(690, lens, H_q=32, H_kv=8, D=128, num_blocks=need, dtype="bf16", new_token=False,
                        shared_prefix_tokens=256)
    dw = DeviceWorkload(wl)
    msl = int(lens.max())
    ws = torch.zeros(B.pa_decode_shared_prefix_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, 256),
                     dtype=torch.uint8, device="cuda")
    dw.seq_lens[1] = 200  # below the prefix
    B.pa_decode_shared_prefix(dw.out, dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.seq_lens, msl, wl.scale, 256,
                              ws)
    torch.cuda.synchronize()
    assert B.pa_get_device_errors(clear=True) & B.PA_DEVERR_LEN_RANGE
