"""CPU checks of the benchmark's host-side logic: the algorithmic bytes and flops it divides by,
the packing of a step's inputs into one buffer per direction, the traffic record's source check
and the single-rank reductions. No device calls."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
from paged_kv_cache_238_gb300 import workloads as W  # noqa: E402


def test_step_bytes_of_a_small_decode_batch_by_hand():
    wl = W.build_decode(900, [1, 16, 17, 40], H_q=8, H_kv=2, D=64, num_blocks=16, dtype="bf16")
    b = bench.step_bytes(wl)
    tok = 2 * 2 * 64 * 2                       # K and V of one token: 2 x H_kv x D x 2 bytes
    keys = 1 + 16 + 17 + 40
    pages = 1 + 1 + 2 + 3                       # ceil(len / 16) block-table entries
    q = 4 * 8 * 64 * 2
    assert b["kv"] == keys * tok
    assert b["decode"] == keys * tok + 2 * q + 4 * pages + 4 * 4
    assert b["reshape"] == 2 * 4 * tok + 8 * 4  # new K/V read and written, plus int64 slots
    assert b["step"] == b["decode"] + b["reshape"]


def test_prefill_flops_count_visible_pairs_only():
    wl = W.build_mixed(901, prior_lens=[0, 10], chunk_lens=[4, 3], decode_lens=[], H_q=4, H_kv=2, D=8,
                       num_blocks=8, dtype="bf16", pad_multiple=0)
    # chunk rows see prior + own causal prefix: (0*4 + 1+2+3+4) + (10*3 + 1+2+3)
    pairs = (1 + 2 + 3 + 4) + (30 + 6)
    assert bench.step_bytes(wl)["prefill_flops"] == 4 * 8 * 4 * pairs


def test_shared_prefix_blocks_count_once_in_the_distinct_bytes():
    wl = W.build_decode(902, [40, 40, 40], H_q=4, H_kv=1, D=8, num_blocks=16, dtype="bf16", new_token=False,
                        shared_prefix_tokens=32)
    b = bench.step_bytes(wl)
    tok = 2 * 1 * 8 * 2
    assert b["kv"] == 120 * tok
    assert b["kv_unique"] == (32 + 3 * 8) * tok  # two shared blocks once, three private tails
    # the decode bytes (value and roofline) count the distinct keys; the logical figure each
    # sequence's keys
    q = 3 * 4 * 8 * 2
    rest = 2 * q + 4 * 3 * 3 + 4 * 3            # Q and output, 3 table entries per row, lengths
    assert b["decode"] == b["kv_unique"] + rest
    assert b["decode_logical"] == b["kv"] + rest


def test_step_inputs_are_packed_and_a_second_buffer_set_mirrors_them():
    wl = W.build_decode(903, [5, 33, 17], H_q=8, H_kv=2, D=64, num_blocks=16, dtype="bf16")
    st = bench.DeviceStep(wl, torch.device("cpu"), 1, None, fuse_append=True)
    assert st.fused_append and st.kernels == ["decode"]
    for t in st.inputs:                      # every input is a view of the one input buffer
        off = t.data_ptr() - st.in_arena.data_ptr()
        assert 0 <= off and off % 256 == 0 and off + t.numel() * t.element_size() <= st.in_arena.numel()
    assert np.array_equal(st.bt.numpy(), wl.block_table)
    assert np.array_equal(st.slots.numpy(), wl.slot_mapping)
    b = st.add_buffer()
    assert b == 1
    assert torch.equal(st.in_arenas[1], st.in_arena)
    for n in st.in_names + st.out_names:
        t0, t1 = st.bufs[0][n], st.bufs[1][n]
        assert t1.shape == t0.shape and t1.dtype == t0.dtype
        assert t1.data_ptr() - st.in_arenas[1].data_ptr() == t0.data_ptr() - st.in_arena.data_ptr() or \
            t1.data_ptr() - st.out_arenas[1].data_ptr() == t0.data_ptr() - st.out_arena.data_ptr()


def test_traffic_record_is_dropped_when_the_kernel_source_changes(monkeypatch):
    rec = bench.recorded_traffic("decode", "gqa_decode")
    if rec is None:
        pytest.skip("no record for the current decode source")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="decode": "0" * 16)
    assert bench.recorded_traffic("decode", "gqa_decode") is None


def test_single_rank_reductions_are_identities():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_rate(1000.0, 1, 0.5) == 2000.0
