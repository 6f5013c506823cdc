"""Shared helpers for the GPU parity tests: moving generator arrays to the device, running the
CUDA path through the binding, and the tolerance check of the attention outputs.

Tolerances (written here once, used by every parity test):
  * fp32: max |gpu - oracle| <= 1e-5 (no TF32 anywhere on the fp32 path);
  * bf16: |gpu - oracle| <= 2e-2 + 1e-2 * |oracle| elementwise, the oracle computed in fp64
    from the same bf16-rounded Q/K/V and the GPU output widened to fp64;
  * reshape_and_cache: bit-exact on every block except the null block 0.
"""
from __future__ import annotations

import functools

import numpy as np

from paged_kv_cache_238_gb300 import workloads as W

FP32_ATOL = 1e-5
BF16_ATOL = 2e-2
BF16_RTOL = 1e-2


def to_dev(a: np.ndarray, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_bits(t) -> np.ndarray:
    """Device tensor -> numpy with the generator's storage types (bf16 as uint16 bits)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def to_f64(t) -> np.ndarray:
    return W.as_f64(to_host_bits(t))


def assert_close(gpu: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> None:
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    if dtype == "f32":
        worst = float(err.max()) if err.size else 0.0
        assert worst <= FP32_ATOL, f"{what}: max abs error {worst:.3e} > {FP32_ATOL}"
    else:
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
        bad = err > bound
        if bad.any():
            i = np.unravel_index(np.argmax(err - bound), err.shape)
            raise AssertionError(f"{what}: {int(bad.sum())} elements outside 2e-2 + 1e-2|ref|; worst at {i}: "
                                 f"gpu {gpu[i]:.6f} ref {ref[i]:.6f}")


class DeviceWorkload:
    """A generator workload copied to the GPU (pool, tables, queries, new tokens)."""

    def __init__(self, wl: W.Workload, device="cuda"):
        import torch
        self.wl = wl
        self.k_cache = to_dev(wl.k_cache, device)
        self.v_cache = to_dev(wl.v_cache, device)
        self.tdtype = self.k_cache.dtype
        if wl.q is not None:
            self.q = to_dev(wl.q, device)
            self.block_table = to_dev(wl.block_table, device)
            self.seq_lens = to_dev(wl.seq_lens, device)
            self.out = torch.empty_like(self.q)
        if wl.q_prefill is not None:
            self.q_prefill = to_dev(wl.q_prefill, device)
            self.block_table_prefill = to_dev(wl.block_table_prefill, device)
            self.seq_lens_prefill = to_dev(wl.seq_lens_prefill, device)
            self.query_start_loc = to_dev(wl.query_start_loc, device)
            self.out_prefill = torch.empty_like(self.q_prefill)
        if wl.slot_mapping is not None:
            self.k_new = to_dev(wl.k_new, device)
            self.v_new = to_dev(wl.v_new, device)
            self.slot_mapping = to_dev(wl.slot_mapping, device)

    def host_pool_after_writes(self):
        """Oracle-side pool: generator pool plus the new tokens written by the oracle."""
        import oracle
        kc, vc = self.wl.k_cache.copy(), self.wl.v_cache.copy()
        if self.wl.slot_mapping is not None:
            oracle.reshape_and_cache(self.wl.k_new, self.wl.v_new, kc, vc, self.wl.slot_mapping)
        return kc, vc


@functools.lru_cache(maxsize=1)
def mixed_step_reference():
    """Oracle results for the whole mixed-step workload, computed once per test session:
    (pool K, pool V after the step's slot writes, every decode row's output, every prefill
    row's output). Both attentions see the pool after all of the step's writes, as the step
    runs them (the writes come first)."""
    import oracle
    wl = W.mixed_step()
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    ref_dec = oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    ref_pre = oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                               query_start_loc=wl.query_start_loc)
    return wl, kc, vc, ref_dec, ref_pre
