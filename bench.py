"""Benchmark of the paged-KV decode step on GB300.

One step = the whole hot path on one batch: reshape_and_cache of the batch's new tokens
(one per sequence) followed by paged decode attention over all of their keys, for the GQA
decode batch of 64 sequences (32 q / 8 kv heads, head_dim 128, bf16, lognormal context
lengths with mean ~195, 16-token blocks, shuffled physical blocks).

Timing: the step's device inputs stay resident; steps rotate through R independent KV pools
(one per "layer", the same block table), so a pool is touched again only after the other
R-1 (> 3 x L2 in between): inputs larger than L2, no flush kernel. K steps are captured in
CUDA graphs (a step is ~20 us, so launches matter) and timed with CUDA events on the launching
stream, barrier + synchronize on both sides, max over ranks. Every 50th step of a graph
brackets each of its kernels with an event pair; the roofline figure uses their average.

value  = algorithmic bytes of the step / step time (TB/s): KV bytes of every visible key,
         Q, output, block-table entries, lengths, and the new tokens' K/V read and written.
e2e    = the same metric with every step's inputs copied host->device from pinned memory and
         its output copied back, inside the timed graph.
--impl reference  times the fp64 CPU oracle (test infrastructure) on a bounded sample of the
         same workload and prints the same line with "impl": "reference".
--workload  measures another workload of the same path instead of the GQA decode batch:
         prefix_sharing (aliased prefix blocks), long_split_kv (8 x 32768 tokens) or
         mixed_step (reshape_and_cache of 8448 slots + chunked prefill + 240-sequence decode;
         its line reports new tokens/s and, per kernel, the HBM or tensor-pipe roofline) or
         prefill_chunks (the mixed step's prefill half alone, in TFLOP/s).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-KV decode attention: achieved HBM TB/s vs peak; seqs/s (bs 64, GQA)"
WORKLOAD = "GQA decode bf16: 64 seqs, 32 q / 8 kv heads, head_dim 128, block 16, lognormal lengths (mean ~195, " \
           "clipped 16-2048), shuffled physical blocks, 4096-block pool, reshape_and_cache of 1 new token per seq"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------------------------------
# workloads and their algorithmic work (per step)
# ------------------------------------------------------------------------------------------

#: name -> (builder in workloads: name or (name, kwargs), description, default steps, KV replicas rotated)
WORKLOADS = {
    "gqa_decode": ("gqa_decode", WORKLOAD, 20000, 10),
    "prefix_sharing": ("prefix_sharing",
                       "Prefix-sharing decode bf16: 128 seqs, first 1024 tokens alias the same 64 physical blocks, "
                       "unique suffix U{0..512}, 32 q / 8 kv heads, head_dim 128, block 16, 8192-block pool", 5000, 3),
    "long_split_kv": ("long_split_kv",
                      "Long-context split-KV decode bf16: 8 seqs x 32768 tokens, 64 q / 8 kv heads, head_dim 128, "
                      "block 16, 20000-block pool, one new token per seq", 2000, 1),
    "mixed_step": ("mixed_step",
                   "Mixed step bf16: 16 chunked-prefill seqs of 512 new tokens on prior context U{0..4096} + 240 "
                   "decode seqs with context U{64..4096}, 32 q / 8 kv heads, head_dim 128, block 16, slot_mapping "
                   "for all new tokens padded to 8448 with padding slots in the null block", 300, 1),
    "prefill_chunks": (("mixed_step", {"n_decode": 0, "num_blocks": 0}),
                       "Chunked prefill bf16: the mixed step's 16 chunks of 512 new tokens on prior context "
                       "U{0..4096}, 32 q / 8 kv heads, head_dim 128, block 16, pool sized to those sequences", 300, 1),
}


def build_workload(name: str):
    from paged_kv_cache_238_gb300 import workloads as W
    builder = WORKLOADS[name][0]
    fn, kw = (builder, {}) if isinstance(builder, str) else builder
    return getattr(W, fn)(**kw)


def _kv_token_bytes(wl) -> int:
    el = 2 if wl.dtype == "bf16" else 4
    return 2 * wl.H_kv * wl.D * el


def step_bytes(wl) -> dict:
    """Algorithmic bytes of one step: every distinct visible key's K and V once (a prefix that
    several sequences alias counts once: it need leave HBM only once), Q and output, the
    block-table entries a kernel must read, lengths, and the new tokens' K/V read and written
    (plus their slots). Prefill flops count visible (query, key) pairs only. "decode_logical"
    counts each sequence's keys instead."""
    el = 2 if wl.dtype == "bf16" else 4
    tok = _kv_token_bytes(wl)
    res = {"decode": 0, "prefill": 0, "reshape": 0, "kv": 0, "prefill_flops": 0, "kv_unique": 0}
    if wl.seq_lens is not None and wl.S > 0:
        lens = wl.seq_lens.astype(np.int64)
        kv = int(lens.sum()) * tok
        q = wl.S * wl.H_q * wl.D * el
        bt = int(np.sum(-(-lens // 16))) * 4
        res["kv"] += kv
        # distinct (block, row) pairs actually holding visible keys: aliased prefixes count once
        seen = {}
        for i in range(wl.S):
            n = int(lens[i])
            for j in range(-(-n // 16)):
                b = int(wl.block_table[i, j])
                seen[b] = max(seen.get(b, 0), min(16, n - 16 * j))
        kv_u = sum(seen.values()) * tok
        res["kv_unique"] += kv_u
        res["decode"] = kv_u + 2 * q + bt + wl.S * 4
        res["decode_logical"] = kv + 2 * q + bt + wl.S * 4
    if wl.seq_lens_prefill is not None:
        L = wl.seq_lens_prefill.astype(np.int64)
        C = np.diff(wl.query_start_loc).astype(np.int64)
        kv = int(L.sum()) * tok
        Tp = int(C.sum())
        q = Tp * wl.H_q * wl.D * el
        bt = int(np.sum(-(-L // 16))) * 4
        res["prefill"] = kv + 2 * q + bt + 4 * (2 * len(L) + 1)
        res["kv"] += kv
        res["kv_unique"] += kv
        pairs = int(np.sum((L - C) * C + C * (C + 1) // 2))
        res["prefill_flops"] = 4 * wl.D * wl.H_q * pairs
    if wl.slot_mapping is not None:
        T = wl.slot_mapping.shape[0]
        new = T * tok                               # new K and V read ...
        res["reshape"] = 2 * new + 8 * T            # ... and written, plus the slots
    res["step"] = res["decode"] + res["prefill"] + res["reshape"]
    return res


def _peaks_file() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except Exception:
        return {}


def load_peaks() -> tuple:
    """HBM copy bandwidth (GB/s) measured on this GPU model, else the fallback figure."""
    p = _peaks_file()
    if "hbm_gbs" in p:
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak() -> tuple:
    """Dense bf16 tensor throughput (TFLOP/s): the measured burst figure (a kernel timed
    between memory-bound kernels, not a seconds-long GEMM loop), else the fallback."""
    p = _peaks_file()
    if "bf16_tflops" in p:
        return float(p["bf16_tflops"]), "measured (burst)"
    return FALLBACK_BF16_TFLOPS, "fallback"


#: sources each kernel is built from (a recorded ncu traffic figure is valid only for them)
KERNEL_SOURCES = {
    "decode": ("decode.cu", "decode_balanced.cu", "pa_device.cuh"),
    "prefill": ("prefill.cu", "pa_tcgen05.cuh", "pa_device.cuh"),
    "reshape": ("reshape_and_cache.cu", "pa_device.cuh"),
}


def kernel_source_hash(kernel: str = "decode") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_238_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str = "decode", workload: str = "gqa_decode") -> "float | None":
    """DRAM bytes (read + written) per launch of `kernel` on `workload`, from the committed ncu
    summary, if it was taken on the kernel's current source (null otherwise)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(f"{kernel}/{workload}")
    except Exception:
        return None
    if not rec or rec.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.samples.append(parts)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in self.samples:
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest value over the job's ranks: a job's time is that of its slowest rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes its own units (replicas,
    no exchange), so the job's units are world x the per-rank units over the slowest time."""
    return units_per_rank * world / seconds


def to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def count_launches_per_step(step_fn) -> "int | None":
    """Kernels of libpa launched by one eager step, counted from the CUDA activity trace."""
    import torch
    try:
        from torch.profiler import ProfilerActivity, profile
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            step_fn(0)
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        ours = [n for n in names if "pa::" in n or "reshape_and_cache" in n or "decode_" in n or "prefill_" in n]
        return len(ours) if ours else None
    except Exception:
        return None


def _subset(wl, n_dec: int, n_pre: int):
    """The first n_dec decode and n_pre prefill sequences of a workload, with their new tokens."""
    from paged_kv_cache_238_gb300 import workloads as W
    d = dict(wl.__dict__)
    if wl.seq_lens is not None:
        d.update(q=wl.q[:n_dec], block_table=wl.block_table[:n_dec], seq_lens=wl.seq_lens[:n_dec])
    tok = []
    if wl.seq_lens_prefill is not None:
        qsl = wl.query_start_loc[:n_pre + 1]
        d.update(q_prefill=wl.q_prefill[:qsl[-1]], block_table_prefill=wl.block_table_prefill[:n_pre],
                 seq_lens_prefill=wl.seq_lens_prefill[:n_pre], query_start_loc=qsl)
        tok.append(np.arange(int(qsl[-1])))
    if wl.slot_mapping is not None:
        # decode workloads: one new token per sequence, in sequence order; mixed: the prefill
        # chunks' tokens first, then one per decode sequence, then padding
        if wl.seq_lens_prefill is not None:
            tok.append(int(wl.query_start_loc[-1]) + np.arange(n_dec))
        else:
            tok.append(np.arange(n_dec))
        idx = np.concatenate(tok)
        d.update(k_new=wl.k_new[idx], v_new=wl.v_new[idx], slot_mapping=wl.slot_mapping[idx])
    return W.Workload(**d)


def _oracle_pass(wl, cores: int):
    import oracle
    kc, vc = wl.k_cache, wl.v_cache
    if wl.slot_mapping is not None and wl.slot_mapping.shape[0] > 0:
        oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    if wl.seq_lens_prefill is not None and len(wl.seq_lens_prefill) > 0:
        oracle.attention(wl.q_prefill, kc, vc, wl.block_table_prefill, wl.seq_lens_prefill, wl.scale,
                         query_start_loc=wl.query_start_loc, num_threads=cores)
    if wl.seq_lens is not None and wl.S > 0:
        oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale, num_threads=cores)


def oracle_sample(wl, budget_s: float):
    """A bounded sample of one step of the workload for the fp64 oracle: the largest leading
    fraction of its sequences (decode and prefill alike) whose oracle pass fits ~budget_s."""
    cores = os.cpu_count() or 1
    n_dec = wl.S if wl.seq_lens is not None else 0
    n_pre = len(wl.seq_lens_prefill) if wl.seq_lens_prefill is not None else 0
    p_dec, p_pre = min(n_dec, 1), min(n_pre, 1)
    t0 = time.perf_counter()
    _oracle_pass(_subset(wl, p_dec, p_pre), cores)
    one = time.perf_counter() - t0
    # a probe of one decode and one prefill sequence; scale by the larger count
    est_full = one * max(n_dec, n_pre, 1)
    frac = 1.0 if est_full <= budget_s else budget_s / est_full
    sd = n_dec if frac >= 1 else max(p_dec, int(n_dec * frac))
    sp = n_pre if frac >= 1 else max(p_pre, int(n_pre * frac))
    return _subset(wl, sd, sp), sd, sp, cores


def cpu_baseline(wl, budget_s: float = 10.0, value_key: str = "step") -> dict:
    """The fp64 oracle (test infrastructure), as it stands, on the host cores, over a bounded
    sample of one step of the same workload, repeated until ~budget_s."""
    sub, sd, sp, cores = oracle_sample(wl, budget_s / 2)
    b = step_bytes(sub)
    passes, t0 = 0, time.perf_counter()
    while True:
        _oracle_pass(sub, cores)
        passes += 1
        if time.perf_counter() - t0 > budget_s or passes >= 50:
            break
    dt = time.perf_counter() - t0
    tokens = sd + (int(sub.query_start_loc[-1]) if sp else 0)
    # the same oracle on one core, over a sixteenth of the sample (rate per sequence kept)
    sd1, sp1 = (max(1, sd // 16) if sd else 0), (max(1, sp // 16) if sp else 0)
    sub1 = _subset(wl, sd1, sp1)
    t1 = time.perf_counter()
    _oracle_pass(sub1, 1)
    dt1 = time.perf_counter() - t1
    tokens1 = sd1 + (int(sub1.query_start_loc[-1]) if sp1 else 0)
    res = {"unit": "TB/s", "cores": cores, "kind": "oracle",
           "sample": f"{passes} passes over {sd} decode + {sp} prefill sequences of one step "
                     f"(reshape_and_cache + attention, fp64) in {dt:.1f} s",
           "seqs_per_s": (sd + sp) * passes / dt, "tokens_per_s": tokens * passes / dt}
    b1 = step_bytes(sub1)
    if value_key == "tokens":
        res["value"], res["unit"] = tokens * passes / dt, "tokens/s"
        one_core = tokens1 / dt1
    elif value_key == "flops":
        res["value"], res["unit"] = b["prefill_flops"] * passes / dt / 1e12, "TFLOP/s"
        one_core = b1["prefill_flops"] / dt1 / 1e12
    else:
        res["value"] = b["step"] * passes / dt / 1e12
        one_core = b1["step"] / dt1 / 1e12
    res["one_core"] = {"value": one_core, "sample": f"1 pass over {sd1} decode + {sp1} prefill sequences on 1 core "
                                                    f"in {dt1:.2f} s"}
    return res


class DeviceStep:
    """The workload's device tensors (R rotated KV pools) and one step of the hot path:
    reshape_and_cache of the step's new tokens, then chunked prefill and decode attention."""

    def __init__(self, wl, dev, R: int, stream, whole_step: bool = False, decode_sms: int = 0,
                 fuse_append: bool = False, pool_ready: bool = False, shared_prefix: bool = False):
        import torch
        from paged_kv_cache_238_gb300 import binding as B
        self.B, self.wl, self.stream, self.R = B, wl, stream, R
        self.pool_ready = pool_ready
        self.decode_sms = decode_sms
        kc0, vc0 = to_dev(wl.k_cache, dev), to_dev(wl.v_cache, dev)
        self.kcs = [kc0] + [kc0.clone() for _ in range(R - 1)]
        self.vcs = [vc0] + [vc0.clone() for _ in range(R - 1)]
        self.has_new = wl.slot_mapping is not None and wl.slot_mapping.shape[0] > 0
        self.has_dec = wl.seq_lens is not None and wl.S > 0
        self.has_pre = wl.seq_lens_prefill is not None and len(wl.seq_lens_prefill) > 0
        self.inputs, self.outputs = [], []
        if self.has_new:
            self.k_new, self.v_new, self.slots = (to_dev(wl.k_new, dev), to_dev(wl.v_new, dev),
                                                  to_dev(wl.slot_mapping, dev))
            self.inputs += [self.k_new, self.v_new, self.slots]
        if self.has_dec:
            self.q, self.bt, self.lens = to_dev(wl.q, dev), to_dev(wl.block_table, dev), to_dev(wl.seq_lens, dev)
            self.out = torch.empty_like(self.q)
            self.msl = int(wl.seq_lens.max())
            dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
            # a prefix that every sequence aliases: attended once (pa_decode_shared_prefix)
            self.prefix = int(wl.info.get("shared_prefix_tokens", 0)) if shared_prefix else 0
            if self.prefix:
                n = B.pa_decode_shared_prefix_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, self.msl, self.prefix)
                if n == 0:
                    self.prefix = 0
            ws_bytes = n if self.prefix else B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, self.msl, dt)
            self.ws = torch.zeros(max(16, ws_bytes), dtype=torch.uint8, device=dev)
            self.inputs += [self.q, self.bt, self.lens]
            self.outputs.append(self.out)
        if self.has_pre:
            self.qp = to_dev(wl.q_prefill, dev)
            self.btp, self.lp = to_dev(wl.block_table_prefill, dev), to_dev(wl.seq_lens_prefill, dev)
            self.qsl = to_dev(wl.query_start_loc, dev)
            self.outp = torch.empty_like(self.qp)
            self.max_chunk = int(np.diff(wl.query_start_loc).max())
            self.msl_p = int(wl.seq_lens_prefill.max())
            self.inputs += [self.qp, self.btp, self.lp, self.qsl]
            self.outputs.append(self.outp)
        self.kernels = [k for k, on in (("reshape", self.has_new), ("prefill", self.has_pre),
                                        ("decode", self.has_dec)) if on]
        # The step's inputs (and its outputs) live in one device arena each, so the end-to-end
        # step moves them with one host->device and one device->host copy.
        in_names = [n for n, on in (("k_new", self.has_new), ("v_new", self.has_new), ("slots", self.has_new),
                                    ("q", self.has_dec), ("bt", self.has_dec), ("lens", self.has_dec),
                                    ("qp", self.has_pre), ("btp", self.has_pre), ("lp", self.has_pre),
                                    ("qsl", self.has_pre)) if on]
        out_names = [n for n, on in (("out", self.has_dec), ("outp", self.has_pre)) if on]
        self.in_arena = self._pack(in_names, dev, copy=True)
        self.out_arena = self._pack(out_names, dev, copy=False)
        self.inputs = [getattr(self, n) for n in in_names]
        self.outputs = [getattr(self, n) for n in out_names]
        # buffer sets: 0 = the tensors above; add_buffer() makes more with the same layout
        self.in_names, self.out_names = in_names, out_names
        self.bufs = [{n: getattr(self, n) for n in in_names + out_names}]
        self.in_arenas, self.out_arenas = [self.in_arena], [self.out_arena]
        # whole step through pa_step: prefill and decode side by side on an SM split
        self.whole_step = whole_step and self.has_pre and self.has_dec
        # decode-only step with one new token per sequence: pa_decode_append (write + attention)
        self.fused_append = (fuse_append and self.has_new and self.has_dec and not self.has_pre and
                             wl.slot_mapping.shape[0] == wl.S)
        if self.fused_append:
            self.kernels = ["decode"]

    def _pack(self, names, dev, copy: bool):
        """Re-home the named tensors as 256-byte-aligned views of one uint8 device buffer."""
        import torch
        if not names:
            return None
        offs, total = [], 0
        for n in names:
            offs.append(total)
            t = getattr(self, n)
            total += -(-t.numel() * t.element_size() // 256) * 256
        arena = torch.zeros(total, dtype=torch.uint8, device=dev)
        for n, o in zip(names, offs):
            t = getattr(self, n)
            v = arena[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            if copy:
                v.copy_(t)
            setattr(self, n, v)
        return arena

    def add_buffer(self) -> int:
        """Another set of input and output buffers (same layout); returns its index."""
        import torch
        ia, oa = torch.empty_like(self.in_arena), torch.empty_like(self.out_arena)
        ia.copy_(self.in_arena)
        views = {}
        for names, old, new in ((self.in_names, self.in_arena, ia), (self.out_names, self.out_arena, oa)):
            for n in names:
                t = self.bufs[0][n]
                off = t.data_ptr() - old.data_ptr()
                views[n] = new[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        self.bufs.append(views)
        self.in_arenas.append(ia)
        self.out_arenas.append(oa)
        return len(self.bufs) - 1

    def __call__(self, i: int, ev=None, buf: int = 0):
        """Step i on pool i % R with buffer set `buf`; ev maps a kernel name to an event pair
        recorded around it."""
        B, r, s, wl = self.B, i % self.R, self.stream, self.wl
        T = self.bufs[buf]

        def rec(k, j):
            if ev is not None and k in ev:
                ev[k][j].record(s)

        if self.whole_step:
            tev = None
            if ev is not None:
                tev = [ev[k][j] if k in ev else None for k in ("reshape", "prefill", "decode") for j in (0, 1)]
            B.pa_step(self.kcs[r], self.vcs[r], wl.scale,
                      k_new=T["k_new"] if self.has_new else None, v_new=T["v_new"] if self.has_new else None,
                      slot_mapping=T["slots"] if self.has_new else None,
                      prefill_out=T["outp"], prefill_q=T["qp"], prefill_block_table=T["btp"], prefill_seq_lens=T["lp"],
                      query_start_loc=T["qsl"], max_chunk_len=self.max_chunk, prefill_max_seq_len=self.msl_p,
                      decode_out=T["out"], decode_q=T["q"], decode_block_table=T["bt"], decode_seq_lens=T["lens"],
                      decode_max_seq_len=self.msl, workspace=self.ws, decode_sms=self.decode_sms,
                      timing_events=tev, stream=s)
            return
        if self.fused_append:
            rec("decode", 0)
            # the tables are written by host copies only, never by the kernel before
            B.pa_decode_append(T["out"], T["q"], T["k_new"], T["v_new"], T["slots"], self.kcs[r], self.vcs[r], T["bt"],
                               T["lens"], self.msl, wl.scale, self.ws, stream=s, tables_ready=True,
                               pool_ready=self.pool_ready)
            rec("decode", 1)
            return
        if self.has_new:
            rec("reshape", 0)
            B.pa_reshape_and_cache(T["k_new"], T["v_new"], self.kcs[r], self.vcs[r], T["slots"], stream=s)
            rec("reshape", 1)
        if self.has_pre:
            rec("prefill", 0)
            B.pa_prefill_chunk(T["outp"], T["qp"], self.kcs[r], self.vcs[r], T["btp"], T["lp"], T["qsl"],
                               self.max_chunk, self.msl_p, wl.scale, stream=s)
            rec("prefill", 1)
        if self.has_dec:
            rec("decode", 0)
            if self.prefix:
                B.pa_decode_shared_prefix(T["out"], T["q"], self.kcs[r], self.vcs[r], T["bt"], T["lens"], self.msl,
                                          wl.scale, self.prefix, self.ws, stream=s, tables_ready=True,
                                          pool_ready=self.pool_ready)
            else:
                B.pa_decode(T["out"], T["q"], self.kcs[r], self.vcs[r], T["bt"], T["lens"], self.msl, wl.scale,
                            self.ws, stream=s)
            rec("decode", 1)


KERNEL_LABEL = {
    "decode_append": "pa_decode_append: balanced TMA + mma.sync decode with the new tokens' K/V write fused in",
    "decode": "pa_decode: balanced TMA + mma.sync decode kernel (split merge in-kernel)",
    "prefill": "pa_prefill_chunk: tcgen05 chunked-prefill kernel (TMA page gather, S/O/P in TMEM)",
    "reshape": "pa_reshape_and_cache: slot scatter",
}
MIXED_METRIC = "mixed step: new tokens/s (16 x 512-token prefill chunks + 240 decode seqs)"
PREFILL_METRIC = "chunked prefill: causal attention TFLOP/s (16 x 512-token chunks, GQA 32/8, head_dim 128)"


def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_238_gb300 import binding as B
    from paged_kv_cache_238_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    desc = WORKLOADS[args.workload][1]
    wl = build_workload(args.workload)
    nbytes = step_bytes(wl)
    R = args.replicas
    stream = torch.cuda.Stream(device=dev)
    step = DeviceStep(wl, dev, R, stream, whole_step=not args.sequential, decode_sms=args.decode_sms,
                      fuse_append=not args.sequential, pool_ready=not args.no_pool_ready,
                      shared_prefix=not args.no_shared_prefix)
    if step.fused_append:
        # one kernel writes the new tokens and attends: its algorithmic bytes are the decode's
        # plus the new rows read once from the input and written once (not read back)
        new = wl.slot_mapping.shape[0] * _kv_token_bytes(wl)
        nbytes = dict(nbytes)
        nbytes["decode"] = nbytes["decode"] + nbytes["reshape"] - new
        nbytes["step"] = nbytes["step"] - new
        nbytes["reshape"] = 0

    # ---- warm-up (eager, untimed) ----------------------------------------------------------
    # NVTX ranges mark the phases for a timeline profiler (no cost without one)
    nvtx = torch.cuda.nvtx
    nvtx.range_push("warm-up")
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    nvtx.range_pop()
    stream.synchronize()
    assert B.pa_get_device_errors(clear=True) == 0
    launches_per_step = None if args.no_cupti else count_launches_per_step(step)
    if launches_per_step is None:
        launches_per_step = len(step.kernels)  # one kernel per call (split merge inside decode)

    # ---- capture K steps in graphs -------------------------------------------------------
    K = args.steps
    chunk = min(K, args.graph_chunk)

    def evpair():
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))

    # Event pairs around each kernel on every `sample`-th step of the graph only: an event node
    # splits the programmatic (early-launch) edge between two kernels, so bracketing every
    # kernel of every step would slow the steps the line reports.
    sample = max(1, min(args.event_every, chunk))
    ev_steps = {i: {k: evpair() for k in step.kernels} for i in range(0, chunk, sample)}
    for pairs in ev_steps.values():  # torch creates events lazily; the library needs handles
        for e in (x for p in pairs.values() for x in p):
            e.record(stream)
    stream.synchronize()

    def capture(fn, n, with_events):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(n):
                    if with_events and i in ev_steps:
                        fn(i, ev_steps[i])
                    else:
                        fn(i)
        return g

    g_main = capture(step, chunk, True)
    rem = K % chunk
    g_rem = capture(step, rem, False) if rem else None
    n_main = K // chunk

    # ---- e2e graph: pinned host inputs in, results out, every step ------------------------
    # The step's inputs and outputs are packed in one device buffer each (DeviceStep), so a
    # step moves them with one copy each way. Steps go in blocks of EB with their own buffer
    # sets, two groups of sets alternating: block j+1's inputs travel host -> device on one
    # copy stream while block j computes, and block j's outputs travel back on another once it
    # is done (the two directions use separate copy engines). Inside a block the kernels follow
    # one another with nothing between them, so each may launch early under the one before
    # (programmatic launch); only the wait on a block's inputs sits between blocks. The first
    # block's inputs travel at the end of the replay before (each replay still moves K steps'
    # inputs and outputs), so a replay does not start with a copy that nothing overlaps.
    # Every step's copies are inside the timed region.
    EB = max(1, min(chunk, args.e2e_block))
    if step.in_arena.numel() * EB > (16 << 20):
        # large per-step inputs (prefill chunks): copy time, not the launch edge, sets the
        # e2e step; one step per group keeps each copy beside the step before it
        EB = 1
    for _ in range(2 * EB - 1):  # two groups of EB buffer sets (the first group of one step uses one)
        step.add_buffer()
    h_in = step.in_arena.cpu().pin_memory()
    h_out = torch.empty(step.out_arena.shape, dtype=torch.uint8, pin_memory=True)
    h2d = h_in.numel()
    d2h = h_out.numel()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_chunk(n):
        ev = torch.cuda.Event
        start = ev()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        # a first group of one step, so that the replay's first input copy (which nothing
        # overlaps) is short; then groups of EB
        starts = [0] + list(range(1, n, EB))
        blocks = [list(range(j, min(n, 1 if j == 0 else j + EB))) for j in starts if j < n]
        nb = len(blocks)
        copied, done, sent = [ev() for _ in range(nb)], [ev() for _ in range(nb)], [ev() for _ in range(nb)]

        def bufs(j):
            return [(j % 2) * EB + k for k in range(len(blocks[j]))]

        def send_inputs(j):
            with torch.cuda.stream(s_in):
                if j >= 2:
                    s_in.wait_event(done[j - 2])  # block j-2 (same buffer group) has read its inputs
                for b in bufs(j):
                    step.in_arenas[b].copy_(h_in, non_blocking=True)
                copied[j].record(s_in)

        # block 0's inputs were sent at the end of the previous replay (or at set-up)
        copied[0].record(s_in)
        for j in range(nb):
            if j + 1 < nb:
                send_inputs(j + 1)
            stream.wait_event(copied[j])          # block j's inputs landed
            if j >= 2:
                stream.wait_event(sent[j - 2])    # block j-2's outputs (same buffer group) have left
            for i, b in zip(blocks[j], bufs(j)):
                step(i, buf=b)
            done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[j])
                for b in bufs(j):
                    h_out.copy_(step.out_arenas[b], non_blocking=True)
                sent[j].record(s_out)
        # the next replay's first step: its inputs travel now, beside this replay's last steps
        with torch.cuda.stream(s_in):
            s_in.wait_event(done[(nb - 1) // 2 * 2])  # the last block on buffer group 0 has run
            for b in bufs(0):
                step.in_arenas[b].copy_(h_in, non_blocking=True)
        for s_ in (s_in, s_out):
            end = ev()
            end.record(s_)
            stream.wait_event(end)

    def capture_e2e(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                e2e_chunk(n)
        return g

    g_e2e = capture_e2e(chunk)
    g_e2e_rem = capture_e2e(rem) if rem else None

    def timed(gm, gr):
        """The K-step graph(s) replayed back to back, at least args.min_replays times and for
        at least args.min_timed_ms in all, each replay between its own pair of events: the
        median replay (K steps), max over ranks, and the number of replays."""
        def run_once(evs):
            with torch.cuda.stream(stream):
                evs[0].record(stream)
                for _ in range(n_main):
                    gm.replay()
                if gr is not None:
                    gr.replay()
                evs[1].record(stream)

        probe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        run_once(probe)
        torch.cuda.synchronize()
        reps = max(args.min_replays, int(np.ceil(args.min_timed_ms / max(probe[0].elapsed_time(probe[1]), 1e-3))))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for r in range(reps):
                for _ in range(n_main):
                    gm.replay()
                if gr is not None:
                    gr.replay()
                evs[r + 1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        per = [evs[r].elapsed_time(evs[r + 1]) for r in range(reps)]
        return max_over_ranks(float(np.median(per)), world, dev), reps, evs[0].elapsed_time(evs[-1])

    sampler = ClockSampler(local)
    sampler.start()
    # steady state before the timed region (clocks settle; untimed)
    t_end = time.perf_counter() + args.preheat_s
    with torch.cuda.stream(stream):
        while time.perf_counter() < t_end:
            g_main.replay()
            stream.synchronize()
    nvtx.range_push(f"timed: {K} steps x replays")
    ms_total, reps, ms_region = timed(g_main, g_rem)
    nvtx.range_pop()
    clocks = sampler.stop()
    # per-kernel durations from the sampled steps of the last replay of the main graph (inside
    # the timed region)
    kern_ms = {k: sum(e[k][0].elapsed_time(e[k][1]) for e in ev_steps.values()) / len(ev_steps)
               for k in step.kernels}
    nvtx.range_push("timed e2e")
    ms_e2e, reps_e2e, _ = timed(g_e2e, g_e2e_rem)
    nvtx.range_pop()
    assert B.pa_get_device_errors(clear=True) == 0

    ms_step = ms_total / K
    # A step of one kernel launches it back to back: its average launch duration is the event
    # pair around the whole timed region over K. A pair around a single launch (kept as
    # us_single_launch) also counts the launch delay that the event node itself causes.
    single = {}
    if len(step.kernels) == 1:
        k1 = step.kernels[0]
        single[k1] = kern_ms[k1]
        kern_ms[k1] = ms_step
    hbm_peak, hbm_kind = load_peaks()
    tc_peak, tc_kind = load_tensor_peak()
    kernels = {}
    for k, ms in kern_ms.items():
        if k == "prefill":
            ach = nbytes["prefill_flops"] / (ms * 1e-3) / 1e12
            kernels[k] = {"us": round(ms * 1e3, 3), "bound": "tensor", "achieved": round(ach, 1), "unit": "TFLOP/s",
                          "peak": tc_peak, "frac": round(ach / tc_peak, 4), "peak_source": tc_kind,
                          "hbm_gbs": round(nbytes["prefill"] / (ms * 1e-3) / 1e9, 1)}
        else:
            ach = nbytes[k] / (ms * 1e-3) / 1e9
            kernels[k] = {"us": round(ms * 1e3, 3), "bound": "hbm", "achieved": round(ach, 1), "unit": "GB/s",
                          "peak": hbm_peak, "frac": round(ach / hbm_peak, 4), "peak_source": hbm_kind}
    for k, ms in single.items():
        kernels[k]["us_single_launch"] = round(ms * 1e3, 3)
    dom = max(kern_ms, key=kern_ms.get)
    roof = {"kernel": KERNEL_LABEL[dom], **{k: v for k, v in kernels[dom].items() if k != "us"},
            "kernel_us": kernels[dom]["us"], "traffic": recorded_traffic(dom, args.workload)}
    if dom == "decode":
        roof["decode_call_us"] = kernels[dom]["us"]

    n_seqs = (wl.S if step.has_dec else 0) + (len(wl.seq_lens_prefill) if step.has_pre else 0)
    tokens = (wl.S if step.has_dec else 0) + (int(wl.query_start_loc[-1]) if step.has_pre else 0)
    if args.workload == "mixed_step":
        metric, unit, nd = MIXED_METRIC, "tokens/s", 1
        value = job_rate(tokens, world, ms_step * 1e-3)
        e2e_value = job_rate(tokens, world, ms_e2e / K * 1e-3)
    elif args.workload == "prefill_chunks":
        metric, unit, nd = PREFILL_METRIC, "TFLOP/s", 2
        value = job_rate(nbytes["prefill_flops"], world, ms_step * 1e-3) / 1e12
        e2e_value = job_rate(nbytes["prefill_flops"], world, ms_e2e / K * 1e-3) / 1e12
    else:
        metric, unit, nd = METRIC, "TB/s", 4
        value = job_rate(nbytes["step"], world, ms_step * 1e-3) / 1e12
        e2e_value = job_rate(nbytes["step"], world, ms_e2e / K * 1e-3) / 1e12
    line = {
        "metric": metric, "value": round(value, nd), "unit": unit, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded generator; no dataset)",
        "config": {"workload": desc, "seqs": n_seqs, "keys": int(nbytes["kv"] // _kv_token_bytes(wl)),
                   "bytes_per_step": nbytes["step"], "kernels_per_step": step.kernels, "kv_pools_rotated": R,
                   "l2": f"inputs larger than L2: {R} KV pool(s) rotated, "
                         f"{R * nbytes['kv_unique'] / 1e6:.0f} MB of distinct KV touched per rotation "
                         f"(L2 {L2_BYTES / 1e6:.0f} MB)",
                   "graph": f"{n_main} x {chunk}-step CUDA graph" + (f" + {rem}-step graph" if rem else ""),
                   "timing": f"median over {reps} back-to-back replays of the {K}-step graph(s), each between "
                             f"its own event pair ({ms_region:.1f} ms timed in all); e2e: median over {reps_e2e}",
                   "kernel_timing": (f"one kernel per step: the event pair around the {K}-step timed region over K "
                                     f"(us_single_launch: pairs around the kernel of every {sample}th step)")
                   if len(step.kernels) == 1 else
                   f"CUDA event pairs around each kernel of every {sample}th step of the timed "
                                    f"graph ({len(ev_steps)} per replay)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "seqs_per_s": round(n_seqs * world / (ms_step * 1e-3), 1),
        "tokens_per_s": round(tokens * world / (ms_step * 1e-3), 1),
        "e2e": {"value": round(e2e_value, nd), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e / K, 6),
                "blocks": f"{EB} steps per input/output copy group, two groups alternating"},
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": launches_per_step * K * reps,
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if step.fused_append:
        line["config"]["step_call"] = "pa_decode_append: one launch writes the new tokens' K/V and attends"
        line["roofline"]["kernel"] = KERNEL_LABEL["decode_append"]
    if step.whole_step:
        line["config"]["step_call"] = (f"pa_step: reshape_and_cache, then prefill and decode side by side "
                                       f"(decode on {args.decode_sms or '27/64 of the'} SMs)")
        line["config"]["kernel_timing"] += "; prefill and decode overlap, so their durations add up to more than the step"
    if args.workload == "gqa_decode":
        line["config"]["decode_bytes_per_call"] = nbytes["decode"]
        line["config"]["mean_len"] = round(float(wl.seq_lens.mean()), 2)
    if nbytes["kv_unique"] < nbytes["kv"]:
        # aliased prefix blocks: value and roofline count the distinct keys (what must leave
        # HBM); the logical figure counts each sequence's keys and is context only
        line["config"]["kv_bytes_logical"] = nbytes["kv"]
        line["config"]["kv_bytes_distinct"] = nbytes["kv_unique"]
        line["config"]["bytes_basis"] = "distinct keys (an aliased prefix counts once)"
        line["decode_logical_tbs"] = round(nbytes["decode_logical"] / (kern_ms["decode"] * 1e-3) / 1e12, 3)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget_s,
                                            {"tokens/s": "tokens", "TFLOP/s": "flops"}.get(unit, "step"))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ------------------------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_cache_238_gb300 import workloads as W

    desc = WORKLOADS[args.workload][1]
    wl = build_workload(args.workload)
    # Size each step's sample so the whole run stays within ~budget seconds.
    per_step_budget = args.reference_budget_s / max(1, args.steps + args.warmup)
    sub, sd, sp, cores = oracle_sample(wl, per_step_budget)
    b = step_bytes(sub)
    tokens = sd + (int(sub.query_start_loc[-1]) if sp else 0)
    for _ in range(args.warmup):
        _oracle_pass(sub, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_pass(sub, cores)
    dt = time.perf_counter() - t0
    if args.workload == "mixed_step":
        metric, unit = MIXED_METRIC, "tokens/s"
        value = tokens * args.steps / dt
    elif args.workload == "prefill_chunks":
        metric, unit = PREFILL_METRIC, "TFLOP/s"
        value = step_bytes(sub)["prefill_flops"] * args.steps / dt / 1e12
    else:
        metric, unit = METRIC, "TB/s"
        value = b["step"] * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator; no dataset)",
        "config": {"workload": desc, "sample_decode_seqs_per_step": sd, "sample_prefill_seqs_per_step": sp},
        "seqs_per_s": (sd + sp) * args.steps / dt,
        "tokens_per_s": tokens * args.steps / dt,
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": f"{sd} decode + {sp} prefill sequences of the step per timed step "
                                   f"(reshape_and_cache + attention), fp64"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gqa_decode",
                    help="the GQA decode batch (default) or another workload of the same path")
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: per workload)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=None, help="KV pools rotated across steps (default: per workload)")
    ap.add_argument("--graph-chunk", type=int, default=500, help="steps per captured graph")
    ap.add_argument("--event-every", type=int, default=50, help="time each kernel on every Nth step of a graph")
    ap.add_argument("--preheat-s", type=float, default=1.0)
    ap.add_argument("--min-replays", type=int, default=20, help="timed replays of the K-step graph (at least)")
    ap.add_argument("--e2e-block", type=int, default=4, help="e2e: steps per input/output copy group")
    ap.add_argument("--min-timed-ms", type=float, default=50.0, help="replay the K-step graph for at least this long")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cupti", action="store_true", help="skip the activity-trace launch count (e.g. under ncu)")
    ap.add_argument("--sequential", action="store_true",
                    help="one call per kernel: no pa_step (mixed step) and no pa_decode_append (decode step)")
    ap.add_argument("--decode-sms", type=int, default=0, help="pa_step: SMs held by decode (0 = 27/64 of them)")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="prefix_sharing: plain pa_decode instead of pa_decode_shared_prefix")
    ap.add_argument("--no-pool-ready", action="store_true",
                    help="decode step without PA_DECODE_POOL_READY (first page copies after the grid-dependency wait)")
    args = ap.parse_args(argv)
    _, _, default_steps, default_replicas = WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = default_steps
    if args.replicas is None:
        args.replicas = default_replicas
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
