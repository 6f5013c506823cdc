"""Benchmark of the paged-KV decode step on GB300.

One step = the whole hot path on one batch: reshape_and_cache of the batch's new tokens
(one per sequence) followed by paged decode attention over all of their keys, for the GQA
decode batch of 64 sequences (32 q / 8 kv heads, head_dim 128, bf16, lognormal context
lengths with mean ~195, 16-token blocks, shuffled physical blocks).

Timing: the step's device inputs stay resident; steps rotate through R independent KV pools
(one per "layer", the same block table), so a pool is touched again only after the other
R-1 (> 3 x L2 in between): inputs larger than L2, no flush kernel. K steps are captured in
CUDA graphs (the step is launch-bound at ~10 us) and timed with CUDA events on the launching
stream, barrier + synchronize on both sides, max over ranks. Each decode call is bracketed
by its own event pair inside the graph; the roofline figure uses their average.

value  = algorithmic bytes of the step / step time (TB/s): KV bytes of every visible key,
         Q, output, block-table entries, lengths, and the new tokens' K/V read and written.
e2e    = the same metric with every step's inputs copied host->device from pinned memory and
         its output copied back, inside the timed graph.
--impl reference  times the fp64 CPU oracle (test infrastructure) on a bounded sample of the
         same workload and prints the same line with "impl": "reference".
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
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------------------------------
# workload bytes (algorithmic, per step)
# ------------------------------------------------------------------------------------------

def step_bytes(wl) -> dict:
    el = 2 if wl.dtype == "bf16" else 4
    lens = wl.seq_lens.astype(np.int64)
    kv = int(lens.sum()) * 2 * wl.H_kv * wl.D * el
    q = wl.S * wl.H_q * wl.D * el
    out = q
    bt = int(np.sum(-(-lens // 16))) * 4
    seq = wl.S * 4
    T = 0 if wl.slot_mapping is None else wl.slot_mapping.shape[0]
    new = 2 * T * wl.H_kv * wl.D * el          # new K and V read ...
    k1 = 2 * new + 8 * T                       # ... and written, plus the slots
    decode = kv + q + out + bt + seq
    return {"kv": kv, "decode": decode, "reshape": k1, "step": decode + k1}


def load_peaks() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_238_gb300", "csrc")
    for f in ("decode.cu", "decode_balanced.cu", "pa_device.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic() -> "float | None":
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current decode kernel source (null otherwise)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_decode_call")


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
        ours = [n for n in names if "pa::" in n or "reshape_and_cache" in n or "decode_" in n]
        return len(ours) if ours else None
    except Exception:
        return None


def cpu_baseline(wl, budget_s: float = 10.0) -> dict:
    """The fp64 oracle (test infrastructure), as it stands, on the host cores: full 64-seq
    passes of the same step until ~budget_s of CPU time."""
    import oracle
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    cores = os.cpu_count() or 1
    b = step_bytes(wl)["step"]
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
        oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale, num_threads=cores)
        passes += 1
        if time.perf_counter() - t0 > budget_s or passes >= 50:
            break
    dt = time.perf_counter() - t0
    return {"value": b * passes / dt / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} full passes of the 64-sequence step (reshape_and_cache + decode) in {dt:.1f} s",
            "seqs_per_s": wl.S * passes / dt}


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

    wl = W.gqa_decode()
    nbytes = step_bytes(wl)
    R = args.replicas
    # one pool per layer: contents come from the generator; replicas are device copies
    kc0, vc0 = to_dev(wl.k_cache, dev), to_dev(wl.v_cache, dev)
    kcs = [kc0] + [kc0.clone() for _ in range(R - 1)]
    vcs = [vc0] + [vc0.clone() for _ in range(R - 1)]
    q, k_new, v_new = to_dev(wl.q, dev), to_dev(wl.k_new, dev), to_dev(wl.v_new, dev)
    slots, bt, lens = to_dev(wl.slot_mapping, dev), to_dev(wl.block_table, dev), to_dev(wl.seq_lens, dev)
    out = torch.empty_like(q)
    msl = int(wl.seq_lens.max())
    ws = torch.zeros(max(16, B.pa_decode_workspace_size(wl.S, wl.H_q, wl.H_kv, wl.D, msl, torch.bfloat16)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, ev=None):
        r = i % R
        B.pa_reshape_and_cache(k_new, v_new, kcs[r], vcs[r], slots, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        B.pa_decode(out, q, kcs[r], vcs[r], bt, lens, msl, wl.scale, ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    # ---- warm-up (eager, untimed) and a parity spot-check of one sequence --------------------
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    stream.synchronize()
    assert B.pa_get_device_errors(clear=True) == 0
    launches_per_step = None if args.no_cupti else count_launches_per_step(step)
    if launches_per_step is None:
        launches_per_step = 2  # reshape_and_cache + the balanced decode kernel (split merge inside)

    # ---- capture K steps in graphs -------------------------------------------------------
    K = args.steps
    chunk = min(K, args.graph_chunk)
    ev_pairs = [(torch.cuda.Event(enable_timing=True, external=True),
                 torch.cuda.Event(enable_timing=True, external=True)) for _ in range(chunk)]

    def capture(n, with_events):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(n):
                    step(i, ev_pairs[i] if with_events else None)
        return g

    g_main = capture(chunk, True)
    rem = K % chunk
    g_rem = capture(rem, False) if rem else None
    n_main = K // chunk

    # ---- e2e graph: pinned host inputs in, result out, every step -------------------------
    h_q = q.cpu().pin_memory()
    h_kn, h_vn = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    h_slots, h_bt, h_lens = slots.cpu().pin_memory(), bt.cpu().pin_memory(), lens.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_slots, h_bt, h_lens))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step(i):
        r = i % R
        for d, h in ((q, h_q), (k_new, h_kn), (v_new, h_vn), (slots, h_slots), (bt, h_bt), (lens, h_lens)):
            d.copy_(h, non_blocking=True)
        B.pa_reshape_and_cache(k_new, v_new, kcs[r], vcs[r], slots, stream=stream)
        B.pa_decode(out, q, kcs[r], vcs[r], bt, lens, msl, wl.scale, ws, stream=stream)
        h_out.copy_(out, non_blocking=True)

    def capture_e2e(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(n):
                    e2e_step(i)
        return g

    g_e2e = capture_e2e(chunk)
    g_e2e_rem = capture_e2e(rem) if rem else None

    def run_graphs(gm, gr):
        for _ in range(n_main):
            gm.replay()
        if gr is not None:
            gr.replay()

    def timed(gm, gr):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t0.record(stream)
            run_graphs(gm, gr)
            t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ms = t0.elapsed_time(t1)
        if world > 1:
            tt = torch.tensor([ms], device=dev, dtype=torch.float64)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            ms = float(tt.item())
        return ms

    sampler = ClockSampler(local)
    sampler.start()
    # steady state before the timed region (clocks settle; untimed)
    t_end = time.perf_counter() + args.preheat_s
    with torch.cuda.stream(stream):
        while time.perf_counter() < t_end:
            g_main.replay()
            stream.synchronize()
    ms_total = timed(g_main, g_rem)
    clocks = sampler.stop()
    # per-call decode duration from the last replay of the main graph (inside the timed region)
    dec_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    ms_e2e = timed(g_e2e, g_e2e_rem)
    assert B.pa_get_device_errors(clear=True) == 0

    ms_step = ms_total / K
    value = nbytes["step"] * world / (ms_step * 1e-3) / 1e12
    e2e_value = nbytes["step"] * world / (ms_e2e / K * 1e-3) / 1e12
    peak, peak_kind = load_peaks()
    achieved_gbs = nbytes["decode"] / (dec_avg_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generator; no dataset)",
        "config": {"workload": WORKLOAD, "seqs": wl.S, "mean_len": round(float(wl.seq_lens.mean()), 2),
                   "keys": int(wl.seq_lens.sum()), "bytes_per_step": nbytes["step"],
                   "decode_bytes_per_call": nbytes["decode"], "kv_layers_rotated": R,
                   "l2": f"inputs larger than L2: {R} KV pools rotated, each touched again only after "
                         f"{(R - 1) * nbytes['step'] / 1e6:.0f} MB of other pools (L2 {L2_BYTES / 1e6:.0f} MB)",
                   "graph": f"{n_main} x {chunk}-step CUDA graph" + (f" + {rem}-step graph" if rem else ""),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "seqs_per_s": round(wl.S * world / (ms_step * 1e-3), 1),
        "tokens_per_s": round(wl.S * world / (ms_step * 1e-3), 1),
        "e2e": {"value": round(e2e_value, 4), "unit": "TB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e / K, 6)},
        "roofline": {"kernel": "pa_decode: balanced TMA + mma.sync decode kernel (split merge in-kernel)",
                     "bound": "hbm",
                     "achieved": round(achieved_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved_gbs / peak, 4), "peak_source": peak_kind,
                     "decode_call_us": round(dec_avg_ms * 1e3, 3), "traffic": recorded_traffic()},
        "gpu_launches": launches_per_step * K,
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget_s)
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
    import oracle
    from paged_kv_cache_238_gb300 import workloads as W

    wl = W.gqa_decode()
    cores = os.cpu_count() or 1
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    # Size each step's sample so the whole run stays within ~budget seconds.
    t0 = time.perf_counter()
    oracle.reshape_and_cache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    oracle.attention(wl.q, kc, vc, wl.block_table, wl.seq_lens, wl.scale, num_threads=cores)
    full_s = time.perf_counter() - t0
    per_step_budget = args.reference_budget_s / max(1, args.steps + args.warmup)
    n_seq = int(max(1, min(wl.S, wl.S * per_step_budget / max(full_s, 1e-9))))
    idx = np.arange(n_seq)
    sub = W.Workload(**{**wl.__dict__, "q": wl.q[idx], "block_table": wl.block_table[idx],
                        "seq_lens": wl.seq_lens[idx], "k_new": wl.k_new[idx], "v_new": wl.v_new[idx],
                        "slot_mapping": wl.slot_mapping[idx]})
    b = step_bytes(sub)["step"]

    def one():
        oracle.reshape_and_cache(sub.k_new, sub.v_new, kc, vc, sub.slot_mapping)
        oracle.attention(sub.q, kc, vc, sub.block_table, sub.seq_lens, sub.scale, num_threads=cores)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    value = b * args.steps / dt / 1e12
    threads = min(cores, n_seq)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator; no dataset)",
        "config": {"workload": WORKLOAD, "sample_seqs_per_step": n_seq},
        "seqs_per_s": n_seq * args.steps / dt,
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_seq} of the 64 sequences per step (reshape_and_cache + decode), fp64"},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=10, help="KV pools rotated across steps")
    ap.add_argument("--graph-chunk", type=int, default=500, help="steps per captured graph")
    ap.add_argument("--preheat-s", type=float, default=1.0)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cupti", action="store_true", help="skip the activity-trace launch count (e.g. under ncu)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
