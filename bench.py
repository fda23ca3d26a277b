"""Benchmark of the Adasum combine on one GB300 (or N independent replicas).

Default workload: K=16 workers, BERT-Large-shaped gradient set (391 tensors, 335,141,888
elements, bf16 storage, fp32 math), the configuration the throughput target is stated
on.  A step is one full adasum_reduce over the whole set (every segment, every tree
level).  Inputs are synthetic, seeded, resident in HBM before timing; they are 10.7 GB,
far larger than the 126 MB L2, so no flush is needed between steps.  (Workloads under
1 GB of input, such as the 1M-element pair, get an L2 flush before every timed step,
outside that step's own event pair.)  Per-kernel times for the roofline come from a
second, instrumented pass over the same steps, so that the timed steps carry no
per-launch events.

Prints one JSON line (rank 0):
  value      input GB/s = K * N * bytes_per_element * steps / time, summed over ranks
  roofline   the dominant streaming kernel's algorithmic bytes per launch (counted by the
             library from its plan: the tiles, segments or pair the launch covers) / its
             mean CUDA-event time, vs the measured HBM copy bandwidth
  e2e        the same metric through the C-ABI host-buffer call adasum_reduce_host: H2D of
             the inputs, the reduction,
             D2H of the result, every step
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload

`--impl reference` times the CPU oracle instead (the reference arm): each step is a
bounded sample of the workload on the host cores.

Multi-GPU: `torchrun --nproc-per-node N bench.py --gpus N`: every rank reduces its own
full replica of the workload (weak scaling, no collective on the data path); the time
is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "Adasum input GB/s (K*N*bytes/time) and % of GB300 HBM roofline, 1 GPU"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------------------ helpers

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML (read-only) while running."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.02):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._period = period_s
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            bus = None
            try:
                p = torch.cuda.get_device_properties(device_index)
                bus = "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            except Exception:
                bus = None
            ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(),
                                                                         ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            m = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = int(m.value)
            self._nvml, self._h = nv, h
        except Exception:
            self._nvml = None
        self._t = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        nv, h = self._nvml, getattr(self, "_h", None)
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv is not None:
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(int(clk.value))
                if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                    for bit, name in self.REASONS.items():
                        if rs.value & bit and name not in ("gpu_idle",):
                            self.reasons.add(name)
            time.sleep(self._period)

    def __enter__(self):
        self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._t.join()

    def summary(self):
        med = statistics.median(self.samples) if self.samples else None
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": "nvml" if self._nvml else "unavailable"}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------- CPU oracle timing

def oracle_sample(wl, target_bytes: int):
    """A prefix of whole segments of the workload whose input bytes reach target_bytes,
    copied to host as oracle inputs.  Returns (grads, offsets, bytes, description)."""
    import oracle  # CPU baseline leg only
    es = torch.tensor([], dtype=wl.dtype).element_size()
    offs = wl.seg_offsets
    # skip the first (largest) segment only if it alone exceeds the target
    s0 = 0
    while s0 < wl.L and (offs[s0 + 1] - offs[s0]) * wl.K * es > 4 * target_bytes:
        s0 += 1
    s1 = s0
    while s1 < wl.L and (offs[s1] - offs[s0]) * wl.K * es < target_bytes:
        s1 += 1
    lo, hi = int(offs[s0]), int(offs[s1])
    grads = []
    for g in wl.grads:
        t = g[lo:hi].detach().cpu()
        grads.append(t.view(torch.int16).numpy().view(np.uint16).copy()
                     if t.dtype == torch.bfloat16 else t.numpy().copy())
    sub = (offs[s0:s1 + 1] - lo).astype(np.int64)
    nbytes = wl.K * (hi - lo) * es
    desc = (f"segments {s0}..{s1 - 1} of {wl.L} ({s1 - s0} segments, {hi - lo:,} positions, "
            f"{nbytes / 1e9:.3f} GB of input), fp64 oracle, single thread")
    oracle.build()
    return grads, sub, nbytes, desc, oracle


def time_oracle(grads, sub, oracle, reps=1):
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.adasum_reduce(grads, sub, want_out=True)
    return (time.perf_counter() - t0) / reps


# ---------------------------------------------------------------------------- main arms

def run_ours(args):
    import adaptive_gradient_summation_gb300 as ags
    from adaptive_gradient_summation_gb300 import workloads

    rank, world, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ags.load_library()
    wl = workloads.make(args.workload, device=dev, shrink=args.shrink)
    es = torch.tensor([], dtype=wl.dtype).element_size()
    in_bytes = wl.K * wl.N * es
    # minimum bytes of a step: every input once, plus the output, or, for the fused
    # Momentum-SGD step (which runs with out=None), fp32 w and v read and written
    min_bytes = in_bytes + (16 * wl.N if wl.master_w is not None else wl.N * es)
    out = torch.empty(wl.N, dtype=wl.dtype, device=dev)

    def step():
        if wl.master_w is not None:
            ags.reduce_momentum_sgd(wl.grads, wl.seg_offsets, wl.master_w, wl.momentum,
                                    lr=wl.lr, mu=wl.mu, out=None)
        else:
            ags.reduce(wl.grads, wl.seg_offsets, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = ags.launch_count()
    barrier(dist)
    torch.cuda.synchronize()
    # Inputs smaller than a few L2s: flush L2 (write 512 MB) before every timed step,
    # outside that step's event pair, and sum the per-step times.
    small_input = in_bytes < (1 << 30)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if small_input else None
    with ClockSampler(local) as clocks:
        if small_input:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(args.steps)]
            for a0, a1 in pairs:
                flush_buf.zero_()
                a0.record(stream)
                step()
                a1.record(stream)
            torch.cuda.synchronize()
            t_steps = sum(a0.elapsed_time(a1) for a0, a1 in pairs) / 1e3
        else:
            ev0.record(stream)
            for _ in range(args.steps):
                step()
            ev1.record(stream)
            torch.cuda.synchronize()
            t_steps = ev0.elapsed_time(ev1) / 1e3
    barrier(dist)
    launches = ags.launch_count() - launches0
    # Per-kernel CUDA-event times come from a second pass over the same K steps: events
    # around every launch would add their own cost to the step timed above (and
    # serialise launches the library lets overlap).
    ags.profile_enable(True)
    ags.profile_collect()
    torch.cuda.synchronize()
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for _ in range(args.steps):
        step()
    ev3.record(stream)
    torch.cuda.synchronize()
    kstats = ags.profile_collect()
    ags.profile_enable(False)
    t_instr = ev2.elapsed_time(ev3) / 1e3
    t_s = t_steps
    t_max = max_over_ranks(t_s, dist)
    total_bytes = sum_over_ranks(in_bytes * args.steps, dist)
    value = total_bytes / t_max / 1e9
    peak, peak_src = read_peaks()

    # dominant kernel: the largest summed event time among the streaming kernels (the
    # Gram and combine passes, the fused pair kernel), with the algorithmic bytes the
    # library counts for each launch from its plan (only the tiles, segments or pair that
    # launch covers).  The small-segment kernels are latency-bound and are not rated here;
    # the tiny-segment kernel runs concurrently on a second stream.
    def launch_bytes(k):
        n, _, b = kstats[k]
        return b / n if n else 0
    streaming = ("gram", "combine", "pair_fused")
    rated = {k: v for k, v in kstats.items() if k.startswith(streaming) and launch_bytes(k)} or kstats
    dom, (dom_n, dom_ms, _) = max(rated.items(), key=lambda kv: kv[1][1])
    dom_bytes = launch_bytes(dom)
    dom_gbs = dom_bytes / (dom_ms / dom_n / 1e3) / 1e9 if dom_bytes else None
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if args.shrink == 1 and os.path.exists(tpath):  # (the figures are per full-size launch)
        try:
            traffic = json.load(open(tpath)).get(args.workload, {}).get(dom)
        except Exception:
            traffic = None

    # end to end through host memory
    e2e = None
    if not args.no_e2e:
        # one C-ABI call per step (adasum_reduce_host): pinned host inputs in, the
        # combined result back in pinned host memory, the call returning when it is there
        host = [g.cpu().pin_memory() for g in wl.grads]
        out_host = torch.empty(wl.N, dtype=wl.dtype, pin_memory=True)
        ags.reduce_from_host(host, wl.seg_offsets, out_host=out_host)
        barrier(dist)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            ags.reduce_from_host(host, wl.seg_offsets, out_host=out_host)
        te = max_over_ranks(time.perf_counter() - t0, dist)
        e2e = {"value": round(sum_over_ranks(in_bytes * args.e2e_steps, dist) / te / 1e9, 3),
               "unit": UNIT, "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": wl.N * es,
               "steps": args.e2e_steps, "entry_point": "adasum_reduce_host"}
        del host

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        grads, sub, nbytes, desc, oracle = oracle_sample(wl, args.cpu_sample_bytes)
        t = time_oracle(grads, sub, oracle)
        cpu = {"value": round(nbytes / t / 1e9, 4), "unit": UNIT, "cores": 1,
               "kind": "oracle", "sample": desc, "seconds": round(t, 2)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_max / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "shrink": args.shrink,
                       "description": wl.description,
                       "K": wl.K, "N": wl.N, "segments": wl.L,
                       "storage_dtype": str(wl.dtype).replace("torch.", ""),
                       "input_bytes_per_step": in_bytes, "min_bytes_per_step": min_bytes,
                       "parallelism": f"replicas{world}",
                       "l2": ("inputs (%.3f GB) smaller than 1 GB: L2 flushed by a 512 MB write "
                              "before every timed step, outside its event pair" % (in_bytes / 1e9))
                             if small_input else
                             "inputs (%.1f GB) far larger than L2; no flush" % (in_bytes / 1e9)},
            "step_roofline": {"min_bytes": min_bytes,
                              "achieved_gbs": round(min_bytes * args.steps / t_max / 1e9, 2),
                              "peak": peak, "frac": round(min_bytes * args.steps / t_max / 1e9 / peak, 4)},
            "roofline": {"bound": "hbm", "kernel": dom,
                         "achieved": round(dom_gbs, 2) if dom_gbs else None, "peak": peak,
                         "peak_source": peak_src, "unit": "GB/s",
                         "frac": round(dom_gbs / peak, 4) if dom_gbs else None,
                         "algorithmic_bytes_per_launch": dom_bytes,
                         "avg_launch_ms": round(dom_ms / dom_n, 4), "traffic": traffic},
            "kernels": {k: {"launches": n, "total_ms": round(ms, 3), "bytes_per_launch": round(b / n) if n else 0}
                        for k, (n, ms, b) in kstats.items()},
            "kernel_timing": ("CUDA events around every launch, in a second pass over the same %d "
                              "steps (%.4f ms per step with the events; the timed steps run without)"
                              % (args.steps, t_instr * 1e3 / args.steps)),
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from adaptive_gradient_summation_gb300 import workloads
    wl = workloads.make(args.workload, device="cuda" if torch.cuda.is_available() else "cpu")
    grads, sub, nbytes, desc, oracle = oracle_sample(wl, args.ref_sample_bytes)
    del wl
    for _ in range(args.warmup):
        time_oracle(grads, sub, oracle)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(grads, sub, oracle)
    t = time.perf_counter() - t0
    value = nbytes * args.steps / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, "sample": desc},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bert_large_k16")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide every tensor of the workload by this (profiling small cases)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-bytes", type=int, default=5 << 30,
                    help="input bytes of the CPU-baseline sample (about 10 s of the fp64 oracle)")
    ap.add_argument("--ref-sample-bytes", type=int, default=64 << 20)
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
