#!/usr/bin/env python3
"""Benchmark of the DLRM sparse forward on B300.

Default workload: the production one-hot forward (B=65,536 samples, T=26 fp32
tables holding ~1.8e8 rows = ~92 GB, D=128, Zipf(1.05) lookups, N=27 -> 351
interaction values).  One step = one call of the fused sparse forward over one
batch (lookup + pooling + interaction + concatenation).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2|3|4|1]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Prints one JSON line (rank 0).  `value` is samples/s with inputs resident in
HBM and L2 flushed between steps; `e2e` is samples/s through the host-buffer
entry point (pinned host inputs copied in and the output copied back inside
the timed region, two streams so adjacent steps overlap).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gen  # noqa: E402

METRIC = "sparse-forward samples/s and effective HBM GB/s (% of B300 peak) at 1 GPU"
N_ROTATE = 8          # distinct pre-generated batches cycled through
FLUSH_BYTES = 512 << 20  # > 4x the 126 MB L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--max-rows", type=int, default=0,
                   help="cap every table at this many rows (a small case of the same kernel, for profiling)")
    p.add_argument("--uniform", action="store_true",
                   help="uniform instead of Zipf indices (every lookup a likely DRAM read)")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the slowest rank sets a job's time).
    Ranks hold no data-path collective; this host-side reduction is the only
    exchange, over the gloo process group."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(w: gen.Workload, batch: gen.Batch) -> int:
    """Bytes one fused forward must move: every looked-up row, the dense input,
    the output, the indices and the offsets (int32)."""
    return (batch.nnz * w.D * w.elem_bytes + w.B * w.D * 4 + w.B * w.out_width * 4 + batch.nnz * 4
            + (w.T * w.B + 1) * 4)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def traffic_for(workload: int):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on the
    kernel sources as they are now (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(str(workload))
    except (ValueError, OSError):
        return None
    if not d or d.get("sources_sha256") != sources_digest():
        return None
    return d.get("dram_bytes_per_launch")


def sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "embedding_bag_lookup_dlrm_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes)."""
    CLOCK_SM = 1
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4), ("hw_power_brake", 0x80))

    def __init__(self, cuda_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
        except Exception:
            pass
        rc = -1
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError(f"no NVML handle ({rc})")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self) -> float:
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v))
        return float(v.value)

    def max_sm_mhz(self) -> float:
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v))
        return float(v.value)

    def reasons(self) -> int:
        v = self.ct.c_ulonglong()
        self._reasons_fn(self.h, self.ct.byref(v))
        return int(v.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event (throttle) reasons, polled through NVML every
    `period` seconds on a background thread while the timed region runs.
    Reading only: nothing here changes a GPU setting."""

    def __init__(self, gpu_index: int, period: float = 0.002):
        self.gpu, self.period = gpu_index, period
        self.samples, self.reasons, self.max_mhz, self.error = [], set(), None, None
        self._nv = None

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        try:
            self._nv = _Nvml(self.gpu)
            self.max_mhz = self._nv.max_sm_mhz()
            self._poll()
        except Exception as e:  # no NVML: report the absence instead of guessing
            self.error = repr(e)
            self._nv = None
            return self
        self._t = threading.Thread(target=self._loop, daemon=True)
        self._t.start()
        return self

    def _poll(self):
        self.samples.append(self._nv.sm_mhz())
        mask = self._nv.reasons()
        for name, bit in _Nvml.REASONS:
            if mask & bit:
                self.reasons.add(name)

    def _loop(self):
        while not self._stop.is_set():
            try:
                self._poll()
            except Exception as e:
                self.error = repr(e)
                return
            time.sleep(self.period)

    def __exit__(self, *exc):
        self._stop.set()
        if self._nv is not None:
            self._t.join(timeout=5)
            try:
                self._poll()
                self._nv.close()
            except Exception:
                pass

    def summary(self):
        d = {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
             "reasons": sorted(self.reasons), "samples": len(self.samples), "source": "NVML, 2 ms polling"}
        if self.error:
            d["error"] = self.error
        return d


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on host cores
# ---------------------------------------------------------------------------
def oracle_baseline(w: gen.Workload, batch: gen.Batch, seconds: float):
    """Time the oracle's sparse forward on whole batches of the workload until
    `seconds` have passed.  Tables: host copies of the rows the batch touches."""
    import oracle
    orc = oracle.get()
    tabs, nr, cidx = gen.compact_tables(w, batch)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    orc.sparse_fwd(tabs, nr, cidx, batch.offsets, batch.dense, w.mode, w.dtype)  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        orc.sparse_fwd(tabs, nr, cidx, batch.offsets, batch.dense, w.mode, w.dtype)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": n * w.B / el, "unit": "samples/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} x one full batch of {w.B} samples (rows the batch touches copied to host memory), "
                      f"{el:.1f} s"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    orc = oracle.get()
    batches = gen.make_batches(w, range(min(N_ROTATE, max(1, args.steps))))
    prepared = [(b, gen.compact_tables(w, b)) for b in batches]
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    # each step: a bounded sample of the batch (first S samples) sized to ~1-2 s
    S = min(w.B, 16384)

    def sub(b, tabs_nr_idx, S):
        tabs, nr, cidx = tabs_nr_idx
        off = b.offsets.astype(np.int64)
        L = np.diff(off).reshape(w.T, w.B)[:, :S]
        new_off = np.zeros(w.T * S + 1, np.int64)
        np.cumsum(L.reshape(-1), out=new_off[1:])
        idx = np.concatenate([cidx[off[t * w.B]:off[t * w.B] + L[t].sum()] for t in range(w.T)])
        return tabs, nr, idx, new_off, b.dense[:S]

    subs = [sub(b, p, S) for b, p in prepared]
    for i in range(args.warmup):
        tabs, nr, idx, off, x = subs[i % len(subs)]
        orc.sparse_fwd(tabs, nr, idx, off, x, w.mode, w.dtype)
    t0 = time.perf_counter()
    for i in range(args.steps):
        tabs, nr, idx, off, x = subs[i % len(subs)]
        orc.sparse_fwd(tabs, nr, idx, off, x, w.mode, w.dtype)
    el = time.perf_counter() - t0
    value = args.steps * S / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "samples/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator)", "config": config_of(w, args),
            "cpu_baseline": {"value": value, "unit": "samples/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: first {S} samples of one of {len(subs)} rotated batches; "
                                       "rows the batch touches copied to host memory"},
            "e2e": {"value": value, "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, args):
    return {"workload": w.name, "global_batch": w.B * args.gpus, "batch_per_gpu": w.B, "tables": w.T, "dim": w.D,
            "table_dtype": w.dtype, "table_rows_total": int(sum(w.num_rows)),
            "table_gb": round(w.table_bytes() / 1e9, 2), "pooling": w.mode,
            "bag_lengths": f"{w.bag_min}..{w.bag_max}", "index_dist": w.index_dist
            + (f"({w.alpha})" if w.index_dist == "zipf" else ""), "interaction_values": w.N * (w.N - 1) // 2,
            "rotated_batches": N_ROTATE, "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MB write)",
            "parallelism": f"replicas x{args.gpus} (no data-path collective)"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import embedding_bag_lookup_dlrm_b300 as dl

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dl.load_library()

    # tables: filled on the device by the seeded generator
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    tabs = []
    stream = torch.cuda.current_stream()
    for t, V in enumerate(w.num_rows):
        x = torch.empty((V, w.D), dtype=dt, device=dev)
        gen.fill_table_device(x.data_ptr(), w.dtype, w.seed, t, 0, V, w.D, stream.cuda_stream)
        tabs.append(x)
    tables = dl.Tables(tabs)
    batches = gen.make_batches(w, [rank * 1000 + i for i in range(N_ROTATE)])
    dev_batches = [tuple(torch.from_numpy(a).to(dev) for a in (b.indices, b.offsets, b.dense)) for b in batches]
    out = torch.empty((w.B, w.out_width), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def step(i, s):
        idx, off, x = dev_batches[i % N_ROTATE]
        dl.dlrm_sparse_fwd(tables, idx, off, x, w.mode, out=out, stream=s)

    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for i in range(args.warmup):
            flush.zero_()
            step(i, s)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    with ClockSampler(local) as clk, torch.cuda.stream(s):
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()                      # evict L2 (outside the timed events)
            starts[i].record(s)
            step(args.warmup + i, s)
            launches += 1                      # one fused kernel per step
            ends[i].record(s)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = w.B * world * args.steps / (total_ms / 1e3)

    # roofline of the fused kernel (the step is that one kernel)
    alg = statistics.mean(algorithmic_bytes(w, b) for b in batches)
    kernel_ms = statistics.mean(step_ms)
    achieved = alg / (kernel_ms / 1e3) / 1e9
    peak, src = peaks()
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic_for(args.workload),
            "kernel": "forward_kernel (fused sparse forward)", "peak_source": f"{src} (hbm_gbs)",
            "algorithmic_bytes_per_launch": int(alg), "frac_of_nominal_8000": round(achieved / 8000.0, 4),
            "median_launch_ms": round(statistics.median(step_ms), 4)}

    # end to end: pinned host inputs -> device -> fused forward -> output to host
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, tables, batches, dev, dl, torch, world)

    cpu = None
    if rank == 0 and not args.no_cpu and world == 1:
        cpu = oracle_baseline(w, batches[0], args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "samples/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded generator, tables filled on device)", "config": config_of(w, args),
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk.summary(), "wall_s_timed_region": round(t_wall, 3),
                "effective_gbs": round(achieved, 1)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, w, tables, batches, dev, dl, torch, world):
    import torch.distributed as dist
    host = []
    for b in batches:
        host.append(tuple(torch.from_numpy(a).pin_memory() for a in (b.indices, b.offsets, b.dense)))
    max_nnz = max(b.nnz for b in batches)
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    stages = [dl.HostStaging(w.B, w.T, w.D, max_nnz, torch.int32, dev) for _ in range(2)]
    outs = [torch.empty((w.B, w.out_width), dtype=torch.float32).pin_memory() for _ in range(2)]
    done = [None, None]

    def step(i):
        k = i % 2
        if done[k] is not None:
            done[k].synchronize()  # the host buffer of two steps ago is free again
        idx, off, x = host[i % N_ROTATE]
        dl.dlrm_sparse_fwd_host(tables, idx, off, x, outs[k], stages[k], w.mode, stream=streams[k])
        ev = torch.cuda.Event()
        ev.record(streams[k])
        done[k] = ev

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    el = max_over_ranks(el, world)
    b0 = batches[0]
    h2d = int(np.mean([b.indices.nbytes + b.offsets.nbytes + b.dense.nbytes for b in batches]))
    d2h = w.B * w.out_width * 4
    return {"value": round(w.B * world * args.steps / el, 1), "unit": "samples/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(el / args.steps * 1e3, 4),
            "how": "dlrm_sparse_fwd_host on pinned host buffers, two streams alternating (copies of one step "
                   "overlap the kernel of the next); wall clock over the timed steps"}


def main():
    args = parse()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    w = gen.workload(args.workload)
    if args.max_rows > 0:
        w.num_rows = [min(v, args.max_rows) for v in w.num_rows]
        w.name += f" [tables capped at {args.max_rows} rows]"
    if args.uniform:
        w.index_dist = "uniform"
        w.name += " [uniform indices]"
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
