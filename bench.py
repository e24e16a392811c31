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
TRAIN_METRIC = ("sparse training-step samples/s (forward, interaction backward, sorted per-row gradient sums, "
                "row-wise Adagrad) and effective HBM GB/s at 1 GPU")
N_ROTATE = 8          # distinct pre-generated batches cycled through
FLUSH_BYTES = 512 << 20  # > 4x the 126 MB L2
DRAIN_BYTES = 256 << 20  # read after the flush write, so its dirty lines reach DRAM before the timed region


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--max-rows", type=int, default=0,
                   help="cap every table at this many rows (a small case of the same kernel, for profiling)")
    p.add_argument("--batch", type=int, default=0,
                   help="override the batch size (a small case of the same kernels, for profiling)")
    p.add_argument("--uniform", action="store_true",
                   help="uniform instead of Zipf indices (every lookup a likely DRAM read)")
    p.add_argument("--rule", choices=["adagrad", "sgd"], default="adagrad",
                   help="row update rule of the training workload")
    p.add_argument("--shards", type=int, default=1,
                   help="G > 1: table-wise model parallelism over G logical shards on this device (the "
                        "embedding-bag lookup per table shard, the exchange, the interaction per sample shard)")
    p.add_argument("--op", choices=["fused", "embbag"], default="fused",
                   help="embbag: time the embedding-bag lookup alone (pooled vectors written to HBM)")
    p.add_argument("--tier", type=float, default=0.0,
                   help="F > 0: the tables live in pinned host memory with a device cache of the fraction F of each "
                        "table's rows (the hottest in separate history batches); each step stages its lookups, then "
                        "runs the forward on the device buffers")
    p.add_argument("--model", action="store_true",
                   help="the whole DLRM training step on the training workload: bottom MLP 13-512-256-D, the sparse "
                        "path, top MLP (D+K)-512-256, a 256-1 sigmoid head with BCE; SGD on the MLPs")
    p.add_argument("--sort-in-backward", action="store_true",
                   help="training workload: the backward's key build and sort run inside the backward call, beside "
                        "the interaction backward, instead of beside the forward (dlrm_sparse_bwd_sort)")
    p.add_argument("--side-priority", choices=["high", "low"], default=None,
                   help="priority of the training step's side stream (key build and sort); default high for the "
                        "sparse step (measured 1.136 against 1.147 ms), low for the whole model step (whose short "
                        "GEMMs the sort's blocks would delay: 2.085 against 2.095 ms)")
    p.add_argument("--hash", action="store_true",
                   help="the bags arrive as raw 64-bit IDs: the hashing pre-pass (ID mod V_t) runs in each step")
    args = p.parse_args()
    if args.side_priority is None:
        args.side_priority = "low" if args.model else "high"
    return args


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


def sort_passes(w: gen.Workload) -> int:
    """LSD radix passes (digits of at most 9 bits) over keys below the total row count."""
    bits = 1
    while (1 << bits) <= sum(w.num_rows):
        bits += 1
    return (bits + 8) // 9


def train_bytes(w: gen.Workload, batch: gen.Batch, rule: str = "adagrad") -> dict:
    """Bytes one training step must move (int32 indices), by phase.
    forward: looked-up rows, x, out, pooled vectors saved, indices, offsets.
    backward, two models that differ only in the reads of dP:
      "per_bag":    dP written once and read once (a read per bag), the model the
                    workload description uses;
      "per_lookup": dP read once per lookup, which is what a reduction of the
                    lookups sorted by row reads: the rows a bag's lookups touch
                    are scattered over the sorted order, so every lookup fetches
                    its bag's dP row, and at B*T*D*4 bytes (436 MB for the
                    training workload) dP does not stay in the 126 MB L2.
    Both count grad_out, x and pooled read, grad_dense written, the lookup keys
    written, (key, value) read and written by each radix pass, and per touched
    row its weights read and written (and for Adagrad its accumulator)."""
    nnz = batch.nnz
    BTD = w.B * w.T * w.D * 4
    off = batch.offsets.astype(np.int64)
    touched = sum(int(np.unique(batch.indices[off[t * w.B]:off[(t + 1) * w.B]]).size) for t in range(w.T))
    fwd = (nnz * w.D * w.elem_bytes + w.B * w.D * 4 + w.B * w.out_width * 4 + BTD + nnz * 4
           + (w.T * w.B + 1) * 4)
    row = 2 * w.D * 4 + (8 if rule == "adagrad" else 0)
    common = (w.B * w.out_width * 4 + w.B * w.D * 4 + BTD + w.B * w.D * 4 + BTD + nnz * 8
              + sort_passes(w) * nnz * 16 + touched * row + nnz * 4 + (w.T * w.B + 1) * 4)
    per_bag = common + BTD
    per_lookup = common + nnz * w.D * 4
    return {"forward": fwd, "backward": per_bag, "backward_per_lookup": per_lookup, "total": fwd + per_bag,
            "touched_rows": touched}


def hash_bytes(w: gen.Workload, batch: gen.Batch) -> int:
    """Bytes of the hashing pre-pass: a raw 8-byte ID read and a 4-byte row written per lookup, and the
    T + 1 table boundaries of the offsets."""
    return batch.nnz * 12 + (w.T + 1) * 4


def exchange_bytes(w: gen.Workload) -> int:
    """Bytes of one exchange of the pooled vectors: every (sample, table) row read once and written once."""
    return 2 * w.B * w.T * w.D * 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


FORWARD_SOURCES = ("common.cuh", "fwd_tc.cu", "tc.cuh")  # the tensor-core forward kernel's own sources


def traffic_record(workload: int):
    """The committed DRAM-traffic record of a workload's forward kernel (profiles/traffic.json), if it was
    taken on the kernel sources as they are now (else None).  Records hold capped-table captures."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(str(workload))
    except (ValueError, OSError):
        return None
    if not d or d.get("sources_sha256") != sources_digest(FORWARD_SOURCES):
        return None
    return d


def traffic_for(workload: int):
    """DRAM bytes per full-size launch, when a committed capture scales to it (else None)."""
    d = traffic_record(workload)
    return d.get("dram_bytes_per_launch") if d and d.get("scales_to_full_size") else None


def sources_digest(files) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "embedding_bag_lookup_dlrm_b300", "csrc")
    for name in sorted(files):
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
def sub_batch(w: gen.Workload, b: gen.Batch, S: int):
    """The first S samples of a batch (all their bags), as a workload of batch S."""
    import dataclasses
    S = min(S, w.B)
    off = b.offsets.astype(np.int64)
    L = np.diff(off).reshape(w.T, w.B)[:, :S]
    new_off = np.zeros(w.T * S + 1, np.int64)
    np.cumsum(L.reshape(-1), out=new_off[1:])
    idx = np.concatenate([b.indices[off[t * w.B]:off[t * w.B] + L[t].sum()] for t in range(w.T)])
    g = b.grad_out[:S] if b.grad_out is not None else None
    return (dataclasses.replace(w, B=S),
            gen.Batch(indices=idx.astype(np.int32), offsets=new_off.astype(np.int32), dense=b.dense[:S], grad_out=g))


class OracleStep:
    """One step of the path on the CPU oracle (plain C, OpenMP over samples):
    the fused forward, and for training also the interaction backward, the
    per-row gradient sums and the row update.  Tables are host copies of the
    rows the batch touches."""

    def __init__(self, w: gen.Workload, b: gen.Batch, rule: str = "adagrad"):
        import oracle
        self.orc = oracle.get()
        self.w, self.b, self.rule = w, b, rule
        self.tabs, self.nr, self.idx = gen.compact_tables(w, b)
        if w.train:
            self.acc = [np.full(n, w.accum_init, np.float32) for n in self.nr] if rule == "adagrad" else None

    def __call__(self):
        w, b = self.w, self.b
        r = self.orc.sparse_fwd(self.tabs, self.nr, self.idx, b.offsets, b.dense, w.mode, w.dtype,
                                with_pooled=w.train)
        if w.train:
            self.orc.sparse_bwd_update(self.tabs, self.nr, self.idx, b.offsets, b.dense, r["pooled"], b.grad_out,
                                       self.rule, w.lr, w.eps, self.acc, w.mode)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def oracle_baseline(w: gen.Workload, batch: gen.Batch, seconds: float, rule: str = "adagrad"):
    """Time the oracle on a bounded part of the workload (the first 16,384
    samples of a forward batch, 4,096 of a training batch) at all host cores,
    then at one thread, each for about half of `seconds`.  The thread count
    changes no arithmetic."""
    S = 4096 if w.train else 16384
    ws, bs = sub_batch(w, batch, S)
    run = OracleStep(ws, bs, rule)
    all_threads = run.orc.set_threads(os.cpu_count() or 1)

    def timed(threads, secs):
        got = run.orc.set_threads(threads)
        run()  # warm
        n, t0 = 0, time.perf_counter()
        while True:
            run()
            n += 1
            el = time.perf_counter() - t0
            if el >= secs:
                return n * ws.B / el, got, f"{n} x the first {ws.B} samples of one batch, {el:.1f} s"

    v_all, c_all, what_all = timed(all_threads, seconds / 2)
    v_one, _, what_one = timed(1, seconds / 2)
    run.orc.set_threads(all_threads)
    return {"value": v_all, "unit": "samples/s", "cores": c_all, "kind": "oracle",
            "sample": what_all + " (rows the batch touches copied to host memory)",
            "one_thread": {"value": v_one, "unit": "samples/s", "sample": what_one},
            "cpu_model": cpu_model(), "nproc": os.cpu_count()}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    batches = gen.make_batches(w, range(min(N_ROTATE, max(1, args.steps))))
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    # each step: a bounded sample of one batch (its first S samples), about a second of CPU work
    S = min(w.B, 4096 if w.train else 16384)
    runs = [OracleStep(*sub_batch(w, b, S), args.rule) for b in batches]
    for i in range(args.warmup):
        runs[i % len(runs)]()
    t0 = time.perf_counter()
    for i in range(args.steps):
        runs[i % len(runs)]()
    el = time.perf_counter() - t0
    value = args.steps * S / el
    line = {"impl": "reference", "metric": TRAIN_METRIC if w.train else METRIC, "value": value,
            "unit": "samples/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generator)", "config": config_of(w, args),
            "cpu_baseline": {"value": value, "unit": "samples/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: first {S} samples of one of {len(runs)} rotated batches; "
                                       "rows the batch touches copied to host memory"},
            "e2e": {"value": value, "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, args):
    return {"workload": w.name, "global_batch": w.B * args.gpus, "batch_per_gpu": w.B, "tables": w.T, "dim": w.D,
            "table_dtype": w.dtype, "table_rows_total": int(sum(w.num_rows)),
            "table_gb": round(w.table_bytes() / 1e9, 2), "pooling": w.mode,
            "bag_lengths": f"{w.bag_min}..{w.bag_max}", "index_dist": w.index_dist
            + (f"({w.alpha})" if w.index_dist == "zipf" else ""), "interaction_values": w.N * (w.N - 1) // 2,
            "rotated_batches": N_ROTATE,
            "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MB write, then a {DRAIN_BYTES >> 20} MB read so "
                  "the flush's dirty lines are written back outside the timed region)",
            "parallelism": f"replicas x{args.gpus} (no data-path collective)"
            + (f"; tables split over {args.shards} logical shards on each device (table-wise model parallel, "
               "all-to-all by the exchange kernel)" if args.shards > 1 else ""),
            **({"update_rule": args.rule} if w.train else {}),
            **({"indices": "raw 64-bit IDs, hashed to rows (ID mod V_t) inside each step"} if args.hash else {}),
            **({"op": "embedding-bag lookup alone (dlrm_embbag_fwd), pooled vectors written"}
               if args.op == "embbag" else {}),
            **({"host_tier": f"tables in pinned host memory; device cache of {args.tier:g} of each table's rows, "
                             "filled with the hottest rows of separate history batches"} if args.tier > 0 else {})}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def phase_bytes(args, w: gen.Workload, b: gen.Batch) -> dict:
    """Algorithmic bytes of each phase of one step of this configuration (int32 indices)."""
    BTD = w.B * w.T * w.D * 4
    rows = b.nnz * w.D * w.elem_bytes
    csr = b.nnz * 4 + (w.T * w.B + 1) * 4
    out = w.B * w.out_width * 4
    x = w.B * w.D * 4
    ph = {}
    if args.hash:
        ph["hash"] = hash_bytes(w, b)
    if args.shards > 1:
        ph["lookup"] = rows + csr + BTD
        ph["exchange"] = exchange_bytes(w)
        ph["interaction"] = BTD + x + out
        if w.train:
            tb = train_bytes(w, b, args.rule)
            ph["interaction_bwd"] = out + x + BTD + x + BTD
            ph["exchange_bwd"] = exchange_bytes(w)
            ph["update"] = tb["backward"] - ph["interaction_bwd"]
        return ph
    if args.op == "embbag":
        ph["lookup"] = rows + csr + BTD
        return ph
    if args.tier > 0:
        ph["stage"] = b.nnz * 12 + b.tier_misses * w.D * w.elem_bytes * 2  # index, map, rewritten index; staged rows
        ph["forward"] = algorithmic_bytes(w, b)
        return ph
    if w.train:
        tb = train_bytes(w, b, args.rule)
        ph["forward"] = tb["forward"]
        ph["backward"] = tb["backward"]
    else:
        ph["forward"] = algorithmic_bytes(w, b)
    return ph


def raw_ids_for(w: gen.Workload, b: gen.Batch, seed: int) -> np.ndarray:
    """Raw 64-bit IDs whose hash (ID mod V_t) is the batch's row: row + V_t * k, k random, so the hashed
    step looks up exactly the rows of the plain step."""
    rng = np.random.default_rng(seed)
    off = b.offsets.astype(np.int64)
    raw = np.empty(b.nnz, np.uint64)
    for t in range(w.T):
        lo, hi = off[t * w.B], off[(t + 1) * w.B]
        V = w.num_rows[t]
        k = rng.integers(0, (1 << 63) // V, size=hi - lo, dtype=np.uint64)
        raw[lo:hi] = b.indices[lo:hi].astype(np.uint64) + k * np.uint64(V)
    return raw.view(np.int64)


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import embedding_bag_lookup_dlrm_b300 as dl
    from embedding_bag_lookup_dlrm_b300 import sharding

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dl.load_library()
    if args.hash and args.shards > 1:
        raise SystemExit("--hash and --shards together are not a configuration of this bench")
    if args.op == "embbag" and args.shards > 1:
        raise SystemExit("--op embbag times the lookup of an unsharded workload")

    # tables: filled on the device by the seeded generator (copied to pinned host memory for the host tier)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    tabs = []
    stream = torch.cuda.current_stream()
    for t, V in enumerate(w.num_rows):
        x = torch.empty((V, w.D), dtype=dt, device=dev)
        gen.fill_table_device(x.data_ptr(), w.dtype, w.seed, t, 0, V, w.D, stream.cuda_stream)
        if args.tier > 0:
            h = torch.empty((V, w.D), dtype=dt).pin_memory()
            h.copy_(x)
            del x
            x = h
        tabs.append(x)
    batches = gen.make_batches(w, [rank * 1000 + i for i in range(N_ROTATE)])
    if args.tier > 0:
        # the cache: each table's hottest rows in separate history batches, not the timed ones
        history = gen.make_batches(w, [rank * 1000 + 500 + i for i in range(N_ROTATE)])
        cap = [max(0, int(args.tier * V)) for V in w.num_rows]
        hot = dl.hot_rows([h.indices for h in history], [h.offsets for h in history], w.B, w.T, cap, w.num_rows)
        stage_rows = [max(int(b.offsets[(t + 1) * w.B]) - int(b.offsets[t * w.B]) for b in batches)
                      for t in range(w.T)]
        tier = dl.TieredTables(tabs, cap, stage_rows, dev)
        for t in range(w.T):
            tier.fill(t, torch.from_numpy(hot[t]).to(dev))
        for b in batches:  # lookups the cache misses (they are copied over the host link in the step)
            off = b.offsets.astype(np.int64)
            b.tier_misses = sum(int((~np.isin(b.indices[off[t * w.B]:off[(t + 1) * w.B]], hot[t])).sum())
                                for t in range(w.T))
        tables = tier.device_tables
        staged = torch.empty(max(b.nnz for b in batches), dtype=torch.int32, device=dev)
    else:
        tables = dl.Tables(tabs)
    dev_batches = [tuple(torch.from_numpy(a).to(dev) for a in (b.indices, b.offsets, b.dense)) for b in batches]
    out = torch.empty((w.B, w.out_width), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(DRAIN_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        """Evict L2: write a buffer 4x its size, then read another, so the flush's
        own dirty lines are written back before (not inside) the timed step."""
        flush.zero_()
        drain.sum()

    if args.op == "embbag":
        pooled_out = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device=dev)
    if args.hash:
        raws = [torch.from_numpy(raw_ids_for(w, b, 77 + i)).to(dev) for i, b in enumerate(batches)]
        hashed = torch.empty(max(b.nnz for b in batches), dtype=torch.int32, device=dev)
    if args.shards > 1:
        plan = sharding.ShardPlan.make(w.num_rows, w.D, w.B, args.shards, w.elem_bytes)
        shard_bags = [[(torch.from_numpy(i).to(dev), torch.from_numpy(o).to(dev))
                       for i, o in sharding.split_bags(plan, b.indices, b.offsets)] for b in batches]
        sharded = sharding.ShardedSparse(tabs, plan)
    if w.train:
        accum = ([torch.full((V,), w.accum_init, dtype=torch.float32, device=dev) for V in w.num_rows]
                 if args.rule == "adagrad" else None)
        grads = [torch.from_numpy(b.grad_out).to(dev) for b in batches]
        pooled = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device=dev)
        grad_dense = torch.empty((w.B, w.D), dtype=torch.float32, device=dev)
        ws_bytes = max(dl.dlrm_sparse_bwd_workspace_size(tables, torch.from_numpy(b.indices), torch.from_numpy(b.offsets))
                       for b in batches)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    s = torch.cuda.Stream(device=dev)
    # the training step's key build and sort run beside its forward and interaction backward, on a stream
    # of the highest priority (or, --side-priority low, the lowest) so that the short dependent sort kernels
    # get SMs as soon as any free up
    side = torch.cuda.Stream(device=dev, priority=0 if args.side_priority == "low" else -100)

    def step(i, rec):
        """Queue step i on stream s; rec(name) records the end of a phase."""
        k = i % N_ROTATE
        idx, off, x = dev_batches[k]
        if args.hash:
            idx = dl.dlrm_hash_indices(w.num_rows, raws[k], off, rows=hashed[:raws[k].numel()], stream=s)
            rec("hash")
        if args.tier > 0:
            idx = tier.stage(idx, off, out=staged[:idx.numel()], stream=s)
            rec("stage")
        if args.shards > 1:
            sharded.forward(shard_bags[k], x, w.mode, out=out, stream=s, after=rec)
            if w.train:
                sharded.backward(shard_bags[k], x, grads[k], args.rule, w.lr, w.eps, accum, w.mode,
                                 grad_dense=grad_dense, stream=s, after=rec)
            return
        if args.op == "embbag":
            dl.dlrm_embbag_fwd(tables, idx, off, w.mode, pooled=pooled_out, stream=s)
            rec("lookup")
            return
        if not w.train:
            dl.dlrm_sparse_fwd(tables, idx, off, x, w.mode, out=out, stream=s)
            rec("forward")
            return
        if args.sort_in_backward:
            dl.dlrm_sparse_fwd(tables, idx, off, x, w.mode, out=out, pooled_save=pooled, stream=s)
            rec("forward")
            dl.dlrm_sparse_bwd_update(tables, idx, off, x, pooled, grads[k], args.rule, w.lr, w.eps, accum, w.mode,
                                      grad_dense=grad_dense, workspace=workspace, stream=s, side_stream=side)
            rec("backward")
            return
        # the sort depends only on the bags: it runs on the side stream beside the forward and the
        # interaction backward; only the backward's per-row sums wait for it
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork.record(s)
        side.wait_event(fork)
        dl.dlrm_sparse_bwd_sort(tables, idx, off, workspace, stream=side)
        join.record(side)
        dl.dlrm_sparse_fwd(tables, idx, off, x, w.mode, out=out, pooled_save=pooled, stream=s)
        rec("forward")
        dl.dlrm_sparse_bwd_update_sorted(tables, idx, off, x, pooled, grads[k], args.rule, w.lr, w.eps, accum,
                                         w.mode, grad_dense=grad_dense, workspace=workspace, sorted=join, stream=s)
        rec("backward")

    with torch.cuda.stream(s):
        for i in range(args.warmup):
            flush_l2()
            step(i, lambda name: None)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    marks = [[] for _ in range(args.steps)]  # (phase, event) per step, in order

    def recorder(i):
        def rec(name):
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(s)
            marks[i].append((name, ev))
        return rec

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # kernels of one step (our library's launches)
    per_step = launches_per_step(args, w, plan if args.shards > 1 else None)
    launches = 0
    with ClockSampler(local) as clk, torch.cuda.stream(s):
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush_l2()                         # evict L2 (outside the timed events)
            starts[i].record(s)
            step(args.warmup + i, recorder(i))
            launches += per_step
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(m[-1][1]) for a, m in zip(starts, marks)]
    phase_ms = {}
    for a, m in zip(starts, marks):
        prev = a
        for name, ev in m:
            phase_ms.setdefault(name, []).append(prev.elapsed_time(ev))
            prev = ev
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = w.B * world * args.steps / (total_ms / 1e3)
    peak, src = peaks()

    pb = [phase_bytes(args, w, b) for b in batches]
    phases = {}
    for name, ms in phase_ms.items():
        by = statistics.mean(p[name] for p in pb)
        gbs = by / (statistics.mean(ms) / 1e3) / 1e9
        phases[name] = {"ms": round(statistics.mean(ms), 4), "bytes": int(by), "gbs": round(gbs, 1),
                        "frac": round(gbs / peak, 4)}
    dom = max(phases, key=lambda n: phases[n]["ms"])
    step_bytes = sum(p["bytes"] for p in phases.values())
    effective = step_bytes / (statistics.mean(step_ms) / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": phases[dom]["gbs"], "peak": peak, "unit": "GB/s",
            "frac": phases[dom]["frac"], "traffic": traffic_for(args.workload) if phase_is_traced(args, dom) else None,
            "kernel": kernel_of_phase(args, w, dom), "phase": dom, "peak_source": f"{src} (hbm_gbs, burst copy)",
            **({"traffic_capped_tables": capped_traffic(traffic_record(args.workload))}
               if phase_is_traced(args, dom) and traffic_record(args.workload) else {}),
            "algorithmic_bytes_per_launch": phases[dom]["bytes"], "frac_of_nominal_8000":
            round(phases[dom]["gbs"] / 8000.0, 4), "median_launch_ms": round(statistics.median(phase_ms[dom]), 4),
            "phases": phases, "step_effective_gbs": round(effective, 1), "step_frac": round(effective / peak, 4)}
    if w.train and args.shards == 1:
        tbs = [train_bytes(w, b, args.rule) for b in batches]
        lookup_model = statistics.mean(t["backward_per_lookup"] for t in tbs)
        bw = lookup_model / (statistics.mean(phase_ms["backward"]) / 1e3) / 1e9
        roof["backward_per_lookup_model"] = {"bytes": int(lookup_model), "gbs": round(bw, 1),
                                             "frac": round(bw / peak, 4)}
        roof["touched_rows"] = int(statistics.mean(t["touched_rows"] for t in tbs))

    if args.tier > 0:
        link = host_link(torch, dev, 256 << 20, 256 << 20)
        st = phases["stage"]
        miss_bytes = statistics.mean(b.tier_misses for b in batches) * w.D * w.elem_bytes
        roof["tier"] = {"cached_fraction": args.tier, "cache_rows": int(sum(tier.C)),
                        "miss_lookups_per_step": int(statistics.mean(b.tier_misses for b in batches)),
                        "lookups_per_step": int(statistics.mean(b.nnz for b in batches)),
                        "host_bytes_per_step": int(miss_bytes),
                        "stage_host_gbs": round(miss_bytes / (st["ms"] / 1e3) / 1e9, 1),
                        "host_link_h2d_gbs": link["h2d_gbs"],
                        "stage_frac_of_host_link": round(miss_bytes / (st["ms"] / 1e3) / 1e9 / link["h2d_gbs"], 4)}

    e2e = None
    if not args.no_e2e and args.shards == 1 and not args.hash and args.op == "fused" and args.tier == 0:
        e2e = (run_e2e_train(args, w, tables, batches, dev, dl, torch, world, side) if w.train
               else run_e2e(args, w, tables, batches, dev, dl, torch, world))
        e2e["host_link"] = host_link(torch, dev, e2e["h2d_bytes_per_step"], e2e["d2h_bytes_per_step"])

    cpu = None
    if rank == 0 and not args.no_cpu and world == 1:
        cpu = oracle_baseline(w, batches[0], args.cpu_seconds, args.rule)

    if rank == 0:
        line = {"metric": TRAIN_METRIC if w.train else METRIC, "value": round(value, 1), "unit": "samples/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded generator, tables filled on device)", "config": config_of(w, args),
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk.summary(), "wall_s_timed_region": round(t_wall, 3),
                "effective_gbs": round(effective, 1)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def passes_for_rows(total_rows: int) -> int:
    bits = 1
    while (1 << bits) <= total_rows:
        bits += 1
    return (bits + 8) // 9


def launches_per_step(args, w, plan=None) -> int:
    """Kernels of this library one step launches."""
    n = (1 if args.hash else 0) + (1 if args.tier > 0 else 0)
    if plan is not None:
        G = plan.G
        n += G + 1 + plan.H  # lookup per table shard, exchange, interaction per sample shard
        if w.train:
            # interaction backward per sample shard, exchange, per table shard: key fill and expansion,
            # 3 per radix pass over that shard's rows, 2 row updates (+ the bag-length scaling in mean mode)
            n += plan.H + 1
            for g in range(G):
                rows = sum(w.num_rows[t] for t in plan.tables_of(g))
                n += 4 + 3 * passes_for_rows(rows) + (1 if w.mode == "mean" else 0)
        return n
    bwd = 5 + 3 * sort_passes(w)  # interaction backward, key fill and expansion, 3 per radix pass, 2 row updates
    if args.op != "fused":
        return n + 1
    return n + forward_launches(w) + (bwd if w.train else 0)


def phase_is_traced(args, phase) -> bool:
    """profiles/traffic.json holds DRAM bytes of the plain forward kernel (capped tables, Zipf and uniform)."""
    return args.shards == 1 and args.max_rows == 0 and phase == "forward"


def capped_traffic(rec: dict) -> dict:
    """The capped-table captures of a traffic record, each with its DRAM GB/s (read + write over the
    captured launch's duration) beside its L2 hit rate."""
    out = {}
    for k in ("small_case", "small_case_uniform"):
        if k in rec:
            c = dict(rec[k])
            c["dram_gbs"] = round((c["dram_read_bytes"] + c["dram_write_bytes"]) / (c["duration_us"] * 1e3), 1)
            out[k] = c
    if "why_null" in rec:
        out["why_null"] = rec["why_null"]
    return out


def kernel_of_phase(args, w, phase) -> str:
    return {"forward": forward_kernel_name(w),
            "backward": ("dlrm_sparse_bwd_update kernels (interaction backward, keys, radix sort, row updates; "
                         f"{args.rule})" if args.sort_in_backward else
                         "dlrm_sparse_bwd_update_sorted kernels (interaction backward, row updates; "
                         f"{args.rule}); the key build and radix sort run on a second stream from the "
                         "step's start, beside the forward and the interaction backward, so the two phases share "
                         "their time (step_frac is the whole step's bytes over its time)"),
            "hash": "hash_kernel (raw ID mod V_t)",
            "stage": "stage_kernel (cache slots, misses copied from host memory)",
            "lookup": "embbag_kernel (embedding-bag lookup, a lane group per bag"
                      + (", once per table shard)" if args.shards > 1 else ")"),
            "exchange": "exchange_kernel (all-to-all of the pooled vectors between logical shards)",
            "interaction": "interaction forward per sample shard (forward_tc_kernel, pooled inputs)",
            "interaction_bwd": "interact_bwd_kernel per sample shard",
            "exchange_bwd": "exchange_kernel (pooled gradients back to the table owners)",
            "update": f"embedding-bag backward per table shard (keys, radix sort, row updates; {args.rule})"}[phase]


def host_link(torch, dev, h2d_bytes, d2h_bytes, reps=5):
    """The host link alone: bare pinned cudaMemcpyAsync copies of one step's input and output bytes, each
    direction timed on its own (CUDA events, best of `reps`), and both directions at once."""
    hi = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    di = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    do = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    ho = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            el = time.perf_counter() - t0
            best = el if best is None else min(best, el)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            di.copy_(hi, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            ho.copy_(do, non_blocking=True)

    t_in, t_out = timed(h2d), timed(d2h)
    t_both = timed(lambda: (h2d(), d2h()))
    return {"h2d_gbs": round(h2d_bytes / t_in / 1e9, 1), "d2h_gbs": round(d2h_bytes / t_out / 1e9, 1),
            "both_ms": round(t_both * 1e3, 4), "h2d_ms": round(t_in * 1e3, 4), "d2h_ms": round(t_out * 1e3, 4),
            "how": "bare pinned copies of one step's bytes, wall clock around synchronised copies, best of 5"}


def forward_kernel_name(w):
    """Which forward kernel the library picks for this workload (mirrors its dispatch)."""
    mean_len = (w.bag_max + w.bag_min) / 2
    tc = w.D in (64, 128) and w.T + 1 <= 128 and mean_len <= 16
    if not tc:
        return "forward_kernel (fused sparse forward, FFMA Gram" + (", two warps per sample)" if mean_len >= 8 else ")")
    if w.train and mean_len > 1.25:
        return ("embbag_list_kernel (lookup, pooled vectors saved for the backward) + forward_tc_kernel "
                "(tcgen05 Gram on the saved vectors)")
    return ("forward_tc_kernel (fused sparse forward, tcgen05 Gram"
            + (", multi-lookup bags)" if mean_len > 1.25 else ")"))


def forward_launches(w) -> int:
    """Kernels of one forward: the training forward of multi-lookup bags is the lookup, then the
    interaction on the saved pooled vectors; every other forward is one kernel."""
    return 2 if forward_kernel_name(w).startswith("embbag_list_kernel") else 1


def run_e2e_train(args, w, tables, batches, dev, dl, torch, world, side):
    """Training steps fed from pinned host memory: indices, offsets, dense and
    grad_out copied in on a copy stream (the next step's copies overlap this
    step's kernels), grad_dense copied back, all inside the timed region."""
    host = [tuple(torch.from_numpy(a).pin_memory() for a in (b.indices, b.offsets, b.dense, b.grad_out))
            for b in batches]
    max_nnz = max(b.nnz for b in batches)
    comp, copy = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    stages = []
    for _ in range(2):
        stages.append((torch.empty(max_nnz, dtype=torch.int32, device=dev),
                       torch.empty(w.T * w.B + 1, dtype=torch.int32, device=dev),
                       torch.empty((w.B, w.D), dtype=torch.float32, device=dev),
                       torch.empty((w.B, w.out_width), dtype=torch.float32, device=dev)))
    accum = ([torch.full((V,), w.accum_init, dtype=torch.float32, device=dev) for V in w.num_rows]
             if args.rule == "adagrad" else None)
    pooled = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device=dev)
    out = torch.empty((w.B, w.out_width), dtype=torch.float32, device=dev)
    gd = torch.empty((w.B, w.D), dtype=torch.float32, device=dev)
    gd_host = [torch.empty((w.B, w.D), dtype=torch.float32).pin_memory() for _ in range(2)]
    ws = torch.empty(max(dl.dlrm_sparse_bwd_workspace_size(tables, torch.from_numpy(b.indices), torch.from_numpy(b.offsets))
                         for b in batches),
                     dtype=torch.uint8, device=dev)
    copied = [None, None]
    used = [None, None]

    def h2d(i):
        k = i % 2
        hi, ho, hx, hg = host[i % N_ROTATE]
        di, do, dx, dg = stages[k]
        with torch.cuda.stream(copy):
            if used[k] is not None:
                copy.wait_event(used[k])
            di[:hi.numel()].copy_(hi, non_blocking=True)
            do.copy_(ho, non_blocking=True)
            dx.copy_(hx, non_blocking=True)
            dg.copy_(hg, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy)
            copied[k] = ev

    def run(i):
        k = i % 2
        hi = host[i % N_ROTATE][0]
        di, do, dx, dg = stages[k]
        comp.wait_event(copied[k])
        if args.sort_in_backward:
            dl.dlrm_sparse_fwd(tables, di[:hi.numel()], do, dx, w.mode, out=out, pooled_save=pooled, stream=comp)
            dl.dlrm_sparse_bwd_update(tables, di[:hi.numel()], do, dx, pooled, dg, args.rule, w.lr, w.eps, accum,
                                      w.mode, grad_dense=gd, workspace=ws, stream=comp, side_stream=side)
        else:  # the sort beside the forward, as in the device-timed step
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record(comp)
            side.wait_event(fork)
            dl.dlrm_sparse_bwd_sort(tables, di[:hi.numel()], do, ws, stream=side)
            join.record(side)
            dl.dlrm_sparse_fwd(tables, di[:hi.numel()], do, dx, w.mode, out=out, pooled_save=pooled, stream=comp)
            dl.dlrm_sparse_bwd_update_sorted(tables, di[:hi.numel()], do, dx, pooled, dg, args.rule, w.lr, w.eps,
                                             accum, w.mode, grad_dense=gd, workspace=ws, sorted=join, stream=comp)
        with torch.cuda.stream(comp):
            gd_host[k].copy_(gd, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(comp)
        used[k] = ev

    def steps(first, count):
        h2d(first)
        for i in range(first, first + count):
            if i + 1 < first + count:
                h2d(i + 1)
            run(i)

    steps(0, args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    steps(args.warmup, args.steps)
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t0, world)
    h2d_b = int(np.mean([b.indices.nbytes + b.offsets.nbytes + b.dense.nbytes + b.grad_out.nbytes for b in batches]))
    return {"value": round(w.B * world * args.steps / el, 1), "unit": "samples/s", "h2d_bytes_per_step": h2d_b,
            "d2h_bytes_per_step": w.B * w.D * 4, "ms_per_step": round(el / args.steps * 1e3, 4),
            "how": "indices, offsets, dense, grad_out from pinned host memory on a copy stream (next step's copies "
                   "overlap this step's kernels); fused forward + training step; grad_dense back to pinned host; "
                   "wall clock over the timed steps"}


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


MODEL_BOTTOM = (13, 512, 256)   # dense features -> ... -> D (the workload's width closes the stack)
MODEL_TOP = (512, 256)          # (D + K) -> ... ; then the 1-wide head


def run_model(args, w):
    """The whole DLRM training step (bench.py --model) on one GPU, timed phase by phase."""
    import torch

    import embedding_bag_lookup_dlrm_b300 as dl

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    dl.load_library()
    tabs = []
    for t, V in enumerate(w.num_rows):
        x = torch.empty((V, w.D), dtype=torch.float32, device=dev)
        gen.fill_table_device(x.data_ptr(), "f32", w.seed, t, 0, V, w.D, torch.cuda.current_stream().cuda_stream)
        tabs.append(x)
    batches = gen.make_batches(w, list(range(N_ROTATE)))
    rng = np.random.default_rng(w.seed)
    dev_b = []
    for b in batches:
        dense_in = rng.standard_normal((w.B, MODEL_BOTTOM[0])).astype(np.float32)
        label = (rng.random(w.B) < 0.25).astype(np.float32)
        dev_b.append(tuple(torch.from_numpy(a).to(dev) for a in (dense_in, label, b.indices, b.offsets)))

    def layer(fin, fout):  # uniform(+-1/sqrt(fan_in)), seeded
        bound = 1.0 / np.sqrt(fin)
        return (torch.from_numpy(rng.uniform(-bound, bound, (fout, fin)).astype(np.float32)).to(dev),
                torch.from_numpy(rng.uniform(-bound, bound, fout).astype(np.float32)).to(dev))

    bot_sizes = list(MODEL_BOTTOM) + [w.D]
    top_sizes = [w.out_width] + list(MODEL_TOP)
    bottom = [layer(a, c) for a, c in zip(bot_sizes, bot_sizes[1:])]
    top = [layer(a, c) for a, c in zip(top_sizes, top_sizes[1:])]
    hw, hb = layer(top_sizes[-1], 1)
    model = dl.DLRMModel(tabs, bottom, top, (hw.reshape(-1).contiguous(), hb))
    accum = [torch.full((V,), w.accum_init, dtype=torch.float32, device=dev) for V in w.num_rows]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    # the sparse backward's key build and sort run there, beside the step up to the per-row sums
    side = torch.cuda.Stream(device=dev, priority=0 if args.side_priority == "low" else -100)

    def step(i, rec):
        dense_in, label, idx, off = dev_b[i % N_ROTATE]
        model.train_step(dense_in, idx, off, label, 0.01, w.lr, w.eps, accum, mode=w.mode, stream=s,
                         side_stream=side, after=rec)

    with torch.cuda.stream(s):
        for i in range(args.warmup):
            flush.zero_()
            step(i, None)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    marks = [[] for _ in range(args.steps)]

    def recorder(i):
        def rec(name):
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(s)
            marks[i].append((name, ev))
        return rec

    with ClockSampler(0) as clk, torch.cuda.stream(s):
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(s)
            step(args.warmup + i, recorder(i))
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(m[-1][1]) for a, m in zip(starts, marks)]
    phase_ms = {}
    for a, m in zip(starts, marks):
        prev = a
        for name, ev in m:
            phase_ms.setdefault(name, []).append(prev.elapsed_time(ev))
            prev = ev
    B = w.B
    mac = lambda sizes: sum(a * c for a, c in zip(sizes, sizes[1:]))
    flops = {"bottom_fwd": 2 * B * mac(bot_sizes), "top_fwd": 2 * B * mac(top_sizes),
             "top_bwd": 4 * B * mac(top_sizes), "bottom_bwd": 4 * B * mac(bot_sizes) - 2 * B * bot_sizes[0] * bot_sizes[1]}
    import json as _json
    peaks_d = _json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"bf16_tflops": 1800.0}
    tpk = float(peaks_d.get("bf16_tflops", 1800.0))
    hbm, src = peaks()
    tb = [train_bytes(w, b) for b in batches]
    phases = {}
    for name, ms in phase_ms.items():
        t = statistics.mean(ms)
        d = {"ms": round(t, 4)}
        if name in flops:
            tf = flops[name] / (t / 1e3) / 1e12
            d.update({"fp32_gemm_tflops": round(tf, 2), "tensor_tflops": round(3 * tf, 2),
                      "tensor_frac": round(3 * tf / tpk, 4)})
        elif name == "sparse_fwd":
            by = statistics.mean(x["forward"] for x in tb)
            d.update({"bytes": int(by), "gbs": round(by / (t / 1e3) / 1e9, 1), "frac": round(by / (t / 1e3) / 1e9 / hbm, 4)})
        elif name == "sparse_bwd":
            by = statistics.mean(x["backward"] for x in tb)
            d.update({"bytes": int(by), "gbs": round(by / (t / 1e3) / 1e9, 1), "frac": round(by / (t / 1e3) / 1e9 / hbm, 4)})
        phases[name] = d
    dom = max(phases, key=lambda n: phases[n]["ms"])
    ms_per_step = statistics.mean(step_ms)
    mlp_flops = sum(flops.values())
    mlp_ms = sum(phases[n]["ms"] for n in flops)
    line = {"metric": "DLRM training-step samples/s (bottom MLP, sparse path, top MLP, BCE) at 1 GPU",
            "value": round(B * args.steps / (sum(step_ms) / 1e3), 1), "unit": "samples/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generator; dense features N(0,1), labels Bernoulli(0.25))",
            "config": dict(config_of(w, args), model=f"bottom {bot_sizes}, top {top_sizes + [1]}, sigmoid + BCE, "
                                                     "SGD lr 0.01 on the MLPs"),
            "roofline": {"phase": dom, "phases": phases,
                         "mlp": {"fp32_gemm_flops": int(mlp_flops), "ms": round(mlp_ms, 4),
                                 "tensor_tflops": round(3 * mlp_flops / (mlp_ms / 1e3) / 1e12, 2),
                                 "peak_bf16_tflops": tpk,
                                 "tensor_frac": round(3 * mlp_flops / (mlp_ms / 1e3) / 1e12 / tpk, 4),
                                 "note": "three bf16 products per fp32 product (split-bf16)"},
                         "peak_source": f"{src} (hbm_gbs; bf16_tflops)"},
            "gpu_launches": None, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    w = gen.workload(args.workload)
    if args.max_rows > 0:
        w.num_rows = [min(v, args.max_rows) for v in w.num_rows]
        w.name += f" [tables capped at {args.max_rows} rows]"
    if args.batch > 0:
        w.B = args.batch
        w.name += f" [batch {args.batch}]"
    if args.uniform:
        w.index_dist = "uniform"
        w.name += " [uniform indices]"
    if w.train and args.rule != "adagrad":
        w.name = w.name.replace("row-wise Adagrad", "plain SGD")
        w.name += f" [{args.rule}]" if "plain SGD" not in w.name else ""
    if args.shards > 1:
        w.name += f" [tables over {args.shards} logical shards]"
    if args.hash:
        w.name += " [raw IDs hashed in the step]"
    if args.op == "embbag":
        w.name += " [embedding-bag lookup alone]"
        w.train = False  # a training workload's bags, looked up only
    if args.tier > 0:
        w.name += f" [tables in pinned host memory, device cache of {args.tier:g} of each table's rows]"
        w.train = False  # the forward of a training workload's bags
    if args.impl == "reference":
        run_reference(args, w)
    elif args.model:
        if not w.train:
            raise SystemExit("--model runs on the training workload (--workload 5)")
        run_model(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
