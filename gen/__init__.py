"""Seeded synthetic inputs for the DLRM sparse path.

This module is shared by the test suite and the benchmark.  It produces the
*inputs* of the method (table contents, bags of indices, dense vectors,
upstream gradients) and holds none of the method's arithmetic: no pooling, no
dot product, no gradient, no optimiser step.

Workloads follow the shapes the pages describe: tens of sparse features, one
embedding table E_t : V_t x D per feature ("DLRM", robocikowo.com, embedding
table paragraph), D = 64-128 ("The embedding table is the model": "say 64
numbers"), multi-valued features pooled over a bag ("The embedding table is the
model"), power-law item popularity, tables of tens of gigabytes ("Deep Learning
Recommendation Model (DLRM)", notes.helloworld.co.in).  The public click-log
benchmark the pages mention is not used; these seeded inputs stand in for it.

Table contents come from a counter-based generator so that any row can be
produced on its own, on the host (numpy or the C loop in ``gen.cu``) or on the
device (the fill kernel in ``gen.cu``), bit-identically:

  SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): gamma = 0x9E3779B97F4A7C15 and the finaliser
      mix64(z): z = (z ^ z>>30) * 0xBF58476D1CE4E5B9
                z = (z ^ z>>27) * 0x94D049BB133111EB
                return z ^ z>>31
  stream of table t:      s_t = mix64(seed + (t+1)*gamma)
  element (r, d):         h   = mix64(s_t + (r*D + d + 1)*gamma)
  fp32 value:             k = (h >> 40) - 2^23  (an integer in [-2^23, 2^23))
                          v = fp32(k) * fp32(0.1) * 2^-24, rounded to nearest
                          even once, so v lies in [-0.05, 0.05)
  bf16 value:             round-to-nearest-even of v's fp32 bits to the upper
                          16 bits.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
SCALE = np.float32(np.float32(0.1) / np.float32(16777216.0))  # exact: power-of-2 divide

BASE_SEED = 20261202

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdlrm_gen.so")


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_seed(seed: int, t: int) -> int:
    """Per-table stream key s_t = mix64(seed + (t+1)*gamma)."""
    with np.errstate(over="ignore"):
        s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + np.uint64(t + 1) * GAMMA
    return int(mix64(np.array([s], dtype=np.uint64))[0])


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of finite fp32 values to bf16 bit patterns."""
    bits = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def table_rows_numpy(seed: int, t: int, rows, D: int, dtype: str = "f32") -> np.ndarray:
    """Rows `rows` of table t, computed with numpy (reference for the C/CUDA fills).

    Returns float32 [len(rows), D] for "f32" or uint16 bf16 bit patterns for "bf16"."""
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    s = np.uint64(stream_seed(seed, t))
    c = rows * np.uint64(D) + np.arange(D, dtype=np.uint64)[None, :] + np.uint64(1)
    with np.errstate(over="ignore"):
        h = mix64(s + c * GAMMA)
    k = (h >> np.uint64(40)).astype(np.int64) - (1 << 23)
    v = k.astype(np.float32) * SCALE
    return f32_to_bf16_bits(v) if dtype == "bf16" else v


# --------------------------------------------------------------------------
# C / CUDA fills (gen.cu): same definition, fast.
# --------------------------------------------------------------------------
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with gen/build.py")
        lib = ctypes.CDLL(LIB_PATH)
        lib.gen_rows_host.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.gen_rows_host.restype = None
        lib.gen_fill_device.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
        lib.gen_fill_device.restype = ctypes.c_int
        _lib = lib
    return _lib


def table_rows(seed: int, t: int, rows, D: int, dtype: str = "f32", threads: int = 0) -> np.ndarray:
    """Rows of table t generated by the C host loop (bit-identical to numpy)."""
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    out = np.empty((rows.size, D), dtype=np.uint16 if dtype == "bf16" else np.float32)
    if rows.size:
        _load().gen_rows_host(out.ctypes.data, 1 if dtype == "bf16" else 0, stream_seed(seed, t),
                              rows.ctypes.data, rows.size, D, threads)
    return out


def fill_table_device(ptr: int, dtype: str, seed: int, t: int, row0: int, nrows: int, D: int,
                      stream: int = 0) -> None:
    """Fill rows [row0, row0+nrows) of table t at device pointer `ptr` (row-major, stride D)."""
    rc = _load().gen_fill_device(ctypes.c_void_p(ptr), 1 if dtype == "bf16" else 0,
                                 stream_seed(seed, t), row0, nrows, D, ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"gen_fill_device failed with CUDA error {rc}")


# --------------------------------------------------------------------------
# Index distributions.
# --------------------------------------------------------------------------
def zipf_ranks(rng: np.random.Generator, V: int, alpha: float, n: int) -> np.ndarray:
    """n exact draws of k in 1..V with p(k) ~ k^-alpha (alpha > 0, alpha != 1).

    Rejection from a continuous envelope: x^-alpha is convex, so its integral
    over [k-1/2, k+1/2] is at least k^-alpha (Hermite-Hadamard).  Draw X with
    density ~ x^-alpha on [1/2, V+1/2] by inverting its antiderivative
    H(x) = x^(1-alpha) / (1-alpha), round to k, and keep k with probability
    k^-alpha / (H(k+1/2) - H(k-1/2)).  (The envelope is the one of Hoermann &
    Derflinger's rejection-inversion, 1996; here with a second uniform.)"""
    a1 = 1.0 - alpha

    def H(x):
        return np.power(x, a1) / a1

    def H_inv(y):
        return np.power(y * a1, 1.0 / a1)

    lo, hi = H(0.5), H(V + 0.5)
    out = np.empty(n, dtype=np.int64)
    filled = 0
    while filled < n:
        m = int((n - filled) * 1.15) + 16
        x = H_inv(lo + rng.random(m) * (hi - lo))
        k = np.clip(np.floor(x + 0.5), 1, V)
        keep = rng.random(m) * (H(k + 0.5) - H(k - 0.5)) <= np.power(k, -alpha)
        got = k[keep].astype(np.int64)[: n - filled]
        out[filled:filled + got.size] = got
        filled += got.size
    return out


def affine_perm_params(seed: int, t: int, V: int) -> tuple[int, int]:
    """Seeded bijection k -> (a*k + c) mod V of [0, V) for table t (gcd(a, V) = 1)."""
    rng = np.random.default_rng([seed, 7919, t])
    while True:
        a = int(rng.integers(1, 1 << 31)) | 1
        if math.gcd(a, V) == 1:
            break
    c = int(rng.integers(0, V))
    return a, c


def permute(ranks_minus_1: np.ndarray, a: int, c: int, V: int) -> np.ndarray:
    return (ranks_minus_1.astype(np.int64) * a + c) % V


# --------------------------------------------------------------------------
# Workloads.
# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    B: int
    T: int
    D: int
    dtype: str              # "f32" | "bf16"
    num_rows: list
    bag_min: int            # bag lengths uniform in [bag_min, bag_max]
    bag_max: int
    index_dist: str         # "uniform" | "zipf"
    alpha: float = 0.0
    mode: str = "sum"       # "sum" | "mean"
    seed: int = BASE_SEED
    train: bool = False
    lr: float = 0.01
    eps: float = 1e-8
    accum_init: float = 0.1
    notes: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return self.T + 1

    @property
    def out_width(self) -> int:
        return self.D + self.N * (self.N - 1) // 2

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def table_bytes(self) -> int:
        return sum(self.num_rows) * self.D * self.elem_bytes


def production_table_sizes(seed: int, T: int = 26, lo: float = 1e3, hi: float = 4e7,
                           total_lo: float = 1.75e8, total_hi: float = 1.85e8):
    """T log-uniform row counts in [lo, hi] whose total lies in [total_lo, total_hi]:
    draws with seeds seed, seed+1, ... and keeps the first that fits."""
    for s in range(seed, seed + 1_000_000):
        rng = np.random.default_rng(s)
        sz = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), T))).astype(np.int64)
        sz = np.clip(sz, int(lo), int(hi))
        if total_lo <= sz.sum() <= total_hi:
            return [int(v) for v in sz], s
    raise RuntimeError("no table-size draw fits")


def workload(cid: int, **overrides) -> Workload:
    """The five named workloads.

    1 tiny forward, 2 production one-hot forward (~92 GB of fp32 tables),
    3 multi-hot bf16 forward, 4 wide interaction (N = 101), 5 training step."""
    seed = BASE_SEED + cid
    if cid == 1:
        w = Workload("tiny forward: B=128, T=4 fp32 tables of 1000 rows, D=16, one-hot uniform, sum",
                     B=128, T=4, D=16, dtype="f32", num_rows=[1000] * 4, bag_min=1, bag_max=1,
                     index_dist="uniform", seed=seed)
    elif cid == 2:
        sizes, s = production_table_sizes(seed)
        w = Workload("production one-hot forward: B=65536, T=26 fp32 tables (log-uniform 1e3..4e7 rows, "
                     "~1.8e8 rows, ~92 GB), D=128, one-hot Zipf(1.05) after a seeded row permutation, sum",
                     B=65536, T=26, D=128, dtype="f32", num_rows=sizes, bag_min=1, bag_max=1,
                     index_dist="zipf", alpha=1.05, seed=seed, notes={"size_seed": s})
    elif cid == 3:
        w = Workload("multi-hot pooled forward: B=16384, T=26 bf16 tables of 5e6 rows, D=128, bags 1..64, "
                     "Zipf(1.1), sum",
                     B=16384, T=26, D=128, dtype="bf16", num_rows=[5_000_000] * 26, bag_min=1, bag_max=64,
                     index_dist="zipf", alpha=1.1, seed=seed)
    elif cid == 4:
        w = Workload("wide interaction forward: B=8192, T=100 fp32 tables of 1e6 rows, D=64, one-hot uniform, "
                     "N=101",
                     B=8192, T=100, D=64, dtype="f32", num_rows=[1_000_000] * 100, bag_min=1, bag_max=1,
                     index_dist="uniform", seed=seed)
    elif cid == 5:
        w = Workload("training step sparse path: B=32768, T=26 fp32 tables of 2e6 rows, D=128, bags 1..8, "
                     "Zipf(1.05), sum, row-wise Adagrad lr=0.01 eps=1e-8 accumulator 0.1",
                     B=32768, T=26, D=128, dtype="f32", num_rows=[2_000_000] * 26, bag_min=1, bag_max=8,
                     index_dist="zipf", alpha=1.05, seed=seed, train=True)
    else:
        raise ValueError(f"unknown workload {cid}")
    for k, v in overrides.items():
        setattr(w, k, v)
    return w


@dataclass
class Batch:
    indices: np.ndarray     # int32 [nnz], rows local to their table
    offsets: np.ndarray     # int32 [T*B+1], table-major CSR
    dense: np.ndarray       # float32 [B, D]
    grad_out: np.ndarray | None = None  # float32 [B, D + N(N-1)/2] (training only)

    @property
    def nnz(self) -> int:
        return int(self.indices.size)


def make_batches(w: Workload, batch_ids, with_grad: bool | None = None) -> list:
    """Seeded batches of workload w, one per id (deterministic in (w.seed, id))."""
    batch_ids = list(batch_ids)
    with_grad = w.train if with_grad is None else with_grad
    rngs = {b: np.random.default_rng([w.seed, 1, b]) for b in batch_ids}
    lengths = {b: [] for b in batch_ids}
    idx = {b: [] for b in batch_ids}
    for t in range(w.T):
        V = int(w.num_rows[t])
        if w.index_dist == "zipf":
            a, c = affine_perm_params(w.seed, t, V)
        for b in batch_ids:
            rng = rngs[b]
            if w.bag_min == w.bag_max:
                L = np.full(w.B, w.bag_min, dtype=np.int64)
            else:
                L = rng.integers(w.bag_min, w.bag_max + 1, size=w.B)
            n = int(L.sum())
            if w.index_dist == "zipf":
                rows = permute(zipf_ranks(rng, V, w.alpha, n) - 1, a, c, V)
            else:
                rows = rng.integers(0, V, size=n)
            lengths[b].append(L)
            idx[b].append(rows.astype(np.int32))
    out = []
    for b in batch_ids:
        rng = rngs[b]
        L = np.concatenate(lengths[b])
        offsets = np.zeros(L.size + 1, dtype=np.int64)
        np.cumsum(L, out=offsets[1:])
        dense = rng.standard_normal((w.B, w.D), dtype=np.float32)
        g = rng.standard_normal((w.B, w.out_width), dtype=np.float32) if with_grad else None
        out.append(Batch(indices=np.concatenate(idx[b]), offsets=offsets.astype(np.int32),
                         dense=dense, grad_out=g))
    return out


def compact_tables(w: Workload, batch: Batch, threads: int = 0):
    """Host copies of only the rows a batch touches, for running the oracle
    without materialising whole tables.

    Returns (tables, num_rows, indices) where table t holds the touched rows of
    E_t in ascending row order and `indices` (int64) is remapped into them.
    Bags, offsets and order are unchanged, so any per-bag computation on the
    compact tables equals the one on the full tables."""
    new_idx = np.empty(batch.nnz, dtype=np.int64)
    tables, nrows = [], []
    off = batch.offsets.astype(np.int64)
    for t in range(w.T):
        lo, hi = int(off[t * w.B]), int(off[(t + 1) * w.B])
        rows = batch.indices[lo:hi].astype(np.int64)
        uniq, inv = np.unique(rows, return_inverse=True)
        new_idx[lo:hi] = inv
        tables.append(table_rows(w.seed, t, uniq, w.D, w.dtype, threads))
        nrows.append(int(uniq.size))
    return tables, nrows, new_idx
