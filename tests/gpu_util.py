"""Helpers for the GPU parity tests: seeded problems, device copies, and the
error measure.  Expected values always come from the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import gen

# Tolerances (relative, see rel_err): fp32 pooling, fp32 interaction,
# bf16 tables with fp32 accumulation, and Adagrad-updated rows.
TOL_POOL_F32 = 1e-5
TOL_INTERACT = 1e-4
TOL_BF16 = 2e-3
TOL_ADAGRAD = 2e-3


def rel_err(y, ref, scale):
    """|y - ref| / max(|ref|, S): S is the sum of |terms| behind ref, so values
    that cancel to near zero are measured against the size of what cancelled."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(y - ref) / np.maximum(np.maximum(np.abs(ref), np.asarray(scale, np.float64)), 1e-30)


def assert_close(y, ref, scale, tol, what):
    e = rel_err(y, ref, scale)
    worst = float(e.max()) if e.size else 0.0
    if worst > tol:
        k = int(np.argmax(e))
        raise AssertionError(f"{what}: max rel err {worst:.3g} > {tol:g} at flat index {k}: "
                             f"got {np.asarray(y).ravel()[k]!r}, want {np.asarray(ref).ravel()[k]!r}")
    return worst


def random_case(seed, B, T, D, V, Lmin, Lmax, dtype="f32", value_scale=1.0):
    """Random tables (V rows each), CSR bags with lengths in [Lmin, Lmax], dense x."""
    rng = np.random.default_rng(seed)
    Vs = [V] * T if np.isscalar(V) else list(V)
    tabs = [(rng.uniform(-1, 1, size=(v, D)) * value_scale).astype(np.float32) for v in Vs]
    if dtype == "bf16":
        tabs = [gen.f32_to_bf16_bits(t) for t in tabs]
    L = rng.integers(Lmin, Lmax + 1, size=T * B)
    off = np.zeros(T * B + 1, dtype=np.int64)
    np.cumsum(L, out=off[1:])
    idx = np.concatenate([rng.integers(0, Vs[t], size=int(L[t * B:(t + 1) * B].sum())) for t in range(T)]
                         ).astype(np.int64)
    dense = rng.standard_normal((B, D)).astype(np.float32)
    return tabs, Vs, idx, off, dense


def dev_tables(tabs, dtype):
    out = []
    for t in tabs:
        if dtype == "bf16":
            out.append(torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).cuda().view(torch.bfloat16))
        else:
            out.append(torch.from_numpy(np.ascontiguousarray(t)).cuda())
    return out


def host_table(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def dev_index(a, itype):
    dt = torch.int32 if itype == "i32" else torch.int64
    return torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()


def workload_tables(w: gen.Workload):
    """Device tables of a workload, filled on the device by the seeded generator."""
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    tabs = []
    for t, V in enumerate(w.num_rows):
        x = torch.empty((V, w.D), dtype=dt, device="cuda")
        gen.fill_table_device(x.data_ptr(), w.dtype, w.seed, t, 0, V, w.D,
                              torch.cuda.current_stream().cuda_stream)
        tabs.append(x)
    torch.cuda.synchronize()
    return tabs


def batch_to_device(batch: gen.Batch):
    return (torch.from_numpy(batch.indices).cuda(), torch.from_numpy(batch.offsets).cuda(),
            torch.from_numpy(batch.dense).cuda())


def free_cuda():
    import gc
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
