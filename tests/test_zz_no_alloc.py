"""The allocation-free training step, dlrm_sparse_bwd_adagrad_static.

It exists for callers that cannot allocate device memory when they run a
step: a plugin handed only its input and output buffers through a C
interface, or a process whose device memory belongs to another framework's
pooled allocator.  It must give the same result as dlrm_sparse_bwd_adagrad
with a caller workspace, on consecutive calls that reuse the same fixed
scratch.  The second call here runs a different, larger batch, so it would
expose anything that depended on scratch contents left by the first call.

This file is collected last so that a run which stops at the first failure
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
from gpu_util import TOL_ADAGRAD, TOL_INTERACT, assert_close, dev_index, dev_tables, random_case

pytestmark = pytest.mark.gpu

T, D, V = 26, 128, 500


def _batch(seed, B, Lmax):
    tabs, Vs, idx, off, dense = random_case(seed, B, T, D, V, 1, Lmax, value_scale=0.05)
    rng = np.random.default_rng(seed + 7)
    g = rng.standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)
    return tabs, Vs, idx, off, dense, g


def _state(tabs, Vs):
    return dev_tables(tabs, "f32"), [torch.full((v,), 0.1, dtype=torch.float32, device="cuda") for v in Vs]


def _step(fn, tabs, acc, batch, **kw):
    _, _, idx, off, dense, g = batch
    B = dense.shape[0]
    di, do = dev_index(idx, "i32"), dev_index(off, "i32")
    dx = torch.from_numpy(dense).cuda()
    ps = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    dl.dlrm_sparse_fwd(tabs, di, do, dx, pooled_save=ps)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gd = fn(tabs, acc, di, do, dx, ps, torch.from_numpy(g).cuda(), 0.01, 1e-8, status=status, **kw)
    torch.cuda.synchronize()
    assert status.item() == 0
    return gd.cpu().numpy()


def test_static_scratch_matches_workspace_entry_point_twice():
    first = _batch(501, 256, 8)
    second = _batch(502, 600, 12)   # a different, larger batch on the second call
    tabs0, Vs = first[0], first[1]

    # the existing entry point, caller workspace
    ref_t, ref_a = _state(tabs0, Vs)
    ref_gd = [_step(dl.dlrm_sparse_bwd_adagrad, ref_t, ref_a, b) for b in (first, second)]
    ref_rows = [t.cpu().numpy() for t in ref_t]
    ref_acc = [a.cpu().numpy() for a in ref_a]

    # the allocation-free entry point, two calls in a row on the same scratch
    got_t, got_a = _state(tabs0, Vs)
    got_gd = []
    for k, b in enumerate((first, second)):
        gd_out = torch.empty((b[4].shape[0], D), dtype=torch.float32, device="cuda")
        got_gd.append(_step(dl.dlrm_sparse_bwd_adagrad_static, got_t, got_a, b, grad_dense=gd_out))
        scale = np.abs(ref_gd[k]) + 1e-6
        assert_close(got_gd[k], ref_gd[k], scale, TOL_INTERACT, f"grad_dense, call {k + 1}")

    for t in range(T):
        w = got_t[t].cpu().numpy()
        scale = np.abs(tabs0[t]) + np.abs(tabs0[t] - ref_rows[t])
        assert_close(w, ref_rows[t], scale, TOL_ADAGRAD, f"rows of table {t} after two calls")
        assert_close(got_a[t].cpu().numpy(), ref_acc[t], 0.0, TOL_ADAGRAD, f"accumulators of table {t}")


def test_static_scratch_rejects_a_batch_too_large():
    """A batch whose scratch exceeds the fixed array is refused before any launch, and it is the size
    that refuses it: the same arguments pass every other host check (the workspace query accepts them
    and reports a need above the array's size)."""
    lib = dl.load_library()
    B, nnz = 1 << 16, 1 << 20   # dP alone is B*T*D*4 = 872 MB
    ptrs = (ctypes.c_void_p * T)(*[0x1000] * T)
    rows = (ctypes.c_int64 * T)(*[V] * T)
    tb = dl.DlrmTables(T, D, 0, ptrs, rows)
    bags = dl.DlrmBags(B, nnz, 0, 0x2000, 0x3000)
    need = ctypes.c_size_t(0)
    assert lib.dlrm_sparse_bwd_workspace_size(ctypes.byref(tb), ctypes.byref(bags), ctypes.byref(need)) == 0
    assert need.value > dl.STATIC_SCRATCH_BYTES
    acc = (ctypes.c_void_p * T)(*[0x4000] * T)
    st = lib.dlrm_sparse_bwd_adagrad_static(ctypes.byref(tb), ctypes.byref(bags), 0, 0x5000, 0x6000, 0x7000,
                                            0x8000, acc, 0.01, 1e-8, None, None)
    assert st == dl.DLRM_ERR_INVALID_ARG


def test_static_scratch_accepts_a_batch_just_under_the_limit():
    """The largest batch (bags of 1..8) whose scratch fits the fixed array runs, and matches the
    workspace entry point; one more sample no longer fits."""
    rng = np.random.default_rng(601)
    Bmax = 4000
    L = rng.integers(1, 9, size=(T, Bmax))
    tb = dl.Tables([torch.empty((V, D), dtype=torch.float32, device="cuda") for _ in range(1)] * T)

    def need(B):
        off = np.zeros(T * B + 1, np.int32)
        np.cumsum(L[:, :B].reshape(-1), out=off[1:])
        idx = np.zeros(int(off[-1]), np.int32)
        return dl.dlrm_sparse_bwd_workspace_size(tb, torch.from_numpy(idx), torch.from_numpy(off))

    lo, hi = 1, Bmax   # need(lo) fits, need(hi) does not
    assert need(hi) > dl.STATIC_SCRATCH_BYTES
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= dl.STATIC_SCRATCH_BYTES else (lo, mid)
    B = lo
    assert dl.STATIC_SCRATCH_BYTES - need(B) < 64 << 10   # within 64 KB of the limit

    tabs = [rng.uniform(-0.05, 0.05, size=(V, D)).astype(np.float32) for _ in range(T)]
    off = np.zeros(T * B + 1, np.int64)
    np.cumsum(L[:, :B].reshape(-1), out=off[1:])
    idx = rng.integers(0, V, size=int(off[-1]))
    dense = rng.standard_normal((B, D)).astype(np.float32)
    g = rng.standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)
    batch = (tabs, [V] * T, idx, off, dense, g)
    ref_t, ref_a = _state(tabs, [V] * T)
    ref_gd = _step(dl.dlrm_sparse_bwd_adagrad, ref_t, ref_a, batch)
    got_t, got_a = _state(tabs, [V] * T)
    got_gd = _step(dl.dlrm_sparse_bwd_adagrad_static, got_t, got_a, batch,
                   grad_dense=torch.empty((B, D), dtype=torch.float32, device="cuda"))
    assert_close(got_gd, ref_gd, np.abs(ref_gd) + 1e-6, TOL_INTERACT, "grad_dense at the size limit")
    for t in range(T):
        scale = np.abs(tabs[t]) + np.abs(tabs[t] - ref_t[t].cpu().numpy())
        assert_close(got_t[t].cpu().numpy(), ref_t[t].cpu().numpy(), scale, TOL_ADAGRAD, f"rows of table {t}")
