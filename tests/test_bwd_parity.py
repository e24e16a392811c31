"""GPU parity of dlrm_sparse_bwd_adagrad (through the C ABI) with the CPU oracle:
grad_dense, every touched row and accumulator, untouched rows bit-identical,
bitwise reproducibility, long runs of one row crossing many reduction chunks."""
import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
import gen
import oracle
from gpu_util import (TOL_ADAGRAD, TOL_INTERACT, TOL_POOL_F32, assert_close, batch_to_device, dev_index, dev_tables,
                      free_cuda, random_case, workload_tables)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def run_case(orc, tabs, Vs, idx, off, dense, mode, itype, lr=0.01, eps=1e-8, acc0=0.1, seed=0):
    B, D = dense.shape
    T = len(tabs)
    N = T + 1
    rng = np.random.default_rng(seed + 1)
    g = rng.standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
    pooled, st = orc.embbag(tabs, Vs, idx, off, B, D, mode)
    new_ref = [t.copy() for t in tabs]
    acc_ref = [np.full(v, acc0, np.float32) for v in Vs]
    gd_ref, st2 = orc.sparse_bwd_adagrad(new_ref, Vs, idx, off, dense, pooled, g, acc_ref, lr, eps, mode)

    dt = dev_tables(tabs, "f32")
    acc = [torch.full((v,), acc0, dtype=torch.float32, device="cuda") for v in Vs]
    di, do = dev_index(idx, itype), dev_index(off, itype)
    dx = torch.from_numpy(dense).cuda()
    ps = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    dl.dlrm_sparse_fwd(dt, di, do, dx, mode, pooled_save=ps)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gd = dl.dlrm_sparse_bwd_adagrad(dt, acc, di, do, dx, ps, torch.from_numpy(g).cuda(), lr, eps, mode,
                                    status=status)
    torch.cuda.synchronize()
    return dict(g=g, pooled=pooled, new_ref=new_ref, acc_ref=acc_ref, gd_ref=gd_ref, st_ref=st | st2,
                dt=dt, acc=acc, gd=gd.cpu().numpy(), status=status.item())


def check(res, tabs, Vs, idx, off, B, dense):
    assert res["status"] == res["st_ref"] == 0
    T = len(tabs)
    D = dense.shape[1]
    g = res["g"]
    # scale of grad_dense: |g_x| + sum_j |g_0j| |V_j|
    Vabs = np.concatenate([np.abs(dense)[:, None], np.abs(res["pooled"])], axis=1)
    s = np.abs(g[:, :D]) + np.einsum("bj,bjd->bd", np.abs(g[:, D:D + T]), Vabs[:, 1:])
    assert_close(res["gd"], res["gd_ref"], s, TOL_INTERACT, "grad_dense")
    for t in range(T):
        got = res["dt"][t].cpu().numpy()
        acc = res["acc"][t].cpu().numpy()
        touched = np.zeros(Vs[t], bool)
        seg = idx[off[t * B]:off[(t + 1) * B]]
        touched[seg[(seg >= 0) & (seg < Vs[t])]] = True
        # untouched rows and accumulators are bit-identical
        assert np.array_equal(got[~touched], tabs[t][~touched])
        assert np.all(acc[~touched] == res["acc_ref"][t][~touched])
        # touched rows: the update is small against the weights, so measure it
        # against |w| + |w - w_new| (the size of the step taken)
        scale = np.abs(tabs[t][touched]) + np.abs(tabs[t][touched] - res["new_ref"][t][touched])
        assert_close(got[touched], res["new_ref"][t][touched], scale, TOL_ADAGRAD, f"rows of table {t}")
        assert_close(acc[touched], res["acc_ref"][t][touched], 0.0, TOL_ADAGRAD, f"accum of table {t}")
        # the update itself, against the step size
        step_ref = res["new_ref"][t][touched].astype(np.float64) - tabs[t][touched]
        step = got[touched].astype(np.float64) - tabs[t][touched]
        assert_close(step, step_ref, np.abs(step_ref).max() * 1e-3 + 1e-12, 1e-2, f"steps of table {t}")


CASES = [
    # D, T, mode, itype, Lmin, Lmax, B, V
    (128, 26, "sum", "i32", 1, 8, 200, 300),
    (128, 26, "mean", "i64", 0, 8, 97, 300),
    (64, 5, "sum", "i32", 0, 30, 301, 40),
    (16, 3, "mean", "i32", 1, 3, 1000, 7),
    (256, 2, "sum", "i64", 1, 1, 33, 1000),
    (32, 100, "sum", "i32", 1, 2, 21, 100),
    # N = 113 at D = 256: eight warps per sample, close to the largest shared-memory layout
    (256, 112, "mean", "i32", 0, 2, 9, 50),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "D{}-T{}-{}-{}-L{}..{}-B{}-V{}".format(*c))
def test_bwd_adagrad_random(case, orc):
    D, T, mode, itype, Lmin, Lmax, B, V = case
    tabs, Vs, idx, off, dense = random_case(200 + CASES.index(case), B, T, D, V, Lmin, Lmax, value_scale=0.05)
    res = run_case(orc, tabs, Vs, idx, off, dense, mode, itype, seed=CASES.index(case))
    check(res, tabs, Vs, idx, off, B, dense)


def test_long_runs_cross_chunks(orc):
    """One row looked up ~5000 times (twenty reduction chunks), others rarely."""
    B, T, D, V = 2500, 2, 128, 50
    rng = np.random.default_rng(3)
    tabs = [rng.uniform(-0.05, 0.05, size=(V, D)).astype(np.float32) for _ in range(T)]
    L = np.full(T * B, 2)
    off = np.concatenate([[0], np.cumsum(L)])
    idx = rng.integers(0, V, size=int(L.sum()))
    idx[: 2 * B] = np.where(rng.random(2 * B) < 0.97, 7, idx[: 2 * B])  # table 0: row 7 dominates
    dense = rng.standard_normal((B, D)).astype(np.float32)
    res = run_case(orc, tabs, [V] * T, idx, off, dense, "sum", "i32", lr=0.05)
    check(res, tabs, [V] * T, idx, off, B, dense)


def test_bwd_bitwise_reproducible():
    B, T, D, V = 4000, 26, 128, 400
    tabs, Vs, idx, off, dense = random_case(31, B, T, D, V, 1, 8, value_scale=0.05)
    rng = np.random.default_rng(1)
    g = torch.from_numpy(rng.standard_normal((B, D + 27 * 13)).astype(np.float32)).cuda()
    di, do, dx = dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda()
    results = []
    for _ in range(2):
        dt = dev_tables(tabs, "f32")
        acc = [torch.full((v,), 0.1, device="cuda") for v in Vs]
        ps = torch.empty((B, T, D), device="cuda")
        dl.dlrm_sparse_fwd(dt, di, do, dx, pooled_save=ps)
        gd = dl.dlrm_sparse_bwd_adagrad(dt, acc, di, do, dx, ps, g, 0.01, 1e-8)
        torch.cuda.synchronize()
        results.append((torch.cat([t.flatten() for t in dt]), torch.cat(acc), gd))
    for a, b in zip(*results):
        assert torch.equal(a, b)


@pytest.mark.parametrize("mode,itype,rule,V,wait", [("sum", "i32", "adagrad", 400, "event"),
                                                    ("mean", "i64", "sgd", 3000, "stream"),
                                                    ("sum", "i64", "adagrad", 1 << 17, "event")])
def test_sort_beside_forward_matches_one_call(mode, itype, rule, V, wait):
    """dlrm_sparse_bwd_sort on a second stream while the forward runs, then dlrm_sparse_bwd_update_sorted
    (waiting for the sort through its event argument, or through the caller's stream wait): tables,
    accumulators and grad_dense bit for bit those of the one-call step (dlrm_sparse_bwd_update), over two
    consecutive steps (the second one's sort overwrites the first one's pairs).  V = 2^17 rows per table
    (3.4 M rows in all) makes 22 key bits: three radix passes, against two for the smaller tables."""
    B, T, D = 3000, 26, 128
    tabs, Vs, idx, off, dense = random_case(41, B, T, D, V, 0, 8, value_scale=0.05)
    rng = np.random.default_rng(5)
    g = [torch.from_numpy(rng.standard_normal((B, D + 27 * 13)).astype(np.float32)).cuda() for _ in range(2)]
    di, do, dx = dev_index(idx, itype), dev_index(off, itype), torch.from_numpy(dense).cuda()
    results = []
    for split in (False, True):
        dt = dev_tables(tabs, "f32")
        acc = [torch.full((v,), 0.1, device="cuda") for v in Vs] if rule == "adagrad" else None
        ws = torch.empty(dl.dlrm_sparse_bwd_workspace_size(dt, di, do), dtype=torch.uint8, device="cuda")
        ws.fill_(0xA5)
        ps = torch.empty((B, T, D), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        main, side = torch.cuda.Stream(), torch.cuda.Stream()
        gds = []
        with torch.cuda.stream(main):
            for k in range(2):
                if split:
                    fork, join = torch.cuda.Event(), torch.cuda.Event()
                    fork.record(main)
                    side.wait_event(fork)
                    dl.dlrm_sparse_bwd_sort(dt, di, do, ws, status=status, stream=side)
                    join.record(side)
                    dl.dlrm_sparse_fwd(dt, di, do, dx, mode, pooled_save=ps, status=status, stream=main)
                    if wait == "stream":
                        main.wait_event(join)
                    gd = dl.dlrm_sparse_bwd_update_sorted(dt, di, do, dx, ps, g[k], rule, 0.01, 1e-8, acc, mode,
                                                          workspace=ws, status=status,
                                                          sorted=join if wait == "event" else None, stream=main)
                else:
                    dl.dlrm_sparse_fwd(dt, di, do, dx, mode, pooled_save=ps, status=status, stream=main)
                    gd = dl.dlrm_sparse_bwd_update(dt, di, do, dx, ps, g[k], rule, 0.01, 1e-8, acc, mode,
                                                   workspace=ws, status=status, stream=main)
                gds.append(gd.clone())
        torch.cuda.synchronize()
        assert status.item() == 0, dl.status_string(status.item())
        results.append([torch.cat([t.flatten() for t in dt])] + ([torch.cat(acc)] if acc else []) + gds)
    for a, b in zip(*results):
        assert torch.equal(a, b)


def test_grad_ready_event_orders_grad_dense():
    """dlrm_sparse_bwd_update_sorted's grad_ready event: a copy of grad_dense queued on another stream after
    waiting for it (while the per-row sums still run on the call's stream) holds the final grad_dense."""
    B, T, D = 3000, 26, 128
    tabs, Vs, idx, off, dense = random_case(61, B, T, D, 2000, 1, 8, value_scale=0.05)
    g = torch.from_numpy(np.random.default_rng(7).standard_normal((B, D + 27 * 13)).astype(np.float32)).cuda()
    di, do, dx = dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda()
    dt = dev_tables(tabs, "f32")
    acc = [torch.full((v,), 0.1, device="cuda") for v in Vs]
    ps = torch.empty((B, T, D), device="cuda")
    dl.dlrm_sparse_fwd(dt, di, do, dx, pooled_save=ps)
    ref = dl.dlrm_interact_bwd(dx, ps, g)[0]  # grad_dense alone
    ws = torch.empty(dl.dlrm_sparse_bwd_workspace_size(dt, di, do), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    main, other = torch.cuda.Stream(), torch.cuda.Stream()
    gd = torch.full((B, D), float("nan"), device="cuda")
    copy = torch.empty_like(gd)
    ready = torch.cuda.Event()
    with torch.cuda.stream(main):
        dl.dlrm_sparse_bwd_sort(dt, di, do, ws, stream=main)
        dl.dlrm_sparse_bwd_update_sorted(dt, di, do, dx, ps, g, "adagrad", 0.01, 1e-8, acc, grad_dense=gd,
                                         workspace=ws, grad_ready=ready, stream=main)
    other.wait_event(ready)
    with torch.cuda.stream(other):
        copy.copy_(gd)
    torch.cuda.synchronize()
    assert torch.equal(copy, ref) and torch.equal(gd, ref)


def test_bwd_flags_bad_index(orc):
    B, T, D, V = 50, 3, 64, 30
    tabs, Vs, idx, off, dense = random_case(41, B, T, D, V, 1, 3, value_scale=0.05)
    idx[4] = V + 5
    dt = dev_tables(tabs, "f32")
    acc = [torch.full((v,), 0.1, device="cuda") for v in Vs]
    ps = torch.empty((B, T, D), device="cuda")
    di, do, dx = dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dlrm_sparse_fwd(dt, di, do, dx, pooled_save=ps, status=status)
    g = torch.randn((B, D + 6), device="cuda")
    dl.dlrm_sparse_bwd_adagrad(dt, acc, di, do, dx, ps, g, 0.01, 1e-8, status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_INDEX_OOB


def test_bwd_flags_bad_offsets(orc):
    """Offsets that go backwards: the backward flags them and touches no memory out of range."""
    B, T, D, V = 50, 3, 64, 30
    tabs, Vs, idx, off, dense = random_case(42, B, T, D, V, 1, 3, value_scale=0.05)
    off = off.copy()
    off[5] = off[6] + 2  # bag 4 ends after bag 5 does
    dt = dev_tables(tabs, "f32")
    acc = [torch.full((v,), 0.1, device="cuda") for v in Vs]
    ps = torch.zeros((B, T, D), device="cuda")
    di, do, dx = dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.randn((B, D + 6), device="cuda")
    dl.dlrm_sparse_bwd_adagrad(dt, acc, di, do, dx, ps, g, 0.01, 1e-8, status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_BAD_OFFSETS


def test_workload_training_step(orc):
    """The full training-step workload: B=32768, T=26 fp32 tables of 2e6 rows, bags 1..8, Zipf(1.05)."""
    w = gen.workload(5)
    batch, = gen.make_batches(w, [0])
    tabs_host, nr, cidx = gen.compact_tables(w, batch)
    fwd_ref = orc.sparse_fwd(tabs_host, nr, cidx, batch.offsets, batch.dense, w.mode, with_abs=True,
                             with_pooled=True)
    pooled_ref, pabs, st = orc.embbag(tabs_host, nr, cidx, batch.offsets, w.B, w.D, w.mode, with_abs=True)
    pooled = fwd_ref["pooled"]
    new_ref = [t.copy() for t in tabs_host]
    acc_ref = [np.full(n, w.accum_init, np.float32) for n in nr]
    gd_ref, st2 = orc.sparse_bwd_adagrad(new_ref, nr, cidx, batch.offsets, batch.dense, pooled, batch.grad_out,
                                         acc_ref, w.lr, w.eps, w.mode)
    assert st == 0 and st2 == 0

    tabs = workload_tables(w)
    acc = [torch.full((V,), w.accum_init, dtype=torch.float32, device="cuda") for V in w.num_rows]
    di, do, dx = batch_to_device(batch)
    ps = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dl.dlrm_sparse_fwd(tabs, di, do, dx, w.mode, pooled_save=ps, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0 and fwd_ref["status"] == 0
    # the forward of the step (the multi-lookup tensor-core kernel), every value against the oracle
    assert_close(out.cpu().numpy(), fwd_ref["out"], fwd_ref["out_abs"], TOL_INTERACT, "training forward out")
    assert_close(ps.cpu().numpy(), pooled_ref, pabs, TOL_POOL_F32, "training forward pooled_save")
    del out
    gd = dl.dlrm_sparse_bwd_adagrad(tabs, acc, di, do, dx, ps, torch.from_numpy(batch.grad_out).cuda(), w.lr,
                                    w.eps, w.mode, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    N = w.T + 1
    Vabs = np.abs(pooled)
    s = np.abs(batch.grad_out[:, :w.D]) + np.einsum("bj,bjd->bd", np.abs(batch.grad_out[:, w.D:w.D + w.T]), Vabs)
    assert_close(gd.cpu().numpy(), gd_ref, s, TOL_INTERACT, "grad_dense")
    off = batch.offsets.astype(np.int64)
    for t in range(w.T):
        rows = np.unique(batch.indices[off[t * w.B]:off[(t + 1) * w.B]]).astype(np.int64)
        got = tabs[t][torch.from_numpy(rows).cuda()].cpu().numpy()
        got_acc = acc[t][torch.from_numpy(rows).cuda()].cpu().numpy()
        scale = np.abs(tabs_host[t]) + np.abs(tabs_host[t] - new_ref[t])
        assert_close(got, new_ref[t], scale, TOL_ADAGRAD, f"rows of table {t}")
        assert_close(got_acc, acc_ref[t], 0.0, TOL_ADAGRAD, f"accum of table {t}")
        # a sample of untouched rows still holds the generator's values
        rng = np.random.default_rng(t)
        probe = rng.integers(0, w.num_rows[t], size=64)
        probe = probe[~np.isin(probe, rows)]
        assert np.array_equal(tabs[t][torch.from_numpy(probe).cuda()].cpu().numpy(),
                              gen.table_rows(w.seed, t, probe, w.D))
        assert torch.all(acc[t][torch.from_numpy(probe).cuda()] == w.accum_init)
    del tabs, acc, ps
    free_cuda()
