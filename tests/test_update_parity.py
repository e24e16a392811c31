"""GPU parity, through the C ABI, of the training step split at the pooled
vectors and of its second update rule, against the CPU oracle:

  dlrm_interact_bwd        grad_dense and grad_pooled
  dlrm_embbag_bwd_update   per-row sums and the Adagrad / SGD row update from a
                           seeded pooled gradient (the same input on both sides)
  dlrm_sparse_bwd_update   the fused training step with plain SGD
  dlrm_hash_indices        raw 64-bit IDs to rows, bit-exact

Untouched rows stay bit-identical; touched rows and accumulators within the
Adagrad-row tolerance."""
import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
import oracle
from gpu_util import TOL_ADAGRAD, TOL_INTERACT, assert_close, dev_index, dev_tables, random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _check_rows(got_tabs, got_acc, tabs, new_ref, acc_ref, idx, off, B, what):
    for t in range(len(tabs)):
        got = got_tabs[t].cpu().numpy()
        touched = np.zeros(tabs[t].shape[0], bool)
        seg = idx[off[t * B]:off[(t + 1) * B]]
        touched[seg] = True
        assert np.array_equal(got[~touched], tabs[t][~touched]), f"{what}: untouched rows of table {t} changed"
        scale = np.abs(tabs[t][touched]) + np.abs(tabs[t][touched] - new_ref[t][touched])
        assert_close(got[touched], new_ref[t][touched], scale, TOL_ADAGRAD, f"{what}: rows of table {t}")
        if got_acc is not None:
            acc = got_acc[t].cpu().numpy()
            assert np.all(acc[~touched] == acc_ref[t][~touched])
            assert_close(acc[touched], acc_ref[t][touched], 0.0, TOL_ADAGRAD, f"{what}: accum of table {t}")


INTERACT_CASES = [(16, 4, 37), (128, 26, 1001), (64, 100, 19), (256, 3, 41), (32, 63, 70)]


@pytest.mark.parametrize("D,T,B", INTERACT_CASES, ids=lambda *a: None)
def test_interact_bwd(D, T, B, orc):
    rng = np.random.default_rng(300 + D + T)
    x = rng.standard_normal((B, D)).astype(np.float32)
    P = rng.uniform(-1, 1, size=(B, T, D)).astype(np.float32)
    N = T + 1
    g = rng.standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
    gd_ref, gp_ref = orc.interact_bwd(x, P, g)
    gd, gp = dl.dlrm_interact_bwd(torch.from_numpy(x).cuda(), torch.from_numpy(P).cuda(), torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    # scale: sum_j |g_ij| |V_j| (+ |g_x| for x)
    V = np.concatenate([np.abs(x)[:, None], np.abs(P)], axis=1).astype(np.float64)
    G = np.zeros((B, N, N))
    iu = np.triu_indices(N, 1)
    G[:, iu[0], iu[1]] = np.abs(g[:, D:])
    G = G + G.transpose(0, 2, 1)
    S = np.einsum("bij,bjd->bid", G, V)
    assert_close(gd.cpu().numpy(), gd_ref, S[:, 0] + np.abs(g[:, :D]), TOL_INTERACT, "grad_dense")
    assert_close(gp.cpu().numpy(), gp_ref, S[:, 1:], TOL_INTERACT, "grad_pooled")


EMB_CASES = [
    # D, T, mode, itype, Lmin, Lmax, B, V, rule
    (128, 26, "sum", "i32", 1, 8, 600, 400, "adagrad"),
    (128, 26, "mean", "i64", 0, 8, 500, 400, "adagrad"),
    (128, 26, "sum", "i32", 1, 8, 600, 400, "sgd"),
    (64, 7, "mean", "i32", 0, 20, 333, 60, "sgd"),
    (16, 3, "sum", "i64", 1, 3, 2000, 9, "sgd"),
    (256, 2, "mean", "i32", 1, 4, 90, 500, "adagrad"),
]


@pytest.mark.parametrize("case", EMB_CASES, ids=lambda c: "D{}-T{}-{}-{}-L{}..{}-B{}-V{}-{}".format(*c))
@pytest.mark.parametrize("two_streams", [False, True], ids=["one-stream", "side-stream"])
def test_embbag_bwd_update(case, two_streams, orc):
    D, T, mode, itype, Lmin, Lmax, B, V, rule = case
    tabs, Vs, idx, off, _ = random_case(400 + EMB_CASES.index(case), B, T, D, V, Lmin, Lmax, value_scale=0.05)
    gp = np.random.default_rng(7).standard_normal((B, T, D)).astype(np.float32)  # the same seeded input for both
    lr, eps = (0.01, 1e-8) if rule == "adagrad" else (0.05, 0.0)
    new_ref = [t.copy() for t in tabs]
    acc_ref = [np.full(v, 0.1, np.float32) for v in Vs] if rule == "adagrad" else None
    assert orc.embbag_bwd_update(new_ref, Vs, idx, off, gp, rule, lr, eps, acc_ref, mode) == 0
    dt = dev_tables(tabs, "f32")
    acc = [torch.full((v,), 0.1, device="cuda") for v in Vs] if rule == "adagrad" else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dlrm_embbag_bwd_update(dt, dev_index(idx, itype), dev_index(off, itype), torch.from_numpy(gp).cuda(), rule,
                              lr, eps, acc, mode, status=status,
                              side_stream=torch.cuda.Stream() if two_streams else None)
    torch.cuda.synchronize()
    assert status.item() == 0
    _check_rows(dt, acc, tabs, new_ref, acc_ref, idx, off, B, f"{rule} {mode}")


SGD_CASES = [
    (128, 26, "sum", "i32", 1, 8, 4000, 2000),
    (128, 26, "mean", "i64", 0, 8, 300, 300),
    (64, 40, "sum", "i32", 0, 3, 257, 100),
    (32, 100, "mean", "i32", 1, 2, 21, 100),
]


@pytest.mark.parametrize("case", SGD_CASES, ids=lambda c: "D{}-T{}-{}-{}-L{}..{}-B{}-V{}".format(*c))
def test_sparse_bwd_sgd(case, orc):
    D, T, mode, itype, Lmin, Lmax, B, V = case
    tabs, Vs, idx, off, dense = random_case(500 + SGD_CASES.index(case), B, T, D, V, Lmin, Lmax, value_scale=0.05)
    N = T + 1
    g = np.random.default_rng(8).standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
    pooled, st = orc.embbag(tabs, Vs, idx, off, B, D, mode)
    new_ref = [t.copy() for t in tabs]
    gd_ref, st2 = orc.sparse_bwd_update(new_ref, Vs, idx, off, dense, pooled, g, "sgd", 0.05, mode=mode)
    assert st == 0 and st2 == 0
    dt = dev_tables(tabs, "f32")
    di, do, dx = dev_index(idx, itype), dev_index(off, itype), torch.from_numpy(dense).cuda()
    ps = torch.empty((B, T, D), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dlrm_sparse_fwd(dt, di, do, dx, mode, pooled_save=ps, status=status)
    gd = dl.dlrm_sparse_bwd_update(dt, di, do, dx, ps, torch.from_numpy(g).cuda(), "sgd", 0.05, mode=mode,
                                   status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Vabs = np.abs(pooled)
    s = np.abs(g[:, :D]) + np.einsum("bj,bjd->bd", np.abs(g[:, D:D + T]), Vabs)
    assert_close(gd.cpu().numpy(), gd_ref, s, TOL_INTERACT, "grad_dense")
    _check_rows(dt, None, tabs, new_ref, None, idx, off, B, "sgd step")


HASH_CASES = [
    # T, B, Lmax, row counts, itype
    (4, 300, 5, [1, 7, 1 << 20, 1 << 31], "i32"),
    (3, 1000, 8, [4_294_967_311, (1 << 62) + 3, 1000], "i64"),
    (26, 2048, 8, [2_000_000] * 26, "i32"),
]


@pytest.mark.parametrize("T,B,Lmax,V,itype", HASH_CASES, ids=lambda *a: None)
def test_hash_indices_bit_exact(T, B, Lmax, V, itype, orc):
    rng = np.random.default_rng(600 + T)
    L = rng.integers(0, Lmax + 1, size=T * B)
    off = np.zeros(T * B + 1, np.int64)
    np.cumsum(L, out=off[1:])
    raw = rng.integers(np.iinfo(np.int64).min, np.iinfo(np.int64).max, size=int(off[-1]), dtype=np.int64)
    raw[:2] = [-1, np.iinfo(np.int64).min]  # 2^64 - 1 and 2^63 as unsigned
    ref, st = orc.hash_indices(V, raw, off, B)
    assert st == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = dl.dlrm_hash_indices(V, torch.from_numpy(raw).cuda(), dev_index(off, itype), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(rows.cpu().numpy().astype(np.int64), ref)


def test_hash_indices_flags_bad_offsets(orc):
    T, B = 3, 10
    off = np.arange(T * B + 1, dtype=np.int64)
    off[B] = 3 * B - 1          # table 1 starts after table 2 does: boundaries go backwards
    raw = np.arange(T * B, dtype=np.int64)
    _, st = orc.hash_indices([5, 6, 7], raw, off, B)
    assert st & oracle.BAD_OFFSETS
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dlrm_hash_indices([5, 6, 7], torch.from_numpy(raw).cuda(), dev_index(off, "i32"), status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_BAD_OFFSETS


def test_hashed_ids_feed_the_forward(orc):
    """The pre-pass output serves as the bags' indices: raw IDs -> rows -> fused forward, against the
    oracle's hash followed by the oracle's forward."""
    B, T, D, V = 513, 26, 128, 3000
    tabs, Vs, _, off, dense = random_case(610, B, T, D, V, 1, 4)
    rng = np.random.default_rng(611)
    raw = rng.integers(0, np.iinfo(np.int64).max, size=int(off[-1]), dtype=np.int64)
    rows_ref, st = orc.hash_indices(Vs, raw, off, B)
    ref = orc.sparse_fwd(tabs, Vs, rows_ref, off, dense, "sum", with_abs=True)
    do = dev_index(off, "i32")
    rows = dl.dlrm_hash_indices(Vs, torch.from_numpy(raw).cuda(), do)
    out = dl.dlrm_sparse_fwd(dev_tables(tabs, "f32"), rows, do, torch.from_numpy(dense).cuda())
    torch.cuda.synchronize()
    assert st == 0 and ref["status"] == 0
    assert_close(out.cpu().numpy(), ref["out"], ref["out_abs"], TOL_INTERACT, "hashed forward")


@pytest.mark.parametrize("itype", ["i32", "i64"])
def test_hash_indices_unaligned_buffers(itype, orc):
    """IDs and rows 8 bytes off a 16-byte boundary: the one-lookup-per-thread path of the kernel."""
    T, B = 5, 777
    rng = np.random.default_rng(620)
    V = [3, 1000, 65537, 1 << 30, 17]
    L = rng.integers(0, 7, size=T * B)
    off = np.zeros(T * B + 1, np.int64)
    np.cumsum(L, out=off[1:])
    raw = rng.integers(np.iinfo(np.int64).min, np.iinfo(np.int64).max, size=int(off[-1]), dtype=np.int64)
    ref, st = orc.hash_indices(V, raw, off, B)
    buf = torch.empty(raw.size + 1, dtype=torch.int64, device="cuda")
    buf[1:] = torch.from_numpy(raw).cuda()
    dt = torch.int32 if itype == "i32" else torch.int64
    rows_buf = torch.empty(raw.size + 2, dtype=dt, device="cuda")
    rows = rows_buf[2:] if itype == "i32" else rows_buf[1:-1]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dlrm_hash_indices(V, buf[1:], dev_index(off, itype), rows=rows, status=status)
    torch.cuda.synchronize()
    assert st == 0 and status.item() == 0
    assert np.array_equal(rows.cpu().numpy().astype(np.int64), ref)
