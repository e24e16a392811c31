"""Tables larger than device memory: rows in pinned host memory, a device cache
of hot rows, and the staging pre-pass (dlrm_tier_*).

CPU: the host-side hot-row policy against brute-force counting.
GPU: a tiered forward (stage, then the ordinary forward on the device buffers)
equals the untiered forward bit for bit and the oracle within the fp32
tolerances; cache refills, a staging area that runs out, out-of-range indices
and an empty cache."""
import collections

import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl


def test_hot_rows_policy_brute_force():
    rng = np.random.default_rng(5)
    B, T = 50, 3
    L = rng.integers(0, 6, size=T * B)
    off = np.concatenate([[0], np.cumsum(L)])
    idx = (rng.zipf(1.5, size=int(off[-1])) % 40).astype(np.int64)
    hot = dl.hot_rows(idx, off, B, T, 7)
    for t in range(T):
        c = collections.Counter(idx[off[t * B]:off[(t + 1) * B]].tolist())
        want = sorted(c, key=lambda r: (-c[r], r))[:7]
        assert hot[t].tolist() == want


def _pinned(tabs, dtype):
    out = []
    for t in tabs:
        x = torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).view(torch.bfloat16) if dtype == "bf16" \
            else torch.from_numpy(np.ascontiguousarray(t))
        out.append(x.pin_memory())
    return out


CASES = [
    # D, T, dtype, mode, itype, Lmin, Lmax, B, V, cached fraction, stage rows per table (None: every lookup)
    (128, 26, "f32", "sum", "i32", 1, 1, 3001, 4000, 0.25, None),
    (128, 26, "f32", "mean", "i64", 1, 8, 1500, 4000, 0.10, None),
    (64, 40, "bf16", "sum", "i32", 0, 4, 700, 2000, 0.30, None),
    (16, 4, "f32", "sum", "i32", 1, 3, 800, 500, 0.0, None),
    (256, 3, "f32", "mean", "i64", 1, 5, 300, 3000, 0.5, None),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "D{}-T{}-{}-{}-{}-L{}..{}-B{}-V{}-c{}".format(*c[:10]))
def test_tiered_forward_equals_untiered(case):
    import gpu_util
    import oracle
    D, T, dtype, mode, itype, Lmin, Lmax, B, V, frac, M = case
    tabs, Vs, idx, off, dense = gpu_util.random_case(1000 + CASES.index(case), B, T, D, V, Lmin, Lmax, dtype)
    stage_rows = [int(off[(t + 1) * B] - off[t * B]) for t in range(T)] if M is None else M
    tier = dl.TieredTables(_pinned(tabs, dtype), int(frac * V), stage_rows)
    for t, rows in enumerate(dl.hot_rows(idx, off, B, T, int(frac * V))):
        tier.fill(t, torch.from_numpy(rows).cuda())
    di, do = gpu_util.dev_index(idx, itype), gpu_util.dev_index(off, itype)
    dx = torch.from_numpy(dense).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    staged = tier.stage(di, do, status=status)
    out = dl.dlrm_sparse_fwd(tier.device_tables, staged, do, dx, mode, status=status)
    pooled = dl.dlrm_embbag_fwd(tier.device_tables, staged, do, mode, status=status)
    ref = dl.dlrm_sparse_fwd(gpu_util.dev_tables(tabs, dtype), di, do, dx, mode)
    ref_pooled = dl.dlrm_embbag_fwd(gpu_util.dev_tables(tabs, dtype), di, do, mode)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(out, ref) and torch.equal(pooled, ref_pooled)
    orc = oracle.get().sparse_fwd(tabs, Vs, idx, off, dense, mode, dtype, with_abs=True)
    gpu_util.assert_close(out.cpu().numpy(), orc["out"], orc["out_abs"],
                          gpu_util.TOL_INTERACT if dtype == "f32" else gpu_util.TOL_BF16, "tiered out")
    # every cached lookup reads its slot, every miss a staging row
    st = staged.cpu().numpy().astype(np.int64)
    C = int(frac * V)
    for t in range(T):
        seg = slice(off[t * B], off[(t + 1) * B])
        slot_of = tier.slot_of[t].cpu().numpy()
        cached = slot_of[idx[seg]] >= 0
        assert np.array_equal(st[seg][cached], slot_of[idx[seg]][cached])
        assert np.all(st[seg][~cached] >= C)


@pytest.mark.gpu
def test_cache_refill_and_maps():
    import gpu_util
    B, T, D, V = 900, 5, 64, 1000
    tabs, Vs, idx, off, dense = gpu_util.random_case(1100, B, T, D, V, 1, 4)
    tier = dl.TieredTables(_pinned(tabs, "f32"), 300, int(np.diff(off).max()) * B)
    dx = torch.from_numpy(dense).cuda()
    di, do = gpu_util.dev_index(idx, "i32"), gpu_util.dev_index(off, "i32")
    ref = dl.dlrm_sparse_fwd(gpu_util.dev_tables(tabs, "f32"), di, do, dx)
    rng = np.random.default_rng(3)
    for round_ in range(3):
        sets = [rng.choice(V, size=rng.integers(0, 301), replace=False).astype(np.int64) for _ in range(T)]
        for t in range(T):
            tier.fill(t, torch.from_numpy(sets[t]).cuda())
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = dl.dlrm_sparse_fwd(tier.device_tables, tier.stage(di, do, status=status), do, dx, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0 and torch.equal(out, ref), f"round {round_}"
        for t in range(T):
            slot_of = tier.slot_of[t].cpu().numpy()
            want = np.full(V, -1)
            want[sets[t]] = np.arange(sets[t].size)
            assert np.array_equal(slot_of, want), f"map of table {t}, round {round_}"
            cache = tier.cache[t][:sets[t].size].cpu().numpy()
            assert np.array_equal(cache, tabs[t][sets[t]])


@pytest.mark.gpu
def test_staging_capacity_and_bad_indices():
    import gpu_util
    import oracle
    B, T, D, V = 200, 3, 128, 500
    tabs, Vs, idx, off, dense = gpu_util.random_case(1200, B, T, D, V, 1, 3)
    di, do = gpu_util.dev_index(idx, "i32"), gpu_util.dev_index(off, "i32")
    # too few staging rows: flagged
    tier = dl.TieredTables(_pinned(tabs, "f32"), 0, 10)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tier.stage(di, do, status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_CAPACITY
    # out-of-range indices: the forward flags them and pools them as zero, as on the untiered tables
    bad = idx.copy()
    bad[3], bad[-2] = V, -7
    tier = dl.TieredTables(_pinned(tabs, "f32"), 100, int(idx.size))
    status.zero_()
    dbad = gpu_util.dev_index(bad, "i32")
    out = dl.dlrm_sparse_fwd(tier.device_tables, tier.stage(dbad, do, status=status), do,
                             torch.from_numpy(dense).cuda(), status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_INDEX_OOB
    ref = oracle.get().sparse_fwd(tabs, Vs, bad, off, dense, "sum", with_abs=True)
    gpu_util.assert_close(out.cpu().numpy(), ref["out"], ref["out_abs"], gpu_util.TOL_INTERACT, "oob tiered out")
