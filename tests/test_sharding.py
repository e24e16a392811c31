"""Table-wise model parallelism of the sparse path.

CPU (no GPU needed): the partition of the tables, the per-shard bag split, and
the collective exchange between two gloo ranks: each rank pools its own tables
with the oracle, the ranks exchange the pooled vectors with the plan's
all_to_all_single splits, and the interaction and the backward run per sample
shard; the results equal the unsharded oracle's.

GPU: G logical shards on one device through the C ABI (embedding-bag forward
per table shard, the library's exchange kernel, interaction per sample shard)
give dlrm_sparse_fwd's output bit for bit, and the sharded training step
matches the oracle; the unpack after a collective exchange (one sample shard
per device) gives the logical exchange's buffers."""
import os
import sys

import numpy as np
import pytest
import torch

from embedding_bag_lookup_dlrm_b300 import sharding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem(seed, B=40, T=7, D=16, V=(30, 5, 70, 12, 9, 40, 3), Lmin=0, Lmax=4):
    import gpu_util
    return gpu_util.random_case(seed, B, T, D, list(V), Lmin, Lmax, value_scale=0.05)


def test_partition_is_a_balanced_assignment():
    rng = np.random.default_rng(1)
    for G in (1, 2, 3, 4, 8):
        tb = [int(x) for x in rng.integers(1, 10_000, size=26)]
        shard, slot = sharding.partition_tables(tb, G)
        loads = [sum(b for b, s in zip(tb, shard) if s == g) for g in range(G)]
        assert sum(loads) == sum(tb)
        assert max(loads) - min(loads) <= max(tb)            # greedy largest-first bound
        for g in range(G):
            mine = [t for t in range(26) if shard[t] == g]
            assert sorted(slot[t] for t in mine) == list(range(len(mine)))
            assert [slot[t] for t in mine] == list(range(len(mine)))   # slots follow the global order


def test_split_bags_keeps_every_bag():
    tabs, Vs, idx, off, dense = _problem(2)
    B, T = dense.shape[0], len(tabs)
    plan = sharding.ShardPlan.make(Vs, 16, B, 3)
    parts = sharding.split_bags(plan, idx, off)
    for g, (ig, og) in enumerate(parts):
        mine = plan.tables_of(g)
        assert og[0] == 0 and og[-1] == ig.size and og.size == len(mine) * B + 1
        for k, t in enumerate(mine):
            for b in range(B):
                want = idx[off[t * B + b]:off[t * B + b + 1]]
                got = ig[og[k * B + b]:og[k * B + b + 1]]
                assert np.array_equal(want, got)


def test_sample_ranges():
    assert sharding.sample_ranges(10, 4) == [0, 2, 5, 7, 10]
    assert sharding.sample_ranges(3, 3) == [0, 1, 2, 3]


def _pack(plan, h, x):
    """What the library's exchange with to_sample = 0 writes on sample shard h: per table shard g its
    block [n_h, T_g, D] (x: [n_h, T, D])."""
    return np.concatenate([x[:, plan.tables_of(g), :].reshape(-1) for g in range(plan.G)])


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    for p in (ROOT, os.path.join(ROOT, "tests")):
        sys.path.insert(0, p)
    import torch.distributed as dist

    import oracle
    from embedding_bag_lookup_dlrm_b300 import sharding as sh
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        orc = oracle.get()
        tabs, Vs, idx, off, dense = _problem(3)
        B, T, D = dense.shape[0], len(tabs), 16
        N = T + 1
        g_out = np.random.default_rng(4).standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
        plan = sh.ShardPlan.make(Vs, D, B, world)
        # the unsharded reference: the whole step on the oracle
        ref = orc.sparse_fwd(tabs, Vs, idx, off, dense, "mean", with_pooled=True)
        ref_gd, ref_gp = orc.interact_bwd(dense, ref["pooled"], g_out)
        ref_tabs = [t.copy() for t in tabs]
        ref_acc = [np.full(v, 0.1, np.float32) for v in Vs]
        orc.sparse_bwd_update(ref_tabs, Vs, idx, off, dense, ref["pooled"], g_out, "adagrad", 0.02, 1e-8, ref_acc,
                              "mean")

        # this rank as table shard `rank`: pool its tables for all samples
        mine = plan.tables_of(rank)
        idx_g, off_g = sh.split_bags(plan, idx, off)[rank]
        P_g, st = orc.embbag([tabs[t] for t in mine], [Vs[t] for t in mine], idx_g, off_g, B, D, "mean")
        assert st == 0
        recv = torch.empty(sum(plan.recv_counts(rank)), dtype=torch.float32)
        blocks = sh.exchange_all_to_all(plan, rank, torch.from_numpy(P_g), recv)
        lo, hi = plan.samples_of(rank)
        # the unpack's layout: block g holds tables_of(g) of this rank's samples
        Q = np.empty((hi - lo, T, D), np.float32)
        for g in range(plan.G):
            Q[:, plan.tables_of(g), :] = blocks[g].numpy()
        assert np.array_equal(Q, ref["pooled"][lo:hi]), "exchanged pooled vectors"
        out_h = orc.interact(dense[lo:hi], Q)
        assert np.array_equal(out_h, ref["out"][lo:hi]), "interaction of the sample shard"

        # backward: interaction backward per sample shard, reverse exchange, row update per table shard
        gd_h, gp_h = orc.interact_bwd(dense[lo:hi], Q, g_out[lo:hi])
        assert np.array_equal(gd_h, ref_gd[lo:hi])
        dP_g = torch.empty((B, len(mine), D), dtype=torch.float32)
        sh.exchange_all_to_all_reverse(plan, rank, torch.from_numpy(_pack(plan, rank, gp_h)), dP_g)
        assert np.array_equal(dP_g.numpy(), ref_gp[:, mine, :]), "pooled gradients back at the table owner"
        new = [tabs[t].copy() for t in mine]
        acc = [np.full(Vs[t], 0.1, np.float32) for t in mine]
        assert orc.embbag_bwd_update(new, [Vs[t] for t in mine], idx_g, off_g, dP_g.numpy(), "adagrad", 0.02, 1e-8,
                                     acc, "mean") == 0
        for k, t in enumerate(mine):
            # float gradients of the pooled vectors vs the unsharded step's double ones: one rounding apart
            scale = np.abs(tabs[t]) + np.abs(tabs[t] - ref_tabs[t])
            err = np.abs(new[k] - ref_tabs[t]) / np.maximum(np.maximum(np.abs(ref_tabs[t]), scale), 1e-30)
            assert err.max() <= 1e-5, f"rows of table {t}: {err.max()}"
        q.put((rank, "ok"))
    except BaseException as e:  # report, then let the other rank finish its collectives
        q.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


def test_exchange_two_gloo_ranks():
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: "ok", 1: "ok"}, res


# ---------------------------------------------------------------------------
# GPU
# ---------------------------------------------------------------------------
def _gpu_problem(seed, B, T, D, V, Lmin, Lmax):
    import gpu_util
    return gpu_util.random_case(seed, B, T, D, V, Lmin, Lmax, value_scale=0.05)


def _shard_inputs(plan, idx, off):
    import gpu_util
    return [(gpu_util.dev_index(i, "i32"), gpu_util.dev_index(o, "i32")) for i, o in sharding.split_bags(plan, idx, off)]


@pytest.mark.gpu
@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("Lmin,Lmax,mode", [(1, 1, "sum"), (1, 8, "sum"), (0, 8, "mean")])
def test_logical_shards_forward_bit_exact(G, Lmin, Lmax, mode):
    import embedding_bag_lookup_dlrm_b300 as dl
    import gpu_util
    B, T, D = 1003, 26, 128
    Vs = [int(v) for v in np.random.default_rng(G).integers(50, 5000, size=T)]
    tabs, Vs, idx, off, dense = _gpu_problem(800 + G, B, T, D, Vs, Lmin, Lmax)
    dt = gpu_util.dev_tables(tabs, "f32")
    dx = torch.from_numpy(dense).cuda()
    ref = dl.dlrm_sparse_fwd(dt, gpu_util.dev_index(idx, "i32"), gpu_util.dev_index(off, "i32"), dx, mode)
    plan = sharding.ShardPlan.make(Vs, D, B, G)
    step = sharding.ShardedSparse(dt, plan)
    out = step.forward(_shard_inputs(plan, idx, off), dx, mode)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("G,rule,mode", [(2, "adagrad", "sum"), (4, "adagrad", "mean"), (4, "sgd", "sum")])
def test_logical_shards_training_step(G, rule, mode):
    import embedding_bag_lookup_dlrm_b300 as dl  # noqa: F401
    import gpu_util
    import oracle
    orc = oracle.get()
    B, T, D, V = 777, 26, 128, 600
    tabs, Vs, idx, off, dense = _gpu_problem(900 + G, B, T, D, V, 1, 8)
    N = T + 1
    g = np.random.default_rng(G).standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
    pooled, _ = orc.embbag(tabs, Vs, idx, off, B, D, mode)
    new_ref = [t.copy() for t in tabs]
    acc_ref = [np.full(v, 0.1, np.float32) for v in Vs] if rule == "adagrad" else None
    lr = 0.01 if rule == "adagrad" else 0.05
    gd_ref, st = orc.sparse_bwd_update(new_ref, Vs, idx, off, dense, pooled, g, rule, lr, 1e-8, acc_ref, mode)
    assert st == 0

    dt = gpu_util.dev_tables(tabs, "f32")
    acc = [torch.full((v,), 0.1, device="cuda") for v in Vs] if rule == "adagrad" else None
    dx = torch.from_numpy(dense).cuda()
    plan = sharding.ShardPlan.make(Vs, D, B, G)
    step = sharding.ShardedSparse(dt, plan)
    bags = _shard_inputs(plan, idx, off)
    step.forward(bags, dx, mode)
    gd = step.backward(bags, dx, torch.from_numpy(g).cuda(), rule, lr, 1e-8, acc, mode)
    torch.cuda.synchronize()
    s = np.abs(g[:, :D]) + np.einsum("bj,bjd->bd", np.abs(g[:, D:D + T]), np.abs(pooled))
    gpu_util.assert_close(gd.cpu().numpy(), gd_ref, s, gpu_util.TOL_INTERACT, "sharded grad_dense")
    for t in range(T):
        got = dt[t].cpu().numpy()
        scale = np.abs(tabs[t]) + np.abs(tabs[t] - new_ref[t])
        gpu_util.assert_close(got, new_ref[t], scale, gpu_util.TOL_ADAGRAD, f"sharded rows of table {t}")
        if acc is not None:
            gpu_util.assert_close(acc[t].cpu().numpy(), acc_ref[t], 0.0, gpu_util.TOL_ADAGRAD, f"accum {t}")


@pytest.mark.gpu
def test_unpack_after_collective_matches_logical_exchange():
    """On each sample shard, the blocks a collective all-to-all would deliver (its samples' rows of every
    table shard), unpacked by the library with the one-sample-shard plan, equal the logical exchange's
    buffer; packing that buffer back gives the blocks again."""
    import gpu_util
    B, T, D, G = 301, 26, 64, 4
    tabs, Vs, idx, off, dense = _gpu_problem(950, B, T, D, 300, 1, 4)
    dt = gpu_util.dev_tables(tabs, "f32")
    plan = sharding.ShardPlan.make(Vs, D, B, G)
    step = sharding.ShardedSparse(dt, plan)
    step.forward(_shard_inputs(plan, idx, off), torch.from_numpy(dense).cuda())
    for h in range(G):
        lo, hi = plan.samples_of(h)
        received = [step.by_table[g][lo:hi].contiguous() for g in range(G)]  # what the collective delivers
        unpacked = torch.empty((hi - lo, T, D), device="cuda")
        c = plan.local_unpack_plan(h)
        sharding.pooled_exchange(c, received, [unpacked], 1)
        packed = [torch.empty_like(r) for r in received]
        sharding.pooled_exchange(c, packed, [unpacked], 0)
        torch.cuda.synchronize()
        assert torch.equal(unpacked, step.by_sample[h])
        for a, b in zip(packed, received):
            assert torch.equal(a, b)
