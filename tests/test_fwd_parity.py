"""GPU parity of the forward entry points (through the C ABI) with the CPU oracle.

Shapes span several CTAs with a ragged tail; bags include empty, single and
duplicate lookups; every supported width and both element and index types
appear.  Full-size workloads compare every output value."""
import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
import gen
import oracle
from gpu_util import (TOL_BF16, TOL_INTERACT, TOL_POOL_F32, assert_close, batch_to_device, dev_index,
                      dev_tables, free_cuda, random_case, workload_tables)

pytestmark = pytest.mark.gpu

CASES = [
    # D, T, dtype, mode, itype, Lmin, Lmax, B
    (16, 4, "f32", "sum", "i32", 1, 1, 37),
    (128, 26, "f32", "sum", "i32", 1, 1, 133),
    (128, 26, "bf16", "sum", "i32", 0, 9, 67),
    (128, 26, "f32", "mean", "i64", 0, 6, 45),
    (64, 100, "f32", "sum", "i64", 1, 1, 19),
    (32, 7, "f32", "mean", "i32", 0, 40, 70),
    (256, 3, "bf16", "mean", "i64", 0, 3, 41),
    (128, 1, "f32", "sum", "i32", 0, 4, 29),
    (64, 128, "f32", "sum", "i32", 0, 2, 9),
    (256, 40, "f32", "mean", "i32", 1, 3, 11),
    (16, 13, "bf16", "sum", "i32", 1, 70, 23),
    (64, 20, "bf16", "mean", "i32", 1, 1, 50),
    # bags of 0..2 lookups: the tensor-core kernel, with its row-by-row pooling of the longer bags
    (128, 26, "f32", "mean", "i32", 0, 2, 50),
    (128, 26, "bf16", "sum", "i64", 0, 2, 37),
    (64, 40, "bf16", "sum", "i64", 0, 2, 33),
    (128, 100, "f32", "mean", "i32", 0, 2, 7),
    (64, 63, "f32", "sum", "i32", 1, 1, 13),
    (128, 31, "f32", "sum", "i32", 1, 1, 9),
    # long fp32 bags (mean 25): the FFMA kernel, two warps per sample
    (128, 26, "f32", "sum", "i64", 10, 40, 21),
]


def ids(c):
    return "D{}-T{}-{}-{}-{}-L{}..{}-B{}".format(*c)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_fused_embbag_interact(case, orc):
    D, T, dtype, mode, itype, Lmin, Lmax, B = case
    tabs, Vs, idx, off, dense = random_case(100 + CASES.index(case), B, T, D, 50, Lmin, Lmax, dtype)
    ref = orc.sparse_fwd(tabs, Vs, idx, off, dense, mode, dtype, with_abs=True, with_pooled=True)
    pooled_ref, pabs, st = orc.embbag(tabs, Vs, idx, off, B, D, mode, dtype, with_abs=True)
    assert st == 0 and ref["status"] == 0

    dt = dev_tables(tabs, dtype)
    di, do = dev_index(idx, itype), dev_index(off, itype)
    dx = torch.from_numpy(dense).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pooled_save = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    out = dl.dlrm_sparse_fwd(dt, di, do, dx, mode, pooled_save=pooled_save, status=status)
    pooled = dl.dlrm_embbag_fwd(dt, di, do, mode, status=status)
    out2 = dl.dlrm_interact_fwd(dx, torch.from_numpy(ref["pooled"]).cuda())
    torch.cuda.synchronize()
    assert status.item() == 0

    tol_pool = TOL_BF16 if dtype == "bf16" else TOL_POOL_F32
    assert_close(pooled.cpu().numpy(), pooled_ref, pabs, tol_pool, "embbag pooled")
    assert_close(pooled_save.cpu().numpy(), pooled_ref, pabs, tol_pool, "fused pooled_save")
    o = out.cpu().numpy()
    assert np.array_equal(o[:, :D].view(np.uint32), dense.view(np.uint32)), "dense part not copied exactly"
    assert_close(o, ref["out"], ref["out_abs"], TOL_INTERACT if dtype == "f32" else TOL_BF16, "fused out")
    assert_close(out2.cpu().numpy(), ref["out"], ref["out_abs"], TOL_INTERACT, "interact out")


# More tiles than the tensor-core kernel keeps resident (148 SMs x 3 CTAs = 444), so every CTA walks
# several tiles of its persistent loop: metadata read one and two tiles ahead, the MMA barrier's phase
# flipping, operand buffers reused.  Bags of 1..8 (mean 4.5) take the multi-lookup variant, bags of 0..2
# (mean 1) the one-hot variant with its row-by-row pooling of the longer bags.
MULTI_TILE_CASES = [
    # D, T, dtype, mode, itype, Lmin, Lmax, B, V
    (128, 26, "f32", "sum", "i32", 1, 8, 4001, 5000),
    (128, 26, "f32", "mean", "i64", 1, 8, 4003, 5000),
    (128, 26, "bf16", "sum", "i64", 1, 8, 4005, 5000),
    (128, 26, "bf16", "mean", "i32", 1, 8, 4002, 5000),
    (128, 26, "f32", "mean", "i32", 0, 8, 4000, 300),
    (64, 40, "f32", "sum", "i32", 1, 4, 2001, 2000),
    (64, 40, "bf16", "mean", "i64", 0, 4, 2003, 2000),
    (128, 26, "f32", "sum", "i32", 0, 2, 4007, 5000),
    (128, 80, "f32", "sum", "i64", 1, 3, 501, 1000),
]


@pytest.mark.parametrize("case", MULTI_TILE_CASES, ids=lambda c: "D{}-T{}-{}-{}-{}-L{}..{}-B{}-V{}".format(*c))
def test_fused_multi_tile(case, orc):
    D, T, dtype, mode, itype, Lmin, Lmax, B, V = case
    tabs, Vs, idx, off, dense = random_case(700 + MULTI_TILE_CASES.index(case), B, T, D, V, Lmin, Lmax, dtype)
    ref = orc.sparse_fwd(tabs, Vs, idx, off, dense, mode, dtype, with_abs=True)
    pooled_ref, pabs, st = orc.embbag(tabs, Vs, idx, off, B, D, mode, dtype, with_abs=True)
    assert st == 0 and ref["status"] == 0
    dt = dev_tables(tabs, dtype)
    di, do = dev_index(idx, itype), dev_index(off, itype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pooled_save = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    out = dl.dlrm_sparse_fwd(dt, di, do, torch.from_numpy(dense).cuda(), mode, pooled_save=pooled_save,
                             status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    o = out.cpu().numpy()
    assert np.array_equal(o[:, :D].view(np.uint32), dense.view(np.uint32)), "dense part not copied exactly"
    assert_close(o, ref["out"], ref["out_abs"], TOL_INTERACT if dtype == "f32" else TOL_BF16, "fused out")
    assert_close(pooled_save.cpu().numpy(), pooled_ref, pabs, TOL_BF16 if dtype == "bf16" else TOL_POOL_F32,
                 "fused pooled_save")
    # without pooled_save the multi-lookup bags stay in the one fused kernel (with it, the lookup kernel
    # writes the pooled vectors and the interaction reads them back): both routes against the oracle
    out_inf = dl.dlrm_sparse_fwd(dt, di, do, torch.from_numpy(dense).cuda(), mode, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_close(out_inf.cpu().numpy(), ref["out"], ref["out_abs"], TOL_INTERACT if dtype == "f32" else TOL_BF16,
                 "fused out without pooled_save")


def test_onehot_fp32_bit_exact(orc):
    B, T, D = 77, 26, 128
    tabs, Vs, idx, off, dense = random_case(5, B, T, D, 300, 1, 1)
    tabs[3][7, :3] = [-0.0, 1e-45, -3e38]
    idx[3 * B] = 7
    ref, st = orc.embbag(tabs, Vs, idx, off, B, D)
    dt = dev_tables(tabs, "f32")
    pooled = dl.dlrm_embbag_fwd(dt, dev_index(idx, "i32"), dev_index(off, "i32"))
    ps = torch.empty_like(pooled)
    dl.dlrm_sparse_fwd(dt, dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda(),
                       pooled_save=ps)
    assert np.array_equal(pooled.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(ps.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("D,T,B,Lmax", [(64, 100, 301, 1), (128, 80, 203, 3), (128, 26, 401, 1), (64, 40, 150, 2)])
def test_out_at_every_4_byte_offset(D, T, B, Lmax):
    """`out` need only be 4-byte aligned.  Rows written at 1, 2 and 3 floats past a 16-byte boundary (the
    one-sample tiles of N > 64 send their triangle by a bulk copy whose body must start on a 16-byte
    boundary of out, with plain stores for a head and a tail) equal the rows written to an aligned buffer
    bit for bit, for the fused forward and the interaction-only call; the floats around the rows stay
    untouched."""
    tabs, Vs, idx, off, dense = random_case(900 + T, B, T, D, 700, 1, Lmax, value_scale=0.1)
    dt, di, do = dev_tables(tabs, "f32"), dev_index(idx, "i32"), dev_index(off, "i32")
    dx = torch.from_numpy(dense).cuda()
    N = T + 1
    W = D + N * (N - 1) // 2
    ref = dl.dlrm_sparse_fwd(dt, di, do, dx)
    pooled = torch.empty((B, T, D), device="cuda")
    dl.dlrm_embbag_fwd(dt, di, do, pooled=pooled)
    ref_i = torch.empty((B, W), device="cuda")
    dl.dlrm_interact_fwd(dx, pooled, out=ref_i)
    for shift in (1, 2, 3):
        for call in ("fused", "interact"):
            buf = torch.full((B * W + 8,), -7.0, device="cuda")
            out = buf[shift:shift + B * W].view(B, W)
            if call == "fused":
                dl.dlrm_sparse_fwd(dt, di, do, dx, out=out)
            else:
                dl.dlrm_interact_fwd(dx, pooled, out=out)
            torch.cuda.synchronize()
            want = ref if call == "fused" else ref_i
            assert torch.equal(out.view(torch.int32), want.view(torch.int32)), (call, shift)
            assert torch.all(buf[:shift] == -7.0) and torch.all(buf[shift + B * W:] == -7.0), (call, shift)


def _round_to_16_bits(x):
    """x rounded to 16 significant bits: the sum of two bfloat16 values, which
    is what the tensor-core Gram carries of each fp32 operand."""
    hi = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(x))
    lo = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits((x - hi).astype(np.float32)))
    return (hi + lo).astype(np.float32)


@pytest.mark.parametrize("D,path", [(128, "tensor-core Gram"), (64, "tensor-core Gram"), (32, "FFMA Gram")])
def test_identity_tables_exact_interaction(D, path):
    """E_t = I: embedding-embedding values are [r_i == r_j], x-embedding values x[r_t], exactly.
    The tensor-core path represents each operand as hi + lo (two bf16), so its
    x is drawn with 16 significant bits; the FFMA path takes full fp32 x."""
    B, T = 64, 26
    rng = np.random.default_rng(9)
    tabs = [np.eye(D, dtype=np.float32) for _ in range(T)]
    r = rng.integers(0, D, size=(T, B))
    r[:, 0] = 5  # one sample with every embedding equal
    idx, off = r.reshape(-1), np.arange(T * B + 1)
    x = rng.standard_normal((B, D)).astype(np.float32)
    if path == "tensor-core Gram":
        x = _round_to_16_bits(x)
    out = dl.dlrm_sparse_fwd(dev_tables(tabs, "f32"), dev_index(idx, "i32"), dev_index(off, "i32"),
                             torch.from_numpy(x).cuda()).cpu().numpy()
    iu = torch.triu_indices(T + 1, T + 1, offset=1).numpy()
    for b in (0, 1, 17, 63):
        for k, (i, j) in enumerate(zip(iu[0], iu[1])):
            want = x[b, r[j - 1, b]] if i == 0 else np.float32(r[i - 1, b] == r[j - 1, b])
            assert out[b, D + k] == want


@pytest.mark.parametrize("itype,Lmin,Lmax", [("i32", 1, 4), ("i64", 1, 4), ("i32", 1, 2), ("i32", 0, 2)])
def test_bad_inputs_flag_and_zero(itype, Lmin, Lmax, orc):
    """Out-of-range indices and malformed offsets on the tensor-core kernel: its multi-lookup
    variant (bags of 1..4 or 1..2) and its one-hot variant (bags of 0..2, mean length 1)."""
    B, T, D = 9, 3, 64
    tabs, Vs, idx, off, dense = random_case(11, B, T, D, 20, Lmin, Lmax)
    idx[2] = 20        # == V: out of range
    idx[5] = -1
    idx[-1] = 1 << 30
    ref = orc.sparse_fwd(tabs, Vs, idx, off, dense, "mean", with_abs=True)
    assert ref["status"] == oracle.INDEX_OOB
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dl.dlrm_sparse_fwd(dev_tables(tabs, "f32"), dev_index(idx, itype), dev_index(off, itype),
                             torch.from_numpy(dense).cuda(), "mean", status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_INDEX_OOB
    assert_close(out.cpu().numpy(), ref["out"], ref["out_abs"], TOL_INTERACT, "oob out")

    off_bad = off.copy()
    off_bad[4] = off_bad[5] + 3  # bag 3 runs past bag 4's start: bag 4 reversed
    ref2 = orc.sparse_fwd(tabs, Vs, np.clip(idx, 0, 19), off_bad, dense, "sum", with_abs=True)
    status.zero_()
    out2 = dl.dlrm_sparse_fwd(dev_tables(tabs, "f32"), dev_index(np.clip(idx, 0, 19), itype),
                              dev_index(off_bad, itype), torch.from_numpy(dense).cuda(), "sum", status=status)
    torch.cuda.synchronize()
    assert ref2["status"] & oracle.BAD_OFFSETS and status.item() & dl.DLRM_ERR_BAD_OFFSETS
    assert_close(out2.cpu().numpy(), ref2["out"], ref2["out_abs"], TOL_INTERACT, "bad-offsets out")

    off_end = off.copy()
    off_end[-1] -= 1   # last offset != nnz
    status.zero_()
    dl.dlrm_embbag_fwd(dev_tables(tabs, "f32"), dev_index(np.clip(idx, 0, 19), itype), dev_index(off_end, itype),
                       status=status)
    torch.cuda.synchronize()
    assert status.item() & dl.DLRM_ERR_BAD_OFFSETS


def test_host_entry_point_matches_device_call():
    B, T, D = 300, 26, 128
    tabs, Vs, idx, off, dense = random_case(12, B, T, D, 1000, 1, 3)
    dt = dev_tables(tabs, "f32")
    ref = dl.dlrm_sparse_fwd(dt, dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda())
    ih = torch.from_numpy(idx.astype(np.int32)).pin_memory()
    oh = torch.from_numpy(off.astype(np.int32)).pin_memory()
    xh = torch.from_numpy(dense).pin_memory()
    out_h = torch.empty(ref.shape, dtype=torch.float32).pin_memory()
    stg = dl.HostStaging(B, T, D, idx.size)
    s = torch.cuda.Stream()
    dl.dlrm_sparse_fwd_host(dt, ih, oh, xh, out_h, stg, stream=s)
    s.synchronize()
    assert torch.equal(out_h, ref.cpu())


def test_bitwise_reproducible():
    B, T, D = 1000, 26, 128
    tabs, Vs, idx, off, dense = random_case(13, B, T, D, 5000, 0, 20, "bf16")
    dt = dev_tables(tabs, "bf16")
    args = (dt, dev_index(idx, "i32"), dev_index(off, "i32"), torch.from_numpy(dense).cuda())
    a = dl.dlrm_sparse_fwd(*args)
    b = dl.dlrm_sparse_fwd(*args)
    assert torch.equal(a, b)


def test_device_fill_matches_host_generator():
    rows = np.array([0, 1, 2, 999_999, 123_457, 4_999_999])
    for dtype, V, D in (("f32", 1_000_000, 128), ("bf16", 5_000_000, 128), ("f32", 1000, 16)):
        x = torch.empty((V, D), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
        gen.fill_table_device(x.data_ptr(), dtype, 77, 3, 0, V, D, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        r = rows[rows < V]
        got = x[torch.from_numpy(r).cuda()]
        got = got.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else got.cpu().numpy()
        assert np.array_equal(got, gen.table_rows_numpy(77, 3, r, D, dtype))
        del x


def _workload_parity(cid, orc):
    w = gen.workload(cid)
    batch, = gen.make_batches(w, [0])
    tabs_host, nr, cidx = gen.compact_tables(w, batch)
    ref = orc.sparse_fwd(tabs_host, nr, cidx, batch.offsets, batch.dense, w.mode, w.dtype, with_abs=True,
                         with_pooled=True)
    assert ref["status"] == 0
    tabs = workload_tables(w)
    di, do, dx = batch_to_device(batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pooled_save = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device="cuda")
    out = dl.dlrm_sparse_fwd(tabs, di, do, dx, w.mode, pooled_save=pooled_save, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    tol = TOL_BF16 if w.dtype == "bf16" else TOL_INTERACT
    err = assert_close(out.cpu().numpy(), ref["out"], ref["out_abs"], tol, f"workload {cid} out")
    ps = pooled_save.cpu().numpy()
    if w.bag_max == 1 and w.dtype == "f32":
        assert np.array_equal(ps.view(np.uint32), ref["pooled"].view(np.uint32))
    else:
        pooled_ref, pabs, _ = orc.embbag(tabs_host, nr, cidx, batch.offsets, w.B, w.D, w.mode, w.dtype,
                                         with_abs=True)
        assert_close(ps, pooled_ref, pabs, TOL_BF16 if w.dtype == "bf16" else TOL_POOL_F32, "pooled")
    del tabs, out, pooled_save
    free_cuda()
    return err


def test_workload_tiny(orc):
    _workload_parity(1, orc)


@pytest.mark.parametrize("cid", [2, 3, 4])
def test_workload_full_size(cid, orc):
    """Every output value of the full-size workloads (92 GB of fp32 tables for 2)."""
    _workload_parity(cid, orc)
