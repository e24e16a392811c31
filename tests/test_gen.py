"""The seeded input generators (host side): definition, determinism, shapes."""
import numpy as np
import pytest

import gen


def test_numpy_and_c_fill_agree():
    gen.table_rows(0, 0, [0], 4)  # builds/loads the library
    rows = np.array([0, 1, 7, 999, 4_000_000 - 1, 123_456_789])
    for dtype in ("f32", "bf16"):
        for D in (16, 64, 128):
            a = gen.table_rows_numpy(20261204, 5, rows, D, dtype)
            b = gen.table_rows(20261204, 5, rows, D, dtype)
            assert a.dtype == b.dtype and np.array_equal(a, b)


def test_value_range_and_spread():
    v = gen.table_rows(1, 0, np.arange(4096), 128)
    assert v.min() >= -0.05 and v.max() < 0.05
    assert abs(v.mean()) < 1e-3 and abs(v.std() - 0.1 / np.sqrt(12)) < 1e-3
    # bf16 is the nearest-even rounding of the fp32 value
    h = gen.table_rows(1, 0, np.arange(64), 128, "bf16")
    f = gen.bf16_bits_to_f32(h)
    assert np.all(np.abs(f - v[:64]) <= np.abs(v[:64]) * 2.0 ** -8 + 1e-12)


def test_streams_differ_per_table_and_seed():
    a = gen.table_rows(1, 0, [5], 32)
    assert not np.array_equal(a, gen.table_rows(1, 1, [5], 32))
    assert not np.array_equal(a, gen.table_rows(2, 0, [5], 32))


@pytest.mark.parametrize("V,alpha", [(1000, 1.05), (7, 1.1), (5_000_000, 1.1)])
def test_zipf_frequencies(V, alpha):
    """Rank counts against the exact probabilities k^-alpha / sum_j j^-alpha."""
    rng = np.random.default_rng(0)
    n = 400_000
    k = gen.zipf_ranks(rng, V, alpha, n)
    assert k.min() >= 1 and k.max() <= V
    Z = np.sum(np.arange(1, V + 1, dtype=np.float64) ** -alpha)
    counts = np.bincount(k, minlength=min(V, 200) + 1)
    for r in [1, 2, 3, 5, 7, 10, 100]:
        if r > V:
            continue
        exp = r ** -alpha / Z * n
        assert abs(counts[r] - exp) < 5 * np.sqrt(exp) + 1, (r, counts[r], exp)
    # tail mass beyond rank 100 (or none)
    if V > 100:
        exp_tail = (1 - np.sum(np.arange(1, 101, dtype=np.float64) ** -alpha) / Z) * n
        got_tail = np.sum(k > 100)
        assert abs(got_tail - exp_tail) < 5 * np.sqrt(exp_tail), (got_tail, exp_tail)


def test_affine_permutation_is_bijection():
    for V in (1, 2, 97, 1000, 65536):
        a, c = gen.affine_perm_params(3, 1, V)
        img = gen.permute(np.arange(V), a, c, V)
        assert np.array_equal(np.sort(img), np.arange(V))


def test_production_sizes():
    w = gen.workload(2)
    assert len(w.num_rows) == 26 and 1.75e8 <= sum(w.num_rows) <= 1.85e8
    assert min(w.num_rows) >= 1000 and max(w.num_rows) <= 40_000_000
    assert 88e9 <= w.table_bytes() <= 95e9


@pytest.mark.parametrize("cid", [1, 4])
def test_batch_structure(cid):
    w = gen.workload(cid)
    b1, b2 = gen.make_batches(w, [0, 1])
    b1b, = gen.make_batches(w, [0])
    assert np.array_equal(b1.indices, b1b.indices) and np.array_equal(b1.dense, b1b.dense)
    assert not np.array_equal(b1.indices, b2.indices)
    off = b1.offsets.astype(np.int64)
    assert off.size == w.T * w.B + 1 and off[0] == 0 and off[-1] == b1.nnz
    L = np.diff(off)
    assert L.min() >= w.bag_min and L.max() <= w.bag_max
    for t in range(w.T):
        seg = b1.indices[off[t * w.B]:off[(t + 1) * w.B]]
        assert seg.min() >= 0 and seg.max() < w.num_rows[t]
    assert b1.dense.shape == (w.B, w.D) and b1.dense.dtype == np.float32


def test_multihot_lengths_small():
    w = gen.workload(3, B=256, num_rows=[5000] * 26)
    b, = gen.make_batches(w, [0])
    L = np.diff(b.offsets.astype(np.int64))
    assert L.min() == 1 and L.max() == 64 and abs(L.mean() - 32.5) < 1.0


def test_compact_tables_preserve_rows():
    w = gen.workload(1)
    b, = gen.make_batches(w, [0])
    tabs, nr, idx = gen.compact_tables(w, b)
    full0 = gen.table_rows(w.seed, 0, np.arange(w.num_rows[0]), w.D)
    off = b.offsets.astype(np.int64)
    seg = slice(off[0], off[w.B])
    assert np.array_equal(tabs[0][idx[seg]], full0[b.indices[seg]])
