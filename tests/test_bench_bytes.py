"""The byte models behind bench.py's roofline figures, checked on the CPU
against per-sample counts written out from the workload descriptions (dense
x, one row per lookup, the output row of D + N(N-1)/2 floats, int32 indices
and offsets) and against the training step's parts counted one by one."""
import importlib.util
import os
import sys

import numpy as np
import pytest

import gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


@pytest.mark.parametrize("cid,per_sample", [
    # rows + x + out + indices + offsets, bytes per sample (one-hot workloads: one lookup per bag)
    (1, 4 * 16 * 4 + 16 * 4 + (16 + 10) * 4 + 4 * 4 + 4 * 4),          # 456
    (2, 26 * 128 * 4 + 128 * 4 + (128 + 351) * 4 + 26 * 4 + 26 * 4),  # 15,948
    (4, 100 * 64 * 4 + 64 * 4 + (64 + 5050) * 4 + 100 * 4 + 100 * 4),  # 47,112
])
def test_forward_bytes_per_sample(bench, cid, per_sample):
    w = gen.workload(cid)
    b, = gen.make_batches(w, [0])
    # the closing offset (T*B + 1 entries) is the only term that is not per sample
    assert bench.algorithmic_bytes(w, b) == w.B * per_sample + 4


def test_multi_hot_forward_bytes(bench):
    """Workload 3: bf16 rows, one per lookup, whatever the bag lengths."""
    w = gen.workload(3)
    b, = gen.make_batches(w, [0])
    want = b.nnz * (128 * 2 + 4) + w.B * (128 * 4 + (128 + 351) * 4) + (26 * w.B + 1) * 4
    assert bench.algorithmic_bytes(w, b) == want


@pytest.mark.parametrize("rows,passes", [(10, 1), (511, 1), (512, 2), (1 << 18, 3), (52_000_000, 3),
                                         (178_000_000, 4)])
def test_sort_passes(bench, rows, passes):
    """Digits of at most 9 bits over enough bits that the sentinel key's low bits (all ones) exceed every
    valid key (< total rows): 512 rows take 10 bits, hence two passes."""
    assert bench.passes_for_rows(rows) == passes


def test_training_step_bytes(bench):
    """Workload 5 with a smaller batch: every part of the step counted one by one."""
    w = gen.workload(5, B=512)
    b, = gen.make_batches(w, [0])
    tb = bench.train_bytes(w, b, "adagrad")
    B, T, D, nnz = w.B, w.T, w.D, b.nnz
    K = (T + 1) * T // 2
    BTD = B * T * D * 4
    csr = nnz * 4 + (T * B + 1) * 4
    off = b.offsets.astype(np.int64)
    touched = sum(len(set(b.indices[off[t * B]:off[(t + 1) * B]].tolist())) for t in range(T))
    assert tb["touched_rows"] == touched
    fwd = nnz * D * 4 + B * D * 4 + B * (D + K) * 4 + BTD + csr
    assert tb["forward"] == fwd
    passes = bench.sort_passes(w)
    assert passes == 3  # 26 tables of 2e6 rows: 26 key bits
    common = (B * (D + K) * 4      # grad_out read
              + B * D * 4          # x read
              + BTD                # pooled vectors read
              + B * D * 4          # grad_dense written
              + BTD                # dP written
              + nnz * 8            # lookup keys and values written
              + passes * nnz * 16  # each radix pass reads and writes (key, value)
              + touched * (2 * D * 4 + 8)  # each touched row read and written, its accumulator too
              + csr)               # indices and offsets read for the keys
    assert tb["backward"] == common + BTD                 # dP read once per bag
    assert tb["backward_per_lookup"] == common + nnz * D * 4  # dP read once per lookup
    assert tb["total"] == tb["forward"] + tb["backward"]
    sgd = bench.train_bytes(w, b, "sgd")
    assert tb["backward"] - sgd["backward"] == touched * 8  # no accumulator traffic
