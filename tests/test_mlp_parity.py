"""GPU parity, through the C ABI, of the dense layers around the sparse path
against the float64 oracle (oracle/mlp.py): one FC layer forward (tensor-core
GEMM with bias and ReLU), its backward with SGD, the sigmoid/BCE head, and a
whole DLRM training step (bottom MLP, fused sparse forward, top MLP, head, and
the backward with SGD on the MLPs and row-wise Adagrad on the tables).

Error measure: |y - ref| / max(|ref|, S) with S the sum of |terms| behind ref
(|x| |W|^T + |b| for a layer); the tensor-core products carry about 16
significant bits of each operand (split-bf16), so a layer is held to 1e-4 and
updated weights, like updated rows, to 2e-3 of the step they take."""
import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
import oracle
from gpu_util import TOL_ADAGRAD, assert_close, dev_index, dev_tables, random_case
from oracle import mlp

pytestmark = pytest.mark.gpu

TOL_LAYER = 1e-4


def _layer(rng, fin, fout):
    return (rng.standard_normal((fout, fin)) / np.sqrt(fin)).astype(np.float32), \
        (rng.standard_normal(fout) * 0.1).astype(np.float32)


FC_CASES = [  # M, in, out, relu
    (1000, 13, 512, True), (333, 479, 256, True), (4097, 256, 128, False), (130, 1024, 1000, True),
    (7, 64, 3, False), (20000, 128, 512, True),
]


@pytest.mark.parametrize("M,K,N,relu", FC_CASES)
def test_fc_fwd(M, K, N, relu):
    rng = np.random.default_rng(M + K + N)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w, b = _layer(rng, K, N)
    ref = mlp.fc_fwd(x, w, b, relu)
    S = np.abs(x).astype(np.float64) @ np.abs(w).T.astype(np.float64) + np.abs(b)
    y = dl.dlrm_fc_fwd(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(), relu)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, S, TOL_LAYER, "fc forward")


@pytest.mark.parametrize("M,K,N,relu", FC_CASES)
def test_fc_bwd_sgd(M, K, N, relu):
    rng = np.random.default_rng(7 * M + K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w, b = _layer(rng, K, N)
    y = mlp.fc_fwd(x, w, b, relu).astype(np.float32)
    dy = rng.standard_normal((M, N)).astype(np.float32)
    dx_ref, dW, db = mlp.fc_bwd(x, w, y, dy, relu)
    lr = 0.01
    dwt, dbt = torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda()
    dx = dl.dlrm_fc_bwd_sgd(torch.from_numpy(x).cuda(), dwt, dbt, torch.from_numpy(y).cuda(),
                            torch.from_numpy(dy).cuda(), lr, relu)
    torch.cuda.synchronize()
    dz_abs = np.abs(dy) * ((y > 0) if relu else 1)
    assert_close(dx.cpu().numpy(), dx_ref, dz_abs.astype(np.float64) @ np.abs(w).astype(np.float64), TOL_LAYER, "dx")
    step_w = dwt.cpu().numpy().astype(np.float64) - w
    step_b = dbt.cpu().numpy().astype(np.float64) - b
    assert_close(step_w, -lr * dW, lr * (dz_abs.T.astype(np.float64) @ np.abs(x)) + 1e-7, TOL_ADAGRAD, "W step")
    assert_close(step_b, -lr * db, lr * dz_abs.sum(0) + 1e-7, TOL_ADAGRAD, "b step")


@pytest.mark.parametrize("M,K", [(1000, 256), (4099, 64), (3, 1024)])
def test_head_bce(M, K):
    rng = np.random.default_rng(M * 3 + K)
    h = np.maximum(rng.standard_normal((M, K)), 0).astype(np.float32)
    w = (rng.standard_normal(K) / np.sqrt(K)).astype(np.float32)
    b = np.array([0.2], np.float32)
    label = (rng.random(M) < 0.3).astype(np.float32)
    z, p, loss = mlp.head_fwd(h, w, b[0], label)
    dh, dw, db = mlp.head_bwd(h, w, z, label)
    wt, bt = torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda()
    prob, l, dht = dl.dlrm_head_bce_sgd(torch.from_numpy(h).cuda(), wt, bt, torch.from_numpy(label).cuda(), 0.1)
    torch.cuda.synchronize()
    assert abs(l.item() - loss) <= 1e-5 * max(1.0, abs(loss))
    assert_close(prob.cpu().numpy(), p, 0.0, 1e-5, "probability")
    assert_close(dht.cpu().numpy(), dh, np.abs(dh) + 1e-12, 1e-5, "dh")
    assert_close(wt.cpu().numpy().astype(np.float64) - w, -0.1 * dw, 0.1 * np.abs(h).T @ np.full(M, 1.0 / M) + 1e-9,
                 TOL_ADAGRAD, "w step")
    assert abs((bt.item() - b[0]) - (-0.1 * db)) <= 1e-5


@pytest.mark.parametrize("B,mode,side", [(1500, "sum", False), (3000, "mean", True)])
def test_dlrm_training_step(B, mode, side):
    """The whole step: bottom 13 -> 64 -> 128, T = 26 tables (D = 128, bags 1..8), top 479 -> 256 -> 64,
    head 64 -> 1.  Loss, the interaction output, every MLP weight after SGD and every table row after
    row-wise Adagrad against the oracle; with `side`, the sparse backward's sort runs on a second stream
    beside the forward."""
    orc = oracle.get()
    T, D, V = 26, 128, 400
    rng = np.random.default_rng(B)
    tabs, Vs, idx, off, _ = random_case(B, B, T, D, V, 1, 8, value_scale=0.05)
    dense_in = rng.standard_normal((B, 13)).astype(np.float32)
    label = (rng.random(B) < 0.25).astype(np.float32)
    K = D + (T + 1) * T // 2
    bottom = [_layer(rng, 13, 64), _layer(rng, 64, D)]
    top = [_layer(rng, K, 256), _layer(rng, 256, 64)]
    head = ((rng.standard_normal(64) / 8).astype(np.float32), np.float32(0.05))
    lr_mlp, lr_emb = 0.05, 0.01
    new_tabs = [t.copy() for t in tabs]
    acc_ref = [np.full(v, 0.1, np.float32) for v in Vs]
    ref = mlp.dlrm_step(orc, bottom, top, head, new_tabs, Vs, idx, off, dense_in, label, lr_mlp, lr_emb, 1e-8,
                        acc_ref, mode)
    assert ref["status"] == 0

    cuda = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    model = dl.DLRMModel(dev_tables(tabs, "f32"), [(cuda(w), cuda(b)) for w, b in bottom],
                         [(cuda(w), cuda(b)) for w, b in top], (cuda(head[0]), cuda(np.array([head[1]]))))
    acc = [torch.full((v,), 0.1, device="cuda") for v in Vs]
    loss, prob = model.train_step(cuda(dense_in), dev_index(idx, "i32"), dev_index(off, "i32"), cuda(label), lr_mlp,
                                  lr_emb, 1e-8, acc, mode=mode,
                                  side_stream=torch.cuda.Stream() if side else None)
    torch.cuda.synchronize()
    assert abs(loss.item() - ref["loss"]) <= 1e-4 * max(1.0, ref["loss"])
    # x (the bottom MLP's output) against its layer's scale |h| |W|^T + |b|
    h_prev = mlp.mlp_fwd(dense_in, bottom, relu_last=True)[-2]
    S_x = np.abs(h_prev) @ np.abs(bottom[-1][0]).T.astype(np.float64) + np.abs(bottom[-1][1])
    out = model._buf["out"].cpu().numpy()
    assert_close(out[:, :D], ref["x"], S_x, TOL_LAYER, "x")
    # the interaction values against sum |V_i[d] V_j[d]|; x's rounding (1e-4 of its scale) carries into them
    out_abs = orc.sparse_fwd(tabs, Vs, idx, off, ref["x"], mode, with_abs=True)["out_abs"]
    assert_close(out[:, D:], ref["out"][:, D:], out_abs[:, D:], 1e-3, "interaction out")
    # every layer's SGD step normwise (a single weight's step can cancel to almost nothing; the per-layer tests
    # check each gradient element against its own sum of |terms|), and every updated weight like a table row
    for k, ((wg, bg), (w0, b0), (wr, br)) in enumerate(zip(model.bottom + model.top, bottom + top,
                                                           ref["bottom"] + ref["top"])):
        for got, old, want, what in ((wg, w0, wr, "W"), (bg, b0, br, "b")):
            got = got.cpu().numpy().astype(np.float64)
            err = np.abs((got - old) - (want - old)).max() / np.abs(want - old).max()
            assert err <= 1e-2, f"layer {k} {what}: step error {err:.3g} of the largest step"
            assert_close(got, want, np.abs(old) + np.abs(want - old), TOL_ADAGRAD, f"layer {k} {what} after SGD")
    for t in range(T):
        got = model.tables.tensors[t].cpu().numpy()
        scale = np.abs(tabs[t]) + np.abs(tabs[t] - new_tabs[t])
        assert_close(got, new_tabs[t], scale, TOL_ADAGRAD, f"rows of table {t}")
