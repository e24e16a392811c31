"""Pins of the dense-part oracle (oracle/mlp.py) to facts outside itself:
float64 torch autograd (torch.nn.functional.linear, relu,
binary_cross_entropy_with_logits, embedding_bag, bmm) and closed forms.
Each pin takes the module under test, so that planted mutants of it
(test_mlp_oracle.py) can be run against the same pins."""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _layers(rng, sizes):
    return [(rng.standard_normal((o, i)) / np.sqrt(i), rng.standard_normal(o) * 0.1) for i, o in zip(sizes, sizes[1:])]


def _close(a, b, tol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)
    assert err <= tol, f"{what}: {err:.3g}"


def pin_mlp_vs_autograd(mlp, orc=None):
    """A 3-layer stack and its SGD step against torch autograd of sum(dy * stack(x))."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((9, 5))
    for relu_last in (True, False):
        layers = _layers(rng, [5, 7, 6, 4])
        dy = rng.standard_normal((9, 4))
        outs = mlp.mlp_fwd(x, layers, relu_last)
        xt = torch.tensor(x, requires_grad=True)
        ps = [(torch.tensor(w, requires_grad=True), torch.tensor(b, requires_grad=True)) for w, b in layers]
        h = xt
        for i, (w, b) in enumerate(ps):
            h = F.linear(h, w, b)
            if i < len(ps) - 1 or relu_last:
                h = F.relu(h)
        _close(outs[-1], h.detach().numpy(), 1e-12, "stack output")
        (h * torch.tensor(dy)).sum().backward()
        dx, new = mlp.mlp_bwd_sgd(x, layers, outs, dy, relu_last, lr=0.3)
        _close(dx, xt.grad.numpy(), 1e-12, "dx")
        for (w, b), (wn, bn), (wt, bt) in zip(layers, new, ps):
            _close(wn, w - 0.3 * wt.grad.numpy(), 1e-12, "W after SGD")
            _close(bn, b - 0.3 * bt.grad.numpy(), 1e-12, "b after SGD")


def pin_head_vs_autograd(mlp, orc=None):
    """Logit, sigmoid and mean BCE against binary_cross_entropy_with_logits and its autograd."""
    rng = np.random.default_rng(2)
    h = rng.standard_normal((11, 6)) * 3
    w, b = rng.standard_normal(6), 0.4
    label = rng.integers(0, 2, size=11).astype(np.float64)
    z, p, loss = mlp.head_fwd(h, w, b, label)
    ht, wt, bt = (torch.tensor(a, requires_grad=True) for a in (h, w, np.float64(b)))
    zt = ht @ wt + bt
    lt = F.binary_cross_entropy_with_logits(zt, torch.tensor(label))
    _close(z, zt.detach().numpy(), 1e-12, "logit")
    _close(p, torch.sigmoid(zt).detach().numpy(), 1e-12, "probability")
    _close(loss, lt.item(), 1e-12, "loss")
    lt.backward()
    dh, dw, db = mlp.head_bwd(h, w, z, label)
    _close(dh, ht.grad.numpy(), 1e-12, "dh")
    _close(dw, wt.grad.numpy(), 1e-12, "dw")
    _close(db, bt.grad.numpy(), 1e-12, "db")


def pin_head_closed_forms(mlp, orc=None):
    """z = 0: p = 1/2 and the loss is ln 2 whatever the label; d loss/dz = (1/2 - y)/M; a large |z| of
    the right sign costs about exp(-|z|)."""
    h = np.zeros((4, 3))
    label = np.array([0.0, 1.0, 1.0, 0.0])
    z, p, loss = mlp.head_fwd(h, np.ones(3), 0.0, label)
    assert np.all(z == 0) and np.all(p == 0.5) and abs(loss - np.log(2.0)) < 1e-15
    dh, dw, db = mlp.head_bwd(h, np.ones(3), z, label)
    assert np.allclose(db, np.sum(0.5 - label) / 4) and np.allclose(dh[:, 0], (0.5 - label) / 4)
    _, _, loss_big = mlp.head_fwd(np.array([[40.0]]), np.array([1.0]), 0.0, np.array([1.0]))
    assert 0 < loss_big < 1e-17 and abs(loss_big - np.exp(-40.0)) < 1e-30


def pin_dlrm_step_vs_autograd(mlp, orc):
    """The whole training step against float64 autograd of the loss through the bottom MLP, embedding_bag
    on the tables, the interaction (bmm + triu), the top MLP and the BCE head: every MLP weight after SGD,
    and every table row after row-wise Adagrad (closed form on autograd's row gradient)."""
    rng = np.random.default_rng(3)
    B, F_in, D, T = 6, 5, 4, 3
    V = [7, 5, 9]
    tables = [rng.uniform(-0.5, 0.5, size=(v, D)).astype(np.float32) for v in V]
    L = rng.integers(1, 4, size=T * B)
    off = np.concatenate([[0], np.cumsum(L)])
    idx = np.concatenate([rng.integers(0, V[t], size=int(L[t * B:(t + 1) * B].sum())) for t in range(T)])
    dense_in = rng.standard_normal((B, F_in))
    label = rng.integers(0, 2, size=B).astype(np.float64)
    N = T + 1
    bottom = _layers(rng, [F_in, 8, D])
    top = _layers(rng, [D + N * (N - 1) // 2, 10, 6])
    head = (rng.standard_normal(6) * 0.5, 0.1)
    new_tabs = [t.copy() for t in tables]
    acc0 = [np.full(v, 0.1, np.float32) for v in V]
    acc = [a.copy() for a in acc0]
    res = mlp.dlrm_step(orc, bottom, top, head, new_tabs, V, idx, off, dense_in, label, 0.05, 0.02, 1e-8, acc)
    assert res["status"] == 0

    ps = lambda ls: [(torch.tensor(w, requires_grad=True), torch.tensor(b, requires_grad=True)) for w, b in ls]
    pb, pt = ps(bottom), ps(top)
    hw, hb = torch.tensor(head[0], requires_grad=True), torch.tensor(np.float64(head[1]), requires_grad=True)
    Ws = [torch.tensor(t.astype(np.float64), requires_grad=True) for t in tables]
    h = torch.tensor(dense_in)
    for w, b in pb:
        h = F.relu(F.linear(h, w, b))
    pools = [F.embedding_bag(torch.tensor(idx[off[t * B]:off[(t + 1) * B]], dtype=torch.int64), Ws[t],
                             torch.tensor(off[t * B:(t + 1) * B] - off[t * B], dtype=torch.int64), mode="sum")
             for t in range(T)]
    Vm = torch.cat([h[:, None, :], torch.stack(pools, 1)], 1)
    Z = torch.bmm(Vm, Vm.transpose(1, 2))
    iu = torch.triu_indices(N, N, 1)
    out = torch.cat([h, Z[:, iu[0], iu[1]]], 1)
    _close(res["out"], out.detach().numpy(), 1e-5, "interaction output (fp32 in the oracle)")
    g = out
    for w, b in pt:
        g = F.relu(F.linear(g, w, b))
    zt = g @ hw + hb
    loss = F.binary_cross_entropy_with_logits(zt, torch.tensor(label))
    _close(res["loss"], loss.item(), 1e-5, "loss")
    loss.backward()
    # the oracle rounds x and d(out) to float32 at the sparse boundary: relative 1e-5 covers it
    for (wn, bn), (w, b) in zip(res["bottom"] + res["top"], pb + pt):
        _close(wn, w.detach().numpy() - 0.05 * w.grad.numpy(), 1e-5, "MLP weight after SGD")
        _close(bn, b.detach().numpy() - 0.05 * b.grad.numpy(), 1e-5, "MLP bias after SGD")
    _close(res["head"][0], hw.detach().numpy() - 0.05 * hw.grad.numpy(), 1e-5, "head weight")
    for t in range(T):
        G = Ws[t].grad.numpy()
        for r in range(V[t]):
            if np.any(G[r] != 0) or r in set(idx[off[t * B]:off[(t + 1) * B]].tolist()):
                A = 0.1 + np.mean(G[r] ** 2)
                want = tables[t][r] - 0.02 * G[r] / (np.sqrt(A) + 1e-8)
                _close(new_tabs[t][r], want, 1e-4, f"row {t},{r} after Adagrad")


ALL_MLP_PINS = [pin_mlp_vs_autograd, pin_head_vs_autograd, pin_head_closed_forms, pin_dlrm_step_vs_autograd]
