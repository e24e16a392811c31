"""Plain float64 oracle of the dense parts of a DLRM training step around the
sparse path: the bottom MLP, the top MLP, the sigmoid output and its binary
cross-entropy loss, and plain SGD on their weights.

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg use this module.  It shares no code with the CUDA
library; the sparse part of a step comes from the C oracle (oracle.c).

Sources (web pages, cited by title and section):
  [robocikowo]  "DLRM" (robocikowo.com): "Forward pass" step (1), dense
                features through a bottom MLP of several FC layers with ReLU
                ending in a vector of width D; the bottom-MLP paragraph (2-4
                FC layers with ReLU); step (4) and the top-MLP paragraph: the
                concatenation goes through a top MLP of FC layers with ReLU and
                a sigmoid output (the click-through probability); training
                with SGD/Adagrad; the hardware paragraph (the MLPs are ordinary
                GEMMs).
  [glossary]    "Deep Learning Recommendation Model (DLRM)": dense features
                through a bottom MLP, the top MLP after the interaction.
Readings where the pages are silent:
  - every bottom layer is FC + ReLU (its output x >= 0); every top layer but
    the last is FC + ReLU, the last maps to one logit z, p = sigmoid(z);
  - the loss is the mean binary cross-entropy over the batch,
    -[y log p + (1 - y) log(1 - p)], written in its overflow-free form
    max(z, 0) - z y + log(1 + exp(-|z|));
  - the MLP weights take plain SGD, W -= lr dW, b -= lr db (the embedding rows
    keep their own rule);
  - an FC layer is y = x W^T + b with W of shape [out, in].
"""
from __future__ import annotations

import numpy as np


def fc_fwd(x, w, b, relu: bool):
    """One FC layer, [robocikowo] bottom/top-MLP paragraphs: z = x W^T + b, then ReLU if asked."""
    z = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T + np.asarray(b, np.float64)
    return np.maximum(z, 0.0) if relu else z


def fc_bwd(x, w, y, dy, relu: bool):
    """The layer's backward from the gradient dy of its output y: dz = dy * [y > 0] (ReLU) or dy;
    dx = dz W, dW = dz^T x, db = sum over the batch of dz.  Returns (dx, dW, db)."""
    x, w, dy = (np.asarray(a, np.float64) for a in (x, w, dy))
    dz = dy * (np.asarray(y) > 0) if relu else dy
    return dz @ w, dz.T @ x, dz.sum(axis=0)


def head_fwd(h, w, b, label):
    """The last top layer and the output ([robocikowo] top-MLP paragraph, sigmoid output):
    z = h w + b (w of shape [in]), p = sigmoid(z), loss = mean BCE(p, label).  Returns (z, p, loss)."""
    h, w, label = np.asarray(h, np.float64), np.asarray(w, np.float64), np.asarray(label, np.float64)
    z = h @ w + np.float64(b)
    p = 1.0 / (1.0 + np.exp(-z))
    loss = np.mean(np.maximum(z, 0.0) - z * label + np.log1p(np.exp(-np.abs(z))))
    return z, p, loss


def head_bwd(h, w, z, label):
    """d loss / d z = (sigmoid(z) - label) / M; dh = dz w^T, dw = h^T dz, db = sum dz."""
    h, w, z, label = (np.asarray(a, np.float64) for a in (h, w, z, label))
    dz = (1.0 / (1.0 + np.exp(-z)) - label) / z.shape[0]
    return np.outer(dz, w), h.T @ dz, dz.sum()


def mlp_fwd(x, layers, relu_last: bool):
    """A stack of FC layers [(W, b), ...], ReLU after each (after the last only if relu_last).
    Returns the list of every layer's output (float64)."""
    outs, h = [], x
    for i, (w, b) in enumerate(layers):
        h = fc_fwd(h, w, b, relu=(i < len(layers) - 1) or relu_last)
        outs.append(h)
    return outs


def mlp_bwd_sgd(x, layers, outs, dy, relu_last: bool, lr: float):
    """Backward through mlp_fwd's stack from the gradient dy of its last output, with SGD on every
    layer (each layer's dx computed with its weights before their update).  Returns (dx of the input,
    the updated layers as float64)."""
    new = []
    for i in range(len(layers) - 1, -1, -1):
        w, b = layers[i]
        xin = x if i == 0 else outs[i - 1]
        dx, dW, db = fc_bwd(xin, w, outs[i], dy, relu=(i < len(layers) - 1) or relu_last)
        new.append((np.asarray(w, np.float64) - lr * dW, np.asarray(b, np.float64) - lr * db))
        dy = dx
    return dy, new[::-1]


def dlrm_step(orc, bottom, top, head, tables, num_rows, indices, offsets, dense_in, label, lr_mlp, lr_emb, eps,
              accum, mode="sum"):
    """One DLRM training step on the oracles, in the order [robocikowo] "Forward pass" gives:
    (1) bottom MLP on the dense features -> x (width D); (2)-(4) the sparse forward on the C oracle,
    out = [x, interaction]; the top MLP and the sigmoid head; then the backward: head and top MLP (SGD),
    the sparse training step on the C oracle (row-wise Adagrad on the tables, grad of x), the bottom MLP
    (SGD).  The sparse part sees x and d(out) rounded to float32, as the device path carries them.
    tables and accum (lists of float32 arrays) are updated in place; returns a dict with x, out, z, p,
    loss, grad_out, grad_dense and the updated MLP weights (float64)."""
    bot_outs = mlp_fwd(dense_in, bottom, relu_last=True)
    x = bot_outs[-1].astype(np.float32)
    r = orc.sparse_fwd(tables, num_rows, indices, offsets, x, mode, with_pooled=True)
    top_outs = mlp_fwd(r["out"], top, relu_last=True)
    h = top_outs[-1]
    z, p, loss = head_fwd(h, head[0], head[1], label)
    dh, dw_head, db_head = head_bwd(h, head[0], z, label)
    new_head = (np.asarray(head[0], np.float64) - lr_mlp * dw_head, np.float64(head[1]) - lr_mlp * db_head)
    d_out, new_top = mlp_bwd_sgd(r["out"], top, top_outs, dh, relu_last=True, lr=lr_mlp)
    grad_out = d_out.astype(np.float32)
    grad_dense, st = orc.sparse_bwd_update(tables, num_rows, indices, offsets, x, r["pooled"], grad_out, "adagrad",
                                           lr_emb, eps, accum, mode)
    _, new_bottom = mlp_bwd_sgd(dense_in, bottom, bot_outs, grad_dense, relu_last=True, lr=lr_mlp)
    return {"x": x, "out": r["out"], "pooled": r["pooled"], "z": z, "p": p, "loss": loss, "grad_out": grad_out,
            "grad_dense": grad_dense, "bottom": new_bottom, "top": new_top, "head": new_head,
            "status": r["status"] | st}
