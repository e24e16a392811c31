"""Pins of the CPU oracle to facts outside itself.

Each pin takes a loaded oracle (oracle.Oracle) and raises AssertionError when
the oracle disagrees with something the pages or plain mathematics fix: a
closed form, an invariant, a special case that reduces to a library routine
(float64 torch.nn.functional.embedding_bag, torch.bmm + torch.triu_indices,
torch autograd), central differences, or a worked fixture.  The same pins run
against deliberately altered copies of the oracle (test_oracle_mutants.py) to
show that each plausible mistake is caught.
"""
from __future__ import annotations

import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# small input builders (random but seeded)
# ---------------------------------------------------------------------------
def rand_problem(seed, B=6, T=3, D=8, V=(5, 9, 7), Lmax=4, Lmin=0, dtype="f32"):
    rng = np.random.default_rng(seed)
    V = list(V)[:T] + [V[-1]] * max(0, T - len(V))
    tables = [rng.uniform(-1, 1, size=(v, D)).astype(np.float32) for v in V]
    if dtype == "bf16":
        import gen
        tables = [gen.f32_to_bf16_bits(t) for t in tables]
    L = rng.integers(Lmin, Lmax + 1, size=T * B)
    off = np.zeros(T * B + 1, dtype=np.int64)
    np.cumsum(L, out=off[1:])
    idx = np.concatenate([rng.integers(0, V[t], size=int(L[t * B:(t + 1) * B].sum())) for t in range(T)])
    dense = rng.uniform(-1, 1, size=(B, D)).astype(np.float32)
    return tables, V, idx.astype(np.int64), off, dense


def widen(table, dtype):
    if dtype == "bf16":
        import gen
        return gen.bf16_bits_to_f32(table).astype(np.float64)
    return np.asarray(table, dtype=np.float64)


def torch_pool(tables, idx, off, B, mode, dtype="f32"):
    """float64 pooling with the library routine, table by table -> [B, T, D]."""
    T = len(tables)
    outs = []
    for t in range(T):
        lo = off[t * B]
        seg = torch.from_numpy(np.asarray(idx[off[t * B]:off[(t + 1) * B]], dtype=np.int64))
        offs = torch.from_numpy(np.asarray(off[t * B:(t + 1) * B] - lo, dtype=np.int64))
        w = torch.from_numpy(widen(tables[t], dtype))
        outs.append(F.embedding_bag(seg, w, offs, mode=mode))
    return torch.stack(outs, dim=1)


def torch_interact(dense64, pooled64):
    """float64 [x, triu(V V^T)] with the library Gram and triangle indices."""
    V = torch.cat([dense64[:, None, :], pooled64], dim=1)
    Z = torch.bmm(V, V.transpose(1, 2))
    N = V.shape[1]
    iu = torch.triu_indices(N, N, offset=1)
    return torch.cat([dense64, Z[:, iu[0], iu[1]]], dim=1)


def close(a, b, scale, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b) / np.maximum(np.maximum(np.abs(b), scale), 1e-30)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max relative error {worst:.3g} > {tol:g}"


# ---------------------------------------------------------------------------
# pins: pooling (forward pass step (2), multi-valued features)
# ---------------------------------------------------------------------------
def pin_output_length(orc):
    """Width D + N(N-1)/2 for the shapes in tests/golden/output_lengths.txt."""
    rows = [list(map(int, l.split())) for l in open(os.path.join(GOLDEN, "output_lengths.txt"))
            if l.strip() and not l.startswith("#")]
    for T, D, N, tri, width in rows:
        assert N == T + 1 and width == D + tri
        pooled = np.zeros((1, T, D), dtype=np.float32)
        out = orc.interact(np.zeros((1, D), np.float32), pooled)
        assert out.shape == (1, width), (T, D, out.shape, width)


def pin_onehot_bit_exact(orc):
    """A bag of one row pools to that row, bit for bit (incl. -0.0, subnormals, extremes)."""
    rng = np.random.default_rng(1)
    D, V, B = 16, 12, 24
    t0 = rng.standard_normal((V, D)).astype(np.float32)
    t0[0, :4] = [-0.0, 1e-45, -3.4e38, 1.17549435e-38]
    t1 = rng.uniform(-0.05, 0.05, size=(V, D)).astype(np.float32)
    idx = rng.integers(0, V, size=2 * B)
    off = np.arange(2 * B + 1)
    idx[0] = 0
    for mode in ("sum", "mean"):
        pooled, st = orc.embbag([t0, t1], [V, V], idx, off, B, D, mode)
        assert st == 0
        exp = np.stack([t0[idx[:B]], t1[idx[B:]]], axis=1)
        assert np.array_equal(pooled.view(np.uint32), exp.view(np.uint32)), mode


def pin_k_copies(orc):
    """k copies of row r: sum = k*row (exact in double, rounded once); mean = row."""
    rng = np.random.default_rng(2)
    D, V = 8, 6
    tab = rng.standard_normal((V, D)).astype(np.float32)
    ks = [1, 2, 3, 7, 64]
    rows = [0, 3, 5, 1, 2]
    idx = np.concatenate([[r] * k for r, k in zip(rows, ks)])
    off = np.concatenate([[0], np.cumsum(ks)])
    B = len(ks)
    s, st = orc.embbag([tab], [V], idx, off, B, D, "sum")
    m, _ = orc.embbag([tab], [V], idx, off, B, D, "mean")
    assert st == 0
    for b, (r, k) in enumerate(zip(rows, ks)):
        assert np.array_equal(s[b, 0], (tab[r].astype(np.float64) * k).astype(np.float32)), (r, k)
        assert np.array_equal(m[b, 0], tab[r]), (r, k)


def pin_identity_tables(orc):
    """E_t = I (V_t = D): one-hot bags give unit vectors; the interaction then
    gives [r_i == r_j] between embeddings and x[r_t] against the dense vector."""
    rng = np.random.default_rng(3)
    D, T, B = 8, 4, 16
    tabs = [np.eye(D, dtype=np.float32) for _ in range(T)]
    r = rng.integers(0, D, size=(T, B))
    idx = r.reshape(-1)
    off = np.arange(T * B + 1)
    x = rng.standard_normal((B, D)).astype(np.float32)
    res = orc.sparse_fwd(tabs, [D] * T, idx, off, x, with_pooled=True)
    assert res["status"] == 0
    P = res["pooled"]
    for b in range(B):
        for t in range(T):
            assert np.array_equal(P[b, t], np.eye(D, dtype=np.float32)[r[t, b]])
    N = T + 1
    iu = torch.triu_indices(N, N, offset=1).numpy()
    for b in range(B):
        tri = res["out"][b, D:]
        assert np.array_equal(res["out"][b, :D].view(np.uint32), x[b].view(np.uint32))
        for k, (i, j) in enumerate(zip(iu[0], iu[1])):
            if i == 0:
                want = x[b, r[j - 1, b]]
            else:
                want = np.float32(r[i - 1, b] == r[j - 1, b])
            assert tri[k] == want, (b, i, j, tri[k], want)


def pin_pool_vs_embedding_bag(orc):
    """Random bags (lengths 0..6, duplicates allowed), fp32 and bf16, sum and mean,
    against float64 torch embedding_bag."""
    for seed, dtype in [(10, "f32"), (11, "bf16"), (12, "f32")]:
        tables, V, idx, off, dense = rand_problem(seed, B=9, T=3, D=12, Lmax=6, dtype=dtype)
        for mode in ("sum", "mean"):
            pooled, pabs, st = orc.embbag(tables, V, idx, off, 9, 12, mode, dtype, with_abs=True)
            assert st == 0
            ref = torch_pool(tables, idx, off, 9, mode, dtype).numpy()
            close(pooled, ref, pabs, 1e-7, f"pool {dtype} {mode}")


def pin_empty_and_bad_inputs(orc):
    """Empty bags pool to zero; an out-of-range index contributes zero but counts
    in the mean's L and raises the index flag; a reversed bag range is empty and
    raises the offsets flag."""
    D, V, B = 4, 5, 3
    tab = np.arange(V * D, dtype=np.float32).reshape(V, D) + 1
    # bags: [], [1, 7(oob), 2], [4]
    idx = np.array([1, 7, 2, 4])
    off = np.array([0, 0, 3, 4])
    s, st = orc.embbag([tab], [V], idx, off, B, D, "sum")
    m, _ = orc.embbag([tab], [V], idx, off, B, D, "mean")
    assert st == 2, st
    assert np.array_equal(s[0, 0], np.zeros(D, np.float32))
    assert np.array_equal(s[1, 0], tab[1] + tab[2])
    assert np.array_equal(m[1, 0], ((tab[1].astype(np.float64) + tab[2]) / 3).astype(np.float32))
    assert np.array_equal(s[2, 0], tab[4])
    idx2 = np.array([-1, 0])
    s2, st2 = orc.embbag([tab], [V], idx2, np.array([0, 2, 2, 2]), B, D, "sum")
    assert st2 == 2 and np.array_equal(s2[0, 0], tab[0])
    off_bad = np.array([0, 3, 1, 4])  # bag 1 reversed
    s3, st3 = orc.embbag([tab], [V], idx, off_bad, B, D, "sum")
    assert st3 & 4
    assert np.array_equal(s3[1, 0], np.zeros(D, np.float32))
    assert np.array_equal(s3[2, 0], tab[2] + tab[4])  # bag 2 = [7 (out of range), 2, 4]
    off_end = np.array([0, 1, 2, 3])  # last offset != nnz
    _, st4 = orc.embbag([tab], [V], idx, off_end, B, D, "sum")
    assert st4 & 4


# ---------------------------------------------------------------------------
# pins: interaction (forward pass steps (3)-(4))
# ---------------------------------------------------------------------------
def pin_interact_vs_bmm(orc):
    """Random V against float64 torch.bmm + triu_indices(N, N, 1)."""
    for seed, (B, T, D) in [(20, (5, 3, 8)), (21, (3, 7, 16)), (22, (2, 26, 128)), (23, (2, 1, 4))]:
        rng = np.random.default_rng(seed)
        P = rng.standard_normal((B, T, D)).astype(np.float32)
        x = rng.standard_normal((B, D)).astype(np.float32)
        out, oabs = orc.interact(x, P, with_abs=True)
        ref = torch_interact(torch.from_numpy(x.astype(np.float64)), torch.from_numpy(P.astype(np.float64)))
        close(out, ref.numpy(), oabs, 1e-7, f"interact {B, T, D}")
        assert np.array_equal(out[:, :D].view(np.uint32), x.view(np.uint32))


def pin_n2_closed_form(orc):
    """N = 2 (one table): one triangle value, x . P_0."""
    rng = np.random.default_rng(30)
    B, D = 7, 10
    P = rng.standard_normal((B, 1, D)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32)
    out = orc.interact(x, P)
    assert out.shape == (B, D + 1)
    for b in range(B):
        want = np.float32(np.dot(x[b].astype(np.float64), P[b, 0].astype(np.float64)))
        assert out[b, D] == want, (out[b, D], want)


def pin_orthogonal_zero(orc):
    """Mutually orthogonal vectors give an all-zero triangle (so no diagonal
    |v|^2 term and no cross term leaks in)."""
    D = 8
    H = np.array([[1]], dtype=np.float32)
    while H.shape[0] < D:
        H = np.block([[H, H], [H, -H]])
    x = H[0:1].copy()
    P = H[1:5][None, :, :]
    out = orc.interact(x, P)
    assert np.array_equal(out[0, D:], np.zeros(10, np.float32)), out[0, D:]


def pin_permutation_symmetry(orc):
    """Reordering the tables permutes the triangle as the symmetric Gram says:
    z'(i, j) = z(pi(i), pi(j)) with pi fixing the dense vector 0."""
    rng = np.random.default_rng(31)
    B, T, D = 4, 5, 6
    P = rng.standard_normal((B, T, D)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32)
    perm = np.array([3, 0, 4, 1, 2])
    out = orc.interact(x, P)
    out2 = orc.interact(x, P[:, perm])
    N = T + 1
    pi = np.concatenate([[0], perm + 1])
    iu = torch.triu_indices(N, N, offset=1).numpy()
    pos = {(int(i), int(j)): k for k, (i, j) in enumerate(zip(iu[0], iu[1]))}
    for k, (i, j) in enumerate(zip(iu[0], iu[1])):
        a, b = sorted((int(pi[i]), int(pi[j])))
        assert np.array_equal(out2[:, D + k], out[:, D + pos[(a, b)]]), (i, j)


def pin_cauchy_schwarz(orc):
    """|z(i,j)| <= |v_i| |v_j|."""
    rng = np.random.default_rng(32)
    B, T, D = 6, 4, 9
    P = rng.standard_normal((B, T, D)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32)
    out = orc.interact(x, P)
    V = np.concatenate([x[:, None], P], axis=1).astype(np.float64)
    nrm = np.linalg.norm(V, axis=2)
    iu = torch.triu_indices(T + 1, T + 1, offset=1).numpy()
    bound = nrm[:, iu[0]] * nrm[:, iu[1]]
    assert np.all(np.abs(out[:, D:]) <= bound * (1 + 1e-6))


# ---------------------------------------------------------------------------
# pins: backward and Adagrad (training with SGD/Adagrad)
# ---------------------------------------------------------------------------
def pin_bwd_vs_autograd(orc):
    """dx, dP against float64 autograd of <g, out(x, P)>."""
    for seed, (B, T, D) in [(40, (4, 3, 8)), (41, (3, 26, 16))]:
        rng = np.random.default_rng(seed)
        P = rng.standard_normal((B, T, D)).astype(np.float32)
        x = rng.standard_normal((B, D)).astype(np.float32)
        N = T + 1
        g = rng.standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
        gd, gp = orc.interact_bwd(x, P, g)
        xt = torch.from_numpy(x.astype(np.float64)).requires_grad_()
        Pt = torch.from_numpy(P.astype(np.float64)).requires_grad_()
        out = torch_interact(xt, Pt)
        (out * torch.from_numpy(g.astype(np.float64))).sum().backward()
        scale_x = np.abs(g[:, :D]) + np.abs(np.einsum("bk,bkd->bd", np.abs(g[:, D:D + T]), np.abs(P)))
        close(gd, xt.grad.numpy(), scale_x, 1e-6, "dx")
        scale_p = np.abs(gp).max()
        close(gp, Pt.grad.numpy(), scale_p, 1e-6, "dP")


def pin_bwd_finite_differences(orc):
    """<g, out> is quadratic in V, so central differences of the oracle's own
    forward are exact up to rounding."""
    rng = np.random.default_rng(42)
    B, T, D = 2, 3, 4
    P = rng.standard_normal((B, T, D)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32)
    N = T + 1
    g = rng.standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
    gd, gp = orc.interact_bwd(x, P, g)
    h = 0.25  # exactly representable; perturbed values stay exact in fp32

    def f(xx, PP):
        return float((orc.interact(xx, PP).astype(np.float64) * g).sum())

    for b in range(B):
        for d in range(D):
            xp, xm = x.copy(), x.copy()
            xp[b, d] += h
            xm[b, d] -= h
            fd = (f(xp, P) - f(xm, P)) / (2 * h)
            assert abs(fd - gd[b, d]) <= 1e-4 * (1 + abs(fd)), ("dx", b, d, fd, gd[b, d])
        for t in range(T):
            for d in range(D):
                Pp, Pm = P.copy(), P.copy()
                Pp[b, t, d] += h
                Pm[b, t, d] -= h
                fd = (f(x, Pp) - f(x, Pm)) / (2 * h)
                assert abs(fd - gp[b, t, d]) <= 1e-4 * (1 + abs(fd)), ("dP", b, t, d, fd, gp[b, t, d])


def pin_bwd_n2_closed_form(orc):
    """N = 2: dv0 = g_x + g*v1, dv1 = g*v0."""
    rng = np.random.default_rng(43)
    B, D = 3, 5
    P = rng.standard_normal((B, 1, D)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32)
    g = rng.standard_normal((B, D + 1)).astype(np.float32)
    gd, gp = orc.interact_bwd(x, P, g)
    for b in range(B):
        want_x = (g[b, :D].astype(np.float64) + g[b, D].astype(np.float64) * P[b, 0]).astype(np.float32)
        want_p = (np.float64(g[b, D]) * x[b].astype(np.float64)).astype(np.float32)
        assert np.array_equal(gd[b], want_x)
        assert np.array_equal(gp[b, 0], want_p)


def _adagrad_closed(w, A, g, lr, eps):
    """Row-wise Adagrad on one row, float64: A' = A + mean(g^2); w' = w - lr g/(sqrt(A')+eps)."""
    A2 = np.float64(A) + np.mean(g * g)
    return (w.astype(np.float64) - lr * g / (np.sqrt(A2) + eps)).astype(np.float32), np.float32(A2)


def pin_adagrad_single_row(orc):
    """One row touched by one lookup: closed form with g = dP of that bag."""
    rng = np.random.default_rng(50)
    B, T, D, V = 1, 2, 6, 4
    tabs = [rng.uniform(-0.05, 0.05, size=(V, D)).astype(np.float32) for _ in range(T)]
    idx = np.array([2, 1])
    off = np.array([0, 1, 2])
    x = rng.standard_normal((B, D)).astype(np.float32)
    P = np.stack([tabs[0][[2]], tabs[1][[1]]], axis=1)
    N = T + 1
    g = rng.standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
    _, _, dV = orc.interact_bwd(x, P, g, with_dV=True)
    acc = [np.full(V, 0.1, np.float32) for _ in range(T)]
    new = [t.copy() for t in tabs]
    # a large eps so that where it sits (outside the square root) matters
    orc.sparse_bwd_adagrad(new, [V] * T, idx, off, x, P, g, acc, 0.5, 0.3)
    # independent dP: autograd
    xt = torch.from_numpy(x.astype(np.float64))
    Pt = torch.from_numpy(P.astype(np.float64)).requires_grad_()
    (torch_interact(xt, Pt) * torch.from_numpy(g.astype(np.float64))).sum().backward()
    for t, r in [(0, 2), (1, 1)]:
        gr = Pt.grad.numpy()[0, t]
        w2, A2 = _adagrad_closed(tabs[t][r], 0.1, gr, 0.5, 0.3)
        close(new[t][r], w2, np.abs(tabs[t][r]), 1e-6, "adagrad row")
        close(acc[t][r], A2, 0.1, 1e-6, "adagrad accum")
        for rr in range(V):
            if rr != r:
                assert np.array_equal(new[t][rr], tabs[t][rr]) and acc[t][rr] == np.float32(0.1)


def pin_row_grads_vs_autograd(orc):
    """Per-row gradient of <g, out> with respect to the whole tables (float64
    autograd through embedding_bag, which sums over every lookup of a row), then
    one row-wise Adagrad step, against the oracle's updated tables."""
    for seed, mode in [(60, "sum"), (61, "mean")]:
        tables, V, idx, off, dense = rand_problem(seed, B=8, T=3, D=6, V=(4, 3, 6), Lmax=5)
        B, T, D = 8, 3, 6
        pooled, _ = orc.embbag(tables, V, idx, off, B, D, mode)
        N = T + 1
        rng = np.random.default_rng(seed + 100)
        g = rng.standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
        acc0 = [rng.uniform(0.05, 0.2, size=v).astype(np.float32) for v in V]
        new = [t.copy() for t in tables]
        acc = [a.copy() for a in acc0]
        lr, eps = 0.05, 1e-8
        orc.sparse_bwd_adagrad(new, V, idx, off, dense, pooled, g, acc, lr, eps, mode)
        Ws = [torch.from_numpy(t.astype(np.float64)).requires_grad_() for t in tables]
        pools = []
        for t in range(T):
            lo = off[t * B]
            seg = torch.from_numpy(idx[off[t * B]:off[(t + 1) * B]].astype(np.int64))
            offs = torch.from_numpy((off[t * B:(t + 1) * B] - lo).astype(np.int64))
            pools.append(F.embedding_bag(seg, Ws[t], offs, mode=mode))
        Pt = torch.stack(pools, 1)
        # the oracle's backward sees the pooled vectors rounded to fp32
        Pt_f = Pt + (torch.from_numpy(pooled.astype(np.float64)) - Pt).detach()
        out = torch_interact(torch.from_numpy(dense.astype(np.float64)), Pt_f)
        (out * torch.from_numpy(g.astype(np.float64))).sum().backward()
        for t in range(T):
            G = Ws[t].grad.numpy()
            touched = set(idx[off[t * B]:off[(t + 1) * B]].tolist())
            for r in range(V[t]):
                if r in touched:
                    w2, A2 = _adagrad_closed(tables[t][r], acc0[t][r], G[r], lr, eps)
                    close(new[t][r], w2, np.abs(tables[t][r]) + 1e-3, 1e-6, f"row {t},{r} {mode}")
                    close(acc[t][r], A2, acc0[t][r], 1e-6, f"acc {t},{r} {mode}")
                else:
                    assert np.array_equal(new[t][r], tables[t][r]) and acc[t][r] == acc0[t][r]


def pin_duplicates_one_update(orc):
    """Two lookups of the same row (same bag and across samples) give ONE update
    with the summed gradient, not two sequential updates."""
    rng = np.random.default_rng(70)
    B, T, D, V = 2, 1, 4, 3
    tab = rng.uniform(-0.05, 0.05, size=(V, D)).astype(np.float32)
    idx = np.array([1, 1, 1])  # sample 0: [1, 1], sample 1: [1]
    off = np.array([0, 2, 3])
    pooled, _ = orc.embbag([tab], [V], idx, off, B, D, "sum")
    x = rng.standard_normal((B, D)).astype(np.float32)
    g = rng.standard_normal((B, D + 1)).astype(np.float32)
    acc = [np.full(V, 0.1, np.float32)]
    new = [tab.copy()]
    orc.sparse_bwd_adagrad(new, [V], idx, off, x, pooled, g, acc, 0.01, 1e-8)
    # N = 2: dP_b = g_b * x_b; row 1 gets 2*dP_0 + dP_1
    grow = 2 * g[0, D] * x[0].astype(np.float64) + g[1, D] * x[1].astype(np.float64)
    w2, A2 = _adagrad_closed(tab[1], 0.1, grow, 0.01, 1e-8)
    close(new[0][1], w2, np.abs(tab[1]), 1e-6, "dup row")
    close(acc[0][1], A2, 0.1, 1e-6, "dup acc")


def _table_grads(tables, idx, off, B, mode, grad_pooled):
    """float64 autograd: d<grad_pooled, pooled(W)>/dW per table (sums over every lookup of a row)."""
    T = len(tables)
    Ws = [torch.from_numpy(t.astype(np.float64)).requires_grad_() for t in tables]
    pools = []
    for t in range(T):
        lo = off[t * B]
        seg = torch.from_numpy(np.asarray(idx[off[t * B]:off[(t + 1) * B]], dtype=np.int64))
        offs = torch.from_numpy(np.asarray(off[t * B:(t + 1) * B] - lo, dtype=np.int64))
        pools.append(F.embedding_bag(seg, Ws[t], offs, mode=mode))
    (torch.stack(pools, 1) * torch.from_numpy(np.asarray(grad_pooled, np.float64))).sum().backward()
    return [w.grad.numpy() for w in Ws]


def pin_sgd_vs_autograd(orc):
    """Plain SGD on the embedding rows, w' = w - lr * dL/dw, with dL/dw from float64 autograd of
    <g, out> through embedding_bag and the interaction; untouched rows unchanged."""
    for seed, mode in [(80, "sum"), (81, "mean")]:
        tables, V, idx, off, dense = rand_problem(seed, B=7, T=3, D=6, V=(4, 3, 6), Lmax=5)
        B, T, D = 7, 3, 6
        pooled, _ = orc.embbag(tables, V, idx, off, B, D, mode)
        N = T + 1
        g = np.random.default_rng(seed + 1).standard_normal((B, D + N * (N - 1) // 2)).astype(np.float32)
        new = [t.copy() for t in tables]
        lr = 0.25
        gd, st = orc.sparse_bwd_update(new, V, idx, off, dense, pooled, g, "sgd", lr, mode=mode)
        assert st == 0
        Pt = torch.from_numpy(pooled.astype(np.float64)).requires_grad_()
        (torch_interact(torch.from_numpy(dense.astype(np.float64)), Pt) * torch.from_numpy(g.astype(np.float64))
         ).sum().backward()
        G = _table_grads(tables, idx, off, B, mode, Pt.grad.numpy())
        for t in range(T):
            want = (tables[t].astype(np.float64) - lr * G[t]).astype(np.float32)
            close(new[t], want, np.abs(tables[t]) + 1e-3, 1e-6, f"sgd table {t} {mode}")
            touched = set(idx[off[t * B]:off[(t + 1) * B]].tolist())
            for r in range(V[t]):
                if r not in touched:
                    assert np.array_equal(new[t][r], tables[t][r])


def pin_embbag_bwd_vs_autograd(orc):
    """The row update from a given gradient of the pooled vectors: per-row gradient from float64
    autograd through embedding_bag, then the Adagrad and the SGD closed forms."""
    for seed, mode in [(82, "sum"), (83, "mean")]:
        tables, V, idx, off, _ = rand_problem(seed, B=9, T=3, D=5, V=(6, 2, 5), Lmax=4)
        B, T, D = 9, 3, 5
        rng = np.random.default_rng(seed + 7)
        gp = rng.standard_normal((B, T, D)).astype(np.float32)
        G = _table_grads(tables, idx, off, B, mode, gp)
        acc0 = [rng.uniform(0.05, 0.2, size=v).astype(np.float32) for v in V]
        new_a, acc = [t.copy() for t in tables], [a.copy() for a in acc0]
        assert orc.embbag_bwd_update(new_a, V, idx, off, gp, "adagrad", 0.1, 0.2, acc, mode) == 0
        new_s = [t.copy() for t in tables]
        assert orc.embbag_bwd_update(new_s, V, idx, off, gp, "sgd", 0.1, mode=mode) == 0
        for t in range(T):
            touched = set(idx[off[t * B]:off[(t + 1) * B]].tolist())
            for r in range(V[t]):
                if r in touched:
                    w2, A2 = _adagrad_closed(tables[t][r], acc0[t][r], G[t][r], 0.1, 0.2)
                    close(new_a[t][r], w2, np.abs(tables[t][r]) + 1e-3, 1e-6, f"adagrad row {t},{r}")
                    close(acc[t][r], A2, acc0[t][r], 1e-6, f"adagrad acc {t},{r}")
                    close(new_s[t][r], (tables[t][r] - 0.1 * G[t][r]).astype(np.float32),
                          np.abs(tables[t][r]) + 1e-3, 1e-6, f"sgd row {t},{r}")
                else:
                    assert np.array_equal(new_a[t][r], tables[t][r]) and acc[t][r] == acc0[t][r]
                    assert np.array_equal(new_s[t][r], tables[t][r])


def pin_hash_brute_force(orc):
    """rows = raw ID mod V_t with Python's unbounded integers, the ID as an unsigned 64-bit value (IDs
    at and above 2^63 included), each position hashed with the row count of the table holding it."""
    rng = np.random.default_rng(90)
    V = [1, 7, 1 << 20, 4_294_967_311, (1 << 62) + 3]
    B = 5
    L = rng.integers(0, 6, size=len(V) * B)
    off = np.zeros(len(V) * B + 1, np.int64)
    np.cumsum(L, out=off[1:])
    raw = rng.integers(0, 1 << 63, size=int(off[-1]), dtype=np.uint64) * np.uint64(2) + \
        rng.integers(0, 2, size=int(off[-1]), dtype=np.uint64)
    raw[:3] = [0, (1 << 64) - 1, 1 << 63]
    rows, st = orc.hash_indices(V, raw, off, B)
    assert st == 0
    for t in range(len(V)):
        for p in range(off[t * B], off[(t + 1) * B]):
            assert rows[p] == int(raw[p]) % V[t], (t, p, int(raw[p]), rows[p])
    assert all(0 <= rows[p] for p in range(rows.size))


ALL_PINS = [
    pin_output_length, pin_onehot_bit_exact, pin_k_copies, pin_identity_tables,
    pin_pool_vs_embedding_bag, pin_empty_and_bad_inputs, pin_interact_vs_bmm,
    pin_n2_closed_form, pin_orthogonal_zero, pin_permutation_symmetry, pin_cauchy_schwarz,
    pin_bwd_vs_autograd, pin_bwd_finite_differences, pin_bwd_n2_closed_form,
    pin_adagrad_single_row, pin_row_grads_vs_autograd, pin_duplicates_one_update,
    pin_sgd_vs_autograd, pin_embbag_bwd_vs_autograd, pin_hash_brute_force,
]
