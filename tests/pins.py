"""Checks that pin the oracle to things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle module(s) it is given
disagree with a value fixed independently of the oracle's own formulas: a closed
form, a brute-force enumeration, central finite differences of the scalar loss, or
torch's autograd. They take the oracle modules as arguments so that
``test_oracle_mutations.py`` can run them against copies with a planted mistake.
"""
from __future__ import annotations

import numpy as np

import oracle.ffn as _ffn
import oracle.formats as _formats
import oracle.sparse as _sparse


def tiny_problem(T=4, d=8, I=16, gated=True, seed=0, min_gap=2e-3):
    """Small float64 problem whose gate pre-activations stay at least ``min_gap`` away
    from the ReLU kink (finite differences are then well defined)."""
    for s in range(1000):
        rng = np.random.default_rng([seed, s, 77])
        x = rng.standard_normal((T, d))
        x[:, 0] = 1.0
        Wg = rng.standard_normal((I, d)) / np.sqrt(d)
        Wg[:, 0] -= 0.4                      # about a third of neurons active
        Wu = rng.standard_normal((I, d)) / np.sqrt(d) if gated else None
        Wd = rng.standard_normal((I, d)) / np.sqrt(I)
        dy = rng.standard_normal((T, d))
        g = x @ Wg.T
        if np.abs(g).min() > min_gap and (g > 0).any():
            return x, Wg, Wu, Wd, dy
    raise RuntimeError("no kink-free tiny problem found")


# ---------------------------------------------------------------- forward pins

def pin_forward_permutation(ffn=_ffn, gated=True):
    """Closed form: Wg rows are unit vectors e_{p(j)}, Wu rows are e_0 (so u == 1
    because x[:, 0] == 1), Wd rows are unit vectors e_{q(j)}. Then
    y[t, q(j)] = max(x[t, p(j)], 0) for every j, and 0 in columns no q(j) hits."""
    rng = np.random.default_rng(5)
    T, d, I = 6, 10, 7
    x = rng.standard_normal((T, d))
    x[:, 0] = 1.0
    p = rng.choice(np.arange(1, d), I, replace=False)
    q = rng.choice(np.arange(d), I, replace=False)
    Wg = np.zeros((I, d)); Wg[np.arange(I), p] = 1.0
    Wu = np.zeros((I, d)); Wu[:, 0] = 1.0
    Wd = np.zeros((I, d)); Wd[np.arange(I), q] = 1.0
    y = ffn.forward(x, Wg, Wu if gated else None, Wd)["y"]
    expected = np.zeros((T, d))
    for j in range(I):
        for t in range(T):
            expected[t, q[j]] = x[t, p[j]] if x[t, p[j]] > 0 else 0.0
    np.testing.assert_allclose(y, expected, rtol=0, atol=1e-15)


def pin_forward_scaled_up(ffn=_ffn):
    """Closed form: Wu[j] = s_j * e_0 gives u[:, j] == s_j, so the gated y equals the
    non-gated y computed with Wd rows scaled by s_j."""
    x, Wg, Wu, Wd, _ = tiny_problem(T=5, d=6, I=9, seed=3)
    s = np.linspace(-2.0, 3.0, Wg.shape[0])
    Wu = np.zeros_like(Wg); Wu[:, 0] = s
    yg = ffn.forward(x, Wg, Wu, Wd)["y"]
    yn = ffn.forward(x, Wg, None, Wd * s[:, None])["y"]
    np.testing.assert_allclose(yg, yn, rtol=1e-13, atol=1e-14)


def pin_forward_brute_force(ffn=_ffn, gated=True):
    """Plain loops over every (t, j, c) on a tiny problem."""
    x, Wg, Wu, Wd, _ = tiny_problem(T=3, d=5, I=6, gated=gated, seed=9)
    T, d = x.shape
    I = Wg.shape[0]
    y = np.zeros((T, d))
    for t in range(T):
        for j in range(I):
            g = sum(x[t, c] * Wg[j, c] for c in range(d))
            if g <= 0:
                continue
            h = g * (sum(x[t, c] * Wu[j, c] for c in range(d)) if gated else 1.0)
            for c in range(d):
                y[t, c] += h * Wd[j, c]
    np.testing.assert_allclose(ffn.forward(x, Wg, Wu, Wd)["y"], y, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- backward pins

def _fd_grad(f, arr, eps=1e-6):
    grad = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + eps
        fp = f()
        arr[i] = old - eps
        fm = f()
        arr[i] = old
        grad[i] = (fp - fm) / (2 * eps)
    return grad


def pin_backward_finite_differences(ffn=_ffn, gated=True, l1=0.3):
    """Central differences of L = sum(dy*y) + l1*sum(a) against ``backward``."""
    x, Wg, Wu, Wd, dy = tiny_problem(gated=gated)
    b = ffn.backward(x, Wg, Wu, Wd, dy, l1)
    loss = lambda: ffn.loss(x, Wg, Wu, Wd, dy, l1)  # noqa: E731
    names = [("dx", x), ("dWg", Wg), ("dWd", Wd)] + ([("dWu", Wu)] if gated else [])
    for name, arr in names:
        fd = _fd_grad(loss, arr)
        np.testing.assert_allclose(b[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def pin_backward_l1_on_h(ffn=_ffn, gated=True, l1=0.3):
    """The reference-only reading with the penalty on |h|: central differences of
    its loss, and torch autograd of the same loss, against ``backward``."""
    import torch
    x, Wg, Wu, Wd, dy = tiny_problem(gated=gated)
    b = ffn.backward(x, Wg, Wu, Wd, dy, l1, penalise="h")
    loss = lambda: ffn.loss(x, Wg, Wu, Wd, dy, l1, penalise="h")  # noqa: E731
    names = [("dx", x), ("dWg", Wg), ("dWd", Wd)] + ([("dWu", Wu)] if gated else [])
    for name, arr in names:
        fd = _fd_grad(loss, arr)
        np.testing.assert_allclose(b[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)
    tt = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
          for k, v in dict(x=x, Wg=Wg, Wd=Wd, **({"Wu": Wu} if gated else {})).items()}
    a = torch.relu(tt["x"] @ tt["Wg"].T)
    h = a * (tt["x"] @ tt["Wu"].T) if gated else a
    L = (torch.tensor(dy) * (h @ tt["Wd"])).sum() + l1 * h.abs().sum()
    L.backward()
    leaf = {"dx": "x", "dWg": "Wg", "dWd": "Wd", "dWu": "Wu"}
    for name, _ in names:
        np.testing.assert_allclose(b[name], tt[leaf[name]].grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)
    if gated:
        # the two readings differ on this problem (u takes both signs)
        assert not np.allclose(b["dWg"], ffn.backward(x, Wg, Wu, Wd, dy, l1)["dWg"])


def pin_backward_l1_closed_form(ffn=_ffn, gated=True):
    """dy = 0, l1 = 1: the gradient is that of sum(a) alone, so dWg[j] = sum of x_t
    over tokens with g_tj > 0, dx_t = sum of Wg[j] over its active neurons, and
    dWu = dWd = 0."""
    x, Wg, Wu, Wd, dy = tiny_problem(T=5, d=7, I=11, gated=gated, seed=4)
    dy = np.zeros_like(dy)
    b = ffn.backward(x, Wg, Wu, Wd, dy, 1.0)
    T, I = x.shape[0], Wg.shape[0]
    act = [[float(x[t] @ Wg[j]) > 0 for j in range(I)] for t in range(T)]
    dWg = np.array([sum((x[t] for t in range(T) if act[t][j]), np.zeros(x.shape[1])) for j in range(I)])
    dx = np.array([sum((Wg[j] for j in range(I) if act[t][j]), np.zeros(x.shape[1])) for t in range(T)])
    np.testing.assert_allclose(b["dWg"], dWg, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(b["dx"], dx, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(b["dWd"], 0.0)
    if gated:
        np.testing.assert_array_equal(b["dWu"], 0.0)


def pin_backward_torch_autograd(ffn=_ffn, gated=True, l1=0.05):
    """torch autograd (fp64, CPU) differentiating the loss independently."""
    import torch
    x, Wg, Wu, Wd, dy = tiny_problem(T=9, d=16, I=24, gated=gated, seed=6)
    tt = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
          for k, v in dict(x=x, Wg=Wg, Wd=Wd, **({"Wu": Wu} if gated else {})).items()}
    g = tt["x"] @ tt["Wg"].T
    a = torch.relu(g)
    h = a * (tt["x"] @ tt["Wu"].T) if gated else a
    L = (torch.tensor(dy) * (h @ tt["Wd"])).sum() + l1 * a.sum()
    L.backward()
    b = ffn.backward(x, Wg, Wu, Wd, dy, l1)
    np.testing.assert_allclose(b["dx"], tt["x"].grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["dWg"], tt["Wg"].grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["dWd"], tt["Wd"].grad.numpy(), rtol=1e-12, atol=1e-12)
    if gated:
        np.testing.assert_allclose(b["dWu"], tt["Wu"].grad.numpy(), rtol=1e-12, atol=1e-12)


def pin_backward_weight_rows(ffn=_ffn, gated=True, l1=0.2):
    """Sampled weight-gradient rows agree with finite differences of the loss."""
    x, Wg, Wu, Wd, dy = tiny_problem(T=4, d=6, I=10, gated=gated, seed=8)
    J = np.array([1, 4, 9])
    r = ffn.backward_weight_rows(x, Wg, Wu, Wd, dy, l1, J)
    loss = lambda: ffn.loss(x, Wg, Wu, Wd, dy, l1)  # noqa: E731
    for name, arr in [("dWg", Wg), ("dWd", Wd)] + ([("dWu", Wu)] if gated else []):
        fd = _fd_grad(loss, arr)[J]
        np.testing.assert_allclose(r[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


# ------------------------------------------------------------ format-level pins

def pin_sparse_equals_dense(ffn=_ffn, sparse=_sparse, gated=True, l1=0.25):
    """The packed computation (TwELL inference, Hybrid training) reaches the dense
    definition, on a problem where some rows overflow and some go to the backup."""
    x, Wg, Wu, Wd, dy = tiny_problem(T=12, d=8, I=32, gated=gated, seed=12)
    W, C = 8, 4
    dense_f = ffn.forward(x, Wg, Wu, Wd)
    nnz = np.sort((x @ Wg.T > 0).sum(1))
    R = int(nnz[len(nnz) // 2])          # about half the rows exceed R
    y_tw, tw = sparse.twell_forward(x, Wg, Wu, Wd, W, C)
    assert tw["ovf"].any() and not tw["ovf"].all()
    np.testing.assert_allclose(y_tw, dense_f["y"], rtol=1e-12, atol=1e-13)
    y_hy, hy = sparse.hybrid_forward(x, Wg, Wu, Wd, W, C, R)
    assert hy["backup"].any() and not hy["backup"].all()
    np.testing.assert_allclose(y_hy, dense_f["y"], rtol=1e-12, atol=1e-13)
    b_dense = ffn.backward(x, Wg, Wu, Wd, dy, l1)
    b_sp = sparse.hybrid_backward(x, Wg, Wu, Wd, dy, l1, hy)
    for k in ("dx", "dWg", "dWd") + (("dWu",) if gated else ()):
        np.testing.assert_allclose(b_sp[k], b_dense[k], rtol=1e-12, atol=1e-13, err_msg=k)
