"""The FFN computed entry by entry from the packed formats, in fp64.

Test infrastructure only (see ``oracle/__init__.py``).

This restates the method's own order of work, to check that it reaches exactly
the dense definition of ``oracle.ffn`` (the pages' method is exact: it skips only
multiplications by zero):

* inference (gist.science explainer 2.B "Inference Kernels"): the gate projection
  is packed into TwELL; for every stored entry (t, j) of a non-overflow row the
  up-projection is a dot product u = x_t . Wu[j] and the down-projection adds
  (a * u) * Wd[j] to y_t; overflow rows take the dense path;
* training (explainer 2.B "Training Kernels"): the Hybrid keeps a and u on the
  support of ELL rows and in full for backup rows; the backward computes, per ELL
  entry, dh = dy_t . Wd[j], du = dh * a, dg = dh * u + l1 (the L1 subgradient is
  1 on the support), adds dg * Wg[j] + du * Wu[j] to dx_t, and accumulates the
  weight gradients over the transposed Hybrid; backup rows use dense products.
"""
from __future__ import annotations

import numpy as np

from . import formats
from .ffn import as_f64, relu


def twell_forward(x, Wg, Wu, Wd, W: int, C: int) -> tuple[np.ndarray, dict]:
    """y from the TwELL of a = ReLU(x Wg^T). Returns (y, twell)."""
    x, Wg, Wu, Wd = (as_f64(t) for t in (x, Wg, Wu, Wd))
    T, d = x.shape
    g = x @ Wg.T
    a = relu(g)
    tw = formats.twell_pack(a, W, C)
    y = np.zeros((T, d))
    for t in range(T):
        if tw["ovf"][t]:
            h = a[t] if Wu is None else a[t] * (Wu @ x[t])
            y[t] = h @ Wd
            continue
        k, s = np.nonzero(tw["valid"][t])
        j = k * W + tw["idx"][t, k, s]
        av = tw["val"][t, k, s]
        h = av if Wu is None else av * (Wu[j] @ x[t])
        y[t] = h @ Wd[j]
    return y, tw


def hybrid_forward(x, Wg, Wu, Wd, W: int, C: int, R: int) -> tuple[np.ndarray, dict]:
    """y and the saved Hybrid (a and u on the support / full backup rows)."""
    x, Wg, Wu, Wd = (as_f64(t) for t in (x, Wg, Wu, Wd))
    T, d = x.shape
    a = relu(x @ Wg.T)
    # u is only needed on the support; the dense product is the definition of its values
    U = None if Wu is None else x @ Wu.T
    hy = formats.hybrid_pack(a, U, W, C, R)
    y = np.zeros((T, d))
    for t in range(T):
        if hy["backup"][t]:
            b = hy["backup_slot"][t]
            h = hy["backup_a"][b] if U is None else hy["backup_a"][b] * hy["backup_u"][b]
            y[t] = h @ Wd
            continue
        n = hy["ell_nnz"][t]
        j = hy["ell_idx"][t, :n]
        h = hy["ell_a"][t, :n] if U is None else hy["ell_a"][t, :n] * hy["ell_u"][t, :n]
        y[t] = h @ Wd[j]
    return y, hy


def hybrid_backward(x, Wg, Wu, Wd, dy, l1: float, hy: dict) -> dict:
    """dx, dWg, dWu, dWd from the saved Hybrid."""
    x, Wg, Wu, Wd, dy = (as_f64(t) for t in (x, Wg, Wu, Wd, dy))
    T, d = x.shape
    I = Wg.shape[0]
    gated = Wu is not None
    dx = np.zeros((T, d))
    dWg = np.zeros((I, d))
    dWu = np.zeros((I, d)) if gated else None
    dWd = np.zeros((I, d))
    # per-entry coefficients of the ELL part, laid out like the ELL itself
    R = hy["R"]
    dg_ell = np.zeros((T, R))
    du_ell = np.zeros((T, R))
    h_ell = np.zeros((T, R))
    for t in range(T):
        if hy["backup"][t]:
            b = hy["backup_slot"][t]
            a = hy["backup_a"][b]
            act = (a > 0).astype(np.float64)
            dh = Wd @ dy[t]
            if gated:
                u = hy["backup_u"][b]
                du = dh * a
                dg = (dh * u + l1) * act
                dx[t] = dg @ Wg + du @ Wu
                dWu += np.outer(du, x[t])
                h = a * u
            else:
                dg = (dh + l1) * act
                dx[t] = dg @ Wg
                h = a
            dWg += np.outer(dg, x[t])
            dWd += np.outer(h, dy[t])
            continue
        n = hy["ell_nnz"][t]
        j = hy["ell_idx"][t, :n]
        a = hy["ell_a"][t, :n]
        dh = Wd[j] @ dy[t]
        if gated:
            u = hy["ell_u"][t, :n]
            du = dh * a
            dg = dh * u + l1
            dx[t] = dg @ Wg[j] + du @ Wu[j]
            du_ell[t, :n] = du
            h_ell[t, :n] = a * u
        else:
            dg = dh + l1
            dx[t] = dg @ Wg[j]
            h_ell[t, :n] = a
        dg_ell[t, :n] = dg
    # weight gradients of the ELL part over the transposed Hybrid
    tr = formats.hybrid_transpose(hy)
    for j in range(I):
        lo, hi = tr["col_ptr"][j], tr["col_ptr"][j + 1]
        if lo == hi:
            continue
        tk, sl = tr["tok"][lo:hi], tr["slot"][lo:hi]
        dWg[j] += dg_ell[tk, sl] @ x[tk]
        if gated:
            dWu[j] += du_ell[tk, sl] @ x[tk]
        dWd[j] += h_ell[tk, sl] @ dy[tk]
    return {"dx": dx, "dWg": dWg, "dWu": dWu, "dWd": dWd}
