"""Dense fp64 definition of the ReLU feedforward layer and its gradient.

Test infrastructure only (see ``oracle/__init__.py``).

Problem statement followed here (gist.science explainer "Sparser, Faster, Lighter
Transformer Language Models", section 2.B "Kernel Design" and 2.C "Training
Recipe"; Table 2 of the thelatestinai listing for the gated / non-gated forms):

    gated:      g = x Wg^T,  a = ReLU(g),  u = x Wu^T,  h = a * u,  y = h Wd
    non-gated:  g = x W1^T,  a = ReLU(g),               h = a,      y = h W2

with every weight stored [I, d] (row j belongs to hidden neuron j), so ``x Wg^T``
is the gate projection and ``h Wd`` sums the rows of Wd weighted by h.

Training adds an L1 penalty on the hidden activations (explainer 2.C
"Regularization"). The activation penalised is a = ReLU(g): it is the one whose
support the formats compress, and it is non-negative so |a| = a. The scalar whose
gradient ``backward`` returns is

    L = sum_{t,c} dy[t,c] * y[t,c]  +  l1 * sum_{t,j} a[t,j]

(``dy`` plays the role of the upstream gradient; no 1/T normalisation is applied
to the L1 term -- a caller wanting one folds it into ``l1``). ReLU'(0) is taken
as 0, i.e. the active set is the strict set g > 0.

The pages leave open which activation the penalty acts on. ``penalise="h"`` takes
the other reading, l1 * sum |h| with h = a * u (sign(0) = 0), for reference only:
the library implements the penalty on a. Without a gate, h = a and both readings
coincide.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64. A bf16 value is the upper half of
    an IEEE float32, so shifting the 16 bits up and reinterpreting is exact."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def as_f64(t) -> np.ndarray | None:
    if t is None:
        return None
    t = np.asarray(t)
    if t.dtype == np.uint16:
        return bf16_to_f64(t)
    return t.astype(np.float64)


def relu(g: np.ndarray) -> np.ndarray:
    return np.where(g > 0.0, g, 0.0)


def forward(x, Wg, Wu, Wd) -> dict:
    """Dense forward. ``Wu is None`` selects the non-gated form. Returns g, a, u
    (None when non-gated), h and y, all float64."""
    x, Wg, Wu, Wd = (as_f64(t) for t in (x, Wg, Wu, Wd))
    g = x @ Wg.T
    a = relu(g)
    u = None if Wu is None else x @ Wu.T
    h = a if u is None else a * u
    y = h @ Wd
    return {"g": g, "a": a, "u": u, "h": h, "y": y}


def loss(x, Wg, Wu, Wd, dy, l1: float, penalise: str = "a") -> float:
    """L = sum(dy * y) + l1 * sum(a)  (or + l1 * sum |h| with penalise="h")."""
    f = forward(x, Wg, Wu, Wd)
    pen = np.sum(f["a"]) if penalise == "a" else np.sum(np.abs(f["h"]))
    return float(np.sum(as_f64(dy) * f["y"]) + l1 * pen)


def backward(x, Wg, Wu, Wd, dy, l1: float, fwd: dict | None = None, penalise: str = "a") -> dict:
    """Gradient of L with respect to x and the three weights, by the chain rule:

        dh  = dy Wd^T                      dWd = h^T dy
        gated:     du = dh * a,   dg = (dh * u + l1) * [g > 0]
                   dWu = du^T x,  dWg = dg^T x,  dx = dg Wg + du Wu
        non-gated: dg = (dh + l1) * [g > 0],  dW1 = dg^T x,  dx = dg W1

    The sparse backward of the pages (explainer 2.B "Backpropagation": inject the
    L1 gradient, transpose the hybrid format for the weight gradients) computes
    exactly these quantities restricted to the active set.

    With penalise="h" the penalty's gradient enters through h instead:
    dh' = dh + l1 * sign(h), then du = dh' * a and dg = dh' * u * [g > 0] (gated;
    non-gated h = a >= 0, the same as the default)."""
    x, Wg, Wu, Wd, dy = (as_f64(t) for t in (x, Wg, Wu, Wd, dy))
    f = fwd if fwd is not None else forward(x, Wg, Wu, Wd)
    g, a, u, h = f["g"], f["a"], f["u"], f["h"]
    active = (g > 0.0).astype(np.float64)
    dh = dy @ Wd.T
    dWd = h.T @ dy
    if penalise == "h" and Wu is not None:
        dh_h = dh + l1 * np.sign(h)
        du = dh_h * a
        dg = dh_h * u * active
        return {"dx": dg @ Wg + du @ Wu, "dWg": dg.T @ x, "dWu": du.T @ x, "dWd": dWd, "dh": dh, "dg": dg, "du": du}
    if Wu is None:
        du = None
        dg = (dh + l1) * active
        dWu = None
        dx = dg @ Wg
    else:
        du = dh * a
        dg = (dh * u + l1) * active
        dWu = du.T @ x
        dx = dg @ Wg + du @ Wu
    dWg = dg.T @ x
    return {"dx": dx, "dWg": dWg, "dWu": dWu, "dWd": dWd, "dh": dh, "dg": dg, "du": du}


def backward_weight_rows(x, Wg, Wu, Wd, dy, l1: float, rows) -> dict:
    """Rows ``rows`` of dWg, dWu, dWd only, for sampled checks at full size.

    Row j of every weight gradient depends only on column j of g, u, dh (over all
    tokens), so this evaluates the same formulas as ``backward`` on the selected
    neurons: g[:, J] = x Wg[J]^T, u[:, J] = x Wu[J]^T, dh[:, J] = dy Wd[J]^T."""
    x, Wg, Wu, Wd, dy = (as_f64(t) for t in (x, Wg, Wu, Wd, dy))
    J = np.asarray(rows)
    g = x @ Wg[J].T
    a = relu(g)
    active = (g > 0.0).astype(np.float64)
    dh = dy @ Wd[J].T
    if Wu is None:
        h = a
        dg = (dh + l1) * active
        dWu = None
    else:
        u = x @ Wu[J].T
        h = a * u
        du = dh * a
        dg = (dh * u + l1) * active
        dWu = du.T @ x
    return {"dWg": dg.T @ x, "dWu": dWu, "dWd": h.T @ dy}
