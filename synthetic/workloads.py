"""Seeded synthetic inputs for the ReLU activation-sparse feedforward layer.

This module only draws numbers: it holds none of the FFN's arithmetic, so both the
fp64 oracle (``oracle/``) and the CUDA path can take their inputs from it.

Recipe (stated once here and in the design notes):

* x ~ N(0, 1) per entry, then column 0 is set to 1 so that column 0 of the gate
  weight acts as a per-neuron bias.
* A seeded choice of ``round(outlier_frac * T)`` distinct token rows has its
  non-constant features (columns 1:) multiplied by ``outlier_scale`` before
  rounding. These "outlier" tokens activate many more neurons than ordinary ones,
  standing in for the high-information tokens the pages describe (wispaper blog,
  Figure 2 caption; gist.science explainer, section 4 "Sparsity Patterns").
* Wg, Wu (or W1) ~ N(0, 1/d); Wd (or W2) ~ N(0, 1/I). All weights are stored
  [I, d] row-major: row j of Wg/Wu is the input weight vector of neuron j and row j
  of Wd is the output vector neuron j adds to y.
* Wg[:, 0] (the bias, because x[:, 0] == 1) is set to
  -Phi^{-1}(1 - m/I) * sqrt((d-1)/d) so that an ordinary token activates m neurons
  on average (m = ``mean_active``, the "# non-zeros" statistic of the pages'
  Tables 3 and 5).
* dy ~ N(0, dy_std^2).
* Every tensor is rounded to bfloat16 (round to nearest, ties to even) and returned
  as its raw 16-bit patterns (``numpy.uint16``).

Each tensor comes from its own generator ``numpy.random.default_rng([seed, cfg_id,
layer, tensor_id])`` so that any tensor can be regenerated alone.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from statistics import NormalDist

import numpy as np

# tensor ids for the per-tensor generators
_TID_X, _TID_OUTLIERS, _TID_WG, _TID_WU, _TID_WD, _TID_DY = range(6)


def round_to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """float values -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    f = np.ascontiguousarray(values, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def roundup(v: int, m: int) -> int:
    return (v + m - 1) // m * m


@dataclass(frozen=True)
class FFNSpec:
    """Shape and statistics of one synthetic FFN workload."""

    name: str
    T: int                      # tokens
    d: int                      # model width
    I: int                      # intermediate (hidden) width
    gated: bool = True
    mean_active: float = 29.0   # mean active neurons per ordinary token
    outlier_frac: float = 0.0
    outlier_scale: float = 3.0
    W: int = 128                # TwELL tile width
    C: int = 16                 # TwELL slots per (row, tile)
    R: int = 64                 # Hybrid ELL slots per row
    l1: float = 2e-5            # L1 coefficient on the hidden activations
    dy_std: float = 0.1
    seed: int = 0
    cfg_id: int = 0

    @property
    def n_tiles(self) -> int:
        return self.I // self.W

    @property
    def bias(self) -> float:
        """Gate bias before bf16 rounding: -Phi^{-1}(1 - m/I) * sqrt((d-1)/d)."""
        p = self.mean_active / self.I
        return -NormalDist().inv_cdf(1.0 - p) * math.sqrt((self.d - 1) / self.d)

    def with_(self, **kw) -> "FFNSpec":
        return replace(self, **kw)


def stack_layer_mean_active(layer: int, n_layers: int = 28) -> float:
    """Per-layer mean actives of the 28-layer stack workload: 15 rising to 120 over layers
    0-7, a plateau of 120 on layers 8-14 (the early-middle hump the pages report), then a
    linear fall back to 15 at the last layer."""
    if layer < 8:
        return 15.0 + 105.0 * layer / 8.0
    if layer <= 14:
        return 120.0
    return 120.0 - 105.0 * (layer - 14) / (n_layers - 1 - 14)


def _sweep_R(m: float) -> int:
    return roundup(int(round(2 * m)), 32)


# Named workloads. Sizes follow the pages' 1.5B model FFN shapes (hidden 2048,
# intermediate 5632 gated / 8192 non-gated; Table 2 of the thelatestinai listing).
WORKLOADS: dict[str, FFNSpec] = {
    # tiny gated forward: ~1% active neurons, 2% outlier tokens that overflow the ELL
    "tiny_fwd": FFNSpec("tiny_fwd", T=256, d=256, I=704, mean_active=0.01 * 704,
                        outlier_frac=0.02, W=64, C=8, R=32, cfg_id=1),
    # gated forward at the 1.5B shape, 29 actives per ordinary token, 0.5% outliers
    "gated_fwd_d2048_i5632": FFNSpec("gated_fwd_d2048_i5632", T=16384, d=2048, I=5632,
                                     mean_active=29, outlier_frac=0.005, W=128, C=16,
                                     R=64, cfg_id=2),
    # non-gated forward, intermediate 8192, 40 actives, 1% outliers
    "nongated_fwd_d2048_i8192": FFNSpec("nongated_fwd_d2048_i8192", T=16384, d=2048, I=8192,
                                        gated=False, mean_active=40, outlier_frac=0.01,
                                        W=128, C=16, R=96, cfg_id=3),
}
# Hybrid training step of the non-gated form (shapes and inputs of the non-gated forward)
WORKLOADS["train_nongated_d2048_i8192_m40_o1"] = FFNSpec(
    "train_nongated_d2048_i8192_m40_o1", T=16384, d=2048, I=8192, gated=False, mean_active=40, outlier_frac=0.01,
    W=128, C=16, R=96, l1=2e-5, cfg_id=3)
# Hybrid training step sweep at the 1.5B gated shape
for _m in (29, 108, 911):
    for _f in (0.0, 0.01, 0.05):
        _n = f"train_d2048_i5632_m{_m}_o{int(round(_f * 100))}"
        WORKLOADS[_n] = FFNSpec(_n, T=16384, d=2048, I=5632, mean_active=_m, outlier_frac=_f,
                                W=128, C=16, R=_sweep_R(_m), l1=2e-5, cfg_id=4)


def stack_layer_spec(layer: int, T: int = 8192, seed: int = 0, d: int = 2048, I: int = 5632, W: int = 128,
                     C: int = 16, profile_layer: int | None = None) -> FFNSpec:
    """Layer `layer` of the residual stack workload. Its mean actives follow the
    28-layer profile at `profile_layer` (default: the same index), scaled by I / 5632
    for narrower test shapes."""
    m = stack_layer_mean_active(layer if profile_layer is None else profile_layer) * I / 5632.0
    return FFNSpec(f"stack28_l{layer}", T=T, d=d, I=I, mean_active=m,
                   outlier_frac=0.01, W=W, C=C, R=_sweep_R(m), cfg_id=5, seed=seed)


STACK_WD_SCALE = 1.0 / 16.0


def make_stack(specs: list[FFNSpec]) -> dict:
    """Inputs of a residual stack x_{l+1} = x_l + FFN_l(x_l): the first layer's x (with
    its outlier tokens), every layer's weights, and the gradient arriving at the top.
    Column 0 of every Wd is zero, so feature 0 of the residual stream stays exactly 1
    and each layer's bias (Wg[:, 0]) keeps its meaning. Wd is scaled by 1/16
    (variance 1/(256 I)): a gated FFN is quadratic in its input, and without the
    branch scaling the outlier tokens (3x inputs) grow without bound within a few
    layers; with it their |x| stays below ~13 over 28 layers while the ordinary
    tokens' residual stream keeps unit variance."""
    layers = []
    for l, sp in enumerate(specs):
        w = make_weights(sp, l)
        wd = bf16_bits_to_float32(w["Wd"]) * np.float32(STACK_WD_SCALE)
        wd[:, 0] = 0.0
        w["Wd"] = round_to_bf16_bits(wd)
        layers.append(w)
    return {"x0": make_x(specs[0], 0), "outliers": outlier_rows(specs[0], 0), "layers": layers,
            "dy": make_dy(specs[-1], len(specs) - 1)}


def _rng(spec: FFNSpec, layer: int, tid: int) -> np.random.Generator:
    return np.random.default_rng([spec.seed, spec.cfg_id, layer, tid])


def outlier_rows(spec: FFNSpec, layer: int = 0) -> np.ndarray:
    n = int(round(spec.outlier_frac * spec.T))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(spec, layer, _TID_OUTLIERS).choice(spec.T, n, replace=False))


def make_x(spec: FFNSpec, layer: int = 0, rows: np.ndarray | None = None) -> np.ndarray:
    x = _rng(spec, layer, _TID_X).standard_normal((spec.T, spec.d), dtype=np.float32)
    x[:, 0] = 1.0
    out = outlier_rows(spec, layer)
    if out.size:
        x[out, 1:] *= np.float32(spec.outlier_scale)
    if rows is not None:
        x = x[rows]
    return round_to_bf16_bits(x)


def make_weights(spec: FFNSpec, layer: int = 0) -> dict[str, np.ndarray | None]:
    d, I = spec.d, spec.I
    wg = _rng(spec, layer, _TID_WG).standard_normal((I, d), dtype=np.float32)
    wg *= np.float32(1.0 / math.sqrt(d))
    wg[:, 0] = np.float32(spec.bias)
    wu = None
    if spec.gated:
        wu = _rng(spec, layer, _TID_WU).standard_normal((I, d), dtype=np.float32)
        wu *= np.float32(1.0 / math.sqrt(d))
    wd = _rng(spec, layer, _TID_WD).standard_normal((I, d), dtype=np.float32)
    wd *= np.float32(1.0 / math.sqrt(I))
    return {
        "Wg": round_to_bf16_bits(wg),
        "Wu": None if wu is None else round_to_bf16_bits(wu),
        "Wd": round_to_bf16_bits(wd),
    }


def make_dy(spec: FFNSpec, layer: int = 0) -> np.ndarray:
    dy = _rng(spec, layer, _TID_DY).standard_normal((spec.T, spec.d), dtype=np.float32)
    dy *= np.float32(spec.dy_std)
    return round_to_bf16_bits(dy)


def make_inputs(spec: FFNSpec, layer: int = 0, with_dy: bool = False) -> dict:
    """All tensors of one workload as bf16 bit patterns plus the outlier row list."""
    out = {"x": make_x(spec, layer), **make_weights(spec, layer), "outliers": outlier_rows(spec, layer)}
    out["dy"] = make_dy(spec, layer) if with_dy else None
    return out


def random_bf16_matrix(shape, density: float, seed: int, negative_zero_frac: float = 0.0,
                       signed: bool = False, subnormal_frac: float = 0.0) -> np.ndarray:
    """A bf16 matrix whose entries are nonzero with probability ``density`` (values ~ |N(0,1)|,
    i.e. post-ReLU-like). A fraction of the zero entries can be written as -0.0 (0x8000).

    ``signed`` gives each nonzero a random sign (a general matrix for the standalone
    packer, whose nonzero test is on the magnitude bits); ``subnormal_frac`` of the
    nonzeros become bf16 subnormals: the smallest (0x0001) and the largest (0x007F)
    magnitudes, with the sign the entry had."""
    rng = np.random.default_rng([seed, 9001])
    vals = np.abs(rng.standard_normal(shape, dtype=np.float32)) + np.float32(1e-3)
    keep = rng.random(shape) < density
    bits = round_to_bf16_bits(np.where(keep, vals, np.float32(0.0)))
    if negative_zero_frac > 0:
        negz = (~keep) & (rng.random(shape) < negative_zero_frac)
        bits[negz] = 0x8000
    if subnormal_frac > 0:
        sub = keep & (rng.random(shape) < subnormal_frac)
        bits[sub] = np.where(rng.random(shape) < 0.5, 0x0001, 0x007F).astype(np.uint16)[sub]
    if signed:
        neg = keep & (rng.random(shape) < 0.5)
        bits[neg] |= np.uint16(0x8000)
    return bits
