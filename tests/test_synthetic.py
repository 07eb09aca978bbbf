"""The seeded generator hits the sparsity statistics it is built for (CPU only)."""
import math
from statistics import NormalDist

import numpy as np
import pytest

from oracle import ffn
from synthetic import WORKLOADS, bf16_bits_to_float32, make_inputs, make_x, outlier_rows


def _expected_active_fraction(spec, scale=1.0):
    """Closed form for the generator's bias: P(g > 0) = 1 - Phi(-b / sigma) with the
    bf16-rounded bias b and sigma^2 = scale^2 (d-1)/d."""
    from synthetic.workloads import round_to_bf16_bits
    b = float(bf16_bits_to_float32(round_to_bf16_bits(np.array([spec.bias])))[0])
    sigma = scale * math.sqrt((spec.d - 1) / spec.d)
    return 1.0 - NormalDist().cdf(-b / sigma)


def test_generator_is_deterministic():
    spec = WORKLOADS["tiny_fwd"]
    a, b = make_inputs(spec), make_inputs(spec)
    for k in ("x", "Wg", "Wu", "Wd"):
        np.testing.assert_array_equal(a[k], b[k])
    assert not np.array_equal(a["x"], make_x(spec.with_(seed=1)))


def test_generator_structure():
    spec = WORKLOADS["tiny_fwd"]
    inp = make_inputs(spec, with_dy=True)
    x = bf16_bits_to_float32(inp["x"])
    assert (x[:, 0] == 1.0).all()
    assert inp["outliers"].size == round(spec.outlier_frac * spec.T) == 5
    assert inp["Wg"].shape == (spec.I, spec.d) and inp["Wd"].shape == (spec.I, spec.d)
    assert inp["dy"].shape == (spec.T, spec.d)
    assert 0.09 < np.std(bf16_bits_to_float32(inp["dy"])) < 0.11


@pytest.mark.parametrize("name,T", [("tiny_fwd", None), ("gated_fwd_d2048_i5632", 1024),
                                    ("train_d2048_i5632_m108_o1", 512)])
def test_mean_actives_match_closed_form(name, T):
    spec = WORKLOADS[name]
    if T is not None:
        spec = spec.with_(T=T)
    inp = make_inputs(spec)
    g = ffn.forward(inp["x"], inp["Wg"], None, inp["Wd"])["g"]
    act = (g > 0).sum(1)
    ordinary = np.setdiff1d(np.arange(spec.T), outlier_rows(spec))
    p = _expected_active_fraction(spec)
    m_exp = p * spec.I
    n = ordinary.size
    band = 4 * math.sqrt(m_exp * (1 - p) / n) + 0.05 * m_exp     # binomial 4 sigma + per-neuron spread
    assert abs(act[ordinary].mean() - m_exp) < band, (act[ordinary].mean(), m_exp)
    out = outlier_rows(spec)
    if out.size:
        p_out = _expected_active_fraction(spec, scale=spec.outlier_scale)
        assert abs(act[out].mean() - p_out * spec.I) < 0.15 * p_out * spec.I + 10


def test_stack_generator_structure_and_profile():
    """The residual stack: Wd column 0 is zero (feature 0 of the stream stays 1), Wd is
    the layer's N(0, 1/I) draw scaled by 1/16, and the ordinary tokens' activity follows
    the 28-layer profile through the residual stream (checked over three layers)."""
    from synthetic import make_stack, round_to_bf16_bits, stack_layer_mean_active, stack_layer_spec

    profile = (0, 9, 27)
    specs = [stack_layer_spec(l, T=512, d=512, I=1408, W=64, C=16, profile_layer=p)
             for l, p in enumerate(profile)]
    st = make_stack(specs)
    ordinary = np.setdiff1d(np.arange(512), st["outliers"])
    x = st["x0"]
    for l, (sp, w) in enumerate(zip(specs, st["layers"])):
        wd = bf16_bits_to_float32(w["Wd"])
        assert (wd[:, 0] == 0).all()
        assert abs(wd[:, 1:].std() * 16 * math.sqrt(sp.I) - 1) < 0.02
        assert sp.mean_active == stack_layer_mean_active(profile[l]) * sp.I / 5632
        f = ffn.forward(x, w["Wg"], w["Wu"], w["Wd"])
        act = (f["g"] > 0).sum(1)[ordinary].mean()
        assert abs(act - sp.mean_active) < 0.15 * sp.mean_active + 1, (l, act, sp.mean_active)
        y = round_to_bf16_bits(np.asarray(f["y"], dtype=np.float32))
        x = round_to_bf16_bits(bf16_bits_to_float32(x) + bf16_bits_to_float32(y))
        assert (bf16_bits_to_float32(x)[:, 0] == 1.0).all()
