"""Pins for the oracle's dense forward / backward and its sparse restatement (CPU only)."""
import numpy as np
import pytest

import pins
from oracle import ffn


@pytest.mark.parametrize("gated", [True, False])
def test_forward_permutation_closed_form(gated):
    pins.pin_forward_permutation(gated=gated)


def test_forward_gated_with_constant_up_equals_nongated():
    pins.pin_forward_scaled_up()


@pytest.mark.parametrize("gated", [True, False])
def test_forward_brute_force(gated):
    pins.pin_forward_brute_force(gated=gated)


@pytest.mark.parametrize("gated", [True, False])
def test_backward_finite_differences(gated):
    pins.pin_backward_finite_differences(gated=gated)


@pytest.mark.parametrize("gated", [True, False])
def test_backward_l1_on_h_reading(gated):
    pins.pin_backward_l1_on_h(gated=gated)


@pytest.mark.parametrize("gated", [True, False])
def test_backward_l1_closed_form(gated):
    pins.pin_backward_l1_closed_form(gated=gated)


@pytest.mark.parametrize("gated", [True, False])
def test_backward_torch_autograd(gated):
    pins.pin_backward_torch_autograd(gated=gated)


@pytest.mark.parametrize("gated", [True, False])
def test_backward_weight_rows(gated):
    pins.pin_backward_weight_rows(gated=gated)


@pytest.mark.parametrize("gated", [True, False])
def test_sparse_formats_reach_dense_result(gated):
    pins.pin_sparse_equals_dense(gated=gated)


def test_bf16_conversion_exact():
    # 1.0 = 0x3F80, -2.0 = 0xC000, smallest normal 2^-126 = 0x0080, -0.0 = 0x8000
    bits = np.array([0x3F80, 0xC000, 0x0080, 0x8000, 0x4049], dtype=np.uint16)
    v = ffn.bf16_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 2.0 ** -126
    assert v[3] == 0.0 and np.signbit(v[3])
    assert v[4] == 3.140625


def test_active_set_is_strict():
    # ReLU'(0) = 0: a neuron with g exactly 0 is inactive and gets no L1 gradient
    x = np.array([[1.0, 0.0]])
    Wg = np.array([[0.0, 1.0], [0.5, 0.0]])        # g = [0, 0.5]
    Wd = np.eye(2)
    b = ffn.backward(x, Wg, None, Wd, np.zeros((1, 2)), 1.0)
    np.testing.assert_array_equal(b["dg"], [[0.0, 1.0]])
