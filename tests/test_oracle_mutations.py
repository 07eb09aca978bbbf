"""Planted-mistake tests: each case copies one oracle module, introduces a plausible
error (a dropped term, a wrong sign, a wrong operand, an off-by-one, a transposed
index), and checks that at least one pin rejects the copy. The mistakes are planted
in the oracle only, on the CPU.
"""
import importlib
import inspect
import types

import numpy as np
import pytest

import pins
import oracle
from synthetic import random_bf16_matrix


def _mutant(modname: str, old: str, new: str) -> types.ModuleType:
    mod = importlib.import_module(f"oracle.{modname}")
    src = inspect.getsource(mod)
    assert src.count(old) >= 1, f"snippet not found in oracle.{modname}: {old!r}"
    m = types.ModuleType(f"oracle._mutant_{modname}")
    m.__package__ = "oracle"
    exec(compile(src.replace(old, new, 1), f"<mutant {modname}>", "exec"), m.__dict__)
    return m


def _fails(fn, *args, **kw) -> bool:
    try:
        fn(*args, **kw)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


FFN_MUTANTS = [
    # (description, old, new)
    ("L1 sign flipped", "dg = (dh * u + l1) * active\n        dWu = du.T @ x", "dg = (dh * u - l1) * active\n        dWu = du.T @ x"),
    ("L1 term dropped (gated)", "dg = (dh * u + l1) * active\n        dWu = du.T @ x", "dg = (dh * u) * active\n        dWu = du.T @ x"),
    ("wrong operand in du", "du = dh * a\n        dg = (dh * u + l1) * active\n        dWu", "du = dh * u\n        dg = (dh * u + l1) * active\n        dWu"),
    ("dx drops the up-projection term", "dx = dg @ Wg + du @ Wu", "dx = dg @ Wg"),
    ("dWd uses a instead of h", "dWd = h.T @ dy", "dWd = a.T @ dy"),
    ("ReLU mask dropped", "active = (g > 0.0).astype(np.float64)\n    dh", "active = np.ones_like(g)\n    dh"),
    ("forward ReLU dropped", "h = a if u is None else a * u", "h = a if u is None else g * u"),
    ("forward down-projection rows reversed", "y = h @ Wd\n", "y = h @ Wd[::-1]\n"),
    ("forward gate transposed index", "g = x @ Wg.T\n    a = relu(g)\n    u = None", "g = x @ Wg[::-1].T\n    a = relu(g)\n    u = None"),
    ("sampled rows drop L1", "dg = (dh * u + l1) * active\n        dWu = du.T @ x\n    return", "dg = (dh * u) * active\n        dWu = du.T @ x\n    return"),
    ("sampled rows h without gate", "h = a * u\n        du", "h = a\n        du"),
]

FFN_PINS = [
    pins.pin_forward_permutation,
    pins.pin_forward_scaled_up,
    pins.pin_forward_brute_force,
    pins.pin_backward_finite_differences,
    pins.pin_backward_l1_closed_form,
    pins.pin_backward_weight_rows,
]


@pytest.mark.parametrize("desc,old,new", FFN_MUTANTS, ids=[m[0] for m in FFN_MUTANTS])
def test_ffn_mutant_is_caught(desc, old, new):
    m = _mutant("ffn", old, new)
    assert any(_fails(p, ffn=m) for p in FFN_PINS), f"no pin caught: {desc}"


def test_unmutated_ffn_passes_all_pins():
    for p in FFN_PINS:
        p(ffn=oracle.ffn)


SPARSE_MUTANTS = [
    ("ELL L1 injection dropped", "dg = dh * u + l1\n", "dg = dh * u\n"),
    ("ELL dx misses Wu term", "dx[t] = dg @ Wg[j] + du @ Wu[j]", "dx[t] = dg @ Wg[j]"),
    ("backup uses wrong slot", "b = hy[\"backup_slot\"][t]\n            a = hy", "b = hy[\"backup_slot\"][t] - 1\n            a = hy"),
    ("TwELL local index not offset by tile", "j = k * W + tw[\"idx\"][t, k, s]", "j = tw[\"idx\"][t, k, s]"),
    ("transposed weight grads use ELL u as h", "h_ell[t, :n] = a * u", "h_ell[t, :n] = u"),
]


@pytest.mark.parametrize("desc,old,new", SPARSE_MUTANTS, ids=[m[0] for m in SPARSE_MUTANTS])
def test_sparse_mutant_is_caught(desc, old, new):
    m = _mutant("sparse", old, new)
    assert _fails(pins.pin_sparse_equals_dense, sparse=m), f"not caught: {desc}"


FORMAT_MUTANTS = [
    ("slot order reversed", "order = np.argsort(~nz, axis=-1, kind=\"stable\")",
     "order = np.argsort(~nz, axis=-1, kind=\"stable\")[..., ::-1]"),
    ("overflow at cnt == C", "ovf = (cnt > C).any(axis=1)", "ovf = (cnt >= C).any(axis=1)"),
    ("-0.0 counted as nonzero", "return (A & 0x7FFF) != 0", "return A != 0"),
    ("routing ignores TwELL overflow", "backup = tw[\"ovf\"] | (tw[\"row_nnz\"] > R)", "backup = tw[\"row_nnz\"] > R"),
    ("capped count stored", "cnt = nz.sum(axis=2).astype(np.int64)", "cnt = np.minimum(nz.sum(axis=2), C).astype(np.int64)"),
    ("negative values not counted", "return (A & 0x7FFF) != 0", "return ((A & 0x7FFF) != 0) & ((A & 0x8000) == 0)"),
    ("subnormals not counted", "return (A & 0x7FFF) != 0", "return (A & 0x7F80) != 0"),
]


def _format_pins(fm):
    import test_oracle_formats as tf
    orig = tf.formats
    tf.formats = fm
    try:
        tf.test_twell_golden_worked_example()
        tf.test_hybrid_golden_worked_example()
        tf.test_twell_capacity_boundary()
        for args in [((7, 16), 4, 2, 0.3, 1, False), ((9, 256), 128, 16, 0.08, 3, False),
                     ((8, 128), 64, 6, 0.3, 6, True)]:
            tf.test_twell_matches_brute_force(*args)
    finally:
        tf.formats = orig


@pytest.mark.parametrize("desc,old,new", FORMAT_MUTANTS, ids=[m[0] for m in FORMAT_MUTANTS])
def test_format_mutant_is_caught(desc, old, new):
    m = _mutant("formats", old, new)
    assert _fails(_format_pins, m), f"not caught: {desc}"


def test_unmutated_formats_pass():
    _format_pins(oracle.formats)
    assert random_bf16_matrix((2, 2), 0.5, 0).dtype == np.uint16


NEURON_MUTANTS = [
    ("bf16 by truncation", "return ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)",
     "return (bits >> np.uint64(16)).astype(np.uint16)"),
    ("product in float32", "w = (np.float64(np.float32(std)) * z).astype(np.float32)",
     "w = np.float32(std) * z.astype(np.float32)"),
    # bf16 straight from the float64 product (round half to even at 8 significant
    # bits), skipping the float32 rounding the definition states
    ("no float32 step", "w = (np.float64(np.float32(std)) * z).astype(np.float32)",
     "w = np.float64(np.float32(std)) * z\n"
     "    e = np.floor(np.log2(np.abs(np.where(w == 0, 1.0, w))))\n"
     "    w = (np.round(np.ldexp(w, (7 - e).astype(np.int64))) * np.exp2(e - 7)).astype(np.float32)"),
    ("uniforms from the wrong bits", ">> np.uint64(40)).astype(np.int64)", ">> np.uint64(41)).astype(np.int64)"),
    ("counter offset", "base + np.uint64(i)", "base + np.uint64(i + 1)"),
]


def _neuron_pins(nm):
    import test_oracle_neurons as tn
    orig = tn.neurons
    tn.neurons = nm
    try:
        tn.test_reinit_known_answers()
        tn.test_irwin_hall_draw_moments_and_support()
        tn.test_reinit_touches_dead_rows_only()
    finally:
        tn.neurons = orig


@pytest.mark.parametrize("desc,old,new", NEURON_MUTANTS, ids=[m[0] for m in NEURON_MUTANTS])
def test_neuron_mutant_is_caught(desc, old, new):
    m = _mutant("neurons", old, new)
    assert _fails(_neuron_pins, m), f"not caught: {desc}"


def test_unmutated_neurons_pass():
    _neuron_pins(oracle.neurons)
