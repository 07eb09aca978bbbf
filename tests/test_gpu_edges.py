"""Edge cases of the whole path against the fp64 oracle: an empty batch, a single
token, tokens without any active neuron, the longest per-token entry lists the
sparse forward accepts ((I / W) * C = 10240 entries with every neuron active, which
fills one CTA's shared memory and runs the backward in 40 windows), and a hidden
layer too wide for the backward's shared-memory column histogram."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import assert_close, f64_of, to_dev  # noqa: E402
from oracle import ffn  # noqa: E402
from synthetic import FFNSpec, make_inputs, round_to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _dev(inp):
    return {k: (to_dev(inp[k]) if inp.get(k) is not None else None) for k in ("x", "Wg", "Wu", "Wd", "dy")}


def _check_against_oracle(spec, inp, y_twell, y, grads, what):
    f = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])
    b = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, fwd=f)
    assert_close(f64_of(y_twell), f["y"], f"{what}: TwELL y")
    assert_close(f64_of(y), f["y"], f"{what}: Hybrid y")
    dx, dWg, dWu, dWd = grads
    assert_close(f64_of(dx), b["dx"], f"{what}: dx")
    assert_close(dWg.cpu().numpy(), b["dWg"], f"{what}: dWg")
    assert_close(dWd.cpu().numpy(), b["dWd"], f"{what}: dWd")
    if spec.gated:
        assert_close(dWu.cpu().numpy(), b["dWu"], f"{what}: dWu")


def _run(spec, inp, ovf_cap, backup_cap, route="sparse"):
    dv = _dev(inp)
    f = tw.TwellFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=ovf_cap)
    y_twell = f(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated, route=route)
    y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    grads = h.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1)
    torch.cuda.synchronize()
    tw.raise_if_device_error(f.status, "TwELL forward")
    tw.raise_if_device_error(h.status, "Hybrid step")
    return f, h, y_twell, y, grads


def test_empty_batch():
    # forwards do nothing; the backward's weight gradients are sums over no tokens: 0
    spec = FFNSpec("empty", T=0, d=256, I=704, W=64, C=8, R=32, seed=3)
    dv = {k: torch.empty((0, spec.d), dtype=torch.bfloat16, device="cuda") for k in ("x", "dy")}
    w = make_inputs(spec.with_(T=4))
    Wg, Wu, Wd = (to_dev(w[k]) for k in ("Wg", "Wu", "Wd"))
    f = tw.TwellFFN(0, spec.d, spec.I, spec.W, spec.C, ovf_cap=0)
    assert f(dv["x"], Wg, Wu, Wd).shape == (0, spec.d)
    h = tw.HybridFFN(0, spec.d, spec.I, spec.W, spec.C, spec.R, 0, gated=True)
    assert h.forward(dv["x"], Wg, Wu, Wd).shape == (0, spec.d)
    dx, dWg, dWu, dWd = h.backward(dv["dy"], dv["x"], Wg, Wu, Wd, spec.l1)
    torch.cuda.synchronize()
    tw.raise_if_device_error(h.status)
    assert dx.shape == (0, spec.d)
    for g in (dWg, dWu, dWd):
        assert not bool(g.any())


@pytest.mark.parametrize("route", ["sparse", "dense"])
@pytest.mark.parametrize("gated", [True, False])
def test_single_token(gated, route):
    """One token. On the dense route every GEMM runs one 256-row unit on a CTA pair
    with a single valid row, and the weight-gradient GEMM has K = 1 (its 64-row K
    boxes read zeros past the token)."""
    spec = FFNSpec("one_token", T=1, d=512, I=1280, gated=gated, mean_active=40, W=128, C=8, R=64, seed=4)
    inp = make_inputs(spec, with_dy=True)
    _, h, y_twell, y, grads = _run(spec, inp, ovf_cap=1, backup_cap=1, route=route)
    assert h.saved.took_dense_route() == (route == "dense")
    _check_against_oracle(spec, inp, y_twell, y, grads, f"one token, {route} route")


def test_tokens_without_active_neurons():
    # about one active neuron in 50 tokens: nearly every row has an empty list
    spec = FFNSpec("idle", T=300, d=256, I=704, mean_active=0.02, W=64, C=8, R=32, seed=6)
    inp = make_inputs(spec, with_dy=True)
    f, h, y_twell, y, grads = _run(spec, inp, ovf_cap=8, backup_cap=8)
    empty = int((h.saved.row_nnz[:spec.T] == 0).sum().item())
    assert empty >= spec.T - 20
    _check_against_oracle(spec, inp, y_twell, y, grads, "idle tokens")


def test_wide_hidden_layer():
    # I = 49216 (769 tiles of 64) is past the 48K columns of the backward count
    # pass's shared-memory histogram, so its column counts go to global atomics;
    # three outlier tokens overflow a tile and go to the dense backup (checked on the
    # oracle's activations when the case was chosen).
    spec = FFNSpec("wide", T=128, d=256, I=49216, mean_active=60, outlier_frac=0.02, W=64, C=8, R=256, seed=8)
    inp = make_inputs(spec, with_dy=True)
    f, h, y_twell, y, grads = _run(spec, inp, ovf_cap=8, backup_cap=8)
    assert int(h.saved.n_backup.item()) == 3
    _check_against_oracle(spec, inp, y_twell, y, grads, "wide hidden layer")


def _bf16(v):
    return ffn.bf16_to_f64(round_to_bf16_bits(np.asarray(v, dtype=np.float32)))


def _f16(v):
    """fp16 (IEEE binary16) rounding, round to nearest even: the Hybrid's storage of u."""
    return np.asarray(v, dtype=np.float64).astype(np.float16).astype(np.float64)


def _close_to_stored_precision(got, ref, what):
    """|got - ref| <= 2^-8 |ref| (the bf16 output) + 2e-3 rms(ref) (fp32 sums, and a
    rare one-ulp difference where the GPU's fp32 g rounds to another bf16 a)."""
    got = np.asarray(got, dtype=np.float64)
    slack = 2e-3 * np.sqrt(np.mean(ref ** 2))
    bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + slack
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements off; first at {np.argwhere(bad)[0].tolist()} "
                           f"got {got[bad][0]} ref {ref[bad][0]}")


@pytest.mark.parametrize("gated", [True, False])
def test_longest_entry_lists(gated):
    # every neuron active: (I / W) * C = 160 * 64 = 10240 entries a token, C = W so no
    # tile overflows, and R = I keeps every row in the ELL part
    spec = FFNSpec("longest", T=24, d=256, I=10240, gated=gated, mean_active=10230, W=64, C=64, R=10240, seed=7)
    inp = make_inputs(spec, with_dy=True)
    f, h, y_twell, y, grads = _run(spec, inp, ovf_cap=0, backup_cap=0)
    nnz = h.saved.row_nnz[:spec.T].cpu().numpy()
    assert nnz.min() >= 10000                   # the lists are (almost) full
    assert int(h.saved.n_backup.item()) == 0
    o = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])
    b = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, fwd=o)
    x, Wg, Wu, Wd, dyv = (ffn.as_f64(inp[k]) for k in ("x", "Wg", "Wu", "Wd", "dy"))
    # With every one of 10240 neurons active, a ~ 3 and the sums are long: the bf16
    # storage of a (TwELL values, Hybrid ELL a) and, in the backward, the fp16 storage
    # of u (Hybrid ELL u) move y, dx and dW by ~0.2 % of their terms' scale, more
    # than 1e-2 (1 + |ref|) allows where an element nearly cancels. The reference
    # therefore stores a in bf16 and u in fp16 as the formats do; the rest is the
    # plain definition in fp64.
    a16 = _bf16(o["a"])
    u = o["u"]
    y_ref = (a16 * u if gated else a16) @ Wd
    _close_to_stored_precision(f64_of(y_twell), y_ref, "TwELL y")
    _close_to_stored_precision(f64_of(y), y_ref, "Hybrid y")
    active = (o["g"] > 0).astype(np.float64)
    dh = dyv @ Wd.T
    dx, dWg, dWu, dWd = grads
    if gated:
        u16 = _f16(u)
        dg = (dh * u16 + spec.l1) * active
        du = dh * a16
        dx_ref = dg @ Wg + du @ Wu
        h16 = a16 * u16
        assert_close(dWu.cpu().numpy(), du.T @ x, "dWu", rel_frob=2e-3, elem=np.inf)
    else:
        dg = (dh + spec.l1) * active
        dx_ref = dg @ Wg
        h16 = a16
    _close_to_stored_precision(f64_of(dx), dx_ref, "dx")
    # The weight gradients sum over the 24 tokens only, so a one-ulp difference in
    # a stored a or u (the GPU rounds its fp32 g and u, the reference its fp64 ones)
    # is not averaged away elementwise. They are checked against the same
    # stored-precision reference by a tight relative Frobenius bound, which a dropped
    # token (~20 %) or neuron column (~1 %) would still exceed.
    assert_close(dWg.cpu().numpy(), dg.T @ x, "dWg", rel_frob=2e-3, elem=np.inf)
    assert_close(dWd.cpu().numpy(), h16.T @ dyv, "dWd", rel_frob=2e-3, elem=np.inf)
    # and against the plain oracle the relative Frobenius bound holds
    assert_close(f64_of(y), o["y"], "Hybrid y (Frobenius)", elem=np.inf)
    assert_close(f64_of(dx), b["dx"], "dx (Frobenius)", elem=np.inf)
    assert_close(dWd.cpu().numpy(), b["dWd"], "dWd (Frobenius)", elem=np.inf)
