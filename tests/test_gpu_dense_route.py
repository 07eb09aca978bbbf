"""GPU parity of the dense route of the Hybrid training step: the ELL rows' up and
down projections and their backward as dense tensor-core GEMMs over all neurons,
with the TwELL / Hybrid masks applied in the GEMM epilogues, against the fp64
oracle at the usual tolerances; the saved Hybrid equals the sparse route's; the
automatic route is decided on the device from the rows' activity (an ELL row counts
its nonzeros, a backup row twice the threshold)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import (assert_close, assert_close_by_row_class, bits_of, f64_of, kernel_active_set,  # noqa: E402
                      oracle_on_kernel_branch, to_dev)
from oracle import ffn  # noqa: E402
from synthetic import FFNSpec, WORKLOADS, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


CASES = [
    FFNSpec("dense_gated", T=777, d=512, I=1280, mean_active=40, outlier_frac=0.03, W=128, C=16, R=96, seed=21),
    FFNSpec("dense_nongated", T=600, d=768, I=1024, gated=False, mean_active=30, outlier_frac=0.02, W=64, C=8,
            R=64, seed=22),
    # I = 704: 64-wide column tiles in the up and grad GEMMs; d = 2048
    FFNSpec("dense_i704_d2048", T=300, d=2048, I=704, mean_active=20, outlier_frac=0.02, W=64, C=8, R=48, seed=23),
    # long ELL rows (the grad epilogue's row search and walk over many entries per tile)
    FFNSpec("dense_long_rows", T=513, d=512, I=1280, mean_active=200, outlier_frac=0.02, W=128, C=40, R=320,
            seed=24),
    # 8 x 22 = 176 units of 256 x 256 on CTA pairs in the gate, up and grad GEMMs (more
    # than one round, the last partly empty); d = 256: one column of units for down, dx
    FFNSpec("dense_mixed_tail", T=2048, d=256, I=5632, mean_active=100, outlier_frac=0.01, W=128, C=16, R=224,
            seed=30),
    # I = 1152: 128-wide column tiles, one CTA each, in the gate, up and grad GEMMs;
    # 18 x 9 = 162 tiles on 152 SMs, so the last 10 run as half-width units
    FFNSpec("dense_i1152_tail", T=2300, d=512, I=1152, mean_active=60, outlier_frac=0.01, W=128, C=16, R=160,
            seed=31),
]


def _dev(inp):
    return {k: to_dev(v) for k, v in inp.items() if k in ("x", "Wg", "Wu", "Wd", "dy")}


def _step(spec, dv, route, l1, backup_cap, dense_above=64.0):
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated, route=route,
                     dense_above=dense_above)
    y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    grads = [None if g is None else g.clone()
             for g in h.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], l1)]
    torch.cuda.synchronize()
    tw.raise_if_device_error(h.status, f"{route} route")
    return h, y, grads


def _oracle(inp, h, l1, rows=None):
    """Oracle forward and backward on the kernel's side of the ReLU kink (rows: a
    sample of the tokens)."""
    x, dyi = (inp["x"], inp["dy"]) if rows is None else (inp["x"][rows], inp["dy"][rows])
    act = kernel_active_set(h.saved)
    f = oracle_on_kernel_branch(ffn.forward(x, inp["Wg"], inp["Wu"], inp["Wd"]),
                                act if rows is None else act[rows], inp["Wd"])
    return f, ffn.backward(x, inp["Wg"], inp["Wu"], inp["Wd"], dyi, l1, fwd=f)


def _check_oracle(spec, inp, h, y, grads, l1, rows=None):
    dx, dWg, dWu, dWd = grads
    f, b = _oracle(inp, h, l1, rows)
    yy, dd = (f64_of(y), f64_of(dx)) if rows is None else (f64_of(y)[rows], f64_of(dx)[rows])
    assert_close(yy, f["y"], "y")
    assert_close(dd, b["dx"], "dx")
    if rows is None:
        assert_close(dWg.cpu().numpy(), b["dWg"], "dWg")
        assert_close(dWd.cpu().numpy(), b["dWd"], "dWd")
        if spec.gated:
            assert_close(dWu.cpu().numpy(), b["dWu"], "dWu")


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
@pytest.mark.parametrize("l1", [2e-5, 0.05])
def test_dense_route_matches_oracle(spec, l1):
    inp = make_inputs(spec, with_dy=True)
    h, y, grads = _step(spec, _dev(inp), "dense", l1, spec.T // 4)
    assert h.saved.took_dense_route()
    nb = int(h.saved.n_backup.item())
    assert 0 < nb <= spec.T // 4
    _check_oracle(spec, inp, h, y, grads, l1)
    # y and dx of the ELL rows and of the backup rows, each class on its own
    f, b = _oracle(inp, h, l1)
    backup = h.saved.backup_tok[:nb].cpu().numpy()
    assert_close_by_row_class(f64_of(y), f["y"], backup, "y")
    assert_close_by_row_class(f64_of(grads[0]), b["dx"], backup, "dx")


@pytest.mark.parametrize("spec", CASES[:2], ids=lambda s: s.name)
def test_dense_route_without_backup_capacity_rows(spec):
    """No backup rows: the dense weight-gradient GEMM writes dW instead of adding."""
    spec = spec.with_(outlier_frac=0.0, R=spec.I)
    inp = make_inputs(spec, with_dy=True)
    h, y, grads = _step(spec, _dev(inp), "dense", spec.l1, 0)
    assert int(h.saved.n_backup.item()) == 0
    _check_oracle(spec, inp, h, y, grads, spec.l1)


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_dense_route_saves_the_sparse_routes_hybrid(spec):
    inp = make_inputs(spec, with_dy=True)
    dv = _dev(inp)
    hs, ys, gs = _step(spec, dv, "sparse", spec.l1, spec.T // 4)
    hd, yd, gd = _step(spec, dv, "dense", spec.l1, spec.T // 4)
    for name in ("row_nnz", "ell_nnz", "backup_slot", "n_backup"):
        assert torch.equal(getattr(hs.saved, name), getattr(hd.saved, name)), name
    nb = int(hs.saved.n_backup.item())
    assert torch.equal(hs.saved.backup_tok[:nb], hd.saved.backup_tok[:nb])
    n = hs.saved.ell_nnz[:spec.T].long()
    valid = (torch.arange(spec.R, device="cuda")[None, :] < n[:, None]).cpu().numpy()
    for name in ("ell_idx", "ell_a"):
        np.testing.assert_array_equal(bits_of(getattr(hs.saved, name))[valid], bits_of(getattr(hd.saved, name))[valid])
    if spec.gated:
        # u: the same fp32 dot product of d terms summed in another order, rounded to
        # fp16 once: one fp16 unit in the last place apart (adjacent fp16 values of one
        # sign have adjacent bit patterns), or, where the sum cancels to a small value,
        # apart by no more than the summation-order error of terms of size ~|x||Wu|
        bs = hs.saved.ell_u.view(torch.int16).cpu().numpy().astype(np.int32)[valid]
        bd = hd.saved.ell_u.view(torch.int16).cpu().numpy().astype(np.int32)[valid]
        us = hs.saved.ell_u.double().cpu().numpy()[valid]
        ud = hd.saved.ell_u.double().cpu().numpy()[valid]
        ok = (np.abs(bs - bd) <= 1) | (np.abs(us - ud) <= 1e-5)
        bad = np.flatnonzero(~ok)
        assert bad.size == 0, (f"{bad.size} of {ok.size} u values differ by more than one fp16 ulp; first: "
                               f"{[(float(us[i]), float(ud[i])) for i in bad[:5]]}")
    # the two routes' outputs agree with each other as closely as each with the oracle
    assert_close(f64_of(yd), f64_of(ys), "y: dense vs sparse route")
    assert_close(f64_of(gd[0]), f64_of(gs[0]), "dx: dense vs sparse route")


def _route_work(h, T, dense_above):
    """The automatic route's measure: mean over rows of the ELL nonzeros, a backup row
    counting 2 dense_above."""
    ell = h.saved.ell_nnz[:T].double()
    backup = (h.saved.backup_slot[:T] != -1)
    return float((torch.where(backup, torch.full_like(ell, 2.0 * dense_above), ell)).mean())


@pytest.mark.parametrize("dense_above,expect_dense", [(10.0, True), (1000.0, False)])
def test_auto_route_is_decided_on_the_device(dense_above, expect_dense):
    spec = CASES[0]                                   # ELL rows hold ~40 nonzeros on average
    inp = make_inputs(spec, with_dy=True)
    h, y, grads = _step(spec, _dev(inp), "auto", spec.l1, spec.T // 4, dense_above=dense_above)
    assert h.saved.took_dense_route() == expect_dense
    assert (_route_work(h, spec.T, dense_above) > dense_above) == expect_dense
    _check_oracle(spec, inp, h, y, grads, spec.l1)


# every row overflows its TwELL (~19 nonzeros per 64-wide tile against C = 4): the
# whole layer is backup rows
ALL_BACKUP = [
    FFNSpec("all_backup_gated", T=300, d=512, I=1024, mean_active=300, outlier_frac=0.0, W=64, C=4, R=64, seed=25),
    FFNSpec("all_backup_nongated", T=260, d=768, I=1024, gated=False, mean_active=300, outlier_frac=0.0, W=64,
            C=4, R=64, seed=26),
]


# backups above 512 rows: a and u stored by the grouped full-width launch (the dense
# route's up GEMM saving u), rather than the split-K form
LARGE_BACKUP = [
    FFNSpec("large_backup_gated", T=700, d=512, I=1024, mean_active=300, outlier_frac=0.0, W=64, C=4, R=64, seed=27),
    FFNSpec("large_backup_nongated", T=660, d=768, I=1024, gated=False, mean_active=300, outlier_frac=0.0, W=64,
            C=4, R=64, seed=28),
    # a mix: 60 % outliers over ordinary rows, so ELL rows and backup rows share tiles
    FFNSpec("large_backup_mixed", T=900, d=512, I=1280, mean_active=40, outlier_frac=0.6, W=128, C=16, R=96,
            seed=29),
]


@pytest.mark.parametrize("route", ["sparse", "dense"])
@pytest.mark.parametrize("spec", LARGE_BACKUP, ids=lambda s: s.name)
def test_large_backup_matches_oracle(spec, route):
    inp = make_inputs(spec, with_dy=True)
    h, y, grads = _step(spec, _dev(inp), route, spec.l1, spec.T)
    nb = int(h.saved.n_backup.item())
    assert nb > 512, nb
    _check_oracle(spec, inp, h, y, grads, spec.l1)
    # the saved fp32 rows: a = ReLU(g) and u of the backup tokens
    rows = h.saved.backup_tok[:nb].cpu().numpy()
    f = ffn.forward(inp["x"][rows], inp["Wg"], inp["Wu"], inp["Wd"])
    assert_close(h.saved.backup_a[:nb].double().cpu().numpy(), f["a"], "backup a")
    if spec.gated:
        assert_close(h.saved.backup_u[:nb].double().cpu().numpy(), f["u"], "backup u")


@pytest.mark.parametrize("spec", ALL_BACKUP, ids=lambda s: s.name)
def test_auto_route_takes_the_dense_route_when_every_row_is_backup(spec):
    """No ELL rows: the sparse route would run the whole layer on the split-operand
    backup GEMMs; the automatic route takes the dense route, whose forward forms the
    backup rows' h from their saved fp32 a, and both agree with the oracle."""
    inp = make_inputs(spec, with_dy=True)
    dv = _dev(inp)
    h, y, grads = _step(spec, dv, "auto", spec.l1, spec.T)
    assert int(h.saved.n_backup.item()) == spec.T
    assert h.saved.took_dense_route()
    assert _route_work(h, spec.T, 64.0) == 128.0
    _check_oracle(spec, inp, h, y, grads, spec.l1)
    hs, ys, gs = _step(spec, dv, "sparse", spec.l1, spec.T)
    assert not hs.saved.took_dense_route()
    _check_oracle(spec, inp, hs, ys, gs, spec.l1)
    # the saved fp32 rows do not depend on the route: the same sums, whose split-K
    # partials are added by atomics in an order that varies between launches, so they
    # agree to the size of a reordering of d terms (about sqrt(d) fp32 roundings of the
    # terms' magnitude sum; allowed: eight times that, 2^-16 of it at d = 512-768)
    nb = spec.T
    x = ffn.as_f64(inp["x"])
    for got, ref, W in ((hs.saved.backup_a, h.saved.backup_a, inp["Wg"]),
                        (hs.saved.backup_u, h.saved.backup_u, inp["Wu"] if spec.gated else None)):
        if W is None:
            continue
        terms = np.abs(x) @ np.abs(ffn.as_f64(W)).T
        g, r = got[:nb].double().cpu().numpy(), ref[:nb].double().cpu().numpy()
        assert (np.abs(g - r) <= 1e-4 * np.abs(r) + 2 ** -16 * terms[:nb]).all()


@pytest.mark.parametrize("name,backup_cap", [("train_d2048_i5632_m108_o5", 1280),
                                             ("train_d2048_i5632_m108_o0", 128)])
def test_dense_route_full_size_sampled(name, backup_cap):
    spec = WORKLOADS[name]
    inp = make_inputs(spec, with_dy=True)
    h, y, grads = _step(spec, _dev(inp), "dense", spec.l1, backup_cap)
    assert h.saved.took_dense_route()
    nb = int(h.saved.n_backup.item())
    assert len(inp["outliers"]) <= nb <= backup_cap
    assert int(h.saved.ell_nnz.sum().item()) > 100 * (spec.T - nb)     # ELL rows of ~108 nonzeros
    rows = np.unique(np.concatenate([np.arange(7, spec.T, 1031), inp["outliers"][:10], [spec.T - 1]]))
    _check_oracle(spec, inp, h, y, grads, spec.l1, rows=rows)
    J = np.array([0, 3, 999, 2048, 4095, 5631])
    r = ffn.backward_weight_rows(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, J)
    dx, dWg, dWu, dWd = grads
    assert_close(dWg[J].cpu().numpy(), r["dWg"], "dWg (sampled neurons)")
    assert_close(dWu[J].cpu().numpy(), r["dWu"], "dWu (sampled neurons)")
    assert_close(dWd[J].cpu().numpy(), r["dWd"], "dWd (sampled neurons)")
