"""GPU parity of the whole path against the fp64 oracle: TwELL inference forward,
Hybrid training forward (including the saved Hybrid) and backward."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import (assert_close, assert_close_by_row_class, bits_of, f64_of, kernel_active_set,  # noqa: E402
                      oracle_on_kernel_branch, to_dev)
from oracle import ffn, formats  # noqa: E402
from synthetic import FFNSpec, WORKLOADS, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _dev_inputs(inp):
    return {k: to_dev(v) for k, v in inp.items() if k in ("x", "Wg", "Wu", "Wd", "dy")}


MEDIUM = [
    WORKLOADS["tiny_fwd"],
    FFNSpec("med_gated", T=777, d=512, I=1280, mean_active=20, outlier_frac=0.03, W=128, C=8, R=48, seed=5),
    FFNSpec("med_nongated", T=600, d=768, I=1024, gated=False, mean_active=25, outlier_frac=0.02, W=64, C=8,
            R=64, seed=6),
    FFNSpec("med_w64_d2048", T=300, d=2048, I=704, mean_active=10, outlier_frac=0.02, W=64, C=6, R=24, seed=7),
    # dense-ish regime: long ELL rows (R = 320) and wide TwELL tiles (C = 32)
    FFNSpec("med_long_rows", T=513, d=512, I=1280, mean_active=200, outlier_frac=0.02, W=128, C=32, R=320, seed=8),
    # C = 16 on 128-wide tiles (the vector slot loads of the forward's list building)
    FFNSpec("med_c16", T=700, d=512, I=1024, mean_active=14, outlier_frac=0.02, W=128, C=16, R=64, seed=12),
]


@pytest.mark.parametrize("spec", MEDIUM, ids=lambda s: s.name)
def test_twell_forward_matches_oracle(spec):
    inp = make_inputs(spec)
    dv = _dev_inputs(inp)
    y, twl, status = tw.twell_ffn_fwd(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.W, spec.C)
    tw.raise_if_device_error(status)
    ref = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])
    assert_close(f64_of(y), ref["y"], "y")
    # overflow rows were served by the dense path: check them on their own too
    n = int(twl.n_ovf.item())
    rows = twl.ovf_rows[:n].cpu().numpy()
    assert n > 0 and set(inp["outliers"].tolist()) <= set(rows.tolist())
    assert_close(f64_of(y)[rows], ref["y"][rows], "y (overflow rows)")


def test_twell_forward_full_size_sampled():
    spec = WORKLOADS["gated_fwd_d2048_i5632"]
    inp = make_inputs(spec)
    dv = _dev_inputs(inp)
    y, twl, status = tw.twell_ffn_fwd(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.W, spec.C)
    tw.raise_if_device_error(status)
    rows = np.unique(np.concatenate([np.arange(3, spec.T, 509), inp["outliers"][:12], [0, spec.T - 1]]))
    ref = ffn.forward(inp["x"][rows], inp["Wg"], inp["Wu"], inp["Wd"])
    assert_close(f64_of(y)[rows], ref["y"], "y (sampled rows)")


def test_twell_forward_nongated_full_size_sampled():
    spec = WORKLOADS["nongated_fwd_d2048_i8192"]
    inp = make_inputs(spec)
    dv = _dev_inputs(inp)
    y, twl, status = tw.twell_ffn_fwd(dv["x"], dv["Wg"], None, dv["Wd"], spec.W, spec.C)
    tw.raise_if_device_error(status)
    rows = np.unique(np.concatenate([np.arange(1, spec.T, 1021), inp["outliers"][:8]]))
    ref = ffn.forward(inp["x"][rows], inp["Wg"], None, inp["Wd"])
    assert_close(f64_of(y)[rows], ref["y"], "y (sampled rows)")


def test_twell_forward_capacity_exceeded_is_reported():
    spec = WORKLOADS["tiny_fwd"]
    inp = make_inputs(spec)
    dv = _dev_inputs(inp)
    f = tw.TwellFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=2)   # 5 outliers overflow
    f(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"])
    with pytest.raises(tw.TwellError, match="TW_ECAPACITY"):
        tw.raise_if_device_error(f.status)


def _run_hybrid(spec, inp, backup_cap, l1=None, dy_zero=False):
    dv = _dev_inputs(inp)
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated)
    y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"])
    dy = torch.zeros_like(dv["dy"]) if dy_zero else dv["dy"]
    grads = h.backward(dy, dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1 if l1 is None else l1)
    torch.cuda.synchronize()
    tw.raise_if_device_error(h.status)
    return h, y, grads


@pytest.mark.parametrize("spec", MEDIUM, ids=lambda s: s.name)
@pytest.mark.parametrize("l1", [2e-5, 0.05])
def test_hybrid_forward_backward_match_oracle(spec, l1):
    inp = make_inputs(spec, with_dy=True)
    h, y, (dx, dWg, dWu, dWd) = _run_hybrid(spec, inp, backup_cap=spec.T // 4, l1=l1)
    f = oracle_on_kernel_branch(ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"]),
                                kernel_active_set(h.saved), inp["Wd"])
    b = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], l1, fwd=f)
    backup = h.saved.backup_tok[:int(h.saved.n_backup.item())].cpu().numpy()
    assert_close_by_row_class(f64_of(y), f["y"], backup, "y")
    assert_close_by_row_class(f64_of(dx), b["dx"], backup, "dx")
    assert_close(dWg.cpu().numpy(), b["dWg"], "dWg")
    assert_close(dWd.cpu().numpy(), b["dWd"], "dWd")
    if spec.gated:
        assert_close(dWu.cpu().numpy(), b["dWu"], "dWu")
    nb = int(h.saved.n_backup.item())
    assert 0 < nb <= spec.T // 4


@pytest.mark.parametrize("backup_cap", [0, 64])
def test_hybrid_without_backup_rows(backup_cap):
    """No row needs the dense backup: the weight gradients come from the ELL pass
    alone, whether or not backup capacity exists."""
    spec = FFNSpec("no_backup", T=200, d=512, I=768, mean_active=6, outlier_frac=0.0, W=64, C=12, R=96, seed=9)
    inp = make_inputs(spec, with_dy=True)
    h, y, (dx, dWg, dWu, dWd) = _run_hybrid(spec, inp, backup_cap=backup_cap)
    assert int(h.saved.n_backup.item()) == 0
    f = oracle_on_kernel_branch(ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"]),
                                kernel_active_set(h.saved), inp["Wd"])
    b = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, fwd=f)
    assert_close(f64_of(y), f["y"], "y")
    assert_close(f64_of(dx), b["dx"], "dx")
    assert_close(dWg.cpu().numpy(), b["dWg"], "dWg")
    assert_close(dWu.cpu().numpy(), b["dWu"], "dWu")
    assert_close(dWd.cpu().numpy(), b["dWd"], "dWd")


def test_hybrid_l1_only_gradient_closed_form():
    """dy = 0, l1 = 1: dWg[j] = sum of x_t over tokens where neuron j fires,
    dx_t = sum of Wg[j] over the neurons token t fires, dWu = dWd = 0."""
    spec = MEDIUM[1]
    inp = make_inputs(spec, with_dy=True)
    h, y, (dx, dWg, dWu, dWd) = _run_hybrid(spec, inp, backup_cap=spec.T // 4, l1=1.0, dy_zero=True)
    x = ffn.bf16_to_f64(inp["x"])
    Wg = ffn.bf16_to_f64(inp["Wg"])
    act = (x @ Wg.T) > 0
    assert_close(dWg.cpu().numpy(), act.T.astype(np.float64) @ x, "dWg (L1 only)")
    assert_close(f64_of(dx), act.astype(np.float64) @ Wg, "dx (L1 only)")
    assert float(dWu.abs().max()) == 0.0 and float(dWd.abs().max()) == 0.0


def test_hybrid_saved_format_matches_oracle_packing():
    spec = MEDIUM[1]
    inp = make_inputs(spec, with_dy=True)
    h, y, _ = _run_hybrid(spec, inp, backup_cap=spec.T // 4)
    # reference Hybrid built by the oracle from the gate kernel's own activations
    _, dense = tw.twell_gate_pack(to_dev(inp["x"]), to_dev(inp["Wg"]), spec.W, spec.C, want_dense=True)
    A = bits_of(dense)
    U = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])["u"]
    ref = formats.hybrid_pack(A, U, spec.W, spec.C, spec.R)
    s = h.saved
    np.testing.assert_array_equal(s.row_nnz.cpu().numpy(), ref["row_nnz"])
    np.testing.assert_array_equal(s.backup_slot.cpu().numpy(), ref["backup_slot"])
    np.testing.assert_array_equal(s.ell_nnz.cpu().numpy(), ref["ell_nnz"])
    nb = int(s.n_backup.item())
    np.testing.assert_array_equal(s.backup_tok[:nb].cpu().numpy(), ref["backup_tok"])
    v = ref["ell_valid"]
    np.testing.assert_array_equal(s.ell_idx.cpu().numpy().view(np.uint16).astype(np.int64)[v], ref["ell_idx"][v])
    np.testing.assert_array_equal(bits_of(s.ell_a)[v], ref["ell_a"][v])
    assert_close(s.ell_u.double().cpu().numpy()[v], ref["ell_u"][v], "ell u")
    # backup rows hold fp32 a = ReLU(g) and u. The backup's own GEMM sums g in another
    # order than the gate kernel (a few backup rows take split-K units), so a rounds to
    # the TwELL value except where the two fp32 sums straddle a bf16 rounding boundary:
    # there the two bf16 values are adjacent (bit patterns one apart, same sign); where
    # g is within summation-order error of 0, ReLU may keep a tiny a on one side only
    a32 = s.backup_a[:nb].cpu().numpy()
    a_b = bits_of(s.backup_a[:nb].to(torch.bfloat16)).astype(np.int32)
    diff = np.abs(a_b - ref["backup_a"].astype(np.int32))
    diff[(np.abs(a32) < 1e-6) & (np.abs(ffn.bf16_to_f64(ref["backup_a"])) < 1e-6)] = 0
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3, (int(diff.max()), float((diff > 0).mean()))
    assert_close(s.backup_a[:nb].double().cpu().numpy(), ffn.bf16_to_f64(ref["backup_a"]), "backup a")
    assert_close(s.backup_u[:nb].cpu().numpy(), ref["backup_u"], "backup u")


@pytest.mark.parametrize("name,backup_cap", [("train_d2048_i5632_m29_o1", 256),
                                             ("train_d2048_i5632_m108_o5", 1280),
                                             ("train_d2048_i5632_m911_o0", 16384)])
def test_hybrid_full_size_sampled(name, backup_cap):
    spec = WORKLOADS[name]
    inp = make_inputs(spec, with_dy=True)
    h, y, (dx, dWg, dWu, dWd) = _run_hybrid(spec, inp, backup_cap=backup_cap)
    rows = np.unique(np.concatenate([np.arange(5, spec.T, 1013), inp["outliers"][:10], [spec.T - 1]]))
    f = oracle_on_kernel_branch(ffn.forward(inp["x"][rows], inp["Wg"], inp["Wu"], inp["Wd"]),
                                kernel_active_set(h.saved)[rows], inp["Wd"])
    b = ffn.backward(inp["x"][rows], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"][rows], spec.l1, fwd=f)
    assert_close(f64_of(y)[rows], f["y"], "y (sampled rows)")
    assert_close(f64_of(dx)[rows], b["dx"], "dx (sampled rows)")
    J = np.array([0, 1, 17, 1000, 2047, 4096, 5631])
    r = ffn.backward_weight_rows(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, J)
    assert_close(dWg[J].cpu().numpy(), r["dWg"], "dWg (sampled neurons)")
    assert_close(dWu[J].cpu().numpy(), r["dWu"], "dWu (sampled neurons)")
    assert_close(dWd[J].cpu().numpy(), r["dWd"], "dWd (sampled neurons)")
    assert int(h.saved.n_backup.item()) >= len(inp["outliers"])


@pytest.mark.parametrize("spec", [MEDIUM[0], MEDIUM[2], WORKLOADS["gated_fwd_d2048_i5632"]], ids=lambda s: s.name)
def test_unfused_pipeline_equals_fused_forward(spec):
    """Dense a through memory, then the standalone packer, then the sparse part give
    the fused forward's y: bit for bit on the rows the sparse kernel serves (same
    GEMM, same canonical TwELL, same sparse kernel), and on the overflow rows up to
    the order of the split-K fp32 additions of their dense down projection; both
    match the oracle."""
    inp = make_inputs(spec)
    dv = _dev_inputs(inp)
    f = tw.TwellFFN(spec.T, spec.d, spec.I, spec.W, spec.C)
    y_fused = f(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    st = tw.new_status()
    a = tw.gate_relu_dense(dv["x"], dv["Wg"], status=st)
    packed = tw.twell_pack(a, spec.W, spec.C, status=st)
    sp = tw.TwellSparseFFN(spec.T, spec.d, spec.I, spec.W, spec.C)
    y_unfused = sp(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], packed)
    torch.cuda.synchronize()
    for s_ in (f.status, st, sp.status):
        tw.raise_if_device_error(s_)
    sparse_rows = f.tw.ovf == 0
    assert torch.equal(y_unfused[sparse_rows], y_fused[sparse_rows])
    dense_rows = ~sparse_rows
    if bool(dense_rows.any()):
        # the same fp32 sums in another order, then bf16: a few one-ulp flips at most
        assert_close(f64_of(y_unfused[dense_rows]), f64_of(y_fused[dense_rows]), "overflow rows", rel_frob=1e-3)
    for name in ("cnt", "row_nnz", "ovf"):
        assert torch.equal(getattr(packed, name), getattr(f.tw, name)), name
    # slots past a tile's count are padding (unspecified)
    valid = torch.arange(spec.C, device="cuda")[None, None, :] < packed.cnt.long().clamp(max=spec.C)[:, :, None]
    for name in ("val", "idx"):
        assert torch.equal(getattr(packed, name)[valid], getattr(f.tw, name)[valid]), name
    rows = np.unique(np.concatenate([np.arange(0, spec.T, max(1, spec.T // 300)), inp["outliers"][:8]]))
    ref = ffn.forward(inp["x"][rows], inp["Wg"], inp["Wu"], inp["Wd"])
    assert_close(f64_of(y_unfused)[rows], ref["y"], "y (unfused)")


def test_sparse_part_reports_overflow_beyond_capacity():
    spec = WORKLOADS["tiny_fwd"]
    inp = make_inputs(spec)
    dv = _dev_inputs(inp)
    packed = tw.twell_pack(tw.gate_relu_dense(dv["x"], dv["Wg"]), spec.W, spec.C)
    sp = tw.TwellSparseFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=2)   # 5 rows overflow
    sp(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], packed)
    with pytest.raises(tw.TwellError, match="TW_ECAPACITY"):
        tw.raise_if_device_error(sp.status)


@pytest.mark.parametrize("spec", [MEDIUM[0], MEDIUM[1]], ids=lambda s: s.name)
def test_workspaces_need_no_initial_contents(spec):
    """The library's workspaces hold, among other scratch, the device counters from
    which the gather kernels take their tokens and items; kernels earlier in the same
    call zero them. Workspaces filled with 0xFF bytes (every counter -1, every list
    garbage) must give the same results as fresh ones, twice in a row."""
    inp = make_inputs(spec, with_dy=True)
    dv = _dev_inputs(inp)
    ref = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, spec.T // 4, gated=spec.gated)
    y_ref = ref.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    g_ref = [t.clone() for t in ref.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1)]
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, spec.T // 4, gated=spec.gated)
    f = tw.TwellFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=spec.T // 4)
    y_twell_ref = f(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    for _ in range(2):
        for ws in (h.fwd_ws, h.bwd_ws, f.ws):
            ws.fill_(0xFF)
        y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"])
        grads = h.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1)
        y_twell = f(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"])
        torch.cuda.synchronize()
        for s_ in (ref.status, h.status, f.status):
            tw.raise_if_device_error(s_)
        # the sparse rows' arithmetic is fixed; split-K sums of the dense rows and the
        # column order of the weight-gradient records may differ in the last bits
        assert_close(f64_of(y), f64_of(y_ref), "y with dirty workspaces", rel_frob=1e-3)
        assert_close(f64_of(y_twell), f64_of(y_twell_ref), "TwELL y with dirty workspaces", rel_frob=1e-3)
        for got, want, name in zip(grads, g_ref, ("dx", "dWg", "dWu", "dWd")):
            if got is None:
                continue
            assert_close(got.float().cpu().numpy(), want.float().cpu().numpy(), f"{name} with dirty workspaces",
                         rel_frob=1e-3)


def test_sparse_rows_are_bitwise_reproducible():
    """The token kernels take their tokens from a counter, so which CTA handles a
    token changes from run to run, but a token's arithmetic does not: its list is in
    neuron order and its warps' partial sums are added in a fixed order. Two runs
    give the same TwELL / Hybrid contents and the same y and dx on the ELL rows, bit
    for bit (the dense rows' split-K sums and the weight gradients may differ in the
    last bits)."""
    spec = MEDIUM[0]
    inp = make_inputs(spec, with_dy=True)
    dv = _dev_inputs(inp)
    runs = []
    for _ in range(2):
        h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, spec.T // 4, gated=spec.gated)
        y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
        dx = h.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1)[0].clone()
        torch.cuda.synchronize()
        tw.raise_if_device_error(h.status)
        runs.append((h, y, dx))
    (h0, y0, dx0), (h1, y1, dx1) = runs
    ell = h0.saved.backup_slot[:spec.T] == -1
    assert bool(ell.any()) and bool((~ell).any())
    assert torch.equal(y0[ell], y1[ell])
    assert torch.equal(dx0[ell], dx1[ell])
    for name in ("row_nnz", "ell_nnz", "backup_slot", "n_backup"):
        assert torch.equal(getattr(h0.saved, name), getattr(h1.saved, name)), name
    n = h0.saved.ell_nnz[:spec.T].long()
    valid = torch.arange(spec.R, device="cuda")[None, :] < n[:, None]
    for name in ("ell_idx", "ell_a", "ell_u"):
        a0 = getattr(h0.saved, name).view(torch.int16)
        a1 = getattr(h1.saved, name).view(torch.int16)
        assert torch.equal(a0[valid], a1[valid]), name
