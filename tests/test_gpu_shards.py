"""Token sharding emulated on one GPU. A data-parallel step runs the Hybrid forward
and backward on disjoint token shards and sums the shards' weight gradients (the
all-reduce a multi-GPU run would do); y and dx are per token. The result must match
both the unsharded run and the fp64 oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import assert_close, f64_of, to_dev  # noqa: E402
from oracle import ffn  # noqa: E402
from synthetic import FFNSpec, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _step(spec, x, dy, W, backup_cap):
    T = x.shape[0]
    h = tw.HybridFFN(T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated)
    y = h.forward(x, W["Wg"], W["Wu"], W["Wd"]).clone()
    dx, dWg, dWu, dWd = (None if v is None else v.clone()
                         for v in h.backward(dy, x, W["Wg"], W["Wu"], W["Wd"], spec.l1))
    torch.cuda.synchronize()
    tw.raise_if_device_error(h.status)
    return y, dx, dWg, dWu, dWd, h.saved.backup_slot.clone()


@pytest.mark.parametrize("gated", [True, False])
def test_token_shards_sum_to_unsharded_step(gated):
    spec = FFNSpec("shards", T=640, d=512, I=1280, gated=gated, mean_active=18, outlier_frac=0.03, W=128, C=8,
                   R=48, seed=11)
    inp = make_inputs(spec, with_dy=True)
    x, dy = to_dev(inp["x"]), to_dev(inp["dy"])
    W = {k: (to_dev(inp[k]) if inp[k] is not None else None) for k in ("Wg", "Wu", "Wd")}
    full = _step(spec, x, dy, W, backup_cap=spec.T // 4)
    bounds = [0, 256, 640]   # two shards of unequal size
    parts = [_step(spec, x[a:b].contiguous(), dy[a:b].contiguous(), W, backup_cap=(b - a) // 4)
             for a, b in zip(bounds[:-1], bounds[1:])]
    y = torch.cat([p[0] for p in parts])
    dx = torch.cat([p[1] for p in parts])
    dW = [sum(p[i] for p in parts) if parts[0][i] is not None else None for i in (2, 3, 4)]
    # per-token outputs do not depend on the sharding: bit for bit on the ELL rows,
    # up to the split-K summation order of the dense backup GEMMs on the others. Their
    # fp32 partial sums are added by atomics in an order that varies from launch to
    # launch. A reordering of K terms moves an fp32 sum by about sqrt(K) roundings of
    # the sum of its terms' magnitudes (2^-19 of it at K = 1280; outlier rows sum
    # ~10^3 terms of size up to ~0.3), then bf16 rounds: bounded here by
    # 2^-7 |y| + 2^-16 sum|terms| (eight times that size), the scale from the oracle
    ell = (full[5] == -1).cpu().numpy()
    assert ell.sum() > 0 and (~ell).sum() > 0
    assert np.array_equal(f64_of(y)[ell], f64_of(full[0])[ell])
    assert np.array_equal(f64_of(dx)[ell], f64_of(full[1])[ell])
    f = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])
    b = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, fwd=f)
    Wg, Wd = ffn.as_f64(inp["Wg"]), ffn.as_f64(inp["Wd"])
    y_terms = np.abs(f["h"]) @ np.abs(Wd)
    dx_terms = np.abs(b["dg"]) @ np.abs(Wg)
    if gated:
        dx_terms = dx_terms + np.abs(b["du"]) @ np.abs(ffn.as_f64(inp["Wu"]))
    for got, ref, terms, what in ((f64_of(y), f64_of(full[0]), y_terms, "y"),
                                  (f64_of(dx), f64_of(full[1]), dx_terms, "dx")):
        bad = np.abs(got - ref) > 2 ** -7 * np.abs(ref) + 2 ** -16 * terms
        assert not bad.any(), (what, np.argwhere(bad)[:5].tolist(), got[bad][:5], ref[bad][:5])
    # the summed shard gradients match the unsharded ones up to summation order
    for got, ref in zip(dW, full[2:5]):
        if ref is not None:
            assert_close(got.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64), "dW vs unsharded")
    # and the oracle
    assert_close(f64_of(y), f["y"], "y")
    assert_close(f64_of(dx), b["dx"], "dx")
    assert_close(dW[0].cpu().numpy(), b["dWg"], "dWg")
    assert_close(dW[2].cpu().numpy(), b["dWd"], "dWd")
    if gated:
        assert_close(dW[1].cpu().numpy(), b["dWu"], "dWu")
