"""The residual stack workload x_{l+1} = x_l + FFN_l(x_l) through the Hybrid training
forward and backward, layer after layer, against the fp64 oracle applied layer by
layer with the same bf16 rounding of the residual stream (x_{l+1} and the gradient
g_l = g_{l+1} + dx_l are stored in bf16 on both sides)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import assert_close, f64_of, to_dev  # noqa: E402
from oracle import ffn  # noqa: E402
from synthetic import make_stack, round_to_bf16_bits, stack_layer_spec  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _bf16_sum(a_bits, b_f64):
    """bf16(a + bf16(b)): the stack's residual update on bf16 storage."""
    b_bits = round_to_bf16_bits(np.asarray(b_f64, dtype=np.float32))
    return round_to_bf16_bits((ffn.bf16_to_f64(a_bits) + ffn.bf16_to_f64(b_bits)).astype(np.float32))


@pytest.mark.parametrize("route,shared", [("sparse", False), ("auto", True)], ids=["sparse", "auto_shared_scratch"])
def test_residual_stack_matches_oracle(route, shared):
    """With the automatic route the two middle layers (ELL rows of ~13-15 nonzeros, above
    the threshold of 8) take the dense route and the outer ones (~2) the sparse route;
    with a shared scratch every layer uses the same workspaces and y / dx buffers."""
    # four layers sampling the 28-layer activity profile (rising, plateau, falling)
    specs = [stack_layer_spec(l, T=300, d=256, I=704, W=64, C=8, profile_layer=p)
             for l, p in enumerate((0, 9, 18, 27))]
    st = make_stack(specs)
    n = len(specs)
    # ---------------------------------------------------------------- library
    x = to_dev(st["x0"])
    layers, xs = [], []
    scratch = tw.HybridScratch() if shared else None
    for sp, w in zip(specs, st["layers"]):
        W = {k: to_dev(v) for k, v in w.items()}
        h = tw.HybridFFN(sp.T, sp.d, sp.I, sp.W, sp.C, sp.R, sp.T // 4, gated=True, route=route, dense_above=8.0,
                         scratch=scratch)
        y = h.forward(x, W["Wg"], W["Wu"], W["Wd"])
        xs.append(x)
        layers.append((h, W))
        x = x + y
    out = x
    g = to_dev(st["dy"])
    dWs = [None] * n
    for l in reversed(range(n)):
        h, W = layers[l]
        dx, dWg, dWu, dWd = h.backward(g, xs[l], W["Wg"], W["Wu"], W["Wd"], specs[l].l1)
        dWs[l] = (dWg.clone(), dWu.clone(), dWd.clone())
        g = g + dx
    torch.cuda.synchronize()
    for h, _ in layers:
        tw.raise_if_device_error(h.status)
        assert int(h.saved.n_backup.item()) >= 3   # the outlier tokens stay outliers up the stack
    if route == "auto":
        assert [h.saved.took_dense_route() for h, _ in layers] == [False, True, True, False]
    # ---------------------------------------------------------------- oracle
    xo = st["x0"]
    xos, fs = [], []
    for sp, w in zip(specs, st["layers"]):
        f = ffn.forward(xo, w["Wg"], w["Wu"], w["Wd"])
        xos.append(xo)
        fs.append(f)
        xo = _bf16_sum(xo, f["y"])
    assert_close(f64_of(out), ffn.bf16_to_f64(xo), "stack output")
    go = st["dy"]
    for l in reversed(range(n)):
        w = st["layers"][l]
        b = ffn.backward(xos[l], w["Wg"], w["Wu"], w["Wd"], go, specs[l].l1, fwd=fs[l])
        for got, name in zip(dWs[l], ("dWg", "dWu", "dWd")):
            assert_close(got.cpu().numpy(), b[name], f"layer {l} {name}")
        go = _bf16_sum(go, b["dx"])
    assert_close(f64_of(g), ffn.bf16_to_f64(go), "gradient at the stack input")
