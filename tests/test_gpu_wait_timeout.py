"""A bounded pipeline wait that runs out on the GPU, and the context afterwards.

tw_wait_timeout_probe runs the tcgen05 GEMM with the TMA loads of one K block never
issued, so the MMA issuer waits on a stage barrier that nothing will complete (a
flag nothing sets). The wait gives up after the library's limit (1 s): the call must
come back with TW_ETIMEOUT in the status word, within a few seconds, and the next
calls on the same stream must be correct -- nothing faults, traps or hangs. The same
holds on a CTA pair (tw_wait_timeout_probe_pair): rank 0's MMA issuer times out, the
other CTA's waits end by their own limit, and both meet at the closing cluster
barrier."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from activation_sparse_feedforward_gb300 import _lib  # noqa: E402
from gpu_util import assert_close, f64_of, to_dev  # noqa: E402
from oracle import ffn  # noqa: E402
from synthetic import WORKLOADS, make_inputs, round_to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return tw.load()


def test_withheld_stage_times_out_and_the_stream_recovers(lib):
    rng = np.random.default_rng(4)
    M, N, K = 128, 64, 256
    A = round_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    B = round_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    a, b = to_dev(A), to_dev(B)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = tw.new_status()
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.monotonic()
    code = lib.tw_wait_timeout_probe(a.data_ptr(), b.data_ptr(), M, N, K, 1, D.data_ptr(), st.data_ptr(), stream)
    assert code == _lib.TW_OK, lib.tw_status_str(code)
    torch.cuda.synchronize()                 # the kernel returned: no hang, no fault
    elapsed = time.monotonic() - t0
    assert int(st.item()) == _lib.TW_ETIMEOUT
    assert 0.5 < elapsed < 30.0, elapsed     # about one wait limit (1 s), a few at most

    # the same stream, right after: a normal GEMM is exact to fp32 accumulation ...
    st2 = tw.new_status()
    D2 = tw.dense_gemm(a, b, M, N, K, False, False, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64) @ \
        (B.astype(np.uint32) << 16).view(np.float32).astype(np.float64).T
    np.testing.assert_allclose(D2.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)

    # ... and a whole Hybrid training step matches the oracle
    spec = WORKLOADS["tiny_fwd"]
    inp = make_inputs(spec, with_dy=True)
    dv = {k: to_dev(inp[k]) for k in ("x", "Wg", "Wu", "Wd", "dy")}
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap=32, gated=True)
    y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"])
    dx, dWg, dWu, dWd = h.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1)
    torch.cuda.synchronize()
    tw.raise_if_device_error(h.status, "hybrid step after the timeout")
    f = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])
    bw = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, fwd=f)
    assert_close(f64_of(y), f["y"], "y")
    assert_close(f64_of(dx), bw["dx"], "dx")
    assert_close(dWg.cpu().numpy(), bw["dWg"], "dWg")


def test_withheld_stage_times_out_on_a_cta_pair(lib):
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 256
    A = round_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    B = round_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    a, b = to_dev(A), to_dev(B)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = tw.new_status()
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.monotonic()
    code = lib.tw_wait_timeout_probe_pair(a.data_ptr(), b.data_ptr(), M, N, K, 1, D.data_ptr(), st.data_ptr(),
                                          stream)
    assert code == _lib.TW_OK, lib.tw_status_str(code)
    torch.cuda.synchronize()                 # both CTAs returned: no hang, no fault
    elapsed = time.monotonic() - t0
    assert int(st.item()) == _lib.TW_ETIMEOUT
    assert 0.5 < elapsed < 30.0, elapsed     # a few wait limits (1 s each) at most

    # the same stream, right after: the pair GEMM and the single-CTA one are exact to
    # fp32 accumulation ...
    ref = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64) @ \
        (B.astype(np.uint32) << 16).view(np.float32).astype(np.float64).T
    for pair in (True, False):
        st2 = tw.new_status()
        D2 = tw.dense_gemm(a, b, M, N, K, False, False, status=st2, pair=pair)
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        np.testing.assert_allclose(D2.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)

    # ... and a whole Hybrid training step matches the oracle
    spec = WORKLOADS["tiny_fwd"]
    inp = make_inputs(spec, with_dy=True)
    dv = {k: to_dev(inp[k]) for k in ("x", "Wg", "Wu", "Wd", "dy")}
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap=32, gated=True)
    y = h.forward(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"])
    dx = h.backward(dv["dy"], dv["x"], dv["Wg"], dv["Wu"], dv["Wd"], spec.l1)[0]
    torch.cuda.synchronize()
    tw.raise_if_device_error(h.status, "hybrid step after the pair timeout")
    f = ffn.forward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"])
    bw = ffn.backward(inp["x"], inp["Wg"], inp["Wu"], inp["Wd"], inp["dy"], spec.l1, fwd=f)
    assert_close(f64_of(y), f["y"], "y")
    assert_close(f64_of(dx), bw["dx"], "dx")
