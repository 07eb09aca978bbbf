"""twell_ffn_fwd_fixed_scratch, the TwELL inference forward for callers that cannot
allocate device memory (it takes its scratch from a fixed device array inside the
library instead of a caller workspace), must give what twell_ffn_fwd gives.

Called through the C ABI, twice in a row on the same shape (the second call finds
the first call's data left in the shared array), and compared with the workspace
entry point within the parity tolerance used by the other GPU tests. Kept in a file
of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from activation_sparse_feedforward_gb300 import _lib  # noqa: E402
from gpu_util import assert_close, f64_of, to_dev  # noqa: E402
from synthetic import FFNSpec, WORKLOADS, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return tw.load()


def _fixed_scratch_forward(L, dv, spec, ovf_cap):
    twl = tw.TwELL.empty(spec.T, spec.I, spec.W, spec.C)
    y = torch.empty((spec.T, spec.d), dtype=torch.bfloat16, device="cuda")
    status = tw.new_status()
    s = twl.struct()
    wu = dv["Wu"].data_ptr() if dv["Wu"] is not None else None
    code = L.twell_ffn_fwd_fixed_scratch(dv["x"].data_ptr(), dv["Wg"].data_ptr(), wu, dv["Wd"].data_ptr(),
                                         spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap, ctypes.byref(s),
                                         y.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == _lib.TW_OK, L.tw_status_str(code)
    torch.cuda.synchronize()
    tw.raise_if_device_error(status)
    return y, twl


@pytest.mark.parametrize("spec,ovf_cap", [
    (WORKLOADS["tiny_fwd"], 64),
    (FFNSpec("fixed_ragged", T=777, d=512, I=1280, mean_active=20, outlier_frac=0.03, W=128, C=8, seed=5), 128),
    (WORKLOADS["gated_fwd_d2048_i5632"], 512),
], ids=["tiny", "ragged", "d2048_i5632"])
def test_fixed_scratch_matches_workspace_entry_point(lib, spec, ovf_cap):
    inp = make_inputs(spec)
    dv = {k: to_dev(inp[k]) for k in ("x", "Wg", "Wu", "Wd")}
    ref = tw.TwellFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=ovf_cap)
    y_ref = ref(dv["x"], dv["Wg"], dv["Wu"], dv["Wd"]).clone()
    torch.cuda.synchronize()
    tw.raise_if_device_error(ref.status)
    n_ref = int(ref.tw.n_ovf.item())
    assert n_ref > 0                                 # the dense overflow path (the scratch user) runs
    for call in range(2):
        y, twl = _fixed_scratch_forward(lib, dv, spec, ovf_cap)
        assert_close(f64_of(y), f64_of(y_ref), f"y, fixed-scratch call {call + 1}")
        assert int(twl.n_ovf.item()) == n_ref
        np.testing.assert_array_equal(twl.ovf_rows[:n_ref].cpu().numpy(), ref.tw.ovf_rows[:n_ref].cpu().numpy())


def test_fixed_scratch_rejects_shapes_beyond_its_size(lib):
    # 513 overflow rows at d = 2048, I = 5632 need more than the 20 MiB array: refused on the
    # host before anything is enqueued. Every buffer is a real device buffer of its full
    # size, so even a call that did run would stay inside them.
    T, d, I, W, C = 600, 2048, 5632, 128, 16
    dv = {k: torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
          for k, shape in (("x", (T, d)), ("Wg", (I, d)), ("Wu", (I, d)), ("Wd", (I, d)))}
    twl = tw.TwELL.empty(T, I, W, C)
    y = torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda")
    status = tw.new_status()
    s = twl.struct()
    torch.cuda.synchronize()
    code = lib.twell_ffn_fwd_fixed_scratch(dv["x"].data_ptr(), dv["Wg"].data_ptr(), dv["Wu"].data_ptr(),
                                           dv["Wd"].data_ptr(), T, d, I, W, C, 513, ctypes.byref(s), y.data_ptr(),
                                           status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == _lib.TW_EWORKSPACE, lib.tw_status_str(code)
    torch.cuda.synchronize()
    assert int(status.item()) == 0                   # nothing ran: no device condition raised
    assert bool((y == 7.0).all())                    # and y was not written
    # an argument twell_ffn_fwd rejects gets the same code here, whatever the size
    code = lib.twell_ffn_fwd_fixed_scratch(dv["x"].data_ptr(), dv["Wg"].data_ptr(), dv["Wu"].data_ptr(),
                                           dv["Wd"].data_ptr(), T, d, I, W, C, T + 1, ctypes.byref(s), y.data_ptr(),
                                           status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == _lib.TW_EINVAL, lib.tw_status_str(code)
