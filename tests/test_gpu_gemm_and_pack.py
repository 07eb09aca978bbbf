"""GPU parity: the tcgen05 GEMM engine's operand layouts, the standalone TwELL
packer (bit-exact) and the fused gate-projection + TwELL-pack kernel."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import assert_close, bits_of, check_active_set, to_dev  # noqa: E402
from oracle import ffn, formats  # noqa: E402
from synthetic import FFNSpec, WORKLOADS, make_inputs, random_bf16_matrix, round_to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return round_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


def _check_layout(M, N, K, a_mn, b_mn, pair):
    A = _rand_bf16((K, M) if a_mn else (M, K), 1)
    B = _rand_bf16((K, N) if b_mn else (N, K), 2)
    D = tw.dense_gemm(to_dev(A), to_dev(B), M, N, K, bool(a_mn), bool(b_mn), pair=pair)
    torch.cuda.synchronize()
    a = ffn.bf16_to_f64(A)
    b = ffn.bf16_to_f64(B)
    ref = (a.T if a_mn else a) @ (b if b_mn else b.T)
    np.testing.assert_allclose(D.cpu().numpy(), ref, rtol=1e-4, atol=1e-4 * np.sqrt(K))


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
# 128 x 64 tiles, one CTA each; (3072, 1792, 64) is 672 tiles, several rounds
@pytest.mark.parametrize("M,N,K", [(256, 192, 320), (192, 64, 64), (512, 256, 1024), (3072, 1792, 64)])
def test_dense_gemm_layouts(a_mn, b_mn, M, N, K):
    _check_layout(M, N, K, a_mn, b_mn, pair=False)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
# 256 x 256 units on CTA pairs: one unit whose second CTA's rows are all past M
# (M 192), whole units, and (3072, 1792, 64): 84 units on at most 76 pairs
@pytest.mark.parametrize("M,N,K", [(192, 256, 64), (512, 512, 1024), (3072, 1792, 64)])
def test_dense_gemm_pair_layouts(a_mn, b_mn, M, N, K):
    _check_layout(M, N, K, a_mn, b_mn, pair=True)


def test_dense_gemm_pair_ragged_rows():
    """M = 300: the second unit's first CTA holds rows 256..299, its second CTA none."""
    _check_layout(300, 256, 192, 0, 0, pair=True)


def test_dense_gemm_ragged_rows():
    M, N, K = 200, 128, 192
    A = _rand_bf16((M, K), 3)
    B = _rand_bf16((N, K), 4)
    D = tw.dense_gemm(to_dev(A), to_dev(B), M, N, K, False, False)
    torch.cuda.synchronize()
    ref = ffn.bf16_to_f64(A) @ ffn.bf16_to_f64(B).T
    np.testing.assert_allclose(D.cpu().numpy(), ref, rtol=1e-4, atol=1e-4 * np.sqrt(K))


def _assert_twell_equal(gpu: "tw.TwELL", ref: dict, rows=None):
    T = ref["T"]
    cnt = gpu.cnt.cpu().numpy().view(np.uint16).astype(np.int64)
    np.testing.assert_array_equal(cnt, ref["cnt"])
    np.testing.assert_array_equal(gpu.row_nnz.cpu().numpy(), ref["row_nnz"])
    np.testing.assert_array_equal(gpu.ovf.cpu().numpy().astype(bool), ref["ovf"])
    n = int(gpu.n_ovf.item())
    assert n == ref["ovf_rows"].size
    np.testing.assert_array_equal(gpu.ovf_rows[:n].cpu().numpy(), ref["ovf_rows"])
    val = bits_of(gpu.val)
    idx = gpu.idx.cpu().numpy().astype(np.int64)
    v = ref["valid"]
    np.testing.assert_array_equal(idx[v], ref["idx"][v])
    np.testing.assert_array_equal(val[v], ref["val"][v])
    assert T == gpu.T


@pytest.mark.parametrize("T,I,W,C,density,signed", [(1, 64, 64, 1, 0.5, False), (77, 640, 64, 8, 0.05, False),
                                                    (300, 1024, 128, 16, 0.1, False), (513, 768, 128, 4, 0.02, False),
                                                    (64, 256, 128, 128, 1.0, False), (50, 256, 64, 8, 0.0, False),
                                                    # negative nonzeros and bf16 subnormals count, -0.0 does not
                                                    (129, 512, 64, 8, 0.1, True), (200, 1024, 128, 16, 0.3, True)])
def test_twell_pack_bit_exact(T, I, W, C, density, signed):
    A = random_bf16_matrix((T, I), density, seed=T + I, negative_zero_frac=0.3, signed=signed,
                           subnormal_frac=0.2 if signed else 0.0)
    out = tw.twell_pack(to_dev(A), W, C)
    torch.cuda.synchronize()
    _assert_twell_equal(out, formats.twell_pack(A, W, C))


def _gate_case(spec: FFNSpec):
    inp = make_inputs(spec)
    x, Wg = to_dev(inp["x"]), to_dev(inp["Wg"])
    out, dense = tw.twell_gate_pack(x, Wg, spec.W, spec.C, want_dense=True)
    torch.cuda.synchronize()
    return inp, out, dense


@pytest.mark.parametrize("spec", [
    WORKLOADS["tiny_fwd"],                                                        # I=704: 64-wide N tiles
    FFNSpec("gate_ragged_128", T=1000, d=512, I=640, mean_active=12, outlier_frac=0.02, W=128, C=8),
    FFNSpec("gate_ragged_256", T=333, d=768, I=1024, mean_active=20, outlier_frac=0.03, W=64, C=8, seed=3),
    # 256-wide tiles on CTA pairs with one 256-row unit: the second CTA of the pair has
    # no rows (T = 77), or neither CTA has more than one (T = 1)
    FFNSpec("gate_pair_77_rows", T=77, d=256, I=512, mean_active=10, outlier_frac=0.03, W=128, C=8, seed=4),
    FFNSpec("gate_pair_one_row", T=1, d=256, I=256, mean_active=8, outlier_frac=0.0, W=64, C=8, seed=13),
], ids=lambda s: s.name)
def test_gate_pack_values_and_bit_exact_pack(spec):
    inp, out, dense = _gate_case(spec)
    g = ffn.forward(inp["x"], inp["Wg"], None, inp["Wd"])["g"]
    a_gpu = ffn.bf16_to_f64(bits_of(dense))
    assert_close(a_gpu, np.maximum(g, 0), "a = ReLU(x Wg^T)")
    check_active_set(a_gpu > 0, g)
    # the fused epilogue's TwELL is exactly the TwELL of its own dense output
    _assert_twell_equal(out, formats.twell_pack(bits_of(dense), spec.W, spec.C))


def test_gate_pack_full_size_sampled_rows():
    spec = WORKLOADS["gated_fwd_d2048_i5632"]
    inp, out, dense = _gate_case(spec)
    rows = np.unique(np.concatenate([np.arange(0, spec.T, 997), inp["outliers"][:8], [spec.T - 1]]))
    g = ffn.bf16_to_f64(inp["x"][rows]) @ ffn.bf16_to_f64(inp["Wg"]).T
    a_bits = bits_of(dense)[rows]
    check_active_set((a_bits & 0x7FFF) != 0, g)
    assert_close(ffn.bf16_to_f64(a_bits), np.maximum(g, 0), "a (sampled rows)")
    ref = formats.twell_pack(a_bits, spec.W, spec.C)
    cnt = out.cnt.cpu().numpy().view(np.uint16)[rows].astype(np.int64)
    np.testing.assert_array_equal(cnt, ref["cnt"])
    np.testing.assert_array_equal(out.row_nnz.cpu().numpy()[rows], ref["row_nnz"])
    np.testing.assert_array_equal(out.ovf.cpu().numpy()[rows].astype(bool), ref["ovf"])
    v = ref["valid"]
    np.testing.assert_array_equal(out.idx.cpu().numpy()[rows].astype(np.int64)[v], ref["idx"][v])
    np.testing.assert_array_equal(bits_of(out.val)[rows][v], ref["val"][v])
    # the overflow list is the ascending list of flagged rows (whole matrix)
    ovf = out.ovf.cpu().numpy().astype(bool)
    n = int(out.n_ovf.item())
    np.testing.assert_array_equal(out.ovf_rows[:n].cpu().numpy(), np.flatnonzero(ovf))
    # every outlier token overflows at this capacity; ordinary tokens almost never do
    assert set(inp["outliers"].tolist()) <= set(np.flatnonzero(ovf).tolist())
