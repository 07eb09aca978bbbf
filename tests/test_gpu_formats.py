"""GPU parity of the standalone format calls against the oracle's packers: TwELL
unpack, Hybrid pack from a chosen matrix and Hybrid unpack (explainer 2.A "New
Sparse Data Format: TwELL" and "Hybrid Format for Training"; wispaper blog, "1.
TwELL" and "2. The Hybrid Training Algorithm"). Integer and byte results are
compared bit for bit; on hand-placed rows the routing edge cases are all present:
a row with exactly R nonzeros, one with R + 1, a row whose TwELL overflows while
row_nnz <= R, a tile with exactly C nonzeros, an all-zero row, a row of -0.0,
negative values and subnormals, the first and last column."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import bits_of, to_dev  # noqa: E402
from oracle import formats  # noqa: E402
from synthetic import random_bf16_matrix, round_to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _f32_of_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def _u_matrix(rng, shape):
    """bf16 up-projection values ~ N(0, 1) kept at magnitudes >= 1e-3, inside fp16's
    normal range, where the Hybrid's fp16 storage of u is exact."""
    u = rng.standard_normal(shape).astype(np.float32)
    u = np.where(np.abs(u) < 1e-3, np.float32(1e-3), u)
    return round_to_bf16_bits(u)


def _edge_matrix():
    """T = 10, I = 256, W = 64 (four tiles), C = 4, R = 6, with the cases of the
    docstring placed by hand."""
    T, I = 10, 256
    vals = {}

    def put(t, cols, v=1.5):
        for c in cols:
            vals[(t, c)] = v

    put(1, [3, 70, 71, 140, 200, 255])                  # exactly R = 6, <= C per tile: ELL
    put(2, [0, 1, 64, 65, 128, 129, 192])               # R + 1 = 7: backup
    put(3, [10, 11, 12, 13, 14])                         # tile 0 holds C + 1 = 5, row_nnz 5 <= R: backup
    put(4, [64, 80, 96, 127])                            # tile 1 holds exactly C = 4: ELL
    put(6, [5], -2.25)                                   # negative value
    put(6, [77], float(_f32_of_bits(np.array([0x0001]))[0]))     # smallest subnormal
    put(6, [150], -float(_f32_of_bits(np.array([0x007F]))[0]))   # largest subnormal, negative
    put(7, [0, 255], 0.75)                               # first and last column
    put(8, list(range(0, 256, 37)), 3.0)                 # 7 nonzeros, one per tile or so: backup by R
    put(9, [1, 2, 3, 4, 66, 67, 68, 69], -1.0)           # two full tiles: 8 > R, backup
    A = np.zeros((T, I), dtype=np.float32)
    for (t, c), v in vals.items():
        A[t, c] = v
    bits = round_to_bf16_bits(A)
    bits[5, [7, 100, 201]] = 0x8000                      # row 5: -0.0 only, a zero row
    bits[0, 50] = 0x8000                                 # row 0: all zero (one -0.0)
    bits[6, 30] = 0x8000                                 # -0.0 beside nonzeros
    return bits, _u_matrix(np.random.default_rng(3), (T, I)), 64, 4, 6


def _random_case(T, I, W, C, R, density, seed):
    A = random_bf16_matrix((T, I), density, seed, negative_zero_frac=0.2, signed=True, subnormal_frac=0.05)
    # a few dense rows (outlier-like) so that both routing reasons occur
    rng = np.random.default_rng(seed)
    dense_rows = rng.choice(T, size=max(1, T // 50), replace=False)
    A[dense_rows] = random_bf16_matrix((dense_rows.size, I), 0.5, seed + 1, signed=True)
    return A, _u_matrix(rng, (T, I)), W, C, R


CASES = {
    "edges": _edge_matrix,
    "random_w128": lambda: _random_case(300, 1024, 128, 8, 24, 0.015, 11),
    "random_w64": lambda: _random_case(129, 448, 64, 3, 10, 0.02, 12),
}


def _check_hybrid(h, ref, A, U, T, cap):
    n_ref = int(ref["backup_tok"].size)
    assert int(h.n_backup.item()) == n_ref
    np.testing.assert_array_equal(h.row_nnz.cpu().numpy()[:T], ref["row_nnz"])
    np.testing.assert_array_equal(h.ell_nnz.cpu().numpy()[:T], ref["ell_nnz"])
    slot = h.backup_slot.cpu().numpy()[:T]
    exp_slot = ref["backup_slot"].copy()
    exp_slot[exp_slot >= cap] = -2                       # rows past the capacity are not stored
    np.testing.assert_array_equal(slot, exp_slot)
    stored = min(n_ref, cap)
    np.testing.assert_array_equal(h.backup_tok.cpu().numpy()[:stored], ref["backup_tok"][:stored])
    v = ref["ell_valid"]
    idx = h.ell_idx.cpu().numpy().view(np.uint16).astype(np.int64)[:T]
    np.testing.assert_array_equal(idx[v], ref["ell_idx"][v])
    np.testing.assert_array_equal(bits_of(h.ell_a)[:T][v], ref["ell_a"][v])
    if U is not None:
        # fp16 storage of U's bf16 values: exact in fp16's range
        np.testing.assert_array_equal(h.ell_u.float().cpu().numpy()[:T][v], _f32_of_bits(ref["ell_u"][v]))
    # backup rows: the full rows widened exactly to fp32
    np.testing.assert_array_equal(h.backup_a.cpu().numpy()[:stored], _f32_of_bits(ref["backup_a"][:stored]))
    if U is not None:
        np.testing.assert_array_equal(h.backup_u.cpu().numpy()[:stored], _f32_of_bits(ref["backup_u"][:stored]))


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
@pytest.mark.parametrize("gated", [True, False], ids=["gated", "nongated"])
def test_hybrid_pack_and_unpack_bit_exact(case, gated):
    A, U, W, C, R = CASES[case]()
    U = U if gated else None
    T, I = A.shape
    ref = formats.hybrid_pack(A, U, W, C, R)
    cap = int(ref["backup_tok"].size)
    assert 0 < cap < T and (ref["ell_nnz"] > 0).any()
    st = tw.new_status()
    h = tw.hybrid_pack(to_dev(A), to_dev(U), W, C, R, backup_cap=cap, status=st)
    torch.cuda.synchronize()
    tw.raise_if_device_error(st, "hybrid_pack")
    _check_hybrid(h, ref, A, U, T, cap)
    # unpack gives A back on every row, and U on the ELL rows' support and on backup rows
    Ag, Ug = tw.hybrid_unpack(h)
    torch.cuda.synchronize()
    ra, ru = formats.hybrid_unpack(ref)
    np.testing.assert_array_equal(Ag.cpu().numpy(), _f32_of_bits(A & np.where((A & 0x7FFF) != 0, 0xFFFF, 0)))
    np.testing.assert_array_equal(Ag.cpu().numpy(), _f32_of_bits(ra))
    if gated:
        np.testing.assert_array_equal(Ug.cpu().numpy(), _f32_of_bits(ru))
    if case == "edges":
        # the hand-placed routing: rows 2, 3, 8, 9 to the backup; 1, 4, 6, 7 ELL; 0, 5 empty ELL rows
        assert ref["backup_tok"].tolist() == [2, 3, 8, 9]
        assert ref["ell_nnz"].tolist() == [0, 6, 0, 0, 4, 0, 3, 2, 0, 0]


@pytest.mark.parametrize("case", ["random_w128", "edges"])
def test_hybrid_pack_capacity_exceeded(case):
    A, U, W, C, R = CASES[case]()
    T, I = A.shape
    ref = formats.hybrid_pack(A, U, W, C, R)
    n = int(ref["backup_tok"].size)
    cap = max(1, n // 2)
    st = tw.new_status()
    h = tw.hybrid_pack(to_dev(A), to_dev(U), W, C, R, backup_cap=cap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4                           # TW_ECAPACITY
    _check_hybrid(h, ref, A, U, T, cap)


@pytest.mark.parametrize("T,I,W,C,density,signed", [(10, 256, 64, 4, 0.05, True), (300, 1024, 128, 8, 0.03, True),
                                                    (77, 640, 64, 8, 0.3, False), (50, 256, 128, 2, 0.0, True)])
def test_twell_unpack_bit_exact(T, I, W, C, density, signed):
    A = random_bf16_matrix((T, I), density, seed=T + I, negative_zero_frac=0.3, signed=signed,
                           subnormal_frac=0.1 if signed else 0.0)
    packed = tw.twell_pack(to_dev(A), W, C)
    out = tw.twell_unpack(packed)
    torch.cuda.synchronize()
    ref = formats.twell_pack(A, W, C)
    exp = formats.twell_unpack(ref)
    np.testing.assert_array_equal(bits_of(out), exp)
    # the identity on every row without overflow (-0.0 comes back as +0.0)
    keep = ~ref["ovf"]
    clean = np.where((A & 0x7FFF) != 0, A, 0).astype(np.uint16)
    np.testing.assert_array_equal(bits_of(out)[keep], clean[keep])
