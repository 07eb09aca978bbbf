"""Pins for the oracle's TwELL / Hybrid packers (CPU only).

Each packer is checked against (1) a hand-worked fixture, (2) a brute-force
enumeration written as plain loops on small matrices, and (3) the invariants the
format definitions fix: unpack(pack(A)) == A on rows that are not flagged,
sum(cnt) == nnz(A) == sum(row_nnz), ovf <=> some cnt > C, slots ascending and < W,
backup <=> (TwELL overflow or row_nnz > R), backup slots ranked by row.
"""
import json
import os

import numpy as np
import pytest

from oracle import formats
from synthetic import random_bf16_matrix, round_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "twell_hybrid_worked_example.json")


def _golden():
    with open(GOLDEN) as f:
        g = json.load(f)

    def to_bits(rows):
        out = np.zeros((len(rows), len(rows[0])), dtype=np.uint16)
        for i, r in enumerate(rows):
            for j, v in enumerate(r):
                out[i, j] = 0x8000 if v == "-0" else round_to_bf16_bits(np.array([v]))[0]
        return out

    return g, to_bits(g["A"]), to_bits(g["U"])


def _bits_to_float(b):
    return float((np.array([b], dtype=np.uint32) << 16).view(np.float32)[0])


def test_twell_golden_worked_example():
    g, A, _ = _golden()
    tw = formats.twell_pack(A, g["W"], g["C"])
    exp = g["twell"]
    np.testing.assert_array_equal(tw["cnt"], np.array(exp["cnt"]))
    np.testing.assert_array_equal(tw["row_nnz"], exp["row_nnz"])
    np.testing.assert_array_equal(tw["ovf"].astype(int), exp["ovf"])
    np.testing.assert_array_equal(tw["ovf_rows"], exp["ovf_rows"])
    for t, row in enumerate(exp["slots"]):
        for k, slots in enumerate(row):
            assert int(tw["valid"][t, k].sum()) == len(slots)
            for s, (col, v) in enumerate(slots):
                assert tw["idx"][t, k, s] == col
                assert _bits_to_float(tw["val"][t, k, s]) == v


def test_hybrid_golden_worked_example():
    g, A, U = _golden()
    hy = formats.hybrid_pack(A, U, g["W"], g["C"], g["R"])
    exp = g["hybrid"]
    np.testing.assert_array_equal(hy["backup"].astype(int), exp["backup"])
    np.testing.assert_array_equal(hy["backup_tok"], exp["backup_tok"])
    np.testing.assert_array_equal(hy["backup_slot"], exp["backup_slot"])
    np.testing.assert_array_equal(hy["ell_nnz"], exp["ell_nnz"])
    for t, ents in enumerate(exp["ell"]):
        for s, (col, av, uv) in enumerate(ents):
            assert hy["ell_idx"][t, s] == col
            assert _bits_to_float(hy["ell_a"][t, s]) == av
            assert _bits_to_float(hy["ell_u"][t, s]) == uv
    np.testing.assert_array_equal(hy["backup_a"], A[exp["backup_tok"]])
    np.testing.assert_array_equal(hy["backup_u"], U[exp["backup_tok"]])
    tr = formats.hybrid_transpose(hy)
    np.testing.assert_array_equal(tr["col_ptr"], exp["csc"]["col_ptr"])
    np.testing.assert_array_equal(tr["tok"], exp["csc"]["tok"])
    np.testing.assert_array_equal(tr["slot"], exp["csc"]["slot"])


def brute_force_twell(A, W, C):
    """Plain-loop enumeration of the TwELL definition (independent of the numpy packer)."""
    T, I = A.shape
    nT = I // W
    cnt = [[0] * nT for _ in range(T)]
    slots = [[[] for _ in range(nT)] for _ in range(T)]
    for t in range(T):
        for k in range(nT):
            for c in range(W):
                b = int(A[t, k * W + c])
                if b & 0x7FFF:
                    if cnt[t][k] < C:
                        slots[t][k].append((c, b))
                    cnt[t][k] += 1
    ovf = [any(c > C for c in cnt[t]) for t in range(T)]
    return cnt, slots, ovf


@pytest.mark.parametrize("shape,W,C,density,seed,signed", [
    ((7, 16), 4, 2, 0.3, 1, False),
    ((5, 64), 64, 8, 0.1, 2, False),
    ((9, 256), 128, 16, 0.08, 3, False),
    ((3, 12), 4, 4, 0.9, 4, False),
    ((6, 8), 8, 1, 0.2, 5, False),
    # a general matrix: negative nonzeros and bf16 subnormals count, -0.0 does not
    ((8, 128), 64, 6, 0.3, 6, True),
    ((5, 256), 128, 16, 0.15, 7, True),
])
def test_twell_matches_brute_force(shape, W, C, density, seed, signed):
    A = random_bf16_matrix(shape, density, seed, negative_zero_frac=0.3, signed=signed,
                           subnormal_frac=0.2 if signed else 0.0)
    if signed:
        assert ((A & 0x8000) != 0)[(A & 0x7FFF) != 0].any() and (((A & 0x7F80) == 0) & ((A & 0x7FFF) != 0)).any()
    tw = formats.twell_pack(A, W, C)
    cnt, slots, ovf = brute_force_twell(A, W, C)
    np.testing.assert_array_equal(tw["cnt"], np.array(cnt))
    np.testing.assert_array_equal(tw["ovf"], np.array(ovf))
    for t in range(shape[0]):
        for k in range(shape[1] // W):
            n = len(slots[t][k])
            assert int(tw["valid"][t, k].sum()) == n
            for s, (c, b) in enumerate(slots[t][k]):
                assert tw["idx"][t, k, s] == c and tw["val"][t, k, s] == b


@pytest.mark.parametrize("density", [0.0, 0.005, 0.05, 0.3, 1.0])
def test_twell_invariants(density):
    W, C = 64, 8
    A = random_bf16_matrix((40, 320), density, seed=11, negative_zero_frac=0.5, signed=True, subnormal_frac=0.1)
    tw = formats.twell_pack(A, W, C)
    nz = (A & 0x7FFF) != 0
    assert tw["cnt"].sum() == nz.sum() == tw["row_nnz"].sum()
    np.testing.assert_array_equal(tw["row_nnz"], nz.sum(1))
    np.testing.assert_array_equal(tw["ovf"], (tw["cnt"] > C).any(1))
    valid = tw["valid"]
    assert (valid[..., 1:] <= valid[..., :-1]).all()          # stored slots form a prefix
    both = valid[..., 1:] & valid[..., :-1]
    assert (np.diff(tw["idx"], axis=2)[both] > 0).all()      # strictly ascending columns
    np.testing.assert_array_equal(valid.sum(2), np.minimum(tw["cnt"], C))
    assert ((tw["idx"][valid] < W) & (tw["idx"][valid] >= 0)).all()
    dense = formats.twell_unpack(tw)
    keep = ~tw["ovf"]
    # -0.0 entries come back as +0.0; compare as "is nonzero" + exact value on nonzeros
    np.testing.assert_array_equal((dense[keep] & 0x7FFF) != 0, nz[keep])
    np.testing.assert_array_equal(np.where(nz[keep], A[keep], 0), dense[keep])


def test_twell_capacity_boundary():
    W, C = 8, 3
    one = round_to_bf16_bits(np.array([1.0]))[0]
    A = np.zeros((4, 16), dtype=np.uint16)
    A[0, [0, 3, 7]] = one                      # exactly C in tile 0: no overflow
    A[1, [8, 9, 10, 15]] = one                 # C + 1 in tile 1: overflow
    A[2, :] = 0x8000                           # all -0.0: empty row
    A[3, :] = one                              # all active: every tile overflows
    tw = formats.twell_pack(A, W, C)
    np.testing.assert_array_equal(tw["cnt"], [[3, 0], [0, 4], [0, 0], [8, 8]])
    np.testing.assert_array_equal(tw["ovf"], [False, True, False, True])
    np.testing.assert_array_equal(tw["ovf_rows"], [1, 3])
    np.testing.assert_array_equal(tw["idx"][1, 1], [0, 1, 2])
    np.testing.assert_array_equal(tw["idx"][0, 0], [0, 3, 7])


def test_twell_rejects_bad_geometry():
    A = np.zeros((2, 10), dtype=np.uint16)
    with pytest.raises(ValueError):
        formats.twell_pack(A, 4, 2)
    with pytest.raises(ValueError):
        formats.twell_pack(np.zeros((2, 8), dtype=np.uint16), 4, 5)


@pytest.mark.parametrize("R", [1, 3, 12, 400])
def test_hybrid_invariants(R):
    W, C = 16, 4
    A = random_bf16_matrix((30, 64), 0.15, seed=21, negative_zero_frac=0.2)
    U = random_bf16_matrix((30, 64), 1.0, seed=22)
    hy = formats.hybrid_pack(A, U, W, C, R)
    tw = formats.twell_pack(A, W, C)
    nz = (A & 0x7FFF) != 0
    np.testing.assert_array_equal(hy["backup"], tw["ovf"] | (nz.sum(1) > R))
    np.testing.assert_array_equal(hy["backup_tok"], np.flatnonzero(hy["backup"]))
    assert (np.diff(hy["backup_tok"]) > 0).all()
    np.testing.assert_array_equal(hy["backup_slot"][hy["backup_tok"]], np.arange(hy["backup_tok"].size))
    assert (hy["ell_nnz"] <= R).all()
    Ad, Ud = formats.hybrid_unpack(hy)
    np.testing.assert_array_equal(np.where(nz, A, 0), np.where((Ad & 0x7FFF) != 0, Ad, 0))
    np.testing.assert_array_equal(Ud[nz], U[nz])
    np.testing.assert_array_equal(Ud[hy["backup"]], U[hy["backup"]])
    # brute force of the ELL part
    for t in range(30):
        if hy["backup"][t]:
            continue
        cols = [c for c in range(64) if A[t, c] & 0x7FFF]
        assert list(hy["ell_idx"][t, :len(cols)]) == cols
        assert list(hy["ell_a"][t, :len(cols)]) == [A[t, c] for c in cols]
    # transpose: every ELL entry appears once, in its column, tokens ascending per column
    tr = formats.hybrid_transpose(hy)
    seen = set()
    for j in range(64):
        lo, hi = tr["col_ptr"][j], tr["col_ptr"][j + 1]
        toks = tr["tok"][lo:hi]
        assert (np.diff(toks) >= 0).all()
        for t, s in zip(toks, tr["slot"][lo:hi]):
            assert hy["ell_idx"][t, s] == j
            seen.add((int(t), int(s)))
    assert len(seen) == int(hy["ell_nnz"].sum())
