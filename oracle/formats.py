"""TwELL and Hybrid sparse formats: packing and unpacking, written from the pages.

Test infrastructure only (see ``oracle/__init__.py``).

TwELL, tile-wise ELLPACK (gist.science explainer, section 2.A "New Sparse Data
Format: TwELL"; wispaper blog, "1. TwELL: Tile-wise ELLPACK"; Figure 1 caption of
the thelatestinai listing): the columns of the activation matrix are cut into 1D
tiles of width W; inside each (row, tile) the nonzero values and their local column
indices are kept in a small ELL of fixed capacity C. Readings taken where the pages
are silent:

* nonzero: for bf16 bit patterns, any entry whose magnitude bits are not all zero
  (so -0.0 counts as zero); for float arrays, ``!= 0``;
* slots hold the nonzeros in ascending column order (the pages build the format
  with warp atomics, so any order is valid; ascending order is the canonical one);
* ``cnt`` is the true (uncapped) number of nonzeros of the (row, tile); only the
  first min(cnt, C) are stored; a row with any cnt > C "overflows" and is served by
  the dense path, so TwELL is lossless on the rows it does not flag.

Hybrid (explainer 2.A "Hybrid Format for Training"; wispaper blog, "2. The Hybrid
Training Algorithm"; tunx.ai announcement, "Details" -- the dense backup as the
fallback for rows too active for the ELL): every row goes either to a compact
row-wise ELL of capacity R
(global column indices, ascending) or to a dense backup matrix that holds the full
row. The Hybrid is built from the TwELL of the gate activations (explainer 2.B,
"Hybrid Conversion"), so a row whose TwELL overflowed (values beyond C were never
stored) cannot be put in the ELL; the routing rule read from this is

    backup(t)  <=>  ovf_twell(t)  or  row_nnz(t) > R,

and the backup slot of a row is its rank among backup rows in ascending row order.
The transposed Hybrid (explainer 2.B "Backpropagation") lists, per neuron j, the
ELL entries holding column j, in ascending token order.
"""
from __future__ import annotations

import numpy as np


def is_nonzero(A: np.ndarray) -> np.ndarray:
    A = np.asarray(A)
    if A.dtype == np.uint16:
        return (A & 0x7FFF) != 0
    return A != 0


def _first_nonzeros(nz: np.ndarray, k: int) -> np.ndarray:
    """Column positions (along the last axis) of the first k nonzeros, ascending;
    positions past the number of nonzeros point at zero entries."""
    order = np.argsort(~nz, axis=-1, kind="stable")
    return order[..., :k]


def twell_pack(A: np.ndarray, W: int, C: int) -> dict:
    """Pack a [T, I] activation matrix into TwELL with tile width W and capacity C.

    Returns cnt [T, nT] (true counts), idx [T, nT, C] (local column, -1 in unused
    slots), val [T, nT, C] (A's entries, 0 in unused slots), valid [T, nT, C],
    row_nnz [T], ovf [T] (any cnt > C) and ovf_rows (ascending)."""
    A = np.asarray(A)
    T, I = A.shape
    if W <= 0 or I % W != 0:
        raise ValueError("I must be a multiple of the tile width W")
    if not 1 <= C <= W:
        raise ValueError("capacity C must be in [1, W]")
    nT = I // W
    tiles = A.reshape(T, nT, W)
    nz = is_nonzero(tiles)
    cnt = nz.sum(axis=2).astype(np.int64)
    pos = _first_nonzeros(nz, C)
    valid = np.arange(C)[None, None, :] < np.minimum(cnt, C)[:, :, None]
    val = np.take_along_axis(tiles, pos, axis=2)
    val = np.where(valid, val, np.zeros((), dtype=A.dtype))
    idx = np.where(valid, pos, -1).astype(np.int64)
    row_nnz = cnt.sum(axis=1)
    ovf = (cnt > C).any(axis=1)
    return {"T": T, "I": I, "W": W, "C": C, "cnt": cnt, "idx": idx, "val": val,
            "valid": valid, "row_nnz": row_nnz, "ovf": ovf,
            "ovf_rows": np.flatnonzero(ovf).astype(np.int64)}


def twell_unpack(tw: dict) -> np.ndarray:
    """Scatter the stored slots back into a dense [T, I] matrix (zeros elsewhere).
    Equal to the packed matrix on every row with ovf == False."""
    T, I, W = tw["T"], tw["I"], tw["W"]
    out = np.zeros((T, I), dtype=tw["val"].dtype)
    t, k, s = np.nonzero(tw["valid"])
    out[t, k * W + tw["idx"][t, k, s]] = tw["val"][t, k, s]
    return out


def hybrid_pack(A: np.ndarray, U: np.ndarray | None, W: int, C: int, R: int) -> dict:
    """Hybrid format of the activations A (and the up-projection U, gated form).

    ELL rows keep up to R entries: global column ``idx`` ascending, with A's and U's
    values at those columns. Backup rows keep their full A and U rows."""
    A = np.asarray(A)
    T, I = A.shape
    if R < 1:
        raise ValueError("R must be >= 1")
    tw = twell_pack(A, W, C)
    backup = tw["ovf"] | (tw["row_nnz"] > R)
    backup_tok = np.flatnonzero(backup).astype(np.int64)
    backup_slot = np.full(T, -1, dtype=np.int64)
    backup_slot[backup_tok] = np.arange(backup_tok.size)
    nz = is_nonzero(A)
    ell_nnz = np.where(backup, 0, tw["row_nnz"]).astype(np.int64)
    pos = _first_nonzeros(nz, min(R, I))
    if R > I:
        pos = np.concatenate([pos, np.zeros((T, R - I), dtype=pos.dtype)], axis=1)
    valid = np.arange(R)[None, :] < ell_nnz[:, None]
    ell_idx = np.where(valid, pos, -1).astype(np.int64)
    ell_a = np.where(valid, np.take_along_axis(A, np.minimum(pos, I - 1), axis=1),
                     np.zeros((), dtype=A.dtype))
    out = {"T": T, "I": I, "R": R, "W": W, "C": C, "row_nnz": tw["row_nnz"],
           "backup": backup, "backup_tok": backup_tok, "backup_slot": backup_slot,
           "ell_nnz": ell_nnz, "ell_idx": ell_idx, "ell_valid": valid, "ell_a": ell_a,
           "backup_a": A[backup_tok].copy(), "ell_u": None, "backup_u": None}
    if U is not None:
        U = np.asarray(U)
        out["ell_u"] = np.where(valid, np.take_along_axis(U, np.minimum(pos, I - 1), axis=1),
                                np.zeros((), dtype=U.dtype))
        out["backup_u"] = U[backup_tok].copy()
    return out


def hybrid_unpack(hy: dict) -> tuple[np.ndarray, np.ndarray | None]:
    """Dense A and U back from a Hybrid. A is exact on every row; U is exact on the
    support of ELL rows and on the whole of backup rows (zero elsewhere)."""
    T, I = hy["T"], hy["I"]
    A = np.zeros((T, I), dtype=hy["ell_a"].dtype)
    t, s = np.nonzero(hy["ell_valid"])
    A[t, hy["ell_idx"][t, s]] = hy["ell_a"][t, s]
    A[hy["backup_tok"]] = hy["backup_a"]
    U = None
    if hy["ell_u"] is not None:
        U = np.zeros((T, I), dtype=hy["ell_u"].dtype)
        U[t, hy["ell_idx"][t, s]] = hy["ell_u"][t, s]
        U[hy["backup_tok"]] = hy["backup_u"]
    return A, U


def hybrid_transpose(hy: dict) -> dict:
    """Transposed Hybrid over the ELL part: for each neuron j, the (token, slot)
    pairs of the ELL entries holding column j, tokens ascending (CSC layout:
    col_ptr [I + 1], tok [nnz], slot [nnz])."""
    I = hy["I"]
    t, s = np.nonzero(hy["ell_valid"])          # row-major: tokens ascending
    j = hy["ell_idx"][t, s]
    order = np.argsort(j, kind="stable")        # stable keeps tokens ascending per column
    counts = np.bincount(j, minlength=I)
    col_ptr = np.zeros(I + 1, dtype=np.int64)
    np.cumsum(counts, out=col_ptr[1:])
    return {"I": I, "col_ptr": col_ptr, "tok": t[order].astype(np.int64),
            "slot": s[order].astype(np.int64)}
