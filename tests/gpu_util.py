"""Helpers for the GPU parity tests: moving bf16 bit patterns between numpy and
torch, and the agreed tolerance for floating-point results:

* relative Frobenius error <= 5e-3, and
* per element |gpu - ref| <= 1e-2 * (1 + |ref|),

against the fp64 oracle on the same bf16-rounded inputs. Active-set (g > 0)
disagreements are allowed only where the oracle's |g| <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

REL_FROB = 5e-3
ELEM = 1e-2
KINK = 1e-3


def to_dev(bits: np.ndarray | None) -> torch.Tensor | None:
    if bits is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, rel_frob: float = REL_FROB, elem: float = ELEM):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.linalg.norm(got - ref)
    nrm = np.linalg.norm(ref)
    rel = err / nrm if nrm > 0 else err
    assert rel <= rel_frob, f"{what}: relative Frobenius error {rel:.3e} > {rel_frob}"
    bad = np.abs(got - ref) > elem * (1.0 + np.abs(ref))
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside 1e-2*(1+|ref|); first at "
                           f"{np.argwhere(bad)[0].tolist()} got {got[bad][0]} ref {ref[bad][0]}")
    return rel


def assert_close_by_row_class(got: np.ndarray, ref: np.ndarray, backup_rows: np.ndarray, what: str):
    """assert_close over all rows, then separately over the ELL rows and over the dense
    backup rows, so that an error confined to the few backup (outlier) rows cannot hide
    in the Frobenius norm of the whole."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert_close(got, ref, what)
    is_backup = np.zeros(got.shape[0], dtype=bool)
    is_backup[np.asarray(backup_rows, dtype=np.int64)] = True
    if (~is_backup).any():
        assert_close(got[~is_backup], ref[~is_backup], f"{what} (ELL rows)")
    if is_backup.any():
        assert_close(got[is_backup], ref[is_backup], f"{what} (backup rows)")


def check_active_set(active_gpu: np.ndarray, g_ref: np.ndarray, what: str = "active set"):
    """Every disagreement between the GPU's active set and g_ref > 0 sits at |g_ref| <= 1e-3."""
    diff = active_gpu != (g_ref > 0)
    assert not (diff & (np.abs(g_ref) > KINK)).any(), (
        f"{what}: {int((diff & (np.abs(g_ref) > KINK)).sum())} disagreements away from the kink")
    return int(diff.sum())
