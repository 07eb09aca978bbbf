"""Helpers for the GPU parity tests: moving bf16 bit patterns between numpy and
torch, and the agreed tolerance for floating-point results:

* relative Frobenius error <= 5e-3, and
* per element |gpu - ref| <= 1e-2 * (1 + |ref|),

against the fp64 oracle on the same bf16-rounded inputs. Active-set (g > 0)
disagreements are allowed only where the oracle's |g| <= 1e-3; there the
gradients are compared on the side of the kink the kernel took (see
``oracle_on_kernel_branch``).
"""
from __future__ import annotations

import numpy as np
import torch

import activation_sparse_feedforward_gb300 as tw
from oracle import ffn

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


def kernel_active_set(saved) -> np.ndarray:
    """The kernel's ReLU decisions (a != 0) over [T, I], read back from the Hybrid its
    training forward saved: the ELL rows' index lists and the dense backup rows. Needs
    every backup row stored (n_backup <= backup_cap)."""
    assert int(saved.n_backup.item()) <= saved.backup_cap
    A, _ = tw.hybrid_unpack(saved, with_u=False)
    torch.cuda.synchronize()
    return A.cpu().numpy() != 0


def oracle_on_kernel_branch(f: dict, active_gpu: np.ndarray, Wd) -> dict:
    """The oracle's forward values moved to the kernel's side of the ReLU kink.

    The layer's gradient jumps at g = 0: an entry whose |g| is within the fp32
    accumulation error of x Wg^T may fall on either side, and both gradients are
    then correct (dg and dWg differ by that entry's whole (dh u + l1) term). After
    check_active_set has confirmed that every disagreement lies in the kink band
    |g| <= 1e-3, each disagreeing entry gets g of the kernel's sign (same
    magnitude) and a, h and y are re-derived from it as the oracle's forward does.
    The arithmetic stays the oracle's; only the side of the kink is the kernel's."""
    check_active_set(active_gpu, f["g"])
    flip = active_gpu != (f["g"] > 0)
    if not flip.any():
        return f
    g = f["g"].copy()
    mag = np.maximum(np.abs(g[flip]), np.finfo(np.float64).tiny)
    g[flip] = np.where(active_gpu[flip], mag, -mag)
    a = ffn.relu(g)
    h = a if f["u"] is None else a * f["u"]
    return {**f, "g": g, "a": a, "h": h, "y": h @ ffn.as_f64(Wd)}
