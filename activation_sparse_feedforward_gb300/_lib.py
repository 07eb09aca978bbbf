"""ctypes declarations of the C ABI in ``include/twell.h``.

Loading fails loudly when ``libtwell.so`` has not been built: there is no fallback
implementation of any operation.
"""
from __future__ import annotations

import ctypes
import os
import threading

# TW_LIB_PATH selects another build of the same library (the bounds-checked one)
LIB_PATH = os.environ.get("TW_LIB_PATH") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtwell.so")

c_void_p = ctypes.c_void_p
c_int = ctypes.c_int
c_size_t = ctypes.c_size_t
c_float = ctypes.c_float

(TW_OK, TW_EINVAL, TW_EALIGN, TW_EUNSUPPORTED, TW_ECAPACITY, TW_ETIMEOUT, TW_ECUDA, TW_EWORKSPACE,
 TW_EBOUNDS) = range(9)


class TwTwell(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("I", ctypes.c_int32), ("W", ctypes.c_int32), ("C", ctypes.c_int32),
                ("cnt", c_void_p), ("val", c_void_p), ("idx", c_void_p), ("row_nnz", c_void_p),
                ("ovf", c_void_p), ("ovf_rows", c_void_p), ("n_ovf", c_void_p)]


class TwHybrid(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("I", ctypes.c_int32), ("R", ctypes.c_int32),
                ("backup_cap", ctypes.c_int32),
                ("row_nnz", c_void_p), ("ell_nnz", c_void_p), ("ell_idx", c_void_p), ("ell_a", c_void_p),
                ("ell_u", c_void_p), ("backup_slot", c_void_p), ("backup_tok", c_void_p),
                ("backup_a", c_void_p), ("backup_u", c_void_p), ("n_backup", c_void_p),
                ("route", ctypes.c_int32), ("dense_above", ctypes.c_float), ("route_taken", c_void_p)]


TW_ROUTE_SPARSE, TW_ROUTE_DENSE, TW_ROUTE_AUTO = 0, 1, 2
ROUTES = {"sparse": TW_ROUTE_SPARSE, "dense": TW_ROUTE_DENSE, "auto": TW_ROUTE_AUTO}


# name -> (restype, argtypes); every symbol declared in include/twell.h
SIGNATURES = {
    "tw_status_str": (ctypes.c_char_p, [c_int]),
    "tw_abi_version": (c_int, []),
    "twell_pack": (c_int, [c_void_p, c_int, c_int, c_int, c_int, ctypes.POINTER(TwTwell), c_void_p, c_void_p]),
    "twell_unpack": (c_int, [ctypes.POINTER(TwTwell), c_void_p, c_void_p]),
    "hybrid_pack_workspace_size": (c_size_t, [c_int]),
    "hybrid_pack": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, ctypes.POINTER(TwHybrid), c_void_p,
                            c_size_t, c_void_p, c_void_p]),
    "hybrid_unpack": (c_int, [ctypes.POINTER(TwHybrid), c_void_p, c_void_p, c_void_p]),
    "twell_gate_pack": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(TwTwell),
                                c_void_p, c_void_p, c_void_p]),
    "twell_ffn_fwd_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "twell_ffn_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                              ctypes.POINTER(TwTwell), c_void_p, c_size_t, c_void_p, c_void_p, c_void_p]),
    "twell_ffn_fwd_fixed_scratch": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                            c_int, c_int, ctypes.POINTER(TwTwell), c_void_p, c_void_p, c_void_p]),
    "hybrid_ffn_fwd_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int]),
    "hybrid_ffn_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                               ctypes.POINTER(TwHybrid), c_void_p, c_size_t, c_void_p, c_void_p, c_void_p]),
    "hybrid_ffn_bwd_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "hybrid_ffn_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                               ctypes.POINTER(TwHybrid), c_float, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p, c_size_t, c_void_p, c_void_p]),
    "twell_ffn_sparse_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                     ctypes.POINTER(TwTwell), c_void_p, c_size_t, c_void_p, c_void_p, c_void_p]),
    "tw_gate_relu_dense": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "hybrid_neuron_counts": (c_int, [ctypes.POINTER(TwHybrid), c_void_p, c_void_p]),
    "tw_reinit_dead_rows": (c_int, [c_void_p, c_int, c_int, c_void_p, ctypes.c_uint64, c_float, c_void_p, c_void_p]),
    "tw_dense_gemm": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                              c_void_p]),
    "tw_dense_gemm_pair": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                              c_void_p]),
    "tw_l2_gather_probe": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int, c_void_p, c_int,
                                   ctypes.POINTER(ctypes.c_double), c_void_p]),
    "tw_l2_gather_probe_blocks": (c_int, [c_int]),
    "tw_wait_timeout_probe": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "tw_wait_timeout_probe_pair": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "tw_fma_probe": (c_int, [c_void_p, c_int, c_int, ctypes.POINTER(ctypes.c_double), c_void_p]),
    "tw_trace_begin": (c_int, [ctypes.POINTER(c_void_p), c_int]),
    "tw_trace_end": (c_int, []),
    "tw_trace_label": (ctypes.c_char_p, [c_int]),
}

_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load ``libtwell.so`` (once) and declare every entry point's signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libtwell.so not found at {LIB_PATH}: build it first with "
                "`python -m activation_sparse_feedforward_gb300.build` (or __graft_entry__.build()). "
                "There is no non-CUDA fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class TwellError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().tw_status_str(code).decode()
        super().__init__(f"{where}: {msg}")


def check(code: int, where: str) -> None:
    if code != TW_OK:
        raise TwellError(code, where)
