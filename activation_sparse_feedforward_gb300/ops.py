"""Torch-facing binding of the C ABI: allocates outputs and workspaces with torch,
passes raw device pointers and the current CUDA stream, and raises on host-side
error codes. Every step of the computation runs in the library's CUDA kernels.

Device-side conditions (capacity exceeded, a bounded wait timing out) land in an
int32 status tensor; ``raise_if_device_error(status)`` synchronises and checks it.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib

BF16 = torch.bfloat16


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _check_bf16(name: str, t: torch.Tensor, shape: tuple[int, ...] | None = None) -> None:
    if t.dtype != BF16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if shape is not None and tuple(t.shape) != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def raise_if_device_error(status: torch.Tensor, where: str = "device") -> None:
    code = int(status.item())
    if code != _lib.TW_OK:
        raise _lib.TwellError(code, where)


@dataclass
class TwELL:
    """TwELL buffers (see ``tw_twell`` in include/twell.h)."""

    T: int
    I: int
    W: int
    C: int
    cnt: torch.Tensor       # [T, nT] uint16 stored as int16 bits
    val: torch.Tensor       # [T, nT, C] bf16
    idx: torch.Tensor       # [T, nT, C] uint8
    row_nnz: torch.Tensor   # [T] int32
    ovf: torch.Tensor       # [T] uint8
    ovf_rows: torch.Tensor  # [T] int32
    n_ovf: torch.Tensor     # [1] int32

    @staticmethod
    def empty(T: int, I: int, W: int, C: int, device="cuda") -> "TwELL":
        nT = I // W
        return TwELL(T, I, W, C,
                     cnt=torch.empty((T, nT), dtype=torch.int16, device=device),
                     val=torch.empty((T, nT, C), dtype=BF16, device=device),
                     idx=torch.empty((T, nT, C), dtype=torch.uint8, device=device),
                     row_nnz=torch.empty(T, dtype=torch.int32, device=device),
                     ovf=torch.empty(T, dtype=torch.uint8, device=device),
                     ovf_rows=torch.empty(max(T, 1), dtype=torch.int32, device=device),
                     n_ovf=torch.zeros(1, dtype=torch.int32, device=device))

    def struct(self) -> _lib.TwTwell:
        return _lib.TwTwell(self.T, self.I, self.W, self.C, _ptr(self.cnt), _ptr(self.val), _ptr(self.idx),
                            _ptr(self.row_nnz), _ptr(self.ovf), _ptr(self.ovf_rows), _ptr(self.n_ovf))


@dataclass
class Hybrid:
    """Hybrid buffers saved by the training forward (see ``tw_hybrid``)."""

    T: int
    I: int
    R: int
    backup_cap: int
    row_nnz: torch.Tensor      # [T] int32
    ell_nnz: torch.Tensor      # [T] int32
    ell_idx: torch.Tensor      # [T, R] int16 bits of uint16
    ell_a: torch.Tensor        # [T, R] bf16
    ell_u: torch.Tensor | None  # [T, R] fp16
    backup_slot: torch.Tensor  # [T] int32
    backup_tok: torch.Tensor   # [max(cap,1)] int32
    backup_a: torch.Tensor     # [max(cap,1), I] fp32
    backup_u: torch.Tensor | None  # [max(cap,1), I] fp32
    n_backup: torch.Tensor     # [1] int32
    route: int = _lib.TW_ROUTE_SPARSE
    dense_above: float = 0.0
    route_taken: torch.Tensor | None = None  # [1] int32: 0 sparse, 1 dense (written by the forward)

    @staticmethod
    def empty(T: int, I: int, R: int, backup_cap: int, gated: bool, device="cuda", route: str = "sparse",
              dense_above: float = 64.0) -> "Hybrid":
        cap1 = max(backup_cap, 1)
        return Hybrid(T, I, R, backup_cap,
                      row_nnz=torch.empty(max(T, 1), dtype=torch.int32, device=device),
                      ell_nnz=torch.empty(max(T, 1), dtype=torch.int32, device=device),
                      ell_idx=torch.empty((max(T, 1), R), dtype=torch.int16, device=device),
                      ell_a=torch.empty((max(T, 1), R), dtype=BF16, device=device),
                      ell_u=torch.empty((max(T, 1), R), dtype=torch.float16, device=device) if gated else None,
                      backup_slot=torch.empty(max(T, 1), dtype=torch.int32, device=device),
                      backup_tok=torch.empty(cap1, dtype=torch.int32, device=device),
                      backup_a=torch.empty((cap1, I), dtype=torch.float32, device=device),
                      backup_u=torch.empty((cap1, I), dtype=torch.float32, device=device) if gated else None,
                      n_backup=torch.zeros(1, dtype=torch.int32, device=device),
                      route=_lib.ROUTES[route], dense_above=float(dense_above),
                      route_taken=torch.zeros(1, dtype=torch.int32, device=device))

    def struct(self) -> _lib.TwHybrid:
        return _lib.TwHybrid(self.T, self.I, self.R, self.backup_cap, _ptr(self.row_nnz), _ptr(self.ell_nnz),
                             _ptr(self.ell_idx), _ptr(self.ell_a), _ptr(self.ell_u), _ptr(self.backup_slot),
                             _ptr(self.backup_tok), _ptr(self.backup_a), _ptr(self.backup_u),
                             _ptr(self.n_backup), self.route, self.dense_above, _ptr(self.route_taken))

    def took_dense_route(self) -> bool:
        """Whether the last forward took the dense route (synchronises)."""
        return self.route_taken is not None and int(self.route_taken.item()) == 1


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------- ops

def twell_pack(A: torch.Tensor, W: int, C: int, status: torch.Tensor | None = None, out: TwELL | None = None) -> TwELL:
    """TwELL of a dense bf16 [T, I] matrix (into `out` when given)."""
    _check_bf16("A", A)
    T, I = A.shape
    if out is None:
        out = TwELL.empty(T, I, W, C, A.device)
    st = status if status is not None else new_status(A.device)
    s = out.struct()
    _lib.check(_lib.load().twell_pack(_ptr(A), T, I, W, C, s, _ptr(st), _stream()), "twell_pack")
    return out


def twell_unpack(tw_in: TwELL) -> torch.Tensor:
    """Dense bf16 [T, I] matrix of the stored TwELL slots (zeros elsewhere)."""
    A = torch.empty((max(tw_in.T, 1), tw_in.I), dtype=BF16, device=tw_in.cnt.device)
    s = tw_in.struct()
    _lib.check(_lib.load().twell_unpack(s, _ptr(A), _stream()), "twell_unpack")
    return A[:tw_in.T]


def hybrid_pack(A: torch.Tensor, U: torch.Tensor | None, W: int, C: int, R: int, backup_cap: int,
                status: torch.Tensor | None = None) -> "Hybrid":
    """Hybrid of a dense bf16 A [T, I] (and U, gated form) with ELL row capacity R,
    TwELL tile width W and capacity C for the overflow rule, and room for backup_cap
    backup rows."""
    _check_bf16("A", A)
    T, I = A.shape
    if U is not None:
        _check_bf16("U", U, (T, I))
    out = Hybrid.empty(T, I, R, backup_cap, U is not None, A.device)
    st = status if status is not None else new_status(A.device)
    L = _lib.load()
    ws = _workspace(L.hybrid_pack_workspace_size(T), A.device)
    s = out.struct()
    _lib.check(L.hybrid_pack(_ptr(A), _ptr(U), T, I, W, C, s, _ptr(ws), ws.numel(), _ptr(st), _stream()),
               "hybrid_pack")
    return out


def hybrid_unpack(h: "Hybrid", with_u: bool | None = None) -> tuple[torch.Tensor, torch.Tensor | None]:
    """Dense fp32 A (and U when the Hybrid is gated, or with_u) [T, I] from a Hybrid."""
    want_u = (h.ell_u is not None) if with_u is None else with_u
    dev = h.row_nnz.device
    A = torch.empty((max(h.T, 1), h.I), dtype=torch.float32, device=dev)
    U = torch.empty((max(h.T, 1), h.I), dtype=torch.float32, device=dev) if want_u else None
    s = h.struct()
    _lib.check(_lib.load().hybrid_unpack(s, _ptr(A), _ptr(U), _stream()), "hybrid_unpack")
    return A[:h.T], (U[:h.T] if U is not None else None)


def twell_gate_pack(x: torch.Tensor, Wg: torch.Tensor, W: int, C: int, want_dense: bool = False,
                    status: torch.Tensor | None = None, out: TwELL | None = None):
    """a = bf16(ReLU(x Wg^T)) packed into TwELL by the fused tensor-core kernel.
    Returns (TwELL, dense a or None)."""
    _check_bf16("x", x)
    T, d = x.shape
    I = Wg.shape[0]
    _check_bf16("Wg", Wg, (I, d))
    out = out or TwELL.empty(T, I, W, C, x.device)
    dense = torch.empty((T, I), dtype=BF16, device=x.device) if want_dense else None
    st = status if status is not None else new_status(x.device)
    s = out.struct()
    _lib.check(_lib.load().twell_gate_pack(_ptr(x), _ptr(Wg), T, d, I, W, C, s, _ptr(dense), _ptr(st), _stream()),
               "twell_gate_pack")
    return out, dense


class TwellFFN:
    """Preallocated inference forward: y = FFN(x) through TwELL."""

    def __init__(self, T: int, d: int, I: int, W: int, C: int, ovf_cap: int | None = None, device="cuda"):
        self.T, self.d, self.I, self.W, self.C = T, d, I, W, C
        self.ovf_cap = T if ovf_cap is None else ovf_cap
        self.tw = TwELL.empty(T, I, W, C, device)
        self.ws_bytes = int(_lib.load().twell_ffn_fwd_workspace_size(T, d, I, W, C, self.ovf_cap))
        self.ws = _workspace(self.ws_bytes, device)
        self.y = torch.empty((T, d), dtype=BF16, device=device)
        self.status = new_status(device)
        self._tws = self.tw.struct()

    def __call__(self, x, Wg, Wu, Wd) -> torch.Tensor:
        _check_bf16("x", x, (self.T, self.d))
        for n, w in (("Wg", Wg), ("Wu", Wu), ("Wd", Wd)):
            if w is not None:
                _check_bf16(n, w, (self.I, self.d))
        code = _lib.load().twell_ffn_fwd(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), self.T, self.d, self.I, self.W,
                                         self.C, self.ovf_cap, self._tws, _ptr(self.ws), self.ws_bytes,
                                         _ptr(self.y), _ptr(self.status), _stream())
        _lib.check(code, "twell_ffn_fwd")
        return self.y


def twell_ffn_fwd(x, Wg, Wu, Wd, W: int, C: int, ovf_cap: int | None = None):
    """One-shot inference forward. Returns (y, TwELL, status)."""
    T, d = x.shape
    f = TwellFFN(T, d, Wg.shape[0], W, C, ovf_cap, x.device)
    y = f(x, Wg, Wu, Wd)
    return y, f.tw, f.status


class HybridScratch:
    """Buffers several HybridFFN layers can share because each call is done with them
    when the next layer's call starts on the same stream: the forward and backward
    workspaces and the y and dx outputs (a layer's y must be consumed, e.g. by a
    residual add, before the next layer's forward overwrites it). Sized for the
    largest of the layers it serves."""

    def __init__(self, device="cuda"):
        self.device = device
        self.fwd_ws = _workspace(0, device)
        self.bwd_ws = _workspace(0, device)
        self.y = None
        self.dx = None

    def reserve(self, fwd_bytes: int, bwd_bytes: int, T: int, d: int) -> None:
        if self.fwd_ws.numel() < fwd_bytes:
            self.fwd_ws = _workspace(fwd_bytes, self.device)
        if self.bwd_ws.numel() < bwd_bytes:
            self.bwd_ws = _workspace(bwd_bytes, self.device)
        if self.y is None or self.y.shape != (T, d):
            self.y = torch.empty((T, d), dtype=BF16, device=self.device)
            self.dx = torch.empty((T, d), dtype=BF16, device=self.device)


class HybridFFN:
    """Preallocated training forward + backward through the Hybrid format.

    route: "sparse" (the pages' CUDA-core gathers for the ELL rows), "dense" (every
    row's projections as dense tensor-core GEMMs) or "auto" (decided on the device per
    forward: dense when the mean over rows of the ELL nonzeros, a backup row counting
    2 dense_above, exceeds dense_above). scratch: a
    HybridScratch shared with other layers (workspaces, y and dx), or None for own
    buffers."""

    def __init__(self, T: int, d: int, I: int, W: int, C: int, R: int, backup_cap: int, gated: bool = True,
                 device="cuda", route: str = "sparse", dense_above: float = 64.0,
                 scratch: HybridScratch | None = None):
        self.T, self.d, self.I, self.W, self.C, self.R = T, d, I, W, C, R
        self.backup_cap = backup_cap
        self.gated = gated
        L = _lib.load()
        self.saved = Hybrid.empty(T, I, R, backup_cap, gated, device, route=route, dense_above=dense_above)
        self._hs = self.saved.struct()
        rc = _lib.ROUTES[route]
        fwd_bytes = int(L.hybrid_ffn_fwd_workspace_size(T, d, I, W, C, R, backup_cap, rc))
        bwd_bytes = int(L.hybrid_ffn_bwd_workspace_size(T, d, I, R, backup_cap, rc))
        self.scratch = scratch
        if scratch is None:
            self.fwd_ws = _workspace(fwd_bytes, device)
            self.bwd_ws = _workspace(bwd_bytes, device)
            self.y = torch.empty((T, d), dtype=BF16, device=device)
            self.dx = torch.empty((T, d), dtype=BF16, device=device)
        else:
            scratch.reserve(fwd_bytes, bwd_bytes, T, d)
        self.dWg = torch.empty((I, d), dtype=torch.float32, device=device)
        self.dWu = torch.empty((I, d), dtype=torch.float32, device=device) if gated else None
        self.dWd = torch.empty((I, d), dtype=torch.float32, device=device)
        self.status = new_status(device)

    def fix_route(self) -> str:
        """Keep the route the last forward took for the following calls (synchronises
        once): a training loop whose layers change activity slowly decides each layer's
        route on the device in one step and then launches only that route's kernels.
        The workspaces sized for the automatic route serve either fixed route."""
        taken = _lib.TW_ROUTE_DENSE if self.saved.took_dense_route() else _lib.TW_ROUTE_SPARSE
        self.saved.route = taken
        self._hs = self.saved.struct()
        return "dense" if taken == _lib.TW_ROUTE_DENSE else "sparse"

    # the buffers a layer may share with others (see HybridScratch)
    @property
    def _fwd_ws(self):
        return self.scratch.fwd_ws if self.scratch is not None else self.fwd_ws

    @property
    def _bwd_ws(self):
        return self.scratch.bwd_ws if self.scratch is not None else self.bwd_ws

    @property
    def _y(self):
        return self.scratch.y if self.scratch is not None else self.y

    @property
    def _dx(self):
        return self.scratch.dx if self.scratch is not None else self.dx

    def forward(self, x, Wg, Wu, Wd) -> torch.Tensor:
        _check_bf16("x", x, (self.T, self.d))
        if (Wu is not None) != self.gated:
            raise ValueError("Wu must be given exactly for the gated form")
        ws, y = self._fwd_ws, self._y
        code = _lib.load().hybrid_ffn_fwd(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), self.T, self.d, self.I, self.W,
                                          self.C, self._hs, _ptr(ws), ws.numel(), _ptr(y), _ptr(self.status),
                                          _stream())
        _lib.check(code, "hybrid_ffn_fwd")
        return y

    def backward(self, dy, x, Wg, Wu, Wd, l1: float):
        _check_bf16("dy", dy, (self.T, self.d))
        ws, dx = self._bwd_ws, self._dx
        code = _lib.load().hybrid_ffn_bwd(_ptr(dy), _ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), self.T, self.d, self.I,
                                          self._hs, float(l1), _ptr(dx), _ptr(self.dWg), _ptr(self.dWu),
                                          _ptr(self.dWd), _ptr(ws), ws.numel(), _ptr(self.status), _stream())
        _lib.check(code, "hybrid_ffn_bwd")
        return dx, self.dWg, self.dWu, self.dWd


def gate_relu_dense(x: torch.Tensor, Wg: torch.Tensor, status: torch.Tensor | None = None) -> torch.Tensor:
    """Dense a = bf16(ReLU(x Wg^T)) [T, I]: the first stage of the unfused pipeline."""
    _check_bf16("x", x)
    _check_bf16("Wg", Wg)
    T, d = x.shape
    I = Wg.shape[0]
    a = torch.empty((T, I), dtype=BF16, device=x.device)
    st = status if status is not None else new_status(x.device)
    _lib.check(_lib.load().tw_gate_relu_dense(_ptr(x), _ptr(Wg), T, d, I, _ptr(a), _ptr(st), _stream()),
               "tw_gate_relu_dense")
    return a


class TwellSparseFFN:
    """Preallocated sparse part of the inference forward on an already packed TwELL
    (the unfused pipeline's last stage; see twell_ffn_sparse_fwd)."""

    def __init__(self, T: int, d: int, I: int, W: int, C: int, ovf_cap: int | None = None, device="cuda"):
        self.T, self.d, self.I, self.W, self.C = T, d, I, W, C
        self.ovf_cap = T if ovf_cap is None else ovf_cap
        self.ws_bytes = int(_lib.load().twell_ffn_fwd_workspace_size(T, d, I, W, C, self.ovf_cap))
        self.ws = _workspace(self.ws_bytes, device)
        self.y = torch.empty((T, d), dtype=BF16, device=device)
        self.status = new_status(device)

    def __call__(self, x, Wg, Wu, Wd, packed: "TwELL") -> torch.Tensor:
        _check_bf16("x", x, (self.T, self.d))
        s = packed.struct()
        code = _lib.load().twell_ffn_sparse_fwd(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), self.T, self.d, self.I, self.W,
                                                self.C, self.ovf_cap, ctypes.byref(s), _ptr(self.ws), self.ws_bytes,
                                                _ptr(self.y), _ptr(self.status), _stream())
        _lib.check(code, "twell_ffn_sparse_fwd")
        return self.y


def hybrid_neuron_counts(saved: "Hybrid", counts: torch.Tensor | None = None) -> torch.Tensor:
    """counts[j] += tokens with a_tj != 0 in the saved Hybrid (ELL entries and dense
    backup rows). A new zeroed [I] int32 tensor is used when none is given."""
    if counts is None:
        counts = torch.zeros(saved.I, dtype=torch.int32, device=saved.row_nnz.device)
    if counts.dtype != torch.int32 or counts.numel() != saved.I or not counts.is_contiguous():
        raise ValueError("counts must be a contiguous int32 tensor of I elements")
    s = saved.struct()
    _lib.check(_lib.load().hybrid_neuron_counts(ctypes.byref(s), _ptr(counts), _stream()), "hybrid_neuron_counts")
    return counts


def reinit_dead_rows(W: torch.Tensor, counts: torch.Tensor, seed: int, std: float) -> torch.Tensor:
    """Redraw (in place) every row j of the bf16 matrix W [I, d] with counts[j] == 0
    (see tw_reinit_dead_rows). Returns the device int32 count of rows redrawn."""
    _check_bf16("W", W)
    I, d = W.shape
    if counts.dtype != torch.int32 or counts.numel() != I:
        raise ValueError("counts must be an int32 tensor of I elements")
    n = torch.zeros(1, dtype=torch.int32, device=W.device)
    _lib.check(_lib.load().tw_reinit_dead_rows(_ptr(W), I, d, _ptr(counts), int(seed) & ((1 << 64) - 1), float(std),
                                               _ptr(n), _stream()), "tw_reinit_dead_rows")
    return n


def dense_gemm(A: torch.Tensor, B: torch.Tensor, M: int, N: int, K: int, a_mn: bool, b_mn: bool,
               status: torch.Tensor | None = None, pair: bool = False) -> torch.Tensor:
    """D = A B (fp32) on the tcgen05 GEMM engine. A is [M, K] (a_mn False) or stored
    [K, M]; B is stored [N, K] (b_mn False) or [K, N]. pair: on CTA pairs
    (tw_dense_gemm_pair, N % 256 == 0)."""
    _check_bf16("A", A)
    _check_bf16("B", B)
    D = torch.empty((M, N), dtype=torch.float32, device=A.device)
    st = status if status is not None else new_status(A.device)
    name = "tw_dense_gemm_pair" if pair else "tw_dense_gemm"
    _lib.check(getattr(_lib.load(), name)(_ptr(A), _ptr(B), M, N, K, int(a_mn), int(b_mn), _ptr(D), _ptr(st),
                                          _stream()), name)
    return D


def fma_probe(out: torch.Tensor, blocks: int, iters: int) -> float:
    """Launch the fp32 FMA throughput probe (see tw_fma_probe) on the current stream;
    `out` is a float32 device tensor of at least blocks * 256 elements. Returns the
    FLOPs the launch performs."""
    if out.dtype != torch.float32 or not out.is_cuda or out.numel() < blocks * 256:
        raise ValueError("out must be a float32 CUDA tensor of at least blocks * 256 elements")
    flops = ctypes.c_double(0.0)
    _lib.check(_lib.load().tw_fma_probe(_ptr(out), int(blocks), int(iters), ctypes.byref(flops), _stream()),
               "tw_fma_probe")
    return flops.value


def l2_gather_probe(table: torch.Tensor, idx: torch.Tensor, out: torch.Tensor | None = None,
                    blocks: int | None = None) -> tuple[torch.Tensor, float]:
    """Launch the L2 row-gather probe (see tw_l2_gather_probe) on the current stream
    over table [rows, d] bf16 and idx [n] int32; returns (out, bytes gathered)."""
    _check_bf16("table", table)
    rows, d = table.shape
    L = _lib.load()
    nb = blocks if blocks is not None else L.tw_l2_gather_probe_blocks(d)
    if out is None:
        out = torch.empty(nb * d // 8, dtype=torch.float32, device=table.device)
    b = ctypes.c_double(0.0)
    _lib.check(L.tw_l2_gather_probe(_ptr(table), rows, d, _ptr(idx), idx.numel(), _ptr(out), nb, ctypes.byref(b),
                                    _stream()), "tw_l2_gather_probe")
    return out, b.value
