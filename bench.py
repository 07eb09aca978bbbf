"""Benchmark of the activation-sparse FFN hot path on one GB300 (or N replicas).

A step is one Hybrid training step of one gated ReLU FFN layer through the
library's C ABI: hybrid_ffn_fwd (gate GEMM + fused TwELL pack, Hybrid conversion,
sparse up/down on the CUDA cores, dense backup on the tensor cores) followed by
hybrid_ffn_bwd (sparse backward with L1 injection, transposed-Hybrid weight
gradients, dense backup GEMMs). Inputs are seeded synthetic bf16 tensors of the
pages' 1.5B-model FFN shape (see synthetic/workloads.py for the recipe).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--tokens T] [--no-cpu-baseline]
                    [--no-dense] [--no-inference] [--no-stack] [--no-sweep] [--clock-soak S]

Prints ONE JSON line (rank 0). Timing: W untimed warm-up steps, then K steps each
bracketed by CUDA events on the launching stream with a 256 MiB L2 flush between
steps (outside the events); barrier + synchronize around the timed region and the
max over ranks. The same K-step region is then repeated until the clock sampler has
seen a few seconds of it (the `clocks` record and `repeats`); `value` is the first
one. Per-kernel durations come from events the library records after each of its
launches during further timed steps (tw_trace_begin).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse gated-FFN fwd+bwd input tokens/ms (d2048,I5632) and % of roofline"
UNIT = "tokens/ms"
DEFAULT_WORKLOAD = "train_d2048_i5632_m29_o1"
# the automatic route takes the dense tensor-core path above this many nonzeros per ELL
# row (the crossover of the two routes measured across the sweep)
DENSE_ABOVE = 64.0
# seconds of fp64 oracle work the cpu_baseline sample is sized to
CPU_TARGET_S = 12.0
L2_FLUSH_BYTES = 256 << 20


def _peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float, device) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines: list[str] = []
        self.target = self._nvsmi_index(device_index)

    @staticmethod
    def _nvsmi_index(device_index: int) -> str | None:
        try:
            import torch
            p = torch.cuda.get_device_properties(device_index)
            bus = getattr(p, "pci_bus_id", None)
            dom = getattr(p, "pci_domain_id", 0)
            dev = getattr(p, "pci_device_id", 0)
            if bus is not None:
                return f"{dom:08X}:{bus:02X}:{dev:02X}.0"
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return str(device_index)

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.target is not None:
            cmd += ["-i", self.target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines) -> dict:
        """Median SM clock, the highest maximum clock, the throttle reasons seen active
        and the sample count, from nvidia-smi CSV lines of FIELDS (malformed lines and
        unreadable clocks are skipped)."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ algorithmic work per kernel
def kernel_work(label: str, spec, stats: dict) -> tuple[str, float] | None:
    """(bound, algorithmic bytes or FLOPs) of one launch of a kernel, from the step's
    measured active counts. Bytes count each tensor the kernel must read or write
    once; weights are read once per launch."""
    T, d, I, R = spec.T, spec.d, spec.I, spec.R
    nT = I // spec.W
    nnz_ell = stats["nnz_ell"]          # entries in ELL rows
    nb = stats["n_backup"]
    g = 2 if spec.gated else 1          # weight matrices gathered per entry in the forward
    if label == "gate_pack":
        return "tensor", 2.0 * T * d * I
    if label == "sparse_fwd":
        # x (gated) + y + TwELL counts + TwELL entries (val, idx) + ELL written (idx, a, u) + weights
        b = (T * d * 2 if spec.gated else 0) + T * d * 2 + T * nT * 2 + nnz_ell * 3 + nnz_ell * 6 + g * I * d * 2
        return "hbm", float(b)
    if label == "sparse_bwd_token":
        # dy + dx + ELL read (idx, a, u) + one 16-byte column record written per
        # entry + three weight matrices
        return "hbm", float(2 * T * d * 2 + nnz_ell * 6 + nnz_ell * 16 + 3 * I * d * 2)
    if label == "ell_weight_grad":
        # x and dy read + dW written (fp32, 3 matrices) + one 16-byte column record
        # read per entry
        return "hbm", float(2 * T * d * 2 + 3 * I * d * 4 + nnz_ell * 16)
    if label in ("dense_up", "dense_down", "dense_grad"):
        return "tensor", 2.0 * T * d * I
    if label == "dense_dx":
        return "tensor", 2.0 * g * T * d * I
    if label == "dense_weight_grad":
        return "tensor", 2.0 * (g + 1) * T * d * I
    if label == "backup_hidden":
        return "tensor", 2.0 * 2 * nb * d * I
    if label == "backup_grad":
        return "tensor", 2.0 * nb * d * I
    if label == "backup_rows_gemm":
        return "tensor", 2.0 * 2 * nb * I * d      # two K segments: y's (hi, lo), or a non-gated dx
    if label == "backup_rows_gemm4":
        return "tensor", 2.0 * 4 * nb * I * d      # the gated dx: dG and dU, each (hi, lo)
    if label == "backup_weight_grad":
        return "tensor", 2.0 * 2 * nb * I * d
    return None


# L2 figure derived from ncu: lts__throughput read 47-54 % while the token kernels
# moved 11.5-13.1 TB/s of L2 sectors, i.e. 100 % = 24.2 TB/s (see
# profiles/token_kernels_train_d2048_i5632_m29_o1.md). Reported beside the gather
# rate the library's probe measures in the same run, which is the denominator.
L2_NCU_DERIVED_GBS = 24200.0


def measured_traffic(label: str, workload: str) -> float | None:
    """DRAM bytes per launch of `label` from the committed ncu summary for `workload`
    (profiles/dram_traffic_<workload>.txt), or None when there is none or the
    kernel's sources changed since it was taken (their sha256 no longer matches)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if not f or f[0].startswith("#") or f[0] != label or len(f) != 5:
            continue
        m = hashlib.sha256()
        for src in f[3].split(","):
            with open(os.path.join(ROOT, "activation_sparse_feedforward_gb300", "csrc", src), "rb") as fh:
                m.update(fh.read())
        return float(f[1]) + float(f[2]) if m.hexdigest()[:16] == f[4] else None
    return None


def gathered_bytes(label: str, spec, stats: dict) -> float | None:
    """Row-slice bytes a gather kernel must pull through L2 per launch: every ELL entry
    costs whole d-rows of the matrices it touches."""
    row = spec.d * 2
    e = stats["nnz_ell"]
    if label == "sparse_fwd":
        return float((2 if spec.gated else 1) * e * row)
    if label == "sparse_bwd_token":
        return float((3 if spec.gated else 2) * e * row)
    if label == "ell_weight_grad":
        return float(2 * e * row)
    return None


# ------------------------------------------------------------------ oracle timing (CPU)
def oracle_sample_time(spec, inp, n_tokens: int) -> tuple[float, int, str]:
    """Time the fp64 oracle (as it stands) over the whole hot path for a sample of
    n_tokens tokens: dense forward, TwELL and Hybrid packing, dense backward."""
    import numpy as np

    from oracle import ffn, formats

    rows = np.arange(n_tokens)
    x, dy = inp["x"][rows], inp["dy"][rows]
    t0 = time.perf_counter()
    f = ffn.forward(x, inp["Wg"], inp["Wu"], inp["Wd"])
    formats.twell_pack(f["a"], spec.W, spec.C)
    formats.hybrid_pack(f["a"], f["u"], spec.W, spec.C, spec.R)
    ffn.backward(x, inp["Wg"], inp["Wu"], inp["Wd"], dy, spec.l1, fwd=f)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dt, cores, f"first {n_tokens} tokens of {spec.name}, full weights, fp64 numpy (BLAS threads: all cores)"


# ------------------------------------------------------------------ step roofline
def step_roofline(spec, stats: dict, ms_per_step: float, peaks: dict) -> dict:
    """The whole training step's roofline: the slower of (gate + dense backup + sparse
    FLOPs at the sustained bf16 peak) and (algorithmic bytes at HBM peak), from the
    step's measured ELL entries and backup rows."""
    T, d, I = spec.T, spec.d, spec.I
    nw = 3 if spec.gated else 2
    F = (2.0 * T * d * I + (14.0 if spec.gated else 10.0) * d * I * stats["n_backup"]
         + (16.0 if spec.gated else 10.0) * d * stats["nnz_ell"])
    B = (3 * T * d * 2 + 2 * T * d * 2 + 2 * nw * I * d * 2 + nw * I * d * 4 + stats["nnz_ell"] * (6 + 6 + 8 + 4))
    t_roof = max(F / (peaks["bf16_tflops_sustained"] * 1e12), B / (peaks["hbm_gbs"] * 1e9))
    return {"tokens_per_ms": T / (t_roof * 1e3), "frac": (T / ms_per_step) / (T / (t_roof * 1e3)), "flops": F,
            "bytes": B}


def dense_train_step(x, Wg, Wu, Wd, dy, l1):
    """The dense bf16 FFN (torch / cuBLAS) forward + backward with the same L1 term,
    as a closure over fresh leaf copies of the inputs."""
    import torch

    ws = [w.detach().clone().requires_grad_(True) for w in (Wg, Wu, Wd) if w is not None]
    Wg_, Wd_ = ws[0], ws[-1]
    Wu_ = ws[1] if Wu is not None else None
    x_ = x.detach().clone().requires_grad_(True)

    def step():
        a = torch.relu(x_ @ Wg_.T)
        h = a * (x_ @ Wu_.T) if Wu_ is not None else a
        torch.autograd.backward([h @ Wd_, a], [dy, torch.full_like(a, l1)])
        x_.grad = None
        for w in ws:
            w.grad = None

    return step


def measure_l2_gather(dev, stream, d: int = 2048, table_rows: int = 3 * 5632, n_idx: int = 1 << 22) -> dict:
    """Row-slice gather rate of this GPU from an L2-resident table the size of the three
    gated weight matrices at d 2048, I 5632 (66 MiB), with the access pattern and
    residency of the token kernels (tw_l2_gather_probe): the median of 5 timed
    launches after two untimed ones."""
    import torch

    import activation_sparse_feedforward_gb300 as tw

    g = torch.Generator(device=dev)
    g.manual_seed(0)
    table = torch.randn((table_rows, d), generator=g, device=dev).to(torch.bfloat16)
    idx = torch.randint(0, table_rows, (n_idx,), generator=g, device=dev, dtype=torch.int32)
    out, nbytes = tw.l2_gather_probe(table, idx)
    for _ in range(2):
        tw.l2_gather_probe(table, idx, out=out)
    ts = []
    for _ in range(5):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record(stream)
        tw.l2_gather_probe(table, idx, out=out)
        e_.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(s_.elapsed_time(e_))
    ms = statistics.median(ts)
    if not bool(torch.isfinite(out).all()):
        raise RuntimeError("l2 gather probe produced non-finite values")
    return {"gbs": nbytes / (ms * 1e-3) / 1e9, "ms": ms, "bytes": nbytes, "table_mib": table_rows * d * 2 / 2**20,
            "row_slice_bytes": 512, "loads_in_flight_per_warp": 8,
            "ncu_derived_gbs": L2_NCU_DERIVED_GBS}


# ------------------------------------------------------------------ secondary measurements
def _time_steps(fn, steps: int, warmup: int, flush, stream) -> float:
    """Average device ms of fn over `steps` calls, L2 flushed (untimed) before each."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        total += s.elapsed_time(e)
    return total / steps


def measure_fma_peak(dev, stream) -> dict:
    """CUDA-core fp32 FMA rate of this GPU from the library's probe kernel (packed
    two-lane FMAs, 2048 threads per SM): the median of 5 timed launches."""
    import torch

    import activation_sparse_feedforward_gb300 as tw

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = sms * 8, 16384
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    for _ in range(2):
        flops = tw.fma_probe(out, blocks, iters)
    ts = []
    for _ in range(5):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record(stream)
        tw.fma_probe(out, blocks, iters)
        e_.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(s_.elapsed_time(e_))
    ms = statistics.median(ts)
    if not bool(torch.isfinite(out).all()):
        raise RuntimeError("fma probe produced non-finite values")
    return {"tflops": flops / (ms * 1e-3) / 1e12, "ms": ms, "blocks": blocks, "threads": 256, "iters": iters,
            "instruction": "fma.rn.f32x2"}


def measure_inference(dev, flush, stream, steps: int) -> dict:
    """TwELL inference forward at the gated and non-gated 1.5B FFN shapes, next to the
    dense bf16 forward (cuBLAS through torch) on the same inputs."""
    import numpy as np
    import torch

    import activation_sparse_feedforward_gb300 as tw
    from synthetic import WORKLOADS, make_inputs

    out = {}
    for name in ("gated_fwd_d2048_i5632", "nongated_fwd_d2048_i8192"):
        spec = WORKLOADS[name]
        inp = make_inputs(spec)
        x, Wg, Wu, Wd = (None if inp[k] is None else
                         torch.from_numpy(inp[k].view(np.int16)).view(torch.bfloat16).to(dev)
                         for k in ("x", "Wg", "Wu", "Wd"))
        f = tw.TwellFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=512, device=dev)
        ms = _time_steps(lambda: f(x, Wg, Wu, Wd), steps, 3, flush, stream)
        tw.raise_if_device_error(f.status, name)

        def dense():
            a = torch.relu(x @ Wg.T)
            h = a * (x @ Wu.T) if Wu is not None else a
            return h @ Wd

        ms_d = _time_steps(dense, steps, 3, flush, stream)

        # the unfused pipeline: dense a through HBM, standalone packer, sparse part
        a_buf = torch.empty((spec.T, spec.I), dtype=torch.bfloat16, device=dev)
        packed = tw.TwELL.empty(spec.T, spec.I, spec.W, spec.C, dev)
        st = tw.new_status(dev)
        sp = tw.TwellSparseFFN(spec.T, spec.d, spec.I, spec.W, spec.C, ovf_cap=512, device=dev)

        def unfused():
            L = tw.load()
            L.tw_gate_relu_dense(x.data_ptr(), Wg.data_ptr(), spec.T, spec.d, spec.I, a_buf.data_ptr(), st.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
            tw.twell_pack(a_buf, spec.W, spec.C, status=st, out=packed)
            return sp(x, Wg, Wu, Wd, packed)

        ms_u = _time_steps(unfused, steps, 3, flush, stream)
        tw.raise_if_device_error(st, name + " unfused")
        tw.raise_if_device_error(sp.status, name + " unfused")
        out[name] = {"tokens_per_ms": spec.T / ms, "ms": ms, "dense_bf16_tokens_per_ms": spec.T / ms_d,
                     "unfused_tokens_per_ms": spec.T / ms_u, "unfused_ms": ms_u,
                     "n_overflow_rows": int(f.tw.n_ovf.item()),
                     "nnz_per_token": float(f.tw.row_nnz.float().mean().item())}
        del a_buf, packed, sp
    return out


def probe_backup_cap(spec, x, Wg, Wu, Wd, dev) -> int:
    """The dense backup sized to hold a workload's backup rows: counted by one forward
    with room for every row, rounded up to whole 128-row tiles with one spare tile."""
    import torch

    import activation_sparse_feedforward_gb300 as tw

    probe = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, spec.T, gated=spec.gated, device=dev)
    probe.forward(x, Wg, Wu, Wd)
    cap = min(spec.T, 128 * int(math.ceil(int(probe.saved.n_backup.item()) / 128.0)) + 128)
    del probe
    torch.cuda.empty_cache()
    return cap


def measure_sweep(dev, flush, stream, steps: int, peaks: dict) -> list:
    """The training step over the sparsity sweep (mean actives x outlier fraction) and
    the non-gated training step, each next to the dense bf16 step on the same inputs,
    with its ELL / backup split and step roofline fraction."""
    import numpy as np
    import torch

    import activation_sparse_feedforward_gb300 as tw
    from synthetic import WORKLOADS, make_inputs

    names = [f"train_d2048_i5632_m{m}_o{o}" for m in (29, 108, 911) for o in (0, 1, 5)]
    names.append("train_nongated_d2048_i8192_m40_o1")
    rows = []
    for name in names:
        spec = WORKLOADS[name]
        inp = make_inputs(spec, with_dy=True)
        x, Wg, Wu, Wd, dy = (None if inp[k] is None else torch.from_numpy(inp[k].view(np.int16)).view(torch.bfloat16).to(dev)
                             for k in ("x", "Wg", "Wu", "Wd", "dy"))
        cap = probe_backup_cap(spec, x, Wg, Wu, Wd, dev)
        row = {"workload": spec.name, "C": spec.C, "R": spec.R, "backup_cap": cap, "dense_above": DENSE_ABOVE}
        for route in ("auto", "sparse", "dense"):
            h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, cap, gated=spec.gated, device=dev,
                             route=route, dense_above=DENSE_ABOVE)

            def step():
                h.forward(x, Wg, Wu, Wd)
                h.backward(dy, x, Wg, Wu, Wd, spec.l1)

            # the sparse route at high activity takes tens of ms a step: fewer steps
            n = steps if route != "sparse" or spec.mean_active < 200 else 3
            ms = _time_steps(step, n, 3 if n > 3 else 1, flush, stream)
            tw.raise_if_device_error(h.status, f"{spec.name} {route}")
            if route == "auto":
                stats = {"n_backup": int(h.saved.n_backup.item()), "nnz_ell": int(h.saved.ell_nnz.sum().item()),
                         "nnz": float(h.saved.row_nnz[:spec.T].float().mean().item())}
                roof = step_roofline(spec, stats, ms, peaks)
                row.update({"tokens_per_ms": spec.T / ms, "ms": ms,
                            "route_taken": "dense" if h.saved.took_dense_route() else "sparse",
                            "n_backup": stats["n_backup"], "backup_rows_frac": stats["n_backup"] / spec.T,
                            "nnz_ell": stats["nnz_ell"], "nnz_per_token": stats["nnz"],
                            "ell_entries_per_ell_row": stats["nnz_ell"] / max(1, spec.T - stats["n_backup"]),
                            "step_roofline_frac": roof["frac"], "step_roofline_tokens_per_ms": roof["tokens_per_ms"]})
            else:
                row[f"{route}_route_tokens_per_ms"] = spec.T / ms
            del h
            torch.cuda.empty_cache()
        ms_d = _time_steps(dense_train_step(x, Wg, Wu, Wd, dy, spec.l1), steps, 3, flush, stream)
        row["dense_bf16_tokens_per_ms"] = spec.T / ms_d
        row["vs_dense"] = row["tokens_per_ms"] / row["dense_bf16_tokens_per_ms"]
        rows.append(row)
        del x, Wg, Wu, Wd, dy
        torch.cuda.empty_cache()
    return rows


def measure_stack(dev, flush, stream, steps: int, n_layers: int = 28, T: int = 8192) -> dict:
    """The 28-layer residual stack x_{l+1} = x_l + FFN_l(x_l) at the 1.5B shape, with the
    per-layer activity profile: forward alone and forward + backward (the backward
    carries g_l = g_{l+1} + dx_l down the stack), next to the same stack in dense bf16
    torch (cuBLAS + autograd, same L1 term). The residual adds are bf16 torch adds in
    both; every FFN step of the sparse stack runs in the library."""
    import numpy as np
    import torch

    import activation_sparse_feedforward_gb300 as tw
    from synthetic import make_stack, stack_layer_spec

    def to_dev(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)

    specs = [stack_layer_spec(l, T=T) for l in range(n_layers)]
    st = make_stack(specs)
    Ws = [{k: to_dev(v) for k, v in w.items()} for w in st["layers"]]
    x0, dyt = to_dev(st["x0"]), to_dev(st["dy"])
    cap = min(T, 128 * int(math.ceil(1.5 * 0.01 * T / 128.0)) + 128)
    # memory: the peak allocated above the inputs and weights, through the stack's
    # buffers (saved Hybrids, workspaces, outputs, dW of every layer) and one step
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    scratch = tw.HybridScratch(dev)
    ffns = [tw.HybridFFN(T, sp.d, sp.I, sp.W, sp.C, sp.R, cap, gated=True, device=dev, route="auto",
                         dense_above=DENSE_ABOVE, scratch=scratch) for sp in specs]
    xs = [None] * n_layers

    def fwd():
        x = x0
        for l in range(n_layers):
            xs[l] = x
            x = x + ffns[l].forward(x, Ws[l]["Wg"], Ws[l]["Wu"], Ws[l]["Wd"])
        return x

    def bwd():
        g = dyt
        for l in reversed(range(n_layers)):
            g = g + ffns[l].backward(g, xs[l], Ws[l]["Wg"], Ws[l]["Wu"], Ws[l]["Wd"], specs[l].l1)[0]
        return g

    def train():
        fwd()
        bwd()

    train()
    torch.cuda.synchronize(dev)
    peak_ours = torch.cuda.max_memory_allocated(dev) - mem0
    # each layer keeps the route the device chose for it in that first step
    routes = [f.fix_route() for f in ffns]
    ms_f = _time_steps(fwd, steps, 3, flush, stream)
    ms_t = _time_steps(train, steps, 3, flush, stream)
    for l, f in enumerate(ffns):
        tw.raise_if_device_error(f.status, f"stack layer {l}")
    out = {"layers": n_layers, "tokens": T, "fwd_tokens_per_ms": T / ms_f, "train_tokens_per_ms": T / ms_t,
           "fwd_ms": ms_f, "train_ms": ms_t,
           "route": f"auto (dense above {DENSE_ABOVE:g} nonzeros per ELL row) in the first step, then each "
                    "layer's route kept (fix_route)",
           "routes_taken": routes,
           "layer_buffers": "one shared scratch (workspaces, y, dx) for all layers; per layer: saved Hybrid, dW",
           "n_backup": [int(f.saved.n_backup.item()) for f in ffns],
           "nnz_per_token": [round(float(f.saved.row_nnz.float().mean().item()), 2) for f in ffns]}
    del ffns, xs, scratch
    torch.cuda.empty_cache()

    # dense bf16 stack on the same weights
    P = [{k: w.detach().clone().requires_grad_(True) for k, w in W.items()} for W in Ws]
    l1 = specs[0].l1

    def dense_fwd(keep):
        x, acts = x0, []
        for W in P:
            a = torch.relu(x @ W["Wg"].T)
            acts.append(a)
            x = x + (a * (x @ W["Wu"].T)) @ W["Wd"]
        return x, acts

    def dense_fwd_only():
        with torch.no_grad():
            dense_fwd(False)

    def dense_train():
        y, acts = dense_fwd(True)
        torch.autograd.backward([y] + acts, [dyt] + [torch.full_like(a, l1) for a in acts])
        for W in P:
            for w in W.values():
                w.grad = None

    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    dense_train()
    torch.cuda.synchronize(dev)
    peak_dense = torch.cuda.max_memory_allocated(dev) - mem0
    out["memory"] = {"hybrid_stack_peak_bytes": peak_ours, "dense_stack_peak_bytes": peak_dense,
                     "ratio": peak_ours / peak_dense,
                     "what": "torch.cuda.max_memory_allocated during one training step minus the memory held "
                             "before it (inputs, weights); ours includes every layer's preallocated library "
                             "buffers (saved Hybrid, workspaces, y, dx, dW), dense its autograd activations "
                             "and gradients"}
    out["dense_fwd_tokens_per_ms"] = T / _time_steps(dense_fwd_only, steps, 3, flush, stream)
    out["dense_train_tokens_per_ms"] = T / _time_steps(dense_train, steps, 3, flush, stream)
    out["dense_impl"] = "torch bf16 matmul + autograd (cuBLAS)"
    return out


# ------------------------------------------------------------------ our arm
def run_ours(args, dist: Dist) -> dict | None:
    import numpy as np
    import torch

    import activation_sparse_feedforward_gb300 as tw
    from synthetic import WORKLOADS, make_inputs

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    peaks = _peaks()
    spec = WORKLOADS[args.workload].with_(seed=dist.rank)
    if args.tokens:
        spec = spec.with_(T=args.tokens)
    inp = make_inputs(spec, with_dy=True)

    def to_dev(b):
        return None if b is None else torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)

    x, Wg, Wu, Wd, dy = (to_dev(inp[k]) for k in ("x", "Wg", "Wu", "Wd", "dy"))
    backup_cap = probe_backup_cap(spec, x, Wg, Wu, Wd, dev)
    h = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated, device=dev,
                     route=args.route, dense_above=DENSE_ABOVE)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        h.forward(x, Wg, Wu, Wd)
        h.backward(dy, x, Wg, Wu, Wd, spec.l1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    tw.raise_if_device_error(h.status, "warm-up")
    stats = {"n_backup": int(h.saved.n_backup.item()), "nnz_ell": int(h.saved.ell_nnz.sum().item()),
             "nnz": int(h.saved.row_nnz[:spec.T].sum().item()),
             "route": "dense" if h.saved.took_dense_route() else "sparse"}

    # kernel trace events (materialised once so their handles exist)
    per_step_cap = 64
    tev = [torch.cuda.Event(enable_timing=True) for _ in range(per_step_cap * args.steps)]
    for e in tev:
        e.record(stream)
    torch.cuda.synchronize(dev)
    import ctypes
    arr = (ctypes.c_void_p * len(tev))(*[e.cuda_event for e in tev])
    L = tw.load()

    # ---- headline: K steps, L2 flushed (untimed) before each, no trace events. The
    # same K-step region is repeated until the clock sampler has watched it for
    # --clock-soak seconds; `value` is the first region, the others give the spread.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(dist.local_rank)
    regions = []
    clocks.start()
    t_soak = time.monotonic()
    while True:
        dist.barrier()
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
        regions.append([s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)])
        # every rank takes the same decision (rank 0's clock)
        done = dist.max(1.0 if time.monotonic() - t_soak >= args.clock_soak else 0.0, dev) > 0
        if done or len(regions) >= 10000:
            break
    clk = clocks.stop()
    tw.raise_if_device_error(h.status, "timed steps")
    step_ms = regions[0]
    total_ms = dist.max(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    value = spec.T * dist.world * args.steps / total_ms
    region_values = [spec.T * args.steps / sum(r) for r in regions]
    repeats = {"regions": len(regions), "value_median": statistics.median(region_values),
               "value_min": min(region_values), "value_max": max(region_values),
               "seconds": time.monotonic() - t_soak}
    if clk.get("sm_mhz") and clk.get("sm_max_mhz"):
        # the first region's time scaled to the maximum SM clock (time x median MHz)
        repeats["ms_per_step_at_max_clock"] = ms_per_step * clk["sm_mhz"] / clk["sm_max_mhz"]

    # ---- warm L2: the same K steps back to back
    ws_, we_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    ws_.record(stream)
    for i in range(args.steps):
        step()
    we_.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = dist.max(ws_.elapsed_time(we_), dev)
    warm = {"value": spec.T * dist.world * args.steps / warm_ms, "ms_per_step": warm_ms / args.steps,
            "l2": "no flush between steps"}

    # ---- kernel trace: K more flushed steps with an event after every library launch
    tstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    assert L.tw_trace_begin(arr, len(tev)) == 0
    for i in range(args.steps):
        flush.zero_()
        tstarts[i].record(stream)
        step()
    n_ev = L.tw_trace_end()
    torch.cuda.synchronize(dev)
    tw.raise_if_device_error(h.status, "traced steps")

    # per-kernel durations: event i ends launch i; the step's start event precedes launch 0
    labels = [L.tw_trace_label(i).decode() for i in range(n_ev)]
    if n_ev % args.steps != 0 or n_ev == len(tev):
        raise RuntimeError(f"kernel trace incomplete: {n_ev} events for {args.steps} steps")
    per_step = n_ev // args.steps
    per_kernel: dict[str, list[float]] = {}
    launches = 0
    for i in range(args.steps):
        prev = tstarts[i]
        for k in range(i * per_step, (i + 1) * per_step):
            per_kernel.setdefault(labels[k], []).append(prev.elapsed_time(tev[k]))
            launches += labels[k] != "memset"
            prev = tev[k]
    kernels = {lab: {"launches": len(v), "total_ms": sum(v), "avg_us": 1e3 * sum(v) / len(v)}
               for lab, v in per_kernel.items()}
    total_k = sum(v["total_ms"] for v in kernels.values()) or 1.0
    for v in kernels.values():
        v["share"] = v["total_ms"] / total_k
    dom = max((lab for lab in kernels if lab != "memset"), key=lambda lab: kernels[lab]["total_ms"])
    bound, work = kernel_work(dom, spec, stats) or ("hbm", 0.0)
    avg_s = kernels[dom]["avg_us"] * 1e-6
    if bound == "tensor":
        achieved = work / avg_s / 1e12
        peak = peaks["bf16_tflops_sustained"]
        unit = "TFLOP/s"
    else:
        achieved = work / avg_s / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak,
                "traffic": measured_traffic(dom, spec.name) if not args.tokens else None,
                "peak_source": f"{peaks['source']} ({'bf16 sustained' if bound == 'tensor' else 'HBM copy'})"}
    l2 = measure_l2_gather(dev, stream, d=spec.d, table_rows=(3 if spec.gated else 2) * spec.I)
    for lab, v in kernels.items():
        kw = kernel_work(lab, spec, stats)
        if kw:
            b, w = kw
            v["bound"] = b
            v["achieved"] = (w / (v["avg_us"] * 1e-6)) / (1e12 if b == "tensor" else 1e9)
            if b == "hbm":
                v["hbm_frac"] = v["achieved"] / peaks["hbm_gbs"]
        gb = gathered_bytes(lab, spec, stats)
        if gb:
            v["l2_gather_gbs"] = gb / (v["avg_us"] * 1e-6) / 1e9
            v["l2_gather_frac"] = v["l2_gather_gbs"] / l2["gbs"]
    gb = gathered_bytes(dom, spec, stats)
    if gb:
        # what actually bounds a gather kernel: row slices through L2, against the rate
        # the library's gather probe reaches in this run
        roofline["l2_gather"] = {"achieved": gb / avg_s / 1e9, "peak": l2["gbs"], "unit": "GB/s",
                                 "frac": gb / avg_s / 1e9 / l2["gbs"], "bytes": gb,
                                 "peak_source": "measured: tw_l2_gather_probe in this run",
                                 "ncu_derived_peak": L2_NCU_DERIVED_GBS}

    step_roof = step_roofline(spec, stats, ms_per_step, peaks)
    F = step_roof["flops"]
    B = step_roof["bytes"]
    # secondary: the sparse FLOPs priced at the measured CUDA-core fp32 FMA rate (they
    # run on CUDA cores), the gate and backup FLOPs at the tensor peak
    fma = measure_fma_peak(dev, stream)
    F_sparse = (16.0 if spec.gated else 10.0) * spec.d * stats["nnz_ell"]
    t_roof2 = max((F - F_sparse) / (peaks["bf16_tflops_sustained"] * 1e12) + F_sparse / (fma["tflops"] * 1e12),
                  B / (peaks["hbm_gbs"] * 1e9))
    step_roof["cuda_core_sparse"] = {"tokens_per_ms": spec.T / (t_roof2 * 1e3),
                                     "frac": (spec.T / ms_per_step) / (spec.T / (t_roof2 * 1e3)),
                                     "sparse_flops": F_sparse, "fp32_fma": fma}

    # end to end through the public API with host buffers (pinned): every step uploads
    # its x and dy and downloads its y and dx. The steps are pipelined the way a
    # training loop would run them: two sets of device buffers and layer state, step
    # i + 1's upload on one copy stream and step i - 1's download on another while
    # step i computes.
    hx = x.cpu().pin_memory()
    hdy = dy.cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    hs = [h, tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated, device=dev,
                          route=args.route, dense_above=DENSE_ABOVE)]
    xin = [torch.empty_like(x) for _ in range(2)]
    dyin = [torch.empty_like(dy) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}

    def e2e_steps(nsteps):
        for i in range(nsteps):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev["done"][b])      # step i - 2 no longer reads slot b
                xin[b].copy_(hx, non_blocking=True)
                dyin[b].copy_(hdy, non_blocking=True)
                ev["in"][b].record(up)
            stream.wait_event(ev["in"][b])
            if i >= 2:
                stream.wait_event(ev["out"][b])       # step i - 2's outputs have left the device
            hs[b].forward(xin[b], Wg, Wu, Wd)
            hs[b].backward(dyin[b], xin[b], Wg, Wu, Wd, spec.l1)
            ev["done"][b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["done"][b])
                hy.copy_(hs[b].y, non_blocking=True)
                hdx.copy_(hs[b].dx, non_blocking=True)
                ev["out"][b].record(down)
        stream.wait_stream(down)

    e2e_steps(2)
    torch.cuda.synchronize(dev)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    e_s.record(stream)
    up.wait_stream(stream)
    e2e_steps(args.steps)
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = dist.max(e_s.elapsed_time(e_e), dev)
    for f in hs:
        tw.raise_if_device_error(f.status, "e2e steps")
    e2e = {"value": spec.T * dist.world * args.steps / e2e_ms, "unit": UNIT,
           "h2d_bytes_per_step": int(hx.numel() * 2 + hdy.numel() * 2),
           "d2h_bytes_per_step": int(hy.numel() * 2 + hdx.numel() * 2),
           "pipelining": "uploads and downloads on two copy streams, overlapped with the neighbouring steps"}
    del hs[1]

    # dense bf16 FFN (torch/cuBLAS) forward + backward with the same L1 term, same run
    dense = None
    if not args.no_dense:
        dense_step = dense_train_step(x, Wg, Wu, Wd, dy, spec.l1)
        for _ in range(2):
            dense_step()
        torch.cuda.synchronize(dev)
        ds, de = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ds.record(stream)
        for _ in range(max(3, args.steps // 2)):
            dense_step()
        de.record(stream)
        torch.cuda.synchronize(dev)
        dense = {"value": spec.T * max(3, args.steps // 2) / ds.elapsed_time(de), "unit": UNIT,
                 "impl": "torch bf16 matmul + autograd (cuBLAS)"}

    # memory one layer's training step holds beyond x, dy and the weights: for the
    # library, everything HybridFFN preallocates (saved Hybrid, workspaces, y, dx, dW);
    # for dense torch, the peak its forward + backward allocates
    def nbytes(o):
        return sum(t.numel() * t.element_size() for t in vars(o).values() if isinstance(t, torch.Tensor))
    ours_bytes = nbytes(h) + nbytes(h.saved)
    # the library side as a measured peak: a fresh layer object (its preallocated saved
    # Hybrid, workspaces, y, dx, dW) and one training step, above what was held before
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    m0 = torch.cuda.memory_allocated(dev)
    h_m = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, backup_cap, gated=spec.gated, device=dev,
                       route=args.route, dense_above=DENSE_ABOVE)
    h_m.forward(x, Wg, Wu, Wd)
    h_m.backward(dy, x, Wg, Wu, Wd, spec.l1)
    torch.cuda.synchronize(dev)
    ours_peak = torch.cuda.max_memory_allocated(dev) - m0
    tw.raise_if_device_error(h_m.status, "memory step")
    del h_m
    torch.cuda.empty_cache()
    memory = {"hybrid_saved_bytes": nbytes(h.saved), "layer_bytes": ours_bytes, "layer_peak_bytes": ours_peak,
              "dense_saved_bytes_bf16_a_u": 2 * spec.T * spec.I * 2}
    if dense is not None:
        torch.cuda.synchronize(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        m0 = torch.cuda.memory_allocated(dev)
        dense_step()
        torch.cuda.synchronize(dev)
        memory["dense_step_peak_bytes"] = torch.cuda.max_memory_allocated(dev) - m0
        memory["layer_bytes_vs_dense"] = ours_bytes / memory["dense_step_peak_bytes"]
        memory["layer_peak_vs_dense_peak"] = ours_peak / memory["dense_step_peak_bytes"]

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": statistics.median(step_ms),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": spec.name, "tokens": spec.T, "d": spec.d, "I": spec.I, "gated": spec.gated,
                   "mean_active": spec.mean_active, "outlier_frac": spec.outlier_frac, "W": spec.W, "C": spec.C,
                   "R": spec.R, "backup_cap": backup_cap, "l1": spec.l1,
                   "step": "hybrid_ffn_fwd + hybrid_ffn_bwd", "l2": "256 MiB flush between steps (untimed)",
                   "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU"},
        "measured": {"nnz_per_token": stats["nnz"] / spec.T, "nnz_ell": stats["nnz_ell"],
                     "n_backup": stats["n_backup"], "route_taken": stats["route"],
                     "route": args.route + (f" (dense above {DENSE_ABOVE:g} nonzeros per ELL row)"
                                            if args.route == "auto" else "")},
        "roofline": roofline,
        "step_roofline": step_roof,
        "e2e": e2e,
        "gpu_launches": launches,
        "kernels": {k_: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                    for k_, v in sorted(kernels.items(), key=lambda kv: -kv[1]["total_ms"])},
        "clocks": clk,
        "repeats": repeats,
        "l2_gather_probe": l2,
        "dense_bf16": dense,
        "warm_l2": warm,
        "memory": memory,
    }
    # per-neuron activity counts of the step's forward and dead-neuron re-initialisation
    # of (a copy of) the gate projection
    counts = torch.zeros(spec.I, dtype=torch.int32, device=dev)
    Wg_copy = Wg.clone()

    def neuron_pass():
        counts.zero_()
        tw.hybrid_neuron_counts(h.saved, counts)
        return tw.reinit_dead_rows(Wg_copy, counts, 1234, 1.0 / math.sqrt(spec.d))

    n_dead = neuron_pass()
    ms_neur = _time_steps(neuron_pass, max(3, args.steps // 2), 3, flush, stream)
    line["dead_neurons"] = {"counts_and_reinit_us": 1e3 * ms_neur, "dead": int(n_dead.item()),
                            "min_count": int(counts.min().item()), "max_count": int(counts.max().item())}
    if not args.no_inference:
        line["inference"] = measure_inference(dev, flush, stream, max(3, args.steps // 2))
    if not args.no_sweep:
        line["sweep"] = measure_sweep(dev, flush, stream, max(3, min(10, args.steps // 2)), peaks)
    if not args.no_stack:
        line["stack"] = measure_stack(dev, flush, stream, 3)
    if dist.rank == 0 and not args.no_cpu_baseline:
        # a probe sample sizes the timed one to about CPU_TARGET_S of oracle work
        # (capped at the whole batch)
        n_s = args.cpu_sample_tokens
        dt, cores, sample = oracle_sample_time(spec, inp, n_s)
        grow = min(spec.T, 256 * int(n_s * CPU_TARGET_S / max(dt, 1e-3) / 256))
        if grow > n_s:
            n_s = grow
            dt, cores, sample = oracle_sample_time(spec, inp, n_s)
        line["cpu_baseline"] = {"value": n_s / (dt * 1e3), "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample, "seconds": dt}
    return line


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args, dist: Dist) -> dict | None:
    if dist.rank != 0:
        return None
    from synthetic import WORKLOADS, make_inputs

    spec = WORKLOADS[args.workload]
    inp = make_inputs(spec, with_dy=True)
    n_s = args.reference_sample_tokens
    for _ in range(args.warmup):
        oracle_sample_time(spec, inp, min(n_s, 64))
    times = []
    for _ in range(args.steps):
        dt, cores, sample = oracle_sample_time(spec, inp, n_s)
        times.append(dt)
    total = sum(times)
    value = n_s * args.steps / (total * 1e3)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": spec.name, "tokens_per_step": n_s},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-inference", action="store_true", help="skip the TwELL inference forward figures")
    ap.add_argument("--no-sweep", action="store_true", help="skip the training sparsity sweep")
    ap.add_argument("--route", choices=["sparse", "dense", "auto"], default="sparse",
                    help="route of the headline step's ELL rows (the sweep and the stack report all of them)")
    ap.add_argument("--clock-soak", type=float, default=4.0,
                    help="seconds over which the K-step timed region is repeated for the clock record")
    ap.add_argument("--no-stack", action="store_true", help="skip the 28-layer residual stack figures")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (small cases for profiler captures)")
    ap.add_argument("--cpu-sample-tokens", type=int, default=2048)
    ap.add_argument("--reference-sample-tokens", type=int, default=1024)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    if args.impl == "reference":
        line = run_reference(args, dist)
    else:
        import torch
        dist.init("nccl" if torch.cuda.is_available() else "gloo")
        line = run_ours(args, dist)
        dist.close()
    if line is not None and dist.rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
