"""Host-side pieces of bench.py that need no GPU: the committed DRAM-traffic
figures are reported only while the kernel sources they were measured on are
unchanged, and the algorithmic work formulas count what they say."""
import hashlib
import os

import bench


def _tree(tmp_path, src_text):
    csrc = tmp_path / "activation_sparse_feedforward_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(src_text.encode()).hexdigest()[:16]
    (tmp_path / "profiles" / "dram_traffic_wl.txt").write_text(
        "# comment\nkern 100 23 k.cu " + sha + "\n")
    return csrc


def test_traffic_reported_while_sources_match(tmp_path, monkeypatch):
    csrc = _tree(tmp_path, "kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("kern", "wl") == 123.0
    assert bench.measured_traffic("other", "wl") is None
    assert bench.measured_traffic("kern", "missing") is None
    (csrc / "k.cu").write_text("kernel v2\n")
    assert bench.measured_traffic("kern", "wl") is None


def test_committed_traffic_file_parses():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic_train_d2048_i5632_m29_o1.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert rows and all(len(r) == 5 and int(r[1]) > 0 and int(r[2]) >= 0 for r in rows)


def test_gathered_bytes_counts_rows_per_entry():
    from synthetic import WORKLOADS
    spec = WORKLOADS["train_d2048_i5632_m29_o1"]
    stats = {"nnz_ell": 1000, "n_backup": 0, "nnz": 1000}
    row = spec.d * 2
    assert bench.gathered_bytes("sparse_fwd", spec, stats) == 2 * 1000 * row
    assert bench.gathered_bytes("sparse_bwd_token", spec, stats) == 3 * 1000 * row
    assert bench.gathered_bytes("ell_weight_grad", spec, stats) == 2 * 1000 * row
    assert bench.gathered_bytes("gate_pack", spec, stats) is None
    ng = spec.with_(gated=False)
    assert bench.gathered_bytes("sparse_fwd", ng, stats) == 1000 * row


def test_clock_record_summary():
    lines = ["0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, 1800, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 2010, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, [N/A], 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # unreadable clock
             "garbage line"]
    out = bench.ClockSampler.summarize(lines)
    assert out == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = bench.ClockSampler.summarize(["0, 1500, 2070, 1400, 0x48, Active, Not Active, Active, Not Active"])
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and hot["samples"] == 1
    assert bench.ClockSampler.summarize([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_kernel_work_matches_the_documented_bench_figures():
    """The roofline's per-launch work at the bench workload (train_d2048_i5632_m29_o1,
    476079 ELL entries, 164 backup rows): the gate GEMM's 2 T d I = 3.78e11 FLOP and the
    backward token pass's ~214 MB of algorithmic bytes (dy, dx, the ELL, the records,
    three weight matrices), as DESIGN states them."""
    from synthetic import WORKLOADS
    spec = WORKLOADS["train_d2048_i5632_m29_o1"]
    stats = {"nnz_ell": 476079, "n_backup": 164}
    bound, flop = bench.kernel_work("gate_pack", spec, stats)
    assert bound == "tensor" and abs(flop - 3.78e11) / 3.78e11 < 0.005
    bound, b = bench.kernel_work("sparse_bwd_token", spec, stats)
    assert bound == "hbm" and abs(b - 214e6) / 214e6 < 0.01
    assert bench.kernel_work("no_such_kernel", spec, stats) is None
