"""The C-ABI library loads on a CPU-only machine, exports every function that
include/twell.h declares, agrees with the ctypes struct layouts, and rejects bad
arguments on the host before touching the GPU."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import activation_sparse_feedforward_gb300 as tw
from activation_sparse_feedforward_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "twell.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tw.lib_path()):
        from activation_sparse_feedforward_gb300.build import build
        build()
    return tw.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in twell.h but not exported"
        assert n in _lib.SIGNATURES, f"{n} missing from the ctypes binding"
    assert set(_lib.SIGNATURES) == set(names)


def test_abi_version_and_status_strings(lib):
    assert lib.tw_abi_version() == 2
    for code in range(9):
        assert lib.tw_status_str(code).decode().startswith("TW_")


def test_struct_layouts_match_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "twell.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(tw_twell), offsetof(tw_twell, cnt), '
        'offsetof(tw_twell, n_ovf), sizeof(tw_hybrid), offsetof(tw_hybrid, n_backup)); return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    got = [ctypes.sizeof(_lib.TwTwell), _lib.TwTwell.cnt.offset, _lib.TwTwell.n_ovf.offset,
           ctypes.sizeof(_lib.TwHybrid), _lib.TwHybrid.n_backup.offset]
    assert [int(v) for v in out] == got


def test_host_validation_rejects_bad_arguments(lib):
    s = _lib.TwTwell(4, 256, 64, 8, 16, 16, 16, 16, 16, 16, 16)   # fake, aligned, never dereferenced
    assert lib.twell_pack(16, 4, 256, 32, 8, ctypes.byref(s), 16, None) == _lib.TW_EUNSUPPORTED  # W = 32
    assert lib.twell_pack(16, 4, 250, 64, 8, ctypes.byref(s), 16, None) == _lib.TW_EUNSUPPORTED  # I % W
    assert lib.twell_pack(16, 4, 256, 64, 0, ctypes.byref(s), 16, None) == _lib.TW_EINVAL        # C = 0
    assert lib.twell_pack(16, 4, 256, 64, 65, ctypes.byref(s), 16, None) == _lib.TW_EINVAL       # C > W
    assert lib.twell_pack(16, 5, 256, 64, 8, ctypes.byref(s), 16, None) == _lib.TW_EINVAL        # T mismatch
    assert lib.twell_pack(18, 4, 256, 64, 8, ctypes.byref(s), 16, None) == _lib.TW_EALIGN        # misaligned A
    assert lib.twell_pack(None, 4, 256, 64, 8, ctypes.byref(s), 16, None) == _lib.TW_EINVAL
    assert lib.twell_pack(16, 4, 256, 64, 8, None, 16, None) == _lib.TW_EINVAL
    assert lib.twell_gate_pack(16, 16, 4, 320, 256, 64, 8, ctypes.byref(s), None, 16, None) == _lib.TW_EUNSUPPORTED
    # T == 0 is a no-op that succeeds without any launch
    z = _lib.TwTwell(0, 256, 64, 8)
    assert lib.twell_pack(None, 0, 256, 64, 8, ctypes.byref(z), None, None) == _lib.TW_OK
    # workspace too small
    assert lib.twell_ffn_fwd(16, 16, 16, 16, 4, 256, 256, 64, 8, 4, ctypes.byref(s), 16, 0, 16, 16,
                             None) == _lib.TW_EWORKSPACE
    assert lib.tw_dense_gemm(16, 16, 64, 60, 64, 0, 0, 16, 16, None) == _lib.TW_EINVAL
    # the CTA-pair forms: N a multiple of 256; the pair timeout hook one 256 x 256 unit
    assert lib.tw_dense_gemm_pair(16, 16, 64, 128, 64, 0, 0, 16, 16, None) == _lib.TW_EINVAL      # N % 256
    assert lib.tw_dense_gemm_pair(16, 16, 60, 256, 64, 1, 0, 16, 16, None) == _lib.TW_EINVAL      # M % 64, MN-major A
    assert lib.tw_dense_gemm_pair(16, 16, 64, 256, 60, 0, 0, 16, 16, None) == _lib.TW_EINVAL      # K % 64
    assert lib.tw_wait_timeout_probe_pair(16, 16, 300, 256, 64, 0, 16, 16, None) == _lib.TW_EINVAL  # M > 256
    assert lib.tw_wait_timeout_probe_pair(16, 16, 256, 512, 64, 0, 16, 16, None) == _lib.TW_EINVAL  # N != 256
    assert lib.tw_wait_timeout_probe_pair(16, 16, 256, 256, 64, 1, 16, 16, None) == _lib.TW_EINVAL  # K block past K


def test_neuron_functions_validate_on_the_host(lib):
    import math
    assert lib.hybrid_neuron_counts(None, 16, None) == _lib.TW_EINVAL
    assert lib.tw_reinit_dead_rows(16, 4, 0, 16, 1, 0.1, 16, None) == _lib.TW_EINVAL          # d = 0
    assert lib.tw_reinit_dead_rows(16, 4, 8, 16, 1, math.inf, 16, None) == _lib.TW_EINVAL     # std not finite
    assert lib.tw_reinit_dead_rows(None, 4, 8, 16, 1, 0.1, 16, None) == _lib.TW_EINVAL        # no W
    assert lib.tw_reinit_dead_rows(16, 4, 8, 18, 1, 0.1, 16, None) == _lib.TW_EALIGN          # counts misaligned
    h = _lib.TwHybrid(0, 64, 8, 0)
    assert lib.hybrid_neuron_counts(ctypes.byref(h), 16, None) == _lib.TW_OK                  # T = 0: nothing to do


def test_trace_hook_host_side(lib):
    assert lib.tw_trace_begin(None, 4) == _lib.TW_EINVAL
    assert lib.tw_trace_end() == 0
    assert lib.tw_trace_label(0) is None


def test_workspace_sizes_grow_with_capacity(lib):
    a = lib.twell_ffn_fwd_workspace_size(16384, 2048, 5632, 128, 16, 0)
    b = lib.twell_ffn_fwd_workspace_size(16384, 2048, 5632, 128, 16, 200)
    assert b - a >= 256 * (2048 + 5632) * 2
    h0 = lib.hybrid_ffn_fwd_workspace_size(16384, 2048, 5632, 128, 16, 64, 0, 0)
    assert h0 >= 16384 * 44 * (2 + 16 * 3)
    assert lib.hybrid_ffn_bwd_workspace_size(16384, 2048, 5632, 64, 256, 0) > \
        lib.hybrid_ffn_bwd_workspace_size(16384, 2048, 5632, 64, 0, 0)


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no non-CUDA fallback"):
        _lib.load()
