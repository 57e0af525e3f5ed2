"""The C ABI library loads, exports every function include/sv.h declares, and rejects bad
arguments on the host before any CUDA call (these run without a GPU)."""
import ctypes
import os
import subprocess
import sys

import pytest

import speculative_decoding_verification_74_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verification_74_gb300 import build
    try:
        build.build()
    except RuntimeError as e:  # no nvcc on this machine
        if not os.path.exists(sv.LIB_PATH):
            pytest.skip(str(e))
    return sv.lib()


def test_exports_every_header_symbol(L):
    names = sv.header_symbols()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_version_and_strings(L):
    assert L.sv_abi_version() == 2
    assert L.sv_status_string(0) == b"ok"
    assert L.sv_status_string(1) == b"invalid argument"


def test_workspace_sizes(L):
    for dt in (sv.SV_BF16, sv.SV_F32):
        a = L.sv_workspace_size(sv.SV_OP_VERIFY, 16, 3, 151936, dt)
        b = L.sv_workspace_size(sv.SV_OP_VERIFY, 64, 16, 151936, dt)
        assert 0 < a < b
        assert a % 256 == 0
    assert L.sv_workspace_size(sv.SV_OP_SCHEDULE, 64, 16, 1, 1) == 256
    assert L.sv_workspace_size(sv.SV_OP_VERIFY, -1, 3, 100, 0) == 0
    assert L.sv_workspace_size(sv.SV_OP_VERIFY, 4, 5000, 100, 0) == 0
    assert L.sv_workspace_size(sv.SV_OP_VERIFY, 4, 3, 0, 0) == 0
    assert L.sv_workspace_size(9, 4, 3, 10, 0) == 0


def test_host_validation_without_gpu(L):
    INV, WS = sv.SV_ERR_INVALID_ARG, sv.SV_ERR_WORKSPACE
    fake = 1 << 20          # an aligned, never-dereferenced address
    # greedy: NULL target, bad sizes, rows not aligned to the element size, no draft information
    assert L.sv_verify_greedy(None, 100, None, 0, fake, 0, 4, 3, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake, 100, None, 0, fake, 0, 4, -1, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake + 1, 104, None, 0, fake, 0, 4, 3, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake + 2, 104, None, 0, fake, 1, 4, 3, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake, 99, None, 0, fake, 0, 4, 3, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake, 104, None, 0, None, 0, 4, 3, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake, 104, None, 0, fake, 7, 4, 3, 100, fake, fake, fake, 1 << 20, None) == INV
    assert L.sv_verify_greedy(fake, 104, None, 0, fake, 0, 4, 3, 100, None, fake, fake, 1 << 20, None) == INV
    # workspace: NULL, misaligned, too small
    assert L.sv_verify_greedy(fake, 104, None, 0, fake, 0, 4, 3, 100, fake, fake, None, 1 << 20, None) == WS
    assert L.sv_verify_greedy(fake, 104, None, 0, fake, 0, 4, 3, 100, fake, fake, fake + 16, 1 << 20, None) == WS
    assert L.sv_verify_greedy(fake, 104, None, 0, fake, 0, 4, 3, 100, fake, fake, fake, 64, None) == WS
    # B == 0 is a no-op
    assert L.sv_verify_greedy(None, 0, None, 0, None, 0, 0, 3, 100, None, None, None, 0, None) == sv.SV_OK
    # sample: temperature and tokens required
    assert L.sv_verify_sample(fake, 104, fake, 104, None, fake, 0, 0, None, 0, 4, 3, 100, fake, fake, None,
                              None, None, fake, 1 << 20, None) == INV
    assert L.sv_verify_sample(fake, 104, fake, 104, fake, None, 0, 0, None, 0, 4, 3, 100, fake, fake, None,
                              None, None, fake, 1 << 20, None) == INV
    # ragged: offsets required, token stride >= Kmax, row counts >= 0
    assert L.sv_verify_ragged(fake, 104, None, 16, fake, 104, fake, 12, fake, 3, fake, fake, 0, 0, None, 0, 4, 3,
                              100, fake, fake, None, None, None, fake, 1 << 20, None) == INV
    assert L.sv_verify_ragged(fake, 104, fake, 16, fake, 104, None, 12, fake, 3, fake, fake, 0, 0, None, 0, 4, 3,
                              100, fake, fake, None, None, None, fake, 1 << 20, None) == INV
    assert L.sv_verify_ragged(fake, 104, fake, 16, fake, 104, fake, 12, fake, 2, fake, fake, 0, 0, None, 0, 4, 3,
                              100, fake, fake, None, None, None, fake, 1 << 20, None) == INV
    assert L.sv_verify_ragged(fake, 104, fake, -1, fake, 104, fake, 12, fake, 3, fake, fake, 0, 0, None, 0, 4, 3,
                              100, fake, fake, None, None, None, fake, 1 << 20, None) == INV
    assert L.sv_verify_ragged(fake, 104, fake, 16, fake, 104, fake, -1, fake, 3, fake, fake, 0, 0, None, 0, 4, 3,
                              100, fake, fake, None, None, None, fake, 1 << 20, None) == INV
    # schedule: sizes, costs, budget, ratios, objective
    f = ctypes.c_float
    assert L.sv_schedule_depth(fake, 16, None, 0, 16, f(1.0), f(0.05), 0, None, 0, 0, fake, None, fake, None,
                               fake, 256, None) == INV
    assert L.sv_schedule_depth(fake, 16, None, 64, 1024, f(1.0), f(0.05), 0, None, 0, 0, fake, None, fake,
                               None, fake, 256, None) == INV
    assert L.sv_schedule_depth(fake, 16, None, 64, 16, f(-1.0), f(0.05), 0, None, 0, 0, fake, None, fake,
                               None, fake, 256, None) == INV
    assert L.sv_schedule_depth(fake, 16, None, 64, 16, f(1.0), f(0.05), 10, None, 0, 0, fake, None, fake,
                               None, fake, 256, None) == INV
    bad_ratio = (ctypes.c_float * 1)(1.5)
    assert L.sv_schedule_depth(fake, 16, None, 64, 16, f(1.0), f(0.05), 0, ctypes.cast(bad_ratio, ctypes.c_void_p),
                               1, 0, fake, None, fake, None, fake, 256, None) == INV
    assert L.sv_schedule_depth(fake, 16, None, 64, 16, f(1.0), f(0.05), 0, None, 0, 5, fake, None, fake, None,
                               fake, 256, None) == INV
    assert L.sv_schedule_depth(fake, 16, None, 64, 16, f(1.0), f(0.05), 0, None, 0, 0, fake, None, fake, None,
                               None, 256, None) == WS
    # schedule with a latency table: the table's own checks, then the shared ones
    def table(Ks, cs):
        k = (ctypes.c_int32 * max(len(Ks), 1))(*Ks)
        c = (ctypes.c_double * max(len(cs), 1))(*cs)
        return ctypes.cast(k, ctypes.c_void_p), ctypes.cast(c, ctypes.c_void_p), k, c

    def sched_t(Ks, cs, n=None, B=64, ws=fake, null=None):
        k, c, _hold_k, _hold_c = table(Ks, cs)
        if null == "K":
            k = None
        if null == "c":
            c = None
        return L.sv_schedule_depth_table(fake, 16, None, B, 16, k, c, len(Ks) if n is None else n, 0, None, 0, 0,
                                         fake, None, fake, None, ws, 256, None)
    assert sched_t([16, 32], [1.0, 2.0], null="K") == INV
    assert sched_t([16, 32], [1.0, 2.0], null="c") == INV
    assert sched_t([16, 32], [1.0, 2.0], n=0) == INV
    assert sched_t(list(range(1, 34)), [1.0] * 33) == INV
    assert sched_t([0, 32], [1.0, 2.0]) == INV
    assert sched_t([32, 32], [1.0, 2.0]) == INV
    assert sched_t([32, 16], [1.0, 2.0]) == INV
    assert sched_t([16, 32], [1.0, 0.0]) == INV
    assert sched_t([16, 32], [1.0, float("nan")]) == INV
    assert sched_t([16, 32], [float("inf"), 1.0]) == INV
    assert sched_t([16, 32], [1.0, 2.0], B=0) == INV
    assert sched_t(list(range(1, 33)), [1.0] * 32, ws=None) == WS
    assert L.sv_query_status(None, None, None) == INV
    assert b"NULL" in L.sv_last_error_string()


def test_binding_fails_loudly_without_library(tmp_path):
    """The product path has no fallback: a missing library is an import-time-of-use error."""
    code = ("import speculative_decoding_verification_74_gb300 as sv\n"
            "sv.LIB_PATH = '/nonexistent/libsv.so'\n"
            "try:\n    sv.lib()\nexcept RuntimeError as e:\n    print('RAISED', e)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "RAISED" in r.stdout
