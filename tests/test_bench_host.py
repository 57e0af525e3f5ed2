"""Host logic of bench.py (CPU only): algorithmic byte counts, the input-set rotation, the source
hash that gates recorded DRAM traffic, and the clock sampler's windows and throttle reasons."""
import datetime
import json
import os
import shutil
from types import SimpleNamespace

import numpy as np

import bench


def _batch(dtype, B, K, V, temps, tokens=True):
    return SimpleNamespace(dtype=dtype, B=B, V=V, temperature=np.asarray(temps, np.float32),
                           tokens=np.zeros((B, K), np.int32) if tokens else None)


def test_algorithmic_bytes_of_the_workloads():
    # per-round logit bytes of the five workloads (each needed byte once)
    c1 = _batch("bf16", 4, 3, 32000, [0.0] * 4, tokens=False)        # draft argmax fused: draft rows read
    assert bench.algorithmic_bytes(c1, [3] * 4) == 1_792_000
    c2 = _batch("bf16", 16, 3, 151936, [1.0] * 16)
    assert bench.algorithmic_bytes(c2, [3] * 16) == 34_033_664
    c3 = _batch("f32", 64, 16, 151936, [0.6] * 64)
    assert bench.algorithmic_bytes(c3, [16] * 64) == 1_283_555_328
    c4 = _batch("bf16", 64, 16, 151936, [1.0] * 64)
    assert bench.algorithmic_bytes(c4, [16] * 64) == 2112 * 303_872
    # greedy requests with given tokens read target rows only; T > 0 adds the draft rows
    mix = _batch("bf16", 3, 4, 1000, [0.0, 1.0, 0.6])
    assert bench.algorithmic_bytes(mix, [2, 4, 0]) == ((3) + (5 + 4) + (1 + 0)) * 1000 * 2


def test_rotation_flushes_re_read_rows_from_l2():
    # the logits read, and the rows the other sets read again after their stream, both exceed
    # L2 twice over, so no step meets its own rows in L2 from its set's previous turn
    L2 = bench.L2_BYTES
    cases = {  # workload: (batch, re-read rows per request)
        "c2": (_batch("bf16", 16, 3, 151936, [1.0] * 16), 2),
        "c3": (_batch("f32", 64, 16, 151936, [0.6] * 64), 2),
        "t1": (_batch("bf16", 64, 15, 151936, [1.0] * 64), 4),
    }
    for w, (b, rows) in cases.items():
        b.keep_len = np.full(b.B, b.tokens.shape[1], np.int32)
        n = bench.rotation_sets(w, b)
        elt = 2 if b.dtype == "bf16" else 4
        assert n >= 2 and n * bench.algorithmic_bytes(b, b.keep_len) >= 2 * L2, w
        assert (n - 1) * b.B * rows * b.V * elt >= 2 * L2, w
        assert (n - 2) * b.B * rows * b.V * elt < 2 * L2, w  # and no more sets than that needs
    # C4's sets are sized by all 16 drafted positions, whatever the schedule keeps
    c4 = _batch("bf16", 64, 16, 151936, [1.0] * 64)
    c4.keep_len = np.zeros(64, np.int32)
    assert bench.rotation_sets("c4", c4) == 1 + int(np.ceil(2 * L2 / (64 * 2 * 151936 * 2)))


def _copy_sources(tmp_path):
    root = tmp_path / "r"
    csrc = root / "speculative_decoding_verification_74_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "speculative_decoding_verification_74_gb300", "csrc")
    for f in ("sv_device.cuh", "sv_internal.h", "sv_verify.cu"):
        shutil.copy(os.path.join(src, f), csrc / f)
    (root / "profiles").mkdir()
    return root, csrc


def test_source_hash_ignores_comments_and_gates_recorded_traffic(tmp_path, monkeypatch):
    root, csrc = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    (root / "profiles" / "traffic.json").write_text(json.dumps(
        {"c2": {"source_hash": h0, "dram_bytes_per_launch": 123}}))
    assert bench.recorded_traffic("c2") == 123
    assert bench.recorded_traffic("c3") is None
    f = csrc / "sv_verify.cu"
    code = f.read_text()
    f.write_text("// a new comment line\n" + code.replace("\n", "\n  ", 3))   # comments and spacing only
    assert bench.kernel_source_hash() == h0 and bench.recorded_traffic("c2") == 123
    f.write_text(code + "\nstatic int touched = 1;\n")                       # a code change
    assert bench.kernel_source_hash() != h0 and bench.recorded_traffic("c2") is None


def _sampler(tmp_path, rows, marks):
    s = bench.ClockSampler.__new__(bench.ClockSampler)      # no nvidia-smi process
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        for ln in rows:
            f.write(ln + "\n")
    s.marks = marks
    s.proc = SimpleNamespace(terminate=lambda: None, wait=lambda timeout=None: 0)
    s.fh = open(os.devnull, "w")
    return s


def _row(t, sm, reasons=()):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    flags = ["Active" if r in reasons else "Not Active" for r in bench.ClockSampler.REASONS]
    return f"{ts}, 0, {sm} MHz, 2070 MHz, 900.00 W, 0x0, " + ", ".join(flags)


def test_clock_sampler_windows_and_reasons(tmp_path):
    t0 = 1_700_000_000.0
    rows = [_row(t0 + 0.01 * k, 1500 if k < 10 else 2070) for k in range(40)]
    rows[25] = _row(t0 + 0.25, 2070, ("sw_power_cap",))
    out = _sampler(tmp_path, rows, {"timed0": t0 + 0.1, "timed1": t0 + 0.3}).stop()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples_timed"] >= 19 and out["basis"] == "samples inside the timed region"
    # a short timed window: the load replay right after it joins the median
    rows = [_row(t0 + 0.01 * k, 1900 + k) for k in range(40)]
    rows[31] = _row(t0 + 0.31, 1931, ("hw_slowdown",))
    out = _sampler(tmp_path, rows, {"timed0": t0 + 0.095, "timed1": t0 + 0.115,
                                    "load0": t0 + 0.295, "load1": t0 + 0.355}).stop()
    assert out["samples_timed"] == 2 and out["samples_load"] == 6
    assert out["sm_mhz"] == float(np.median([1910, 1911] + list(range(1930, 1936))))
    assert out["reasons"] == ["hw_slowdown"]
    assert not os.path.exists(str(tmp_path / "clocks.csv"))
