"""Host logic of bench.py that needs no GPU: the ncu traffic lookup, the clock record and the
reference (oracle) arm's JSON line."""
import argparse
import io
import json
import contextlib

import pytest

import bench
from gen import configs


def test_profiled_traffic_follows_the_sources(monkeypatch):
    # the committed summary of the headline kernel carries the digest of the sources it was
    # taken on; any other digest (a changed kernel) gives no traffic figure
    value = bench.profiled_traffic("attn_fwd_kernel")
    assert value is None or (isinstance(value, int) and value > 0)
    monkeypatch.setattr(bench, "sources_digest", lambda: "0" * 16)
    assert bench.profiled_traffic("attn_fwd_kernel") is None
    assert bench.profiled_traffic("no_such_kernel") is None


def test_tensor_pipe_lookup_follows_the_sources(monkeypatch):
    # each workload's committed single-launch summary is found while the kernel's code is the one
    # it was taken on, and not after any change
    for i in sorted(configs.WORKLOADS):
        v = bench.profiled_tensor_pipe(configs.WORKLOADS[i])
        assert v is None or 0.0 < v <= 100.0
    monkeypatch.setattr(bench, "sources_digest", lambda files=None: "0" * 16)
    assert all(bench.profiled_tensor_pipe(configs.WORKLOADS[i]) is None
               for i in sorted(configs.WORKLOADS))


def test_source_digest_ignores_comments_only():
    a = "int x = 1; // one\n/* block\n comment */ int  y = 2;\n"
    b = "int x = 1;\nint y = 2; // a different comment\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("2", "3"))


class _DoneProc:
    def terminate(self):
        pass

    def wait(self):
        pass


def _sampler_with(rows):
    s = bench.ClockSampler(0)
    s.proc = _DoneProc()
    s.out.write("\n".join(rows) + "\n")
    s.out.flush()
    return s


def test_clock_record_median_and_reasons():
    rows = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    rec = _sampler_with(rows).stop()
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0 and rec["samples"] == 3
    assert rec["reasons"] == ["sw_power_cap"]


def test_clock_record_flags_slowdowns_and_skips_bad_rows():
    rows = [
        "0, 1400, 2070, 500.0, 0x8, Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1500, 2070, 500.0, 0x40, Not Active, Active, Active, Not Active",
    ]
    rec = _sampler_with(rows).stop()
    assert rec["samples"] == 2 and rec["sm_mhz"] == 1450.0
    assert rec["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_oracle_sample_is_bounded():
    w = configs.custom(901, 1, 2, 384, 64, True)
    q, k, v, _ = w.make()
    tflops, rows, secs = bench.oracle_sample(w, q, k, v, target_s=0.0, max_rows=128)
    assert rows == 128 and secs > 0 and tflops > 0


def test_reference_line_contract(monkeypatch):
    w = configs.custom(902, 1, 1, 256, 64, False)
    args = argparse.Namespace(steps=2, warmup=1, cpu_seconds=0.2)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, w, rank=0, world=1)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["dtype"] == "f64" and line["gpu_launches"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["value"] > 0 and line["steps"] == 2
    # other ranks print nothing
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, w, rank=1, world=2)
    assert buf.getvalue() == ""
