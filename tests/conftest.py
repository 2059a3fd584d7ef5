import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the error every parity check achieved (also on success); write them as JSON lines
    to the file named by ATTN_PARITY_LOG when it is set."""
    mod = sys.modules.get("parity_util")
    if mod is None or not mod.RESULTS:
        return
    import json
    tr = terminalreporter
    tr.section("achieved parity error")
    for r in mod.RESULTS:
        if r["kind"] == "fwd":
            tr.write_line(f"fwd {r['case']}: O max {r['o_max_abs']:.2e} mean {r['o_mean_abs']:.2e}"
                          f" over 1e-2 {r['o_over_1e-2']} (|O|<2: {r['o_over_1e-2_below_2']})"
                          f" vs rounded {r['o_max_abs_vs_rounded']:.2e}"
                          f" rounded {r['o_frac_correctly_rounded']:.4f}"
                          f" LSE max {r['lse_max_abs']:.2e} n {r['n']}")
        else:
            tr.write_line(f"{r['kind']} {r['case']}: " + ", ".join(
                f"{k} {v:.3g}" if isinstance(v, float) else f"{k} {v}"
                for k, v in r.items() if k not in ("kind", "case")))
    path = os.environ.get("ATTN_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            for r in mod.RESULTS:
                f.write(json.dumps(r) + "\n")
