"""Shared pytest set-up: the ``gpu`` marker, the repository on ``sys.path``,
and a report of the achieved parity errors at the end of a GPU run."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Achieved errors against the fp64 oracle (report only): max and mean
    |gpu - ref|, the fraction of bf16 outputs equal to bf16_rn(ref), the
    largest distance from bf16_rn(ref) in bf16 steps, and the largest error
    beyond the output rounding's half step."""
    mod = sys.modules.get("gpu_util")
    log = getattr(mod, "ERROR_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tr.section("parity errors against the fp64 oracle (report only)")
    worst = {}
    for r in log:
        key = r["what"].split(" ")[0]
        w = worst.setdefault(key, dict(r, n=0))
        w["n"] += 1
        for k in ("max", "mean", "max_steps", "excess"):
            if k in r and r[k] > w.get(k, -1.0):
                w[k] = r[k]
        if "exact_frac" in r:
            w["exact_frac"] = min(w.get("exact_frac", 1.0), r["exact_frac"])
    for key, w in sorted(worst.items()):
        extra = ""
        if "exact_frac" in w:
            extra = (f"  =bf16_rn(ref) >= {w['exact_frac']:.4f}  max steps {w['max_steps']:.0f}"
                     f"  excess {w['excess']:.2e}")
        tr.write_line(f"{key:<28} n={w['n']:<4} max {w['max']:.3e}  mean {w['mean']:.3e}{extra}")
