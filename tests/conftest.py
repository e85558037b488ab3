import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Achieved parity of every GPU-vs-oracle comparison of the run: the worst
    relL2 / bound ratio per dtype and the bf16 cases closest to their bound.
    With GQA_PARITY_LOG=<path> every case is also written there as JSON."""
    mod = sys.modules.get("parity_util")
    if mod is None or not getattr(mod, "RESULTS", None):
        return
    res = mod.RESULTS
    tr = terminalreporter
    tr.write_sep("-", f"parity against the oracle: {len(res)} comparisons")
    for dt in ("f16", "bf16"):
        sel = [r for r in res if r[1] == dt]
        if not sel:
            continue
        worst = max(sel, key=lambda r: r[2] / r[3])
        tr.write_line(
            f"{dt}: {len(sel)} cases; relL2 max {max(r[2] for r in sel):.3e}, "
            f"median {sorted(r[2] for r in sel)[len(sel) // 2]:.3e}; worst relL2/bound "
            f"{worst[2] / worst[3]:.3f} ({worst[0]}: {worst[2]:.3e} of {worst[3]:.3e}); "
            f"max_abs max {max(r[4] for r in sel):.3e}; lse err max {max(r[5] for r in sel):.3e}")
    bf = sorted((r for r in res if r[1] == "bf16"), key=lambda r: -r[2] / r[3])[:8]
    for r in bf:
        tr.write_line(f"  bf16 {r[0]}: relL2 {r[2]:.3e} bound {r[3]:.3e} "
                      f"(ratio {r[2] / r[3]:.3f}) max_abs {r[4]:.3e}")
    path = os.environ.get("GQA_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump([{"label": r[0], "dtype": r[1], "rel_l2": r[2], "bound": r[3],
                        "max_abs": r[4], "lse_err": r[5]} for r in res], f, indent=0)
