import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the compiled kernels")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def pytest_collection_modifyitems(config, items):
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def fcp():
    """The package with libfcp.so built (compiles for sm_103a if the sources changed)."""
    from context_parallelism_fcp_gb300 import _build

    _build.build()
    import context_parallelism_fcp_gb300 as pkg

    pkg.lib()
    return pkg


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """How much of each tolerance the observed errors used: per tensor, the largest
    error/bound ratio over all comparisons and where it occurred. With
    FCP_PARITY_RECORD=<path> every comparison is also written there as one JSON line."""
    mod = sys.modules.get("tests.parity_util")
    rec = getattr(mod, "RECORD", None)
    if not rec:
        return
    import json

    path = os.environ.get("FCP_PARITY_RECORD")
    if path:
        with open(path, "w") as f:
            for test, where, name, emax, bmax, emean, bmean in rec:
                f.write(json.dumps({"test": test, "where": where, "tensor": name, "max_err": emax, "max_bound": bmax,
                                    "mean_err": emean, "mean_bound": bmean}) + "\n")
    tr = terminalreporter
    tr.write_sep("-", f"parity headroom ({len(rec)} comparisons): observed error / bound")
    worst = {}
    for test, where, name, emax, bmax, emean, bmean in rec:
        rmax = emax / bmax
        rmean = emean / bmean if emean is not None and bmean else 0.0
        w = worst.setdefault(name, [0.0, "", 0.0, ""])
        if rmax > w[0]:
            w[0], w[1] = rmax, f"{test} {where}"
        if rmean > w[2]:
            w[2], w[3] = rmean, f"{test} {where}"
    for name, (rmax, tmax, rmean, tmean) in sorted(worst.items()):
        tr.write_line(f"{name:4s} max {rmax:6.3f}  ({tmax})")
        if rmean:
            tr.write_line(f"{'':4s} mean {rmean:5.3f}  ({tmean})")
