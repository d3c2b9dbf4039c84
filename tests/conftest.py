import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


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


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report the near-ties the parity checks counted (tests/helpers.py)."""
    from tests import helpers as Hp
    if Hp.NEAR_TIE_LOG:
        tr = terminalreporter
        tr.section("near-ties: oracle gap between the k-th and (k+1)-th score below 1e-5")
        agg = {}
        for tid, T, ties, flips in Hp.NEAR_TIE_LOG:
            a = agg.setdefault(tid, [0, 0, 0])
            a[0] += T
            a[1] += ties
            a[2] += flips
        tot = [sum(v[i] for v in agg.values()) for i in range(3)]
        tr.write_line("total: %d tokens compared, %d near-ties, %d with a different selection"
                      % tuple(tot))
        for tid, (n, ties, flips) in agg.items():
            if ties:
                tr.write_line("  %s: %d tokens, %d near-ties, %d flipped" % (tid, n, ties, flips))
    if Hp.NORM_TIE_LOG:
        tr = terminalreporter
        tr.section("stack step: bf16 rounding ties of the normalised input (1-ulp, allowed)")
        agg = {}
        for tid, n, ties in Hp.NORM_TIE_LOG:
            a = agg.setdefault(tid, [0, 0])
            a[0] += n
            a[1] += ties
        for tid, (n, ties) in agg.items():
            tr.write_line("  %s: %d elements, %d at a rounding tie" % (tid, n, ties))
