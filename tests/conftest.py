import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built engine")
    config.addinivalue_line("markers", "slow: full-shape cases that take tens of seconds")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Observed parity magnitudes of the GPU-vs-oracle comparisons."""
    try:
        from gpu_helpers import RECORDS, summarise
    except Exception:  # pragma: no cover
        return
    if not RECORDS:
        return
    import json
    rows = {k: summarise(v) for k, v in RECORDS.items()}
    tr = terminalreporter
    tr.write_sep("-", "parity magnitudes (GPU logits against the oracle)")
    worst = max(r["worst_rel_l2"] for r in rows.values())
    for k, r in sorted(rows.items(), key=lambda kv: -kv[1]["worst_rel_l2"]):
        line = f"{r['worst_rel_l2']:.2e} worst rel-L2  {r['max_abs_err']:.2e} max abs  n={r['n']}"
        if "agree" in r:
            cm = r["agree_clear_margin"]
            line += (f"  agree {r['agree']:.3f}  clear-margin {'-' if cm is None else f'{cm:.3f}'}"
                     f"  near-ties {r['excluded_near_ties']}")
        tr.write_line(f"{line}  {k}")
    tr.write_line(f"worst rel-L2 over all {len(rows)} tests: {worst:.3e}")
    path = os.environ.get("LF_PARITY_JSON")
    if path:
        with open(path, "w") as f:
            json.dump(rows, f, indent=1, sort_keys=True)
