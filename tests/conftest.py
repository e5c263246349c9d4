import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The measured error of every GPU-vs-oracle comparison of the session."""
    import parity
    rec = parity.RECORD
    if not rec:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity record: {len(rec)} comparisons")
    worst = {}
    for r in rec:
        w = worst.get(r["what"])
        if w is None or r["max_abs"] > w["max_abs"]:
            worst[r["what"]] = r
    for what, r in sorted(worst.items()):
        tr.write_line(f"{what[:70]:70s} max_abs {r['max_abs']:.3e} (bound {r['bound']:.0e}) "
                      f"min_cos {r['min_cos']:.9f} ulp_flips {r['ulp_flips']}/{r['elements']}")
    path = os.environ.get("BM_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump(rec, f, indent=0)
