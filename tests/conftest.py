import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst error against its tolerance for every GPU-vs-oracle comparison
    made in this run (one line per test and quantity), and the same records
    as JSON lines in the file FA_PARITY_REPORT names, if set."""
    parity = sys.modules.get("parity")
    margins = getattr(parity, "MARGINS", None)
    if not margins:
        return
    import json
    worst = {}
    for m in margins:
        key = (m["test"], m["what"])
        if key not in worst or m["err"] > worst[key]["err"]:
            worst[key] = m
    tr = terminalreporter
    tr.write_sep("-", "parity margins: worst error / tolerance")
    for (test, what), m in sorted(worst.items()):
        tr.write_line(f"{m['err'] / m['tol']:7.3f}  {m['err']:.3e} / {m['tol']:.0e}  {what:38s} {test}")
    path = os.environ.get("FA_PARITY_REPORT")
    if path:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            for m in margins:
                f.write(json.dumps(m) + "\n")
