import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def load_golden(name):
    """Parse a tests/golden text fixture into a list of cases (dicts of numpy arrays)."""
    import numpy as np

    path = os.path.join(ROOT, "tests", "golden", name)
    cases, cur, section, rows = [], None, None, []

    def flush():
        if cur is not None and section is not None:
            cur[section] = np.array(rows, dtype=np.float64).reshape(len(rows), -1) if rows else None

    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "case":
                flush()
                cur = {"name": tok[1], "M": int(tok[2]), "N": int(tok[3]), "K": int(tok[4])}
                cases.append(cur)
                section, rows = None, []
            elif tok[0] == "opts":  # general form: transa transb alpha beta
                flush()
                cur["opts"] = {"transa": int(tok[1]), "transb": int(tok[2]), "alpha": float(tok[3]),
                               "beta": float(tok[4])}
                section, rows = None, []
            elif tok[0] in ("A", "B", "C", "CIN", "BOUND"):
                flush()
                section, rows = tok[0], []
            else:
                rows.append([float(t) for t in tok])
        flush()
    return cases
