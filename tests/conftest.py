import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture into (M, N, K, A, B, C) numpy arrays."""
    import numpy as np

    path = os.path.join(ROOT, "tests", "golden", name)
    lines = [ln.strip() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    dims = {}
    i = 0
    while lines[i].split()[0] in ("M", "N", "K"):
        key, val = lines[i].split()
        dims[key] = int(val)
        i += 1
    mats = {}
    while i < len(lines):
        tag = lines[i]
        rows = {"A": dims["M"], "B": dims["K"], "C": dims["M"]}[tag]
        mats[tag] = np.array([[float(x) for x in lines[i + 1 + r].split()] for r in range(rows)])
        i += 1 + rows
    return dims["M"], dims["N"], dims["K"], mats["A"], mats["B"], mats["C"]
