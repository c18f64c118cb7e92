import os
import sys
from fractions import Fraction

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running GPU test at full workload size")


def read_golden(name):
    """Parse a tests/golden fixture: '#' comments, 'case <name>' headers, and
    '<key> <values...>' lines.  Returns a list of dicts (one per case; one dict if the
    file has no case headers).  A key keeps its last line; ``d["_all"][key]`` keeps
    every line of a repeated key in file order."""
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                if cur:
                    cases.append(cur)
                cur = {"name": vals[0]}
                continue
            if key == "step":
                cur.setdefault("steps", []).append((int(vals[0]), vals[1], int(vals[2])))
                continue
            cur[key] = vals
            cur.setdefault("_all", {}).setdefault(key, []).append(vals)
    if cur:
        cases.append(cur)
    return cases


def fracs(num, den):
    if len(den) == 1:
        den = den * len(num)
    return [Fraction(int(n), int(d)) for n, d in zip(num, den)]


def cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def kvc():
    """The C-ABI library through its Python binding (GPU tests only)."""
    if not cuda_ok():
        pytest.skip("no CUDA device")
    import attention_score_kv_snapkv_gb300 as kvc_mod
    return kvc_mod
