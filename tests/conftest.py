import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: `key: v1 v2 ...` lines, '#' comments.
    Repeated keys collect into a list of rows."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            vals = [float(t) for t in rest.split()]
            out.setdefault(key.strip(), []).append(vals)
    return {k: (v[0] if len(v) == 1 else v) for k, v in out.items()}


def pytest_sessionfinish(session, exitstatus):
    """With NV_PARITY_LOG set, write every check_close result of the session
    (what was compared, element count, absolute and mixed errors) as JSON."""
    path = os.environ.get("NV_PARITY_LOG")
    if not path:
        return
    mod = sys.modules.get("gpu_util")
    if mod is None:
        return
    import json
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w", encoding="utf-8") as f:
        json.dump([{"what": w, **st} for w, st in mod.PARITY_LOG], f, indent=1)
