import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.hookimpl(tryfirst=True)
def pytest_configure(config):
    if config.option.basetemp is None:   # keep tmp_path directories inside the repository (git-ignored)
        config.option.basetemp = os.path.join(ROOT, ".pytest_tmp")
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")
    _plant_oracle_mistake()


def _plant_oracle_mistake():
    """For tests/test_oracle_mutants.py only: MOE_ORACLE_MUTANT = JSON [old, new] re-executes the oracle's
    source with that one snippet replaced, in this (child) pytest process, so that its pins run against a
    deliberately wrong oracle."""
    spec = os.environ.get("MOE_ORACLE_MUTANT")
    if not spec:
        return
    import json

    from oracle import moe_oracle
    old, new = json.loads(spec)
    with open(moe_oracle.__file__) as f:
        src = f.read()
    if src.count(old) != 1:
        raise RuntimeError(f"planted mistake: {old!r} occurs {src.count(old)} times in the oracle")
    exec(compile(src.replace(old, new), moe_oracle.__file__, "exec"), moe_oracle.__dict__)


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: 'key v v v' lines, a 'logits' block, 'expect <mode>' sections."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {"expect": {}}
    cur = out
    with open(path) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    i = 0
    while i < len(lines):
        parts = lines[i].split()
        if parts[0] == "logits":
            T, E = out["T"], out["E"]
            out["logits"] = [[float(v) for v in lines[i + 1 + t].split()] for t in range(T)]
            i += 1 + T
            continue
        if parts[0] == "expect":
            cur = {}
            out["expect"][parts[1]] = cur
        elif len(parts) == 2 and parts[0] in ("T", "E", "K", "m_tile"):
            out[parts[0]] = int(parts[1])
        else:
            cur[parts[0]] = [float(v) for v in parts[1:]]
        i += 1
    return out
