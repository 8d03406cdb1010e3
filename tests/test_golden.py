"""The oracle reproduces the stored regression fixtures in tests/golden/.

The fixtures were written by tests/golden/make_golden.py, which calls only the
oracle.  Values are float64 hex strings; the check allows 1e-13 for libm
differences between x86_64 and aarch64 (exp, log and tanh are not correctly
rounded everywhere).
"""
import json
import math
import os
import sys

import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)

import make_golden  # noqa: E402


@pytest.mark.parametrize("case", make_golden.CASES, ids=lambda c: c["name"])
def test_golden_fixture(case):
    with open(os.path.join(HERE, case["name"] + ".json")) as f:
        rec = json.load(f)
    assert rec["cite"]
    out, lse = make_golden.run(case)
    want = [float.fromhex(x) for x in rec["out"]]
    got = out.view(-1).tolist()
    assert len(got) == len(want)
    for g, w in zip(got, want):
        assert abs(g - w) <= 1e-13
    for g, w in zip(lse.view(-1).tolist(), [float.fromhex(x) for x in rec["lse"]]):
        if math.isinf(w):
            assert g == w
        else:
            assert abs(g - w) <= 1e-13


@pytest.mark.parametrize("case", make_golden.BWD_CASES, ids=lambda c: c["name"])
def test_golden_backward_fixture(case):
    with open(os.path.join(HERE, case["name"] + ".json")) as f:
        rec = json.load(f)
    assert rec["cite"]
    for name, t in zip(("dq", "dk", "dv"), make_golden.run_bwd(case)):
        want = [float.fromhex(x) for x in rec[name]]
        got = t.reshape(-1).tolist()
        assert len(got) == len(want) and any(w != 0.0 for w in want)
        for g, w in zip(got, want):
            assert abs(g - w) <= 1e-12
