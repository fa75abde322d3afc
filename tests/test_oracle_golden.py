"""The oracle reproduces its own frozen trajectories bit for bit (regression guard: a
change to the oracle's arithmetic must come with a regenerated fixture)."""
import importlib.util
import json
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
spec = importlib.util.spec_from_file_location("write_golden", os.path.join(HERE, "golden", "write_golden.py"))
wg = importlib.util.module_from_spec(spec)
spec.loader.exec_module(wg)


@pytest.mark.parametrize("name", sorted(wg.CASES))
def test_oracle_matches_frozen_trajectory(name):
    with open(wg.OUT) as f:
        want = json.load(f)[name]
    got = wg.digest(wg.run(wg.CASES[name]))
    assert got == want
