"""Regression fixture: the oracle's tiny-workload results as recorded by
tests/golden/make_golden.py (which calls only the oracle)."""
import os

import pytest


def test_tiny_workload_matches_recorded_oracle(orc):
    import importlib.util
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    recorded = {}
    with open(os.path.join(here, "tiny_oracle.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.rstrip("\n").split(" ", 1)
            recorded[k] = v
    got = mod.compute()
    for k, v in recorded.items():
        assert got[k] == v, k
