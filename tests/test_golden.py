"""Stored fixtures: the pages' workload facts, and the oracle's tiny-session
digests (written by tests/golden/make_golden.py, which calls only the oracle)."""
import os
import re

from workloads import PROD, TINY

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(name):
    out = {}
    for line in open(os.path.join(HERE, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def test_production_shape_matches_the_pages():
    f = _read("pages_workload_facts.txt")
    assert PROD.capacity == int(f["cache_slots_per_call"])
    assert PROD.tokens == PROD.queries == int(f["new_slots_per_call"])
    assert int(f["passes_per_step"]) * int(f["blocks"]) == int(f["attention_calls_per_step"])


def test_oracle_tiny_session_digests_are_stable():
    import sys
    sys.path.insert(0, HERE)
    from make_golden import records
    want = _read("tiny_session_oracle.txt")
    got = records()
    for k, v in got.items():
        assert want[k] == v, k
    assert re.match(r"head=24 n_valid=48", want["state"])
    assert TINY.capacity == 48
