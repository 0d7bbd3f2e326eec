"""The stored schedule tables obey the pages' step rules (FlashOverlap technical summary,
section 2): Flash-AG computes the local slice first, Flash-RS the kept slice last, and
what a rank forwards at a hop is what its ring successor uses at the next step."""
import json
import os

import pytest


@pytest.fixture(scope="module")
def tables(repo_root):
    with open(os.path.join(repo_root, "tests", "golden", "schedules.json")) as f:
        return json.load(f)["tables"]


@pytest.mark.parametrize("P", ["2", "4", "8"])
def test_golden_tables_follow_the_rules(tables, P):
    t = tables[P]
    n = int(P)
    for r in range(n):
        ag, rs, nv = t["ag_slice"][r], t["rs_chunk"][r], t["rs_chunk_naive"][r]
        assert ag[0] == r and sorted(ag) == list(range(n))
        assert rs[-1] == r and sorted(rs) == list(range(n))
        assert nv == list(range(n))
        for s in range(n - 1):
            assert t["ag_slice"][(r + 1) % n][s + 1] == ag[s]
            assert t["rs_chunk"][(r + 1) % n][s + 1] == rs[s]
