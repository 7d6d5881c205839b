"""Golden fixtures (tests/golden/) against the oracle and the path walk."""
import json
import os

import numpy as np

import oracle_pins as pins
from workloads import CONFIGS, make_workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_golden_masks(oracle):
    data = json.load(open(os.path.join(GOLDEN, "masks.json")))
    for name, entry in data["trees"].items():
        parents = entry["parents"]
        stored = [int(x, 16) for x in entry["mask_hex"]]
        assert stored == pins.paths_mask(parents), name
        assert [int(x) for x in oracle.tree_mask(parents)] == stored, name
        for i, seen in enumerate(entry["attends_to"]):
            assert sum(1 << j for j in seen) == stored[i]


def test_golden_tiny_rows(oracle):
    data = json.load(open(os.path.join(GOLDEN, "tiny_rows.json")))
    wl = make_workload(CONFIGS["tiny"])
    assert wl.parents.tolist() == data["parents"]
    out, lse = oracle.verify_rows(wl, oracle.tree_mask(data["parents"]), data["rows"], threads=1)
    np.testing.assert_allclose(lse, data["lse"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, np.array(data["out"]), rtol=0, atol=1e-12)
