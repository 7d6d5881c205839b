"""Write the golden fixtures in this folder from the fp64 oracle alone.

Run from the repository root:  python tests/golden/make_golden.py

* masks.json      -- ancestor-or-self masks of a few small draft trees
                     (tree mask: pith.science review of 2508.08192, "What
                     carries the argument").  Each entry also lists the
                     ancestor sets in words so a reader can check them by eye.
* tiny_rows.json  -- oracle (out, lse) of sampled rows of the 2-sequence tiny
                     workload (B=2, Hq=4, Hkv=1, d=64, L=128, page=16, T=4),
                     a regression anchor for the oracle itself.

Only ``oracle`` and the seeded ``workloads`` generators are used here.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads import CONFIGS, make_workload  # noqa: E402

TREES = {
    "chain4": [-1, 0, 1, 2],
    "star5": [-1, 0, 0, 0, 0],
    "forest3": [-1, -1, -1],
    "binary7": [-1, 0, 0, 1, 1, 2, 2],
    "eagle_like12": [-1, 0, 0, 0, 1, 1, 2, 3, 4, 4, 6, 8],
}


def main():
    orc = oracle.get()
    masks = {}
    for name, parents in TREES.items():
        m = orc.tree_mask(parents)
        masks[name] = {
            "parents": parents,
            "mask_hex": [f"0x{int(x):016x}" for x in m],
            "attends_to": [[j for j in range(len(parents)) if (int(x) >> j) & 1] for x in m],
        }
    with open(os.path.join(HERE, "masks.json"), "w") as f:
        json.dump({"source": "pith.science/paper/2508.08192, 'What carries the argument' "
                             "(tree mask: each draft token sees itself and its ancestors)",
                   "written_by": "tests/golden/make_golden.py (oracle only)",
                   "trees": masks}, f, indent=1)

    wl = make_workload(CONFIGS["tiny"])
    mask = orc.tree_mask(wl.parents.tolist())
    rows = [(0, 0, 0), (0, 3, 1), (1, 1, 2), (1, 2, 3), (1, 3, 0)]
    out, lse = orc.verify_rows(wl, mask, rows, threads=1)
    with open(os.path.join(HERE, "tiny_rows.json"), "w") as f:
        json.dump({"workload": CONFIGS["tiny"].describe(),
                   "written_by": "tests/golden/make_golden.py (oracle only)",
                   "parents": wl.parents.tolist(),
                   "rows": [list(r) for r in rows],
                   "lse": [float(x) for x in lse],
                   "out": [[float(v) for v in o] for o in out]}, f, indent=1)


if __name__ == "__main__":
    main()
