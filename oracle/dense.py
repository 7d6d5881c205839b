"""The explicit mask of one-pass tree attention -- TEST INFRASTRUCTURE ONLY
(oracle; importable by the tests, the smoke check and the benchmark's CPU
legs only).

One explicit mask over every key is the form split tree attention avoids
(pith.science review of arXiv 2508.08192, "What carries the argument"); with
the tree tokens padded into the paged cache (the padded layout of the
pith.science verdict record, desk editor's note) the mask of tree token i of
sequence b over cache position p is written out below.  Pinned through
``oracle_dense_rows`` equalling the split definition (tests/oracle_pins.py);
parity unpinned: none.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np


def dense_mask(tree_masks, seq_lens, T: int, cols: int) -> Tuple[np.ndarray, np.ndarray]:
    """The explicit [B][T][cols] mask of one-pass tree attention with the tree
    tokens in the cache at L_b + j: position p < L_b (the committed prefix) is
    visible to every tree token; position L_b + j is visible to token i when
    bit j of i's tree mask is set; everything else is hidden.  tree_masks is
    uint64 [T] (shared) or [B][T].  Returns (dense uint8, key_lens = L_b + T)."""
    L = [int(x) for x in np.asarray(seq_lens).tolist()]
    tm = np.asarray(tree_masks, dtype=np.uint64)
    B = len(L)
    dense = np.zeros((B, T, cols), dtype=np.uint8)
    for b in range(B):
        rowmask = tm[b] if tm.ndim == 2 else tm
        for i in range(T):
            bits = int(rowmask[i])
            for p in range(L[b]):
                dense[b, i, p] = 1
            for j in range(T):
                if (bits >> j) & 1:
                    dense[b, i, L[b] + j] = 1
    return dense, np.asarray([x + T for x in L], dtype=np.int32)
