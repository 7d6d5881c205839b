"""Greedy tree acceptance and KV commit -- TEST INFRASTRUCTURE ONLY (oracle).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
may import this module; the product path never does, and it shares no code
with the CUDA path.

What it computes (the step after verification):

* "Efficient Speculative Decoding for Llama at Scale" (fdeinterviews.com
  summary, opening paragraph): the draft proposes candidates, the target
  verifies them, and the service commits one accepted path.
* mlsanity.com referee report on arXiv 2508.08192 (Summary): drafting and
  verification are greedy.  So a draft token is accepted when it equals the
  target's greedy (argmax) token at its parent, and only if its parent was
  accepted.
* The same summary page (paragraph on hidden correctness obligations) and the
  report's minor comment on Section 3.3 (KV bookkeeping after rejection): after
  a branch is rejected, the target cache holds the committed history only.
  Here that means the accepted path's K/V sit at positions ``L_b .. L_b+n-1``
  and the sequence length becomes ``L_b + n``.

Readings where the pages are silent:

* A root (parent -1) is the token the target already chose at the previous
  step, so it is accepted unconditionally.
* The committed path ends at the deepest accepted node.  A tie between nodes
  of equal depth goes to the lowest node index.
* ``n`` counts the root.  The bonus token is the target's token at the path's
  last node.
* A forest accepts every root.

Pins live in ``tests/test_oracle_accept_pins.py``.  Parity unpinned: none.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def greedy_accept(parents: Sequence[int], draft: Sequence[int],
                  target: Sequence[int]) -> Tuple[int, List[int], int]:
    """One sequence: (n, path, bonus_token).

    ``parents`` is a topological parent array (parent < child, roots -1);
    ``draft[i]`` is node i's token; ``target[i]`` is the target's greedy
    token after node i.  The walk goes in node order, so a parent's verdict
    is known before its children's.
    """
    T = len(parents)
    accepted = [False] * T
    depth = [0] * T
    for i in range(T):
        p = parents[i]
        if p < 0:
            accepted[i] = True
            depth[i] = 1
        else:
            if not 0 <= p < i:
                raise ValueError(f"node {i}: parent {p} is not an earlier node")
            accepted[i] = accepted[p] and draft[i] == target[p]
            depth[i] = depth[p] + 1
    best = -1
    for i in range(T):
        if accepted[i] and (best < 0 or depth[i] > depth[best]):
            best = i
    path = []
    node = best
    while node >= 0:
        path.append(node)
        node = parents[node]
    path.reverse()
    return len(path), path, int(target[best])


def greedy_accept_batch(parents, draft, target):
    """Every sequence: parents [T] (shared) or [B][T]; draft, target [B][T].
    Returns (accept_len [B], accept_path [B][T] padded with -1, bonus [B])."""
    draft = np.asarray(draft)
    target = np.asarray(target)
    B, T = draft.shape
    par = np.asarray(parents)
    lens = np.zeros(B, dtype=np.int32)
    paths = np.full((B, T), -1, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    for b in range(B):
        pb = par[b] if par.ndim == 2 else par
        n, path, tok = greedy_accept(pb.tolist(), draft[b].tolist(), target[b].tolist())
        lens[b] = n
        paths[b, :n] = path
        bonus[b] = tok
    return lens, paths, bonus


def kv_commit(k_pages: np.ndarray, v_pages: np.ndarray, block_table: np.ndarray,
              seq_lens: np.ndarray, tree_k, tree_v, accept_path: np.ndarray,
              accept_len: np.ndarray, page_size: int):
    """Return (k_pages', v_pages', seq_lens'): copies of the cache with the
    accepted path written at positions L_b + k, k < n_b.

    ``tree_k`` / ``tree_v`` are [B][T][Hkv][d]; pass None for both when the
    tree tokens already sit in the cache at positions L_b + j, in which case
    all sources are read before anything is written.
    """
    k_new = k_pages.copy()
    v_new = v_pages.copy()
    P = page_size
    B = len(seq_lens)

    def slot(b, pos):
        return int(block_table[b, pos // P]), pos % P

    for b in range(B):
        L = int(seq_lens[b])
        n = int(accept_len[b])
        rows_k, rows_v = [], []
        for k in range(n):
            j = int(accept_path[b, k])
            if tree_k is None:
                pg, off = slot(b, L + j)
                rows_k.append(k_pages[pg, :, off].copy())
                rows_v.append(v_pages[pg, :, off].copy())
            else:
                rows_k.append(np.asarray(tree_k[b, j]).copy())
                rows_v.append(np.asarray(tree_v[b, j]).copy())
        for k in range(n):
            pg, off = slot(b, L + k)
            k_new[pg, :, off] = rows_k[k]
            v_new[pg, :, off] = rows_v[k]
    new_lens = np.asarray(seq_lens, dtype=np.int64) + np.asarray(accept_len, dtype=np.int64)
    return k_new, v_new, new_lens.astype(np.int32)
