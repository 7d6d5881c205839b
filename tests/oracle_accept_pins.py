"""Pins of the acceptance / commit oracle (``oracle/accept.py``) to facts
other than itself.  Each pin takes the oracle module so that a mutated copy
can be checked too."""
import itertools
import json
import math
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def pin_golden_cases(acc):
    """Hand-worked cases (tests/golden/accept.json)."""
    data = json.load(open(os.path.join(HERE, "golden", "accept.json")))
    for c in data["cases"]:
        n, path, bonus = acc.greedy_accept(c["parents"], c["draft"], c["target"])
        assert (n, path, bonus) == (c["n"], c["path"], c["bonus"]), c["why"]


def pin_chain_is_linear_speculation(acc):
    """On a chain the rule is linear greedy speculative decoding: the draft
    is accepted up to its first disagreement with the target's next token."""
    rng = np.random.default_rng(11)
    for T in range(1, 9):
        for _ in range(40):
            draft = rng.integers(0, 3, T).tolist()
            target = rng.integers(0, 3, T).tolist()
            k = 1
            while k < T and draft[k] == target[k - 1]:
                k += 1
            n, path, bonus = acc.greedy_accept(list(range(-1, T - 1)), draft, target)
            assert n == k and path == list(range(k)) and bonus == target[k - 1]


def _all_parent_arrays(T):
    for choice in itertools.product(*[range(-1, i) for i in range(T)]):
        yield list(choice)


def pin_bruteforce_paths(acc, max_T=5):
    """Every parent array with T <= max_T, random binary tokens: the result is
    the longest root path whose every edge (u -> w) has draft[w] ==
    target[u], found by checking each node's path on its own."""
    rng = np.random.default_rng(12)
    for T in range(1, max_T + 1):
        for parents in _all_parent_arrays(T):
            draft = rng.integers(0, 2, T).tolist()
            target = rng.integers(0, 2, T).tolist()
            best = None
            for i in range(T):
                path = [i]
                while parents[path[-1]] >= 0:
                    path.append(parents[path[-1]])
                path.reverse()
                ok = all(draft[w] == target[u] for u, w in zip(path, path[1:]))
                if ok and (best is None or len(path) > len(best)):
                    best = path
            n, path, bonus = acc.greedy_accept(parents, draft, target)
            assert path == best and n == len(best) and bonus == target[best[-1]], \
                (parents, draft, target)


def _commit_case(seed, L_list, T, P, tree_in_cache):
    from workloads import Config, make_workload
    cfg = Config("c", B=len(L_list), Hq=4, Hkv=2, d=64, L=(0, 1), page=P, T=T, max_depth=4,
                 max_branch=3, seed=seed)
    # room for the whole tree after each prefix, whichever layout
    width = max((L + T + P - 1) // P for L in L_list)
    wl = make_workload(cfg, seq_lens=L_list, tree_in_cache=True, max_pages_per_seq=width)
    return wl


def _bits(t):
    from workloads import bf16_bits
    return bf16_bits(t)


def pin_commit_then_attend(acc, oracle_c):
    """After committing the accepted path, the last path node's query
    attending the committed prefix of length L + n (no tree) gives the same
    out / lse as the verification call gave it (prefix + its ancestors).  The
    attention side is the C oracle, pinned on its own."""
    from workloads import Workload
    rng = np.random.default_rng(13)
    for seed, L_list, T, P in ((1, [5, 70], 7, 16), (2, [0, 33], 9, 32), (3, [64], 6, 64)):
        wl = _commit_case(seed, L_list, T, P, True)
        B = len(L_list)
        mask = oracle_c.tree_mask(wl.parents.tolist())
        out, lse = oracle_c.verify(wl, mask)
        parents = wl.parents.tolist()
        draft = rng.integers(0, 2, (B, T))
        target = rng.integers(0, 2, (B, T))
        lens, paths, _ = acc.greedy_accept_batch(parents, draft, target)
        for use_cache in (False, True):
            tk = None if use_cache else _bits(wl.tree_k)
            tv = None if use_cache else _bits(wl.tree_v)
            k2, v2, sl2 = acc.kv_commit(_bits(wl.k_pages), _bits(wl.v_pages),
                                        wl.block_table.numpy(), wl.seq_lens.numpy(), tk, tv,
                                        paths, lens, P)
            assert np.array_equal(sl2, wl.seq_lens.numpy() + lens)
            committed = Workload(
                cfg=wl.cfg, parents=torch.zeros(T, dtype=torch.int32),
                seq_lens=torch.from_numpy(sl2.astype(np.int32)), block_table=wl.block_table,
                q=wl.q, k_pages=torch.from_numpy(k2.view(np.int16)).view(torch.bfloat16),
                v_pages=torch.from_numpy(v2.view(np.int16)).view(torch.bfloat16),
                tree_k=wl.tree_k, tree_v=wl.tree_v, scale=wl.scale)
            no_tree = np.zeros(T, dtype=np.uint64)
            for b in range(B):
                last = int(paths[b, lens[b] - 1])
                rows = np.array([(b, last, h) for h in range(wl.cfg.Hq)], dtype=np.int32)
                o2, l2 = oracle_c.verify_rows(committed, no_tree, rows)
                assert np.abs(o2 - out[b, last]).max() < 1e-12
                assert np.abs(l2 - lse[b, last]).max() < 1e-12


def pin_commit_reads_before_writes(acc):
    """With the tree already in the cache, compacting path [0, 2, 3] moves
    position L+2 to L+1 and L+3 to L+2: every row must come from the
    pre-commit cache, exactly as when the rows come from separate buffers."""
    wl = _commit_case(4, [10], 5, 16, True)
    paths = np.array([[0, 2, 3, -1, -1]], dtype=np.int32)
    lens = np.array([3], dtype=np.int32)
    a = acc.kv_commit(_bits(wl.k_pages), _bits(wl.v_pages), wl.block_table.numpy(),
                      wl.seq_lens.numpy(), None, None, paths, lens, 16)
    b = acc.kv_commit(_bits(wl.k_pages), _bits(wl.v_pages), wl.block_table.numpy(),
                      wl.seq_lens.numpy(), _bits(wl.tree_k), _bits(wl.tree_v), paths, lens, 16)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # the row at L + 1 is tree token 2
    pg, off = int(wl.block_table[0, 11 // 16]), 11 % 16
    assert np.array_equal(a[0][pg, :, off], _bits(wl.tree_k)[0, 2])


ALL_PINS = [pin_golden_cases, pin_chain_is_linear_speculation, pin_bruteforce_paths,
            pin_commit_then_attend, pin_commit_reads_before_writes]
