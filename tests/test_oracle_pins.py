"""The fp64 oracle against facts that do not come from the oracle (CPU only)."""
import math

import numpy as np
import pytest
import torch

import oracle_pins as pins
from workloads import CONFIGS, Config, make_workload, random_tree


def test_mask_bruteforce_all_trees_up_to_7(oracle):
    pins.pin_mask_bruteforce(oracle, max_T=7)


def test_mask_random_trees_networkx(oracle):
    nx = pytest.importorskip("networkx")
    g = torch.Generator().manual_seed(5)
    for T in (1, 2, 17, 33, 63, 64):
        for depth, branch in ((3, 3), (8, 2), (64, 1), (2, 64)):
            try:
                parents = random_tree(T, depth, branch, g).tolist()
            except ValueError:
                continue
            graph = nx.DiGraph()
            graph.add_nodes_from(range(T))
            graph.add_edges_from((p, i) for i, p in enumerate(parents) if p >= 0)
            got = oracle.tree_mask(parents)
            for i in range(T):
                want = (1 << i) | sum(1 << a for a in nx.ancestors(graph, i))
                assert int(got[i]) == want


@pytest.mark.parametrize("parents", [[0], [-1, 1], [-1, 0, 3, 1], [-2], [-1, -1, 2]])
def test_mask_rejects_non_topological_parents(oracle, parents):
    with pytest.raises(ValueError):
        oracle.tree_mask(parents)


def test_mask_rejects_more_than_64_nodes(oracle):
    with pytest.raises(ValueError):
        oracle.tree_mask(list(range(-1, 64)))


def test_dense_explicit_mask_random_tree(oracle):
    pins.pin_dense_random_tree(oracle)


def test_dense_explicit_mask_special_trees(oracle):
    pins.pin_dense_special_trees(oracle)


def test_chain_tree_equals_causal_attention(oracle):
    pins.pin_chain_is_causal(oracle)


def test_zero_query_closed_form(oracle):
    pins.pin_zero_query_closed_form(oracle)


def test_constant_values(oracle):
    pins.pin_constant_values(oracle)


def test_split_merge_equals_single_pass(oracle):
    pins.pin_split_merge(oracle)


def test_page_renumbering_bit_identical(oracle):
    pins.pin_page_renumbering(oracle)


def test_empty_prefix_is_tree_only_attention(oracle):
    wl = pins.pin_workload(19, seq_lens=[0, 0, 0])
    mask = pins.paths_mask(wl.parents.tolist())
    got_o, got_l = oracle.verify(wl, mask)
    ref_o, ref_l = pins.dense_reference(wl, mask)
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all()
    np.testing.assert_allclose(got_o, ref_o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(got_l, ref_l, atol=1e-12, rtol=0)


def test_row_with_no_keys_gives_zero_and_minus_inf(oracle):
    wl = pins.pin_workload(20, seq_lens=[0, 5, 0])
    zero_mask = [0] * wl.cfg.T
    o, l = oracle.verify_rows(wl, zero_mask, [(0, 1, 2), (1, 1, 2)])
    assert np.all(o[0] == 0) and l[0] == -math.inf
    assert np.isfinite(l[1])


def test_bad_page_id_is_rejected(oracle):
    wl = pins.pin_workload(21)
    wl.block_table[2, 0] = wl.num_pages
    with pytest.raises(ValueError):
        oracle.verify(wl, pins.paths_mask(wl.parents.tolist()))


def test_thread_count_does_not_change_result(oracle):
    wl = pins.pin_workload(22)
    mask = pins.paths_mask(wl.parents.tolist())
    o1, l1 = oracle.verify(wl, mask, threads=1)
    o4, l4 = oracle.verify(wl, mask, threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)


def test_generators_are_seeded_and_follow_the_recipe():
    c = CONFIGS["llama70b"]
    small = Config("s", B=5, Hq=4, Hkv=2, d=8, L=c.L, page=64, T=c.T, tree="random",
                   max_depth=c.max_depth, max_branch=c.max_branch, seed=c.seed)
    a = make_workload(small)
    b = make_workload(small)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)
    lo, hi = c.L
    assert int(a.seq_lens.min()) >= lo and int(a.seq_lens.max()) <= hi
    # every used physical page appears exactly once
    used = a.block_table[a.block_table >= 0]
    assert used.numel() == a.num_pages and len(set(used.tolist())) == a.num_pages
    # tree limits hold
    depth = {}
    kids = {}
    for i, p in enumerate(a.parents.tolist()):
        depth[i] = 1 if p < 0 else depth[p] + 1
        kids[p] = kids.get(p, 0) + 1
        assert p < i
    assert max(depth.values()) <= c.max_depth
    assert max(v for k, v in kids.items() if k >= 0) <= c.max_branch
