"""The seeded input generator's layout variants (CPU only): per-sequence trees
and tree tokens written into the paged cache at positions L_b + j."""
import torch

from workloads import CONFIGS, Config, make_workload


def gather(wl, b, pos):
    P = wl.cfg.page
    page = int(wl.block_table[b, pos // P])
    return wl.k_pages[page, :, pos % P], wl.v_pages[page, :, pos % P]


def test_tree_tokens_sit_at_the_padding_positions():
    cfg = Config("w", B=3, Hq=8, Hkv=2, d=64, L=(0, 200), page=16, T=9, seed=5)
    wl = make_workload(cfg, seq_lens=[0, 15, 200], tree_in_cache=True)
    for b in range(3):
        L = int(wl.seq_lens[b])
        assert (wl.block_table[b] >= 0).sum() * 16 >= L + 9
        for j in range(9):
            k, v = gather(wl, b, L + j)
            assert torch.equal(k, wl.tree_k[b, j]) and torch.equal(v, wl.tree_v[b, j])


def test_pages_are_distinct_and_cover_prefix_plus_tree():
    cfg = Config("w2", B=4, Hq=8, Hkv=2, d=64, L=(0, 300), page=64, T=12, seed=6)
    wl = make_workload(cfg, tree_in_cache=True)
    used = wl.block_table[wl.block_table >= 0]
    assert used.unique().numel() == used.numel() == wl.num_pages
    for b in range(4):
        n = int((wl.block_table[b] >= 0).sum())
        assert n == (int(wl.seq_lens[b]) + 12 + 63) // 64


def test_per_sequence_trees_are_valid_and_differ():
    cfg = CONFIGS["maverick"]
    small = Config("w3", B=6, Hq=10, Hkv=2, d=64, L=64, page=64, T=cfg.T,
                   max_depth=cfg.max_depth, max_branch=cfg.max_branch, seed=7)
    wl = make_workload(small, per_sequence_trees=True)
    assert wl.parents.shape == (6, cfg.T)
    for row in wl.parents.tolist():
        assert row[0] == -1 and all(0 <= p < i for i, p in enumerate(row) if i)
    assert len({tuple(r) for r in wl.parents.tolist()}) > 1
    s = wl.sequence(2)
    assert s.cfg.B == 1 and torch.equal(s.parents, wl.parents[2])
    assert torch.equal(s.q[0], wl.q[2]) and torch.equal(s.tree_k[0], wl.tree_k[2])


def test_default_draws_do_not_depend_on_the_variant_flags():
    cfg = CONFIGS["tiny"]
    a = make_workload(cfg)
    b = make_workload(cfg, tree_in_cache=False, per_sequence_trees=False)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_pages, b.k_pages)
    assert torch.equal(a.parents, b.parents)
