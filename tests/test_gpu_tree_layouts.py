"""Per-sequence draft trees and tree tokens padded into the paged cache,
through the C ABI, against the fp64 oracle on the same seeded inputs.

The oracle defines both variants by the same formula as the shared-tree case:
sequence ``b`` attends its prefix and the tree tokens its own mask allows.  It
is evaluated one sequence at a time (``Workload.sequence``), with the tree
tokens' K/V taken from ``tree_k`` / ``tree_v`` -- the very values the
generator wrote into the cache positions ``L_b + j``.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_tree_split_gb300 as ta
from workloads import CONFIGS, Config, make_workload, random_tree

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ta.build()
    ta.load()


def dev(wl):
    c = torch.device("cuda")
    return dict(parents=wl.parents.to(c), q=wl.q.to(c), k=wl.k_pages.to(c),
                v=wl.v_pages.to(c), bt=wl.block_table.to(c), sl=wl.seq_lens.to(c),
                tk=wl.tree_k.to(c), tv=wl.tree_v.to(c))


def oracle_per_sequence(oracle, wl):
    """(masks [B][T] uint64, out [B][T][Hq][d], lse [B][T][Hq]) from the oracle."""
    c = wl.cfg
    outs, lses, masks = [], [], []
    for b in range(c.B):
        s = wl.sequence(b)
        m = oracle.tree_mask(s.parents.tolist())
        o, l = oracle.verify(s, m)
        masks.append(m)
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(masks), np.stack(outs), np.stack(lses)


def check(out, lse, ref_o, ref_l):
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    err_o = np.abs(o - ref_o).max()
    err_l = np.abs(l - ref_l).max()
    assert err_o <= OUT_TOL and err_l <= LSE_TOL, (err_o, err_l)


# ---------------------------------------------------------------------------
# batched mask builder
# ---------------------------------------------------------------------------
def test_batched_masks_bit_exact(oracle):
    g = torch.Generator().manual_seed(7)
    for T, depth, branch in ((4, 4, 3), (16, 4, 4), (33, 8, 2), (64, 64, 1), (64, 2, 64)):
        trees = torch.stack([random_tree(T, depth, branch, g) for _ in range(37)])
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        m = ta.mask_build_batched(trees.cuda(), status=status).cpu().numpy().view(np.uint64)
        assert int(status.item()) == 0
        want = np.stack([oracle.tree_mask(t.tolist()) for t in trees])
        assert np.array_equal(m, want), T


def test_batched_masks_flag_the_bad_tree():
    trees = torch.tensor([[-1, 0, 1], [-1, 2, 0], [-1, 0, 0]], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ta.mask_build_batched(trees.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_PARENT


# ---------------------------------------------------------------------------
# one draft tree per sequence
# ---------------------------------------------------------------------------
PER_SEQ = [
    (Config("ps1", B=4, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=12, seed=51),
     [900, 0, 257, 64]),
    (Config("ps2", B=3, Hq=10, Hkv=2, d=64, L=(0, 500), page=16, T=16, max_depth=4,
            max_branch=4, seed=52), [500, 33, 128]),
    (Config("ps3", B=2, Hq=8, Hkv=2, d=128, L=(0, 400), page=32, T=64, max_depth=8,
            max_branch=3, seed=53), [399, 1]),
]


@pytest.mark.parametrize("cfg,lens", PER_SEQ, ids=[c.name for c, _ in PER_SEQ])
def test_per_sequence_trees(oracle, cfg, lens):
    wl = make_workload(cfg, seq_lens=lens, per_sequence_trees=True)
    x = dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    masks = ta.mask_build_batched(x["parents"], status=status)
    out, lse = ta.verify_batched(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                                 masks, status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_m, ref_o, ref_l = oracle_per_sequence(oracle, wl)
    assert np.array_equal(masks.cpu().numpy().view(np.uint64), want_m)
    check(out, lse, ref_o, ref_l)


def test_batched_with_equal_trees_equals_shared_tree():
    cfg = Config("eq", B=3, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=10, seed=54)
    wl = make_workload(cfg, seq_lens=[900, 300, 17])
    x = dev(wl)
    mask = ta.mask_build(x["parents"])
    o1, l1 = ta.verify(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"], mask,
                       softmax_scale=wl.scale)
    o2, l2 = ta.verify_batched(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                               mask.repeat(3, 1), softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------------------
# tree tokens padded into the paged cache
# ---------------------------------------------------------------------------
PAGED = [
    # tree straddles a page boundary (L = 60, P = 64, T = 12)
    (Config("pt1", B=3, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=12, seed=61),
     [60, 900, 0]),
    # page 16: the tree spans two pages; d = 64; GQA 5
    (Config("pt2", B=2, Hq=10, Hkv=2, d=64, L=(0, 300), page=16, T=16, max_depth=4,
            max_branch=4, seed=62), [30, 256]),
    # T = 64 (two 128-row blocks per unit), prefix page aligned
    (Config("pt3", B=1, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=64, max_depth=8,
            max_branch=3, seed=63), [256]),
]


@pytest.mark.parametrize("per_seq", [False, True], ids=["shared", "per_seq"])
@pytest.mark.parametrize("cfg,lens", PAGED, ids=[c.name for c, _ in PAGED])
def test_tree_in_paged_cache(oracle, cfg, lens, per_seq):
    wl = make_workload(cfg, seq_lens=lens, per_sequence_trees=per_seq, tree_in_cache=True)
    x = dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if per_seq:
        mask = ta.mask_build_batched(x["parents"], status=status)
    else:
        mask = ta.mask_build(x["parents"], status=status)
    out, lse = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask,
                                    status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _, ref_o, ref_l = oracle_per_sequence(oracle, wl)
    check(out, lse, ref_o, ref_l)


def test_paged_tree_agrees_with_separate_tree_buffers():
    # same values read from another place (the work line differs: the tree
    # follows the prefix positions instead of a chunk of its own)
    cfg = Config("bi", B=3, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=12, seed=64)
    wl = make_workload(cfg, seq_lens=[900, 63, 200], tree_in_cache=True)
    x = dev(wl)
    mask = ta.mask_build(x["parents"])
    o1, l1 = ta.verify(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"], mask,
                       softmax_scale=wl.scale)
    o2, l2 = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask,
                                  softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= OUT_TOL
    assert (l1 - l2).abs().max().item() <= LSE_TOL


def test_paged_tree_full_size_llama8b(oracle):
    cfg = CONFIGS["llama8b"]
    wl = make_workload(cfg, tree_in_cache=True)
    x = dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = ta.mask_build(x["parents"], status=status)
    out, lse = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask,
                                    status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _, ref_o, ref_l = oracle_per_sequence(oracle, wl)
    check(out, lse, ref_o, ref_l)


def test_paged_tree_past_the_block_table_sets_status():
    # the block table covers L_b + T - 1 positions only: the last tree token
    # has no page
    cfg = Config("ov", B=1, Hq=8, Hkv=2, d=128, L=(0, 200), page=64, T=4, seed=65)
    wl = make_workload(cfg, seq_lens=[120], tree_in_cache=True)
    assert wl.max_pages_per_seq == 2
    x = dev(wl)
    x["sl"] = torch.tensor([126], dtype=torch.int32, device="cuda")   # 126 + 3 >= 128
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = ta.mask_build(x["parents"])
    ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask, status=status,
                         softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_SEQ_LEN


def test_paged_tree_unmapped_page_sets_status():
    cfg = Config("um", B=1, Hq=8, Hkv=2, d=128, L=(0, 200), page=64, T=4, seed=66)
    wl = make_workload(cfg, seq_lens=[62], tree_in_cache=True, max_pages_per_seq=3)
    x = dev(wl)
    bt = wl.block_table.clone()
    bt[0, 1] = -1            # tree tokens 2, 3 fall on logical page 1
    x["bt"] = bt.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = ta.mask_build(x["parents"])
    ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask, status=status,
                         softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_PAGE
