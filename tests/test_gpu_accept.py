"""Greedy acceptance and KV commit through the C ABI against the oracle
(``oracle/accept.py``): integer work, so every result is compared bit for bit
-- accepted lengths, paths, bonus tokens, and the whole paged cache after the
commit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle.accept as acc
import speculative_decoding_tree_split_gb300 as ta
from workloads import Config, bf16_bits, make_workload, random_tree

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ta.build()
    ta.load()


def run_accept(parents, draft, target):
    """parents [T] or [B][T] (CPU int32), draft/target [B][T] -> numpy results."""
    p = parents.cuda()
    mask = ta.mask_build_batched(p) if p.dim() == 2 else ta.mask_build(p)
    n, path, bonus = ta.greedy_accept(mask, draft.cuda(), target.cuda())
    torch.cuda.synchronize()
    return n.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()


def test_golden_cases():
    data = json.load(open(os.path.join(HERE, "golden", "accept.json")))
    for c in data["cases"]:
        n, path, bonus = run_accept(torch.tensor(c["parents"], dtype=torch.int32),
                                    torch.tensor([c["draft"]], dtype=torch.int32),
                                    torch.tensor([c["target"]], dtype=torch.int32))
        T = len(c["parents"])
        assert n[0] == c["n"] and bonus[0] == c["bonus"], c["why"]
        assert path[0].tolist() == c["path"] + [-1] * (T - c["n"]), c["why"]


@pytest.mark.parametrize("T,depth,branch", [(1, 1, 1), (4, 4, 3), (12, 4, 3), (16, 4, 4),
                                            (33, 8, 2), (64, 64, 1), (64, 6, 3)])
@pytest.mark.parametrize("per_seq", [False, True], ids=["shared", "per_seq"])
def test_random_trees_bit_exact(T, depth, branch, per_seq):
    g = torch.Generator().manual_seed(100 + T)
    B = 301
    if per_seq:
        parents = torch.stack([random_tree(T, depth, branch, g) for _ in range(B)])
    else:
        parents = random_tree(T, depth, branch, g)
    # a 2-token alphabet makes long accepted paths common
    draft = torch.randint(0, 2, (B, T), generator=g, dtype=torch.int32)
    target = torch.randint(0, 2, (B, T), generator=g, dtype=torch.int32)
    n, path, bonus = run_accept(parents, draft, target)
    wn, wpath, wbonus = acc.greedy_accept_batch(parents.numpy(), draft.numpy(), target.numpy())
    assert np.array_equal(n, wn) and np.array_equal(path, wpath)
    assert np.array_equal(bonus, wbonus)


def _commit_inputs(cfg, lens, in_cache, seed_tokens):
    wl = make_workload(cfg, seq_lens=lens, per_sequence_trees=True, tree_in_cache=in_cache,
                       tree_room=True)
    g = torch.Generator().manual_seed(seed_tokens)
    B, T = cfg.B, cfg.T
    draft = torch.randint(0, 2, (B, T), generator=g, dtype=torch.int32)
    target = torch.randint(0, 2, (B, T), generator=g, dtype=torch.int32)
    return wl, draft, target


COMMIT = [
    (Config("c1", B=5, Hq=16, Hkv=4, d=128, L=(0, 500), page=64, T=12, seed=71),
     [0, 60, 500, 64, 127]),
    (Config("c2", B=3, Hq=10, Hkv=2, d=64, L=(0, 300), page=16, T=16, max_depth=6,
            max_branch=2, seed=72), [15, 300, 32]),
    (Config("c3", B=2, Hq=8, Hkv=8, d=128, L=(0, 300), page=32, T=64, max_depth=64,
            max_branch=1, seed=73), [31, 0]),
]


@pytest.mark.parametrize("in_cache", [False, True], ids=["tree_buffers", "tree_in_cache"])
@pytest.mark.parametrize("cfg,lens", COMMIT, ids=[c.name for c, _ in COMMIT])
def test_commit_bit_exact(cfg, lens, in_cache):
    wl, draft, target = _commit_inputs(cfg, lens, in_cache, 200 + cfg.seed)
    n_ref, path_ref, _ = acc.greedy_accept_batch(wl.parents.numpy(), draft.numpy(),
                                                 target.numpy())
    k_ref, v_ref, sl_ref = acc.kv_commit(
        bf16_bits(wl.k_pages), bf16_bits(wl.v_pages), wl.block_table.numpy(),
        wl.seq_lens.numpy(), None if in_cache else bf16_bits(wl.tree_k),
        None if in_cache else bf16_bits(wl.tree_v), path_ref, n_ref, cfg.page)

    k = wl.k_pages.cuda()
    v = wl.v_pages.cuda()
    bt = wl.block_table.cuda()
    sl = wl.seq_lens.cuda()
    masks = ta.mask_build_batched(wl.parents.cuda())
    n, path, _ = ta.greedy_accept(masks, draft.cuda(), target.cuda())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl_out = ta.kv_commit(k, v, bt, sl, path, n,
                          tree_k=None if in_cache else wl.tree_k.cuda(),
                          tree_v=None if in_cache else wl.tree_v.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(n.cpu().numpy(), n_ref)
    assert np.array_equal(sl_out.cpu().numpy(), sl_ref)
    assert np.array_equal(bf16_bits(k.cpu()), k_ref)
    assert np.array_equal(bf16_bits(v.cpu()), v_ref)


def test_in_place_compaction_reads_before_writes():
    # path [0, 2, 3]: position L+2 is both a source (for k = 1) and a target
    cfg = Config("h", B=1, Hq=8, Hkv=2, d=128, L=(0, 100), page=16, T=5, seed=74)
    wl = make_workload(cfg, seq_lens=[10], tree_in_cache=True,
                       parents=torch.tensor([-1, 0, 1, 2, 0], dtype=torch.int32))
    path = torch.tensor([[0, 2, 3, -1, -1]], dtype=torch.int32)
    n = torch.tensor([3], dtype=torch.int32)
    k_ref, v_ref, _ = acc.kv_commit(bf16_bits(wl.k_pages), bf16_bits(wl.v_pages),
                                    wl.block_table.numpy(), wl.seq_lens.numpy(), None, None,
                                    path.numpy(), n.numpy(), 16)
    k, v = wl.k_pages.cuda(), wl.v_pages.cuda()
    ta.kv_commit(k, v, wl.block_table.cuda(), wl.seq_lens.cuda(), path.cuda(), n.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(k.cpu()), k_ref)
    assert np.array_equal(bf16_bits(v.cpu()), v_ref)


def test_verify_accept_commit_then_attend():
    """Step n verifies the tree; after accepting and committing, the last
    path node's query over the committed prefix alone (no tree bits) gives
    the out / lse it got during verification."""
    cfg = Config("loop", B=3, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=12, seed=75)
    wl, draft, target = _commit_inputs(cfg, [900, 63, 200], True, 275)
    x = dict(q=wl.q.cuda(), k=wl.k_pages.cuda(), v=wl.v_pages.cuda(),
             bt=wl.block_table.cuda(), sl=wl.seq_lens.cuda())
    masks = ta.mask_build_batched(wl.parents.cuda())
    out, lse = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], masks,
                                    softmax_scale=wl.scale)
    n, path, _ = ta.greedy_accept(masks, draft.cuda(), target.cuda())
    sl2 = ta.kv_commit(x["k"], x["v"], x["bt"], x["sl"], path, n)
    torch.cuda.synchronize()
    n_h, path_h = n.cpu(), path.cpu()
    last = torch.tensor([int(path_h[b, n_h[b] - 1]) for b in range(cfg.B)])
    q1 = x["q"][torch.arange(cfg.B), last].unsqueeze(1).contiguous()    # [B][1][Hq][d]
    no_tree = torch.zeros(1, dtype=torch.int64, device="cuda")
    out2, lse2 = ta.verify_paged_tree(q1, x["k"], x["v"], x["bt"], sl2, no_tree,
                                      softmax_scale=wl.scale)
    torch.cuda.synchronize()
    o1 = out[torch.arange(cfg.B), last].float()
    l1 = lse[torch.arange(cfg.B), last]
    assert (out2[:, 0].float() - o1).abs().max().item() <= OUT_TOL
    assert (lse2[:, 0] - l1).abs().max().item() <= LSE_TOL


def test_bad_path_and_overflow_set_status():
    cfg = Config("st", B=2, Hq=8, Hkv=2, d=128, L=(0, 100), page=16, T=4, seed=76)
    wl = make_workload(cfg, seq_lens=[10, 20], tree_room=True)
    k, v = wl.k_pages.cuda(), wl.v_pages.cuda()
    bt, sl = wl.block_table.cuda(), wl.seq_lens.cuda()
    tk, tv = wl.tree_k.cuda(), wl.tree_v.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    path = torch.tensor([[0, 1, -1, -1], [0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    n = torch.tensor([5, 2], dtype=torch.int32, device="cuda")        # 5 > T
    ta.kv_commit(k, v, bt, sl, path, n, tree_k=tk, tree_v=tv, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_PATH
    status.zero_()
    path2 = torch.tensor([[0, 7, -1, -1], [0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    n2 = torch.tensor([2, 4], dtype=torch.int32, device="cuda")       # node 7 >= T
    ta.kv_commit(k, v, bt, sl, path2, n2, tree_k=tk, tree_v=tv, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_PATH
    status.zero_()
    width = wl.block_table.shape[1]
    sl_far = torch.tensor([16 * width - 2, 0], dtype=torch.int32, device="cuda")
    n3 = torch.tensor([4, 1], dtype=torch.int32, device="cuda")       # runs past the table
    path3 = torch.tensor([[0, 1, 2, 3], [0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    ta.kv_commit(k, v, bt, sl_far, path3, n3, tree_k=tk, tree_v=tv, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) in (ta.STATUS_BAD_SEQ_LEN, ta.STATUS_BAD_PAGE)


@pytest.mark.parametrize("in_cache", [False, True], ids=["tree_buffers", "tree_in_cache"])
@pytest.mark.parametrize("cfg,lens", COMMIT, ids=[c.name for c, _ in COMMIT])
def test_fused_accept_commit_equals_two_calls(cfg, lens, in_cache):
    wl, draft, target = _commit_inputs(cfg, lens, in_cache, 300 + cfg.seed)
    masks = ta.mask_build_batched(wl.parents.cuda())
    tk = None if in_cache else wl.tree_k.cuda()
    tv = None if in_cache else wl.tree_v.cuda()
    bt, sl = wl.block_table.cuda(), wl.seq_lens.cuda()
    d, t = draft.cuda(), target.cuda()
    k1, v1 = wl.k_pages.cuda(), wl.v_pages.cuda()
    n1, p1, b1 = ta.greedy_accept(masks, d, t)
    s1 = ta.kv_commit(k1, v1, bt, sl, p1, n1, tree_k=tk, tree_v=tv)
    k2, v2 = wl.k_pages.cuda(), wl.v_pages.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n2, p2, b2, s2 = ta.accept_commit(masks, d, t, k2, v2, bt, sl, tree_k=tk, tree_v=tv,
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for x, y in ((n1, n2), (p1, p2), (b1, b2), (s1, s2), (k1, k2), (v1, v2)):
        assert torch.equal(x, y)
    # and against the oracle directly
    wn, wpath, wbonus = acc.greedy_accept_batch(wl.parents.numpy(), draft.numpy(),
                                                target.numpy())
    assert np.array_equal(n2.cpu().numpy(), wn) and np.array_equal(p2.cpu().numpy(), wpath)
    assert np.array_equal(b2.cpu().numpy(), wbonus)
