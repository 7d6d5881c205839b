"""CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs.  Masks bit-exact; out within max-abs 1e-2 and lse within 1e-3 (bf16
inputs, fp32 accumulation)."""
import math

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


def attended_values(wl, mask, b, i, hk):
    """float64 [n][d]: the values query node i of sequence b attends under KV
    head hk -- the committed prefix through the block table, then the tree
    tokens whose bits are set in mask[i]."""
    c = wl.cfg
    L = int(wl.seq_lens[b])
    pos = torch.arange(L)
    pages = wl.block_table[b, pos // c.page].long()
    rows = [wl.v_pages[pages, hk, pos % c.page].to(torch.float64)]
    tree = [j for j in range(c.T) if (int(mask[i]) >> j) & 1]
    rows.append(wl.tree_v[b, tree, hk].to(torch.float64))
    return torch.cat(rows).numpy()


def to_dev(wl):
    d = torch.device("cuda")
    return dict(parents=wl.parents.to(d), q=wl.q.to(d), k_pages=wl.k_pages.to(d),
                v_pages=wl.v_pages.to(d), block_table=wl.block_table.to(d),
                seq_lens=wl.seq_lens.to(d), tree_k=wl.tree_k.to(d), tree_v=wl.tree_v.to(d))


def run_gpu(wl, n_ctas=0, dev_inputs=None, mask=None):
    x = dev_inputs or to_dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if mask is None:
        mask = ta.mask_build(x["parents"], status=status)
    out, lse = ta.verify(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                         x["tree_k"], x["tree_v"], mask, status=status,
                         softmax_scale=wl.scale, n_ctas=n_ctas)
    torch.cuda.synchronize()
    return (mask.cpu().numpy().view(np.uint64), out.float().cpu().numpy(), lse.cpu().numpy(),
            int(status.item()))


def compare_all(oracle, wl, n_ctas=0):
    mask, out, lse, status = run_gpu(wl, n_ctas)
    assert status == 0
    want_mask = oracle.tree_mask(wl.parents.tolist())
    assert np.array_equal(mask, want_mask)
    ref_o, ref_l = oracle.verify(wl, want_mask)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    err_o = np.abs(out - ref_o).max()
    err_l = np.abs(lse - ref_l).max()
    assert err_o <= OUT_TOL and err_l <= LSE_TOL, (err_o, err_l)
    return out, lse


# ---------------------------------------------------------------------------
# mask builder
# ---------------------------------------------------------------------------
def test_mask_random_trees_bit_exact(oracle):
    g = torch.Generator().manual_seed(3)
    for T in (1, 2, 4, 12, 16, 31, 32, 33, 63, 64):
        for depth, branch in ((4, 3), (64, 1), (2, 64), (8, 2)):
            try:
                parents = random_tree(T, depth, branch, g)
            except ValueError:
                continue
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            m = ta.mask_build(parents.cuda(), status=status).cpu().numpy().view(np.uint64)
            assert int(status.item()) == 0
            assert np.array_equal(m, oracle.tree_mask(parents.tolist())), (T, depth, branch)


def test_mask_forest_and_chain_64(oracle):
    for parents in ([-1] * 64, list(range(-1, 63))):
        p = torch.tensor(parents, dtype=torch.int32)
        m = ta.mask_build(p.cuda()).cpu().numpy().view(np.uint64)
        assert np.array_equal(m, oracle.tree_mask(parents))


@pytest.mark.parametrize("parents", [[0], [-1, 1], [-1, 0, 5, 1], [-3, -1]])
def test_mask_bad_parent_sets_status(parents):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ta.mask_build(torch.tensor(parents, dtype=torch.int32, device="cuda"), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_PARENT


# ---------------------------------------------------------------------------
# verify: small cases, every row
# ---------------------------------------------------------------------------
def test_tiny_config(oracle):
    compare_all(oracle, make_workload(CONFIGS["tiny"]))


SMALL = [
    # several 64-token chunks, ragged tails, an empty prefix, GQA 4
    (Config("s1", B=3, Hq=16, Hkv=4, d=128, L=(0, 700), page=64, T=10, seed=21), [0, 700, 129]),
    # page 16 (four pages per chunk), d = 64
    (Config("s2", B=2, Hq=8, Hkv=2, d=64, L=(0, 300), page=16, T=6, seed=22), [300, 47]),
    # page 32, d = 128, GQA 5 (Maverick-like grouping)
    (Config("s3", B=2, Hq=10, Hkv=2, d=128, L=(0, 400), page=32, T=16, max_depth=4,
            max_branch=4, seed=23), [385, 64]),
    # page 128 (two chunks per page)
    (Config("s4", B=2, Hq=8, Hkv=1, d=128, L=(0, 600), page=128, T=5, seed=24), [600, 1]),
    # T = 1: plain paged decode
    (Config("s5", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=1, tree="chain", seed=25),
     [257, 64]),
    # chain tree
    (Config("s6", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=7, tree="chain", seed=26),
     [199, 256]),
    # 256 query rows per unit: two 128-row blocks (T = 64, G = 4)
    (Config("s7", B=1, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=64, max_depth=8,
            max_branch=3, seed=27), [300]),
    # G = 1 (multi-head attention), d = 64
    (Config("s8", B=3, Hq=4, Hkv=4, d=64, L=(0, 300), page=64, T=8, seed=28), [65, 128, 3]),
]


@pytest.mark.parametrize("cfg,lens", SMALL, ids=[c.name for c, _ in SMALL])
def test_small_shapes_all_rows(oracle, cfg, lens):
    compare_all(oracle, make_workload(cfg, seq_lens=lens))


def test_all_prefixes_empty(oracle):
    cfg = Config("e", B=3, Hq=8, Hkv=2, d=128, L=(0, 10), page=64, T=9, seed=29)
    compare_all(oracle, make_workload(cfg, seq_lens=[0, 0, 0], extra_pages=1))


def test_forest_tree(oracle):
    cfg = Config("f", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=6, seed=30)
    wl = make_workload(cfg, seq_lens=[100, 200], parents=torch.full((6,), -1, dtype=torch.int32))
    compare_all(oracle, wl)


def test_zero_query_closed_form(oracle):
    cfg = Config("z", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=5, seed=31)
    wl = make_workload(cfg, seq_lens=[130, 7], q_zero=True)
    mask, out, lse, status = run_gpu(wl)
    assert status == 0
    G = cfg.Hq // cfg.Hkv
    for b in range(2):
        for i in range(5):
            n = int(wl.seq_lens[b]) + bin(int(mask[i])).count("1")
            assert np.abs(lse[b, i] - math.log(n)).max() <= LSE_TOL
            # q = 0 gives equal weights: out is the mean of the attended values
            for hk in range(cfg.Hkv):
                want = attended_values(wl, mask, b, i, hk).mean(0)
                got = out[b, i, hk * G:(hk + 1) * G]
                assert np.abs(got - want).max() <= OUT_TOL, (b, i, hk)


@pytest.mark.parametrize("n_ctas", [1, 3, 7, 40, 152, 500])
def test_split_count_invariance(oracle, n_ctas):
    cfg = Config("k", B=3, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=8, seed=32)
    compare_all(oracle, make_workload(cfg, seq_lens=[900, 1, 450]), n_ctas=n_ctas)


def test_page_renumbering_is_bit_identical():
    cfg = Config("p", B=3, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=8, seed=33)
    wl = make_workload(cfg, seq_lens=[900, 333, 64], extra_pages=5)
    _, o1, l1, s1 = run_gpu(wl)
    g = torch.Generator().manual_seed(33)
    perm = torch.randperm(wl.num_pages, generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(wl.num_pages)
    wl.k_pages = wl.k_pages[inv].contiguous()
    wl.v_pages = wl.v_pages[inv].contiguous()
    bt = wl.block_table.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    wl.block_table = bt
    _, o2, l2, s2 = run_gpu(wl)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_repeated_calls_are_deterministic():
    cfg = Config("r", B=2, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=8, seed=34)
    wl = make_workload(cfg, seq_lens=[900, 500])
    x = to_dev(wl)
    _, o1, l1, _ = run_gpu(wl, dev_inputs=x)
    _, o2, l2, _ = run_gpu(wl, dev_inputs=x)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_two_pass_api_matches_oracle_and_verify(oracle):
    # the two-pass form (prefix pass; suffix pass + merge) against the oracle
    # and against tree_attn_verify, which attends the tree inside the prefix
    # pass
    cfg = Config("t", B=2, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=8, seed=35)
    wl = make_workload(cfg, seq_lens=[900, 77])
    x = to_dev(wl)
    mask = ta.mask_build(x["parents"])
    _, o1, l1, _ = run_gpu(wl, dev_inputs=x, mask=mask)
    ws = torch.empty(ta.workspace_size(2, 16, 4, 128, 8, 0, 64), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(x["q"])
    lse = torch.empty(2, 8, 16, dtype=torch.float32, device="cuda")
    ta.prefix_pass(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"], ws)
    ta.suffix_merge(x["q"], x["seq_lens"], x["block_table"].shape[1], 64, x["tree_k"],
                    x["tree_v"], mask, ws, out, lse)
    torch.cuda.synchronize()
    o2, l2 = out.float().cpu().numpy(), lse.cpu().numpy()
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    assert np.abs(o2 - ref_o).max() <= OUT_TOL and np.abs(l2 - ref_l).max() <= LSE_TOL
    assert np.abs(o2 - o1).max() <= OUT_TOL and np.abs(l2 - l1).max() <= LSE_TOL


# ---------------------------------------------------------------------------
# device-side status codes
# ---------------------------------------------------------------------------
def test_bad_page_id_sets_status():
    cfg = Config("bp", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=4, seed=36)
    wl = make_workload(cfg, seq_lens=[200, 100])
    wl.block_table[1, 0] = wl.num_pages + 3
    *_, status = run_gpu(wl)
    assert status == ta.STATUS_BAD_PAGE


def test_too_long_sequence_sets_status():
    cfg = Config("bl", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=4, seed=37)
    wl = make_workload(cfg, seq_lens=[200, 100])
    wl.seq_lens[0] = 64 * wl.max_pages_per_seq + 1
    *_, status = run_gpu(wl)
    assert status == ta.STATUS_BAD_SEQ_LEN


# ---------------------------------------------------------------------------
# CUDA graph capture (caller-owned workspace, no host sync inside)
# ---------------------------------------------------------------------------
def test_graph_capture_replays_identically():
    cfg = Config("g", B=2, Hq=16, Hkv=4, d=128, L=(0, 900), page=64, T=8, seed=38)
    wl = make_workload(cfg, seq_lens=[900, 300])
    x = to_dev(wl)
    ws = torch.empty(ta.workspace_size(2, 16, 4, 128, 8, 0, 64), dtype=torch.uint8,
                     device="cuda")
    mask = torch.empty(8, dtype=torch.int64, device="cuda")
    out = torch.empty_like(x["q"])
    lse = torch.empty(2, 8, 16, dtype=torch.float32, device="cuda")

    def step():
        ta.mask_build(x["parents"], mask_out=mask)
        ta.verify(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                  x["tree_k"], x["tree_v"], mask, out=out, lse=lse, workspace=ws)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    o_eager, l_eager = out.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    lse.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, o_eager) and torch.equal(lse, l_eager)


# ---------------------------------------------------------------------------
# the five workload shapes at full size
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["llama8b", "llama70b", "chain", "maverick"])
def test_full_size_configs(oracle, name):
    cfg = CONFIGS[name]
    wl = make_workload(cfg)
    mask, out, lse, status = run_gpu(wl)
    assert status == 0
    want_mask = oracle.tree_mask(wl.parents.tolist())
    assert np.array_equal(mask, want_mask)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    # every (b, i, h) row: each (sequence, KV head) unit's pieces of the
    # split work line are checked, not a sample of them
    ref_o, ref_l = oracle.verify(wl, want_mask)
    assert np.abs(out - ref_o).max() <= OUT_TOL
    assert np.abs(lse - ref_l).max() <= LSE_TOL


@pytest.mark.parametrize("name", ["llama8b", "llama70b", "chain", "maverick"])
def test_full_size_verify_tree(oracle, name):
    # The call bench.py times: masks built from the parent array inside the
    # call, at each workload's full size, with the kernel selector's own tree
    # placement (prefix pass for llama8b and llama70b, merge kernel for the
    # chain and Maverick); every row against the oracle.
    cfg = CONFIGS[name]
    wl = make_workload(cfg)
    x = to_dev(wl)
    B, T = cfg.B, cfg.T
    p = ta.plan(B, cfg.Hq, cfg.Hkv, cfg.d, T, cfg.page, wl.max_pages_per_seq)
    assert p["tree_in_prefix"] == (1 if name in ("llama8b", "llama70b") else 0)
    mask_out = torch.zeros(T, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = ta.verify_tree(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["tree_k"], x["tree_v"], x["parents"],
                              mask_out=mask_out, status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_mask = oracle.tree_mask(wl.parents.tolist())
    assert np.array_equal(mask_out.cpu().numpy().view(np.uint64), want_mask)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_o, ref_l = oracle.verify(wl, want_mask)
    assert np.abs(out - ref_o).max() <= OUT_TOL
    assert np.abs(lse - ref_l).max() <= LSE_TOL


def test_merge_rows_per_warp(oracle):
    # 16 x 8 units x 64 rows with the tree on the prefix pass (a small call):
    # 2048 single-row merge CTAs would not fit at once, so each merge warp
    # takes several rows in turn; every row against the oracle, both APIs.
    cfg = Config("rpw", B=16, Hq=64, Hkv=8, d=128, L=(0, 300), page=16, T=8, max_depth=3,
                 max_branch=3, seed=96)
    wl = make_workload(cfg)
    p = ta.plan(16, 64, 8, 128, 8, 16, wl.max_pages_per_seq)
    assert p["tree_in_prefix"] == 1 and p["merge_rows_per_warp"] > 1
    out, lse = compare_all(oracle, wl)
    x = to_dev(wl)
    o2, l2 = ta.verify_tree(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                            x["tree_k"], x["tree_v"], x["parents"], softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert np.array_equal(o2.float().cpu().numpy(), out)
    assert np.array_equal(l2.cpu().numpy(), lse)


def test_merge_rows_per_warp_with_many_partials(oracle):
    # 4 x 16 units of 64 rows, 4096-token prefixes: each unit spans about two
    # and a half prefix CTAs, so a row has up to four partials (a straddling
    # CTA leaves its two row copies unfolded); 1024 single-row merge CTAs
    # would not fit at once, so each merge warp takes two rows in turn.
    cfg = Config("rpw2", B=4, Hq=128, Hkv=16, d=128, L=4096, page=64, T=8, max_depth=3,
                 max_branch=3, seed=95)
    wl = make_workload(cfg)
    p = ta.plan(4, 128, 16, 128, 8, 64, wl.max_pages_per_seq)
    assert p["tree_in_prefix"] == 1 and p["merge_rows_per_warp"] == 2
    assert p["merge_warps_per_row"] == 1
    x = to_dev(wl)
    out, lse = ta.verify_tree(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["tree_k"], x["tree_v"], x["parents"],
                              softmax_scale=wl.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    assert np.abs(out.float().cpu().numpy() - ref_o).max() <= OUT_TOL
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= LSE_TOL


@pytest.mark.parametrize("T,G,n_ctas", [(4, 4, 2), (8, 4, 3), (12, 4, 2), (16, 4, 2), (20, 4, 1),
                                        (16, 5, 2)])
def test_row_replication_paths(oracle, T, G, n_ctas):
    # Few CTAs => many steps per CTA => the prefix pass replicates the query
    # rows 4x (M <= 32) or 2x (M <= 64); M > 64 uses one copy.
    cfg = Config(f"rep{T}x{G}", B=2, Hq=2 * G, Hkv=2, d=128, L=(0, 1000), page=64, T=T,
                 max_depth=5, max_branch=4, seed=40 + T)
    compare_all(oracle, make_workload(cfg, seq_lens=[997, 650]), n_ctas=n_ctas)


# ---------------------------------------------------------------------------
# masks built inside the merge kernel (tree_attn_verify_tree)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("per_seq", [False, True], ids=["shared", "per_seq"])
def test_verify_tree_equals_mask_build_then_verify(oracle, per_seq):
    cfg = Config("vt", B=3, Hq=32, Hkv=8, d=128, L=(0, 3000), page=64, T=12, seed=91)
    wl = make_workload(cfg, seq_lens=[3000, 0, 1031], per_sequence_trees=per_seq)
    x = to_dev(wl)
    if per_seq:
        mask = ta.mask_build_batched(x["parents"])
        o1, l1 = ta.verify_batched(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                                   x["seq_lens"], x["tree_k"], x["tree_v"], mask,
                                   softmax_scale=wl.scale)
    else:
        mask = ta.mask_build(x["parents"])
        o1, l1 = ta.verify(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                           x["tree_k"], x["tree_v"], mask, softmax_scale=wl.scale)
    mask_out = torch.zeros_like(mask)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o2, l2 = ta.verify_tree(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                            x["seq_lens"], x["tree_k"], x["tree_v"], x["parents"],
                            mask_out=mask_out, status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(mask_out, mask)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    if not per_seq:
        ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
        assert np.abs(o2.float().cpu().numpy() - ref_o).max() <= OUT_TOL
        assert np.abs(l2.cpu().numpy() - ref_l).max() <= LSE_TOL


def test_verify_tree_bad_parent_sets_status():
    cfg = Config("vb", B=2, Hq=8, Hkv=2, d=128, L=(0, 300), page=64, T=4, seed=92)
    wl = make_workload(cfg, seq_lens=[200, 100], parents=torch.tensor([-1, 0, 3, 1]))
    x = to_dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ta.verify_tree(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                   x["tree_k"], x["tree_v"], x["parents"], status=status,
                   softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_PARENT


@pytest.mark.parametrize("n_ctas", [2, 19, 152])
def test_many_partials_per_row(oracle, n_ctas):
    # one long sequence, few units: rows collect up to ~80 partials, which
    # exercises the merge's batches past the first round trip
    cfg = Config("mp", B=1, Hq=16, Hkv=2, d=128, L=(0, 12000), page=64, T=4, seed=93)
    wl = make_workload(cfg, seq_lens=[11997])
    mask, out, lse, status = run_gpu(wl, n_ctas=n_ctas)
    assert status == 0
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    assert np.abs(out - ref_o).max() <= OUT_TOL
    assert np.abs(lse - ref_l).max() <= LSE_TOL


@pytest.mark.parametrize("n_ctas", [2, 100])
def test_both_tree_placements(oracle, n_ctas):
    # 8 units x 16 steps: with 2 CTAs (64 steps each) the merge kernel attends
    # the tree; with 100 CTAs the prefix pass does (one masked chunk per unit)
    cfg = Config("tp", B=2, Hq=16, Hkv=4, d=128, L=(0, 1000), page=64, T=12, seed=94)
    wl = make_workload(cfg, seq_lens=[1000, 37])
    p = ta.plan(2, 16, 4, 128, 12, 64, wl.max_pages_per_seq, n_ctas)
    assert p["tree_in_prefix"] == (1 if n_ctas == 100 else 0)
    compare_all(oracle, wl, n_ctas=n_ctas)


@pytest.mark.parametrize("per_seq", [False, True], ids=["shared", "per_seq"])
def test_verify_tree_two_pass_form(oracle, per_seq):
    # 24 x 8 = 192 units (more than GB300's 152 SMs) x 64 steps is more than
    # 32 steps per CTA, so the merge kernel attends the tree (masks built
    # there from the parents)
    cfg = Config("vt2", B=24, Hq=32, Hkv=8, d=128, L=4096, page=64, T=8, max_depth=3,
                 max_branch=3, seed=95)
    wl = make_workload(cfg, per_sequence_trees=per_seq)
    p = ta.plan(24, 32, 8, 128, 8, 64, wl.max_pages_per_seq)
    assert p["tree_in_prefix"] == 0
    x = to_dev(wl)
    mask = ta.mask_build_batched(x["parents"]) if per_seq else ta.mask_build(x["parents"])
    verify = ta.verify_batched if per_seq else ta.verify
    o1, l1 = verify(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                    x["tree_k"], x["tree_v"], mask, softmax_scale=wl.scale)
    mask_out = torch.zeros_like(mask)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o2, l2 = ta.verify_tree(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                            x["seq_lens"], x["tree_k"], x["tree_v"], x["parents"],
                            mask_out=mask_out, status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(mask_out, mask)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    got_o, got_l = o2.float().cpu().numpy(), l2.cpu().numpy()
    for b in range(cfg.B):   # every row, sequence by sequence (each with its own tree)
        s = wl.sequence(b)
        ref_o, ref_l = oracle.verify(s, oracle.tree_mask(s.parents.tolist()))
        assert np.abs(got_o[b] - ref_o[0]).max() <= OUT_TOL, b
        assert np.abs(got_l[b] - ref_l[0]).max() <= LSE_TOL, b
