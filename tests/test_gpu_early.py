"""Early start of the prefix pass (tree_attn_set_early_prefix_loads).

Under the setting the prefix pass reads seq_lens and the block table and
issues the loads of its first committed-prefix K/V blocks before it waits for
the kernel before it in the stream; q, the tree K/V (also where they sit in
the paged cache past the prefix), the parent array and the masks are read
after that wait, and the workspace is written after it.

Checked here:
* the setting changes no result: every call layout gives bit-identical out and
  lse with and without it, on small and full-size workloads;
* q and the tree K/V written by a kernel directly before the call (in the
  same stream, no host synchronisation in between) are the values the call
  uses, against the fp64 oracle -- for the tree in its own buffers, for the
  tree inside the paged cache, and behind this library's own mask kernel,
  which lets its successor start before it ends;
* a captured CUDA graph (writer kernel + call, twice with different q)
  replays with the right results.
"""
import dataclasses

import numpy as np
import pytest
import torch

import speculative_decoding_tree_split_gb300 as ta
from workloads import CONFIGS, Config, make_workload

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ta.build()
    ta.load()


@pytest.fixture
def early():
    """Enables the setting for one test and restores it afterwards."""
    prev = ta.set_early_prefix_loads(True)
    try:
        yield
    finally:
        ta.set_early_prefix_loads(prev)


def to_dev(wl):
    c = torch.device("cuda")
    return dict(parents=wl.parents.to(c), q=wl.q.to(c), k=wl.k_pages.to(c), v=wl.v_pages.to(c),
                bt=wl.block_table.to(c), sl=wl.seq_lens.to(c), tk=wl.tree_k.to(c),
                tv=wl.tree_v.to(c))


def check(out, lse, ref_o, ref_l):
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.abs(o - ref_o).max() <= OUT_TOL
    assert np.abs(l - ref_l).max() <= LSE_TOL


def test_setting_is_host_only_and_restorable():
    prev = ta.set_early_prefix_loads(True)
    try:
        assert ta.set_early_prefix_loads(True) is True
        assert ta.set_early_prefix_loads(False) is True
        assert ta.set_early_prefix_loads(False) is False
    finally:
        ta.set_early_prefix_loads(prev)


SMALL = Config("ea", B=3, Hq=16, Hkv=4, d=128, L=(0, 5000), page=64, T=12, seed=71)
SMALL64 = Config("eb", B=2, Hq=10, Hkv=2, d=64, L=(0, 3000), page=16, T=16, max_depth=4,
                 max_branch=4, seed=72)


def _all_layouts(x, wl, n_ctas=0):
    """(name, out, lse) of every call layout on the same inputs (the tree in
    its own buffers; see the paged and explicit-mask variants below)."""
    res = []
    mask = ta.mask_build(x["parents"])
    res.append(("verify",) + ta.verify(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"],
                                       x["tv"], mask, softmax_scale=wl.scale, n_ctas=n_ctas))
    res.append(("verify_tree",) + ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"],
                                                 x["tk"], x["tv"], x["parents"],
                                                 softmax_scale=wl.scale))
    masks = mask.repeat(wl.cfg.B, 1)
    res.append(("verify_batched",) + ta.verify_batched(x["q"], x["k"], x["v"], x["bt"], x["sl"],
                                                       x["tk"], x["tv"], masks,
                                                       softmax_scale=wl.scale))
    return res


@pytest.mark.parametrize("cfg,lens", [(SMALL, [5000, 61, 1290]), (SMALL64, [3000, 17])],
                         ids=["d128", "d64"])
@pytest.mark.parametrize("n_ctas", [0, 3])
def test_results_bit_identical_with_and_without(cfg, lens, n_ctas):
    wl = make_workload(cfg, seq_lens=lens)
    x = to_dev(wl)
    off = _all_layouts(x, wl, n_ctas)
    prev = ta.set_early_prefix_loads(True)
    try:
        on = _all_layouts(x, wl, n_ctas)
    finally:
        ta.set_early_prefix_loads(prev)
    torch.cuda.synchronize()
    for (name, o0, l0), (_, o1, l1) in zip(off, on):
        assert torch.equal(o0, o1) and torch.equal(l0, l1), name


@pytest.mark.parametrize("cfg,lens", [(SMALL, [5000, 61, 1290]), (SMALL64, [3000, 17])],
                         ids=["d128", "d64"])
def test_tree_in_cache_and_explicit_mask_bit_identical_with_and_without(cfg, lens):
    # tree tokens padded into the paged cache (their blocks load after the
    # dependency wait), and the one-pass explicit-mask form (no early start)
    wl = make_workload(cfg, seq_lens=lens, tree_in_cache=True)
    x = to_dev(wl)
    mask = ta.mask_build(x["parents"])
    cols = ta.dense_cols_for(int(wl.seq_lens.max()) + cfg.T)
    dense, kl = ta.dense_mask_build(mask, x["sl"], cfg.T, cols)

    def run():
        a = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask,
                                 softmax_scale=wl.scale)
        b = ta.verify_dense(x["q"], x["k"], x["v"], x["bt"], kl, dense, softmax_scale=wl.scale)
        return a + b

    off = run()
    prev = ta.set_early_prefix_loads(True)
    try:
        on = run()
    finally:
        ta.set_early_prefix_loads(prev)
    torch.cuda.synchronize()
    for t0, t1 in zip(off, on):
        assert torch.equal(t0, t1)


@pytest.mark.parametrize("name", ["llama8b", "llama70b", "maverick"])
def test_full_size_bit_identical_with_and_without(name):
    cfg = CONFIGS[name]
    wl = make_workload(cfg)
    x = to_dev(wl)
    o0, l0 = ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                            x["parents"], softmax_scale=wl.scale)
    prev = ta.set_early_prefix_loads(True)
    try:
        o1, l1 = ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                                x["parents"], softmax_scale=wl.scale)
    finally:
        ta.set_early_prefix_loads(prev)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def _garbage_like(t, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(t.shape, generator=g, device="cuda") * 4).to(t.dtype)


def test_q_and_tree_written_just_before_are_used(oracle, early):
    wl = make_workload(SMALL, seq_lens=[5000, 61, 1290])
    x = to_dev(wl)
    src = {k: x[k].clone() for k in ("q", "tk", "tv")}
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    for it in range(3):
        for k in src:
            x[k].copy_(_garbage_like(x[k], 100 + it))
        torch.cuda.synchronize()
        # the writers: elementwise kernels in the call's stream, no sync after
        for k in src:
            torch.mul(src[k], 1.0, out=x[k])
        out, lse = ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                                  x["parents"], softmax_scale=wl.scale)
        torch.cuda.synchronize()
        check(out, lse, ref_o, ref_l)


def test_q_written_before_the_mask_kernel_is_used(oracle, early):
    # writer kernel -> tree_mask_build (which lets its successor start before
    # it ends) -> the call
    wl = make_workload(SMALL, seq_lens=[700, 4999, 64])
    x = to_dev(wl)
    q_src = x["q"].clone()
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    for it in range(3):
        x["q"].copy_(_garbage_like(x["q"], 200 + it))
        torch.cuda.synchronize()
        torch.mul(q_src, 1.0, out=x["q"])
        mask = ta.mask_build(x["parents"])
        out, lse = ta.verify(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"], mask,
                             softmax_scale=wl.scale)
        torch.cuda.synchronize()
        check(out, lse, ref_o, ref_l)


def test_tree_written_into_the_paged_cache_just_before_is_used(oracle, early):
    cfg = Config("ep", B=3, Hq=16, Hkv=4, d=128, L=(0, 3000), page=64, T=12, seed=73)
    wl = make_workload(cfg, seq_lens=[60, 2900, 1000], tree_in_cache=True)
    x = to_dev(wl)
    # cache positions L_b + j of the tree tokens: (page, row) pairs
    P = cfg.page
    pages, rows, src_b, src_j = [], [], [], []
    for b in range(cfg.B):
        for j in range(cfg.T):
            pos = int(wl.seq_lens[b]) + j
            pages.append(int(wl.block_table[b, pos // P]))
            rows.append(pos % P)
            src_b.append(b)
            src_j.append(j)
    pages = torch.tensor(pages, device="cuda")
    rows = torch.tensor(rows, device="cuda")
    src_b = torch.tensor(src_b, device="cuda")
    src_j = torch.tensor(src_j, device="cuda")
    tree_k = x["tk"][src_b, src_j]   # [B*T][Hkv][d]
    tree_v = x["tv"][src_b, src_j]
    mask = ta.mask_build(x["parents"])
    want = []
    for b in range(cfg.B):
        s = wl.sequence(b)
        want.append(oracle.verify(s, oracle.tree_mask(s.parents.tolist())))
    ref_o = np.concatenate([w[0] for w in want])
    ref_l = np.concatenate([w[1] for w in want])
    for it in range(3):
        gk = _garbage_like(tree_k, 300 + it)
        gv = _garbage_like(tree_v, 400 + it)
        x["k"][pages, :, rows] = gk
        x["v"][pages, :, rows] = gv
        torch.cuda.synchronize()
        # the writer: a scatter kernel into the pages, then the call
        x["k"][pages, :, rows] = tree_k
        x["v"][pages, :, rows] = tree_v
        out, lse = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], mask,
                                        softmax_scale=wl.scale)
        torch.cuda.synchronize()
        check(out, lse, ref_o, ref_l)


def test_graph_replay_with_a_writer_kernel(oracle, early):
    wl = make_workload(SMALL, seq_lens=[3000, 2048, 100])
    wl2 = dataclasses.replace(wl, q=make_workload(SMALL, seed=74, seq_lens=[3000, 2048, 100]).q)
    x = to_dev(wl)
    q_src = x["q"].clone()
    ws = torch.empty(ta.workspace_size(SMALL.B, SMALL.Hq, SMALL.Hkv, SMALL.d, SMALL.T, 0,
                                       SMALL.page), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x["q"])
    lse = torch.empty(SMALL.B, SMALL.T, SMALL.Hq, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        torch.mul(q_src, 1.0, out=x["q"])
        ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"], x["parents"],
                       out=out, lse=lse, workspace=ws, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        torch.mul(q_src, 1.0, out=x["q"])
        ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"], x["parents"],
                       out=out, lse=lse, workspace=ws, softmax_scale=wl.scale)
    mask = oracle.tree_mask(wl.parents.tolist())
    for w in (wl, wl2, wl):
        q_src.copy_(w.q.to("cuda"))
        x["q"].copy_(_garbage_like(x["q"], 500))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.verify(w, mask)
        check(out, lse, ref_o, ref_l)
