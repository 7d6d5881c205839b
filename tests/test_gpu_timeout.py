"""Failure detection in the prefix pass: a pipeline wait that runs out.

Every wait of the prefix kernel on another role of its CTA (copy warp, MMA
warp, softmax warps) is bounded by the library's wait limit.  Here the limit
is set to 1 ns, far below the microseconds a tile takes to arrive from HBM,
so a wait of the call runs out: the kernel must store
TREE_ATTN_STATUS_TIMEOUT in the status word, let its own copies and MMAs in
flight finish, free its tensor memory and return.  Nothing faults, traps or
hangs; the test then shows that the CUDA context is still usable: the next
calls on the same stream, with the default limit, match the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_tree_split_gb300 as ta
from workloads import Config, make_workload

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ta.build()
    ta.load()


def _inputs():
    # two CTAs over two long sequences: each CTA waits for dozens of K/V
    # blocks, every one of which takes far longer than the limit to land
    cfg = Config("to", B=2, Hq=16, Hkv=4, d=128, L=(0, 4000), page=64, T=8, seed=97)
    wl = make_workload(cfg, seq_lens=[4000, 3511])
    d = torch.device("cuda")
    x = dict(parents=wl.parents.to(d), q=wl.q.to(d), k=wl.k_pages.to(d), v=wl.v_pages.to(d),
             bt=wl.block_table.to(d), sl=wl.seq_lens.to(d), tk=wl.tree_k.to(d),
             tv=wl.tree_v.to(d))
    x["mask"] = ta.mask_build(x["parents"])
    return wl, x


def _call(wl, x, status, n_ctas):
    return ta.verify(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"], x["mask"],
                     status=status, softmax_scale=wl.scale, n_ctas=n_ctas)


def _times_out(run):
    """Runs `run(status)` under a 1 ns wait limit (up to three tries) and
    returns the statuses seen; the limit is restored whatever happens."""
    statuses = []
    prev = ta.set_wait_limit_ns(1)
    try:
        for _ in range(3):
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            run(status)
            torch.cuda.synchronize()   # the kernels returned: no hang, no CUDA error
            statuses.append(int(status.item()))
            if statuses[-1] == ta.STATUS_TIMEOUT:
                break
    finally:
        assert ta.set_wait_limit_ns(prev) == 1
    assert ta.STATUS_TIMEOUT in statuses, statuses
    assert set(statuses) <= {0, ta.STATUS_TIMEOUT}, statuses
    return statuses


def test_wait_timeout_reports_status_and_the_context_recovers(oracle):
    wl, x = _inputs()
    torch.cuda.synchronize()
    _times_out(lambda status: _call(wl, x, status, n_ctas=2))

    # same process, same stream, default limit: the results are right again
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    for n_ctas in (2, 0):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = _call(wl, x, status, n_ctas)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.abs(out.float().cpu().numpy() - ref_o).max() <= OUT_TOL
        assert np.abs(lse.cpu().numpy() - ref_l).max() <= LSE_TOL


# Other kernel variants, each with its own exit paths: one row copy (80 query
# rows: the fold stages a single copy), the tree on the prefix pass's work
# line (masks built in the kernel from the parents), and the one-pass form
# under an explicit mask.
ONE_COPY = Config("to1", B=2, Hq=20, Hkv=4, d=128, L=(0, 3000), page=64, T=16, max_depth=4,
                  max_branch=4, seed=98)
VARIANTS = [
    # (name, config, lengths, CTAs (0: the selector's), replicas, tree on the prefix pass)
    ("one_copy_tree_on_prefix", ONE_COPY, [3000, 1999], 0, 1, 1),
    ("one_copy_two_pass", ONE_COPY, [3000, 1999], 2, 1, 0),
    ("two_copies_tree_on_prefix", Config("to2", B=1, Hq=32, Hkv=8, d=128, L=(0, 6000), page=64,
                                         T=12, seed=99), [6000], 0, 2, 1),
]


@pytest.mark.parametrize("name,cfg,lens,n_ctas,copies,tree_in_prefix", VARIANTS,
                         ids=[v[0] for v in VARIANTS])
def test_wait_timeout_in_other_kernel_variants(oracle, name, cfg, lens, n_ctas, copies,
                                               tree_in_prefix):
    wl = make_workload(cfg, seq_lens=lens)
    d = torch.device("cuda")
    x = dict(q=wl.q.to(d), k=wl.k_pages.to(d), v=wl.v_pages.to(d), bt=wl.block_table.to(d),
             sl=wl.seq_lens.to(d), tk=wl.tree_k.to(d), tv=wl.tree_v.to(d),
             parents=wl.parents.to(d))
    x["mask"] = ta.mask_build(x["parents"])
    p = ta.plan(cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.T, cfg.page, wl.max_pages_per_seq, n_ctas)
    assert (p["replicas"], p["tree_in_prefix"]) == (copies, tree_in_prefix)

    def run(status):
        if n_ctas:
            return _call(wl, x, status, n_ctas)
        return ta.verify_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                              x["parents"], status=status, softmax_scale=wl.scale)

    torch.cuda.synchronize()
    _times_out(run)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    assert np.abs(out.float().cpu().numpy() - ref_o).max() <= OUT_TOL
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= LSE_TOL


def test_wait_timeout_in_the_explicit_mask_kernel(oracle):
    from oracle import all_rows
    cfg = Config("to3", B=2, Hq=16, Hkv=4, d=128, L=(0, 3000), page=64, T=8, seed=100)
    wl = make_workload(cfg, seq_lens=[2900, 1500], tree_in_cache=True)
    d = torch.device("cuda")
    q, k, v = wl.q.to(d), wl.k_pages.to(d), wl.v_pages.to(d)
    bt, sl = wl.block_table.to(d), wl.seq_lens.to(d)
    mask = ta.mask_build(wl.parents.to(d))
    cols = ta.dense_cols_for(int(wl.seq_lens.max()) + cfg.T)
    dense, kl = ta.dense_mask_build(mask, sl, cfg.T, cols)
    torch.cuda.synchronize()

    def run(status):
        return ta.verify_dense(q, k, v, bt, kl, dense, status=status, softmax_scale=wl.scale)

    _times_out(run)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = all_rows(cfg.B, cfg.T, cfg.Hq)
    ref_o, ref_l = oracle.dense_rows(wl, kl.cpu().numpy(), dense.cpu().numpy(), rows)
    got_o = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    got_l = lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert np.abs(got_o - ref_o).max() <= OUT_TOL
    assert np.abs(got_l - ref_l).max() <= LSE_TOL
