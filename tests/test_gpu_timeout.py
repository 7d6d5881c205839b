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


def test_wait_timeout_reports_status_and_the_context_recovers(oracle):
    wl, x = _inputs()
    torch.cuda.synchronize()
    statuses = []
    prev = ta.set_wait_limit_ns(1)
    try:
        for _ in range(3):
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            _call(wl, x, status, n_ctas=2)
            torch.cuda.synchronize()   # the kernels returned: no hang, no CUDA error
            statuses.append(int(status.item()))
            if statuses[-1] == ta.STATUS_TIMEOUT:
                break
    finally:
        assert ta.set_wait_limit_ns(prev) == 1
    assert ta.STATUS_TIMEOUT in statuses, statuses
    assert set(statuses) <= {0, ta.STATUS_TIMEOUT}, statuses

    # same process, same stream, default limit: the results are right again
    ref_o, ref_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
    for n_ctas in (2, 0):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = _call(wl, x, status, n_ctas)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.abs(out.float().cpu().numpy() - ref_o).max() <= OUT_TOL
        assert np.abs(lse.cpu().numpy() - ref_l).max() <= LSE_TOL
