"""tree_attn_verify_noalloc: the entry point for callers that cannot allocate
device memory (fixed-budget memory pools, engines that forbid cudaMalloc after
start-up).  It must give the same results as tree_attn_verify with a caller
workspace, and as the fp64 oracle, call after call, although every call
reuses the library's one built-in scratch array.

Kept in its own file, collected last, so a stop-at-first-failure run has
already run every other test; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_tree_split_gb300 as ta
from workloads import Config, make_workload

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3
SCRATCH_LIMIT = -6


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ta.build()
    return ta.load()


def _inputs(cfg, lens):
    wl = make_workload(cfg, seq_lens=lens)
    dev = torch.device("cuda")
    x = dict(parents=wl.parents.to(dev), q=wl.q.to(dev), k=wl.k_pages.to(dev),
             v=wl.v_pages.to(dev), bt=wl.block_table.to(dev), sl=wl.seq_lens.to(dev),
             tk=wl.tree_k.to(dev), tv=wl.tree_v.to(dev))
    x["mask"] = ta.mask_build(x["parents"])
    return wl, x


def _noalloc(lib, wl, x, out, lse, status):
    c = wl.cfg
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.tree_attn_verify_noalloc(
        x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["bt"].data_ptr(),
        x["bt"].shape[1], x["sl"].data_ptr(), x["tk"].data_ptr(), x["tv"].data_ptr(),
        x["mask"].data_ptr(), out.data_ptr(), lse.data_ptr(), c.B, c.Hq, c.Hkv, c.d, c.T,
        c.page, wl.num_pages, float(wl.scale), status.data_ptr(), stream)


CASES = [
    (Config("na1", B=2, Hq=32, Hkv=8, d=128, L=(0, 3000), page=64, T=12, seed=41), [2900, 131]),
    (Config("na2", B=3, Hq=10, Hkv=2, d=64, L=(0, 900), page=16, T=7, seed=42), [0, 901, 64]),
]


def test_noalloc_matches_verify_on_two_calls_in_a_row(lib, oracle):
    prepared = []
    for cfg, lens in CASES:
        wl, x = _inputs(cfg, lens)
        ref_out, ref_lse = ta.verify(x["q"], x["k"], x["v"], x["bt"], x["sl"], x["tk"], x["tv"],
                                     x["mask"], softmax_scale=wl.scale)
        out = torch.full_like(x["q"], float("nan"))
        lse = torch.full((cfg.B, cfg.T, cfg.Hq), float("nan"), dtype=torch.float32,
                         device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        prepared.append((wl, x, ref_out, ref_lse, out, lse, status))
    torch.cuda.synchronize()
    # two calls back to back on the same stream, both using the shared scratch
    for wl, x, _, _, out, lse, status in prepared:
        assert _noalloc(lib, wl, x, out, lse, status) == 0
    torch.cuda.synchronize()
    for wl, x, ref_out, ref_lse, out, lse, status in prepared:
        assert int(status.item()) == 0
        err_o = (out.float() - ref_out.float()).abs().max().item()
        err_l = (lse - ref_lse).abs().max().item()
        assert err_o <= OUT_TOL and err_l <= LSE_TOL, (wl.cfg.name, err_o, err_l)
        # and every row against the fp64 oracle
        want_o, want_l = oracle.verify(wl, oracle.tree_mask(wl.parents.tolist()))
        err_o = np.abs(out.float().cpu().numpy() - want_o).max()
        err_l = np.abs(lse.cpu().numpy() - want_l).max()
        assert err_o <= OUT_TOL and err_l <= LSE_TOL, (wl.cfg.name, err_o, err_l)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # 64 sequences x 8 KV heads need far more than the 16 MiB array
    cfg = Config("big", B=64, Hq=32, Hkv=8, d=128, L=(0, 128), page=64, T=4, seed=43)
    wl, x = _inputs(cfg, [64] * 64)
    out = torch.empty_like(x["q"])
    lse = torch.empty(64, 4, 32, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, wl, x, out, lse, status) == SCRATCH_LIMIT
