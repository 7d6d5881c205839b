"""One-pass tree attention under an explicit mask (the form split attention
replaces), through the C ABI, against the fp64 oracle: the explicit mask
bit-exact, out within max-abs 1e-2 and lse within 1e-3."""
import numpy as np
import pytest
import torch

import speculative_decoding_tree_split_gb300 as ta
from oracle import all_rows
from oracle.dense import dense_mask as oracle_dense_mask
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


def dev(wl):
    c = torch.device("cuda")
    return dict(parents=wl.parents.to(c), q=wl.q.to(c), k=wl.k_pages.to(c), v=wl.v_pages.to(c),
                bt=wl.block_table.to(c), sl=wl.seq_lens.to(c))


def tree_masks(x):
    p = x["parents"]
    return ta.mask_build_batched(p) if p.dim() == 2 else ta.mask_build(p)


def check_rows(oracle, wl, key_lens, dense, out, lse, rows):
    ref_o, ref_l = oracle.dense_rows(wl, key_lens, dense, rows)
    o = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    l = lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(o - ref_o).max() <= OUT_TOL
    assert np.abs(l[fin] - ref_l[fin]).max() <= LSE_TOL if fin.any() else True


CASES = [
    (Config("d1", B=3, Hq=16, Hkv=4, d=128, L=(0, 700), page=64, T=10, seed=81),
     [700, 0, 129], False),
    (Config("d2", B=2, Hq=10, Hkv=2, d=64, L=(0, 300), page=16, T=16, max_depth=4,
            max_branch=4, seed=82), [300, 47], True),
    (Config("d3", B=2, Hq=8, Hkv=2, d=128, L=(0, 400), page=32, T=64, max_depth=8,
            max_branch=3, seed=83), [385, 64], True),
    (Config("d4", B=2, Hq=8, Hkv=8, d=128, L=(0, 300), page=128, T=4, tree="chain", seed=84),
     [255, 1], False),
]


@pytest.mark.parametrize("cfg,lens,per_seq", CASES, ids=[c.name for c, _, _ in CASES])
def test_explicit_mask_path(oracle, cfg, lens, per_seq):
    wl = make_workload(cfg, seq_lens=lens, per_sequence_trees=per_seq, tree_in_cache=True)
    x = dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tm = tree_masks(x)
    cols = ta.dense_cols_for(max(lens) + cfg.T) + 32       # not the minimal width
    dense, key_lens = ta.dense_mask_build(tm, x["sl"], cfg.T, cols, status=status)
    out, lse = ta.verify_dense(x["q"], x["k"], x["v"], x["bt"], key_lens, dense, status=status,
                               softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_dense, want_kl = oracle_dense_mask(tm.cpu().numpy().view(np.uint64), lens, cfg.T, cols)
    assert np.array_equal(dense.cpu().numpy(), want_dense)
    assert np.array_equal(key_lens.cpu().numpy(), want_kl)
    check_rows(oracle, wl, want_kl, want_dense, out, lse, all_rows(cfg.B, cfg.T, cfg.Hq))


def test_random_explicit_mask(oracle):
    cfg = Config("rm", B=2, Hq=16, Hkv=4, d=128, L=(0, 700), page=64, T=12, seed=85)
    wl = make_workload(cfg, seq_lens=[650, 200], tree_in_cache=True)
    x = dev(wl)
    key_lens = wl.seq_lens + cfg.T
    cols = ta.dense_cols_for(int(key_lens.max()))
    g = torch.Generator().manual_seed(85)
    dense = (torch.rand((2, 12, cols), generator=g) < 0.3).to(torch.uint8)
    dense[0, 3, :] = 0                      # a token that sees no key at all
    dense[1, 5, :] = 0
    dense[1, 5, 130] = 1                    # ... and one that sees a single key
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = ta.verify_dense(x["q"], x["k"], x["v"], x["bt"], key_lens.cuda(), dense.cuda(),
                               status=status, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_rows(oracle, wl, key_lens.numpy(), dense.numpy(), out, lse, all_rows(2, 12, 16))
    assert torch.all(lse[0, 3] == float("-inf")) and torch.all(out[0, 3] == 0)


def test_one_pass_agrees_with_split():
    cfg = Config("eq", B=3, Hq=32, Hkv=8, d=128, L=(0, 3000), page=64, T=12, seed=86)
    wl = make_workload(cfg, seq_lens=[3000, 100, 1777], tree_in_cache=True)
    x = dev(wl)
    tm = tree_masks(x)
    o1, l1 = ta.verify_paged_tree(x["q"], x["k"], x["v"], x["bt"], x["sl"], tm,
                                  softmax_scale=wl.scale)
    dense, kl = ta.dense_mask_build(tm, x["sl"], 12, ta.dense_cols_for(3012))
    o2, l2 = ta.verify_dense(x["q"], x["k"], x["v"], x["bt"], kl, dense, softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= OUT_TOL
    assert (l1 - l2).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("name", ["llama8b", "llama70b", "chain", "maverick"])
def test_full_size(oracle, name):
    cfg = CONFIGS[name]
    wl = make_workload(cfg, tree_in_cache=True)
    x = dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tm = tree_masks(x)
    cols = ta.dense_cols_for(int(wl.seq_lens.max()) + cfg.T)
    dense, kl = ta.dense_mask_build(tm, x["sl"], cfg.T, cols, status=status)
    out, lse = ta.verify_dense(x["q"], x["k"], x["v"], x["bt"], kl, dense, status=status,
                               softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # every (b, i, h) row against the one-pass oracle
    check_rows(oracle, wl, kl.cpu().numpy(), dense.cpu().numpy(), out, lse,
               all_rows(cfg.B, cfg.T, cfg.Hq))


def test_statuses():
    cfg = Config("st", B=1, Hq=8, Hkv=2, d=128, L=(0, 200), page=64, T=4, seed=87)
    wl = make_workload(cfg, seq_lens=[120], tree_in_cache=True)
    x = dev(wl)
    tm = tree_masks(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ta.dense_mask_build(tm, x["sl"], 4, 112, status=status)          # 120 + 4 > 112
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_SEQ_LEN
    status.zero_()
    dense, kl = ta.dense_mask_build(tm, x["sl"], 4, 128)
    kl_far = torch.tensor([64 * wl.max_pages_per_seq + 1], dtype=torch.int32, device="cuda")
    ta.verify_dense(x["q"], x["k"], x["v"], x["bt"], kl_far, dense, status=status,
                    softmax_scale=wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == ta.STATUS_BAD_SEQ_LEN
