"""The kernel selector (tree_attn_plan): the launch choices for each workload
shape, computed on the host only (CPU)."""
import pytest

import speculative_decoding_tree_split_gb300 as ta
from workloads import CONFIGS

SMS = 152   # GB300


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ta.build()
    ta.load()


def max_pages(cfg):
    hi = cfg.L[1] if isinstance(cfg.L, tuple) else cfg.L
    return (hi + cfg.page - 1) // cfg.page


# (units, row blocks, replicas, CTAs, merge warps per row), worked out by hand:
#   units = B * Hkv * ceil(T*G/128); replicas 4 for M <= 32, 2 for M <= 64;
#   CTAs = min(152, units * (ceil(max_pages*P/64) + 1)): the tree tokens are one
#   more 64-key chunk of each unit's work;
#   merge warps from CTAs // units + 1 + replicas (prefix CTAs fold their row
#   copies in their last segment): > 12 -> 4, > 6 -> 2, else 1.
EXPECTED = {
    "tiny": (2, 1, 4, 6, 2),          # M = 16; 2 units x 3 steps = 6 CTAs; 3 + 1 + 4 = 8
    "llama8b": (8, 1, 2, 152, 4),     # M = 48; 19 + 1 + 2 = 22
}

def test_plan_tree_placement_by_hand():
    # llama8b: 8 units x 128 steps = 1024 <= 32 x 152 -> tree on the prefix pass;
    # llama70b: 128 units x 128 = 16384 > 4864 steps, but 128 units <= 152 CTAs
    # with 2 row copies -> tree on the prefix pass;
    # chain: 512 units > 152 CTAs; maverick: one row copy (M = 80) -> the merge
    # attends the tree
    for name in ("llama8b", "llama70b"):
        c = CONFIGS[name]
        p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
        assert p["tree_in_prefix"] == 1, name
    for name in ("chain", "maverick"):
        c = CONFIGS[name]
        p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
        assert p["tree_in_prefix"] == 0, name


def test_plan_llama8b_and_tiny_by_hand():
    for name in ("tiny", "llama8b"):
        c = CONFIGS[name]
        p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
        got = (p["units"], p["row_blocks"], p["replicas"], p["n_ctas"], p["merge_warps_per_row"])
        assert got == EXPECTED[name], (name, got)


def test_plan_other_workloads_by_hand():
    # llama70b: M = 8 * 8 = 64 -> 2 replicas; units 16*8 = 128; 152 // 128 = 1 -> 1+1+2 = 4;
    # tree on the prefix pass, merge alone: 128 units x 64/4 CTAs = 2048 > 152 x 6 = 912 CTAs
    # at once -> ceil(2048 / 912) = 3 rows per merge warp
    c = CONFIGS["llama70b"]
    p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
    assert (p["units"], p["replicas"], p["n_ctas"], p["merge_warps_per_row"]) == (128, 2, 152, 1)
    assert p["merge_rows_per_warp"] == 3
    for name in ("tiny", "llama8b", "chain", "maverick"):
        c = CONFIGS[name]
        p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
        assert p["merge_rows_per_warp"] == 1, name
    # chain: M = 4 * 4 = 16 -> 4 replicas; units 512; 0 + 1 + 4 = 5 -> 1 warp
    c = CONFIGS["chain"]
    p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
    assert (p["units"], p["replicas"], p["n_ctas"], p["merge_warps_per_row"]) == (512, 4, 152, 1)
    # maverick: M = 16 * 5 = 80 -> 1 copy; units 32; 4 + 1 + 1 = 6 -> 1 warp
    c = CONFIGS["maverick"]
    p = ta.plan(c.B, c.Hq, c.Hkv, c.d, c.T, c.page, max_pages(c), SMS)
    assert (p["units"], p["replicas"], p["n_ctas"], p["merge_warps_per_row"]) == (32, 1, 152, 1)


@pytest.mark.parametrize("B,Hq,Hkv,d,T,P,maxp", [
    (1, 8, 8, 64, 1, 16, 1), (3, 16, 4, 128, 10, 64, 11), (1, 8, 2, 128, 64, 64, 5),
    (64, 64, 8, 128, 64, 128, 200), (2, 40, 8, 128, 16, 32, 4), (1, 128, 1, 128, 64, 16, 1)])
def test_plan_invariants(B, Hq, Hkv, d, T, P, maxp):
    p = ta.plan(B, Hq, Hkv, d, T, P, maxp, SMS)
    G = Hq // Hkv
    M = T * G
    assert p["row_blocks"] == (M + 127) // 128
    assert p["units"] == B * Hkv * p["row_blocks"]
    prefix_steps = p["units"] * ((maxp * P + 63) // 64)
    # small calls (<= 32 steps per CTA), and calls with no more units than
    # CTAs and at least two row copies, attend the tree in the prefix pass:
    # one extra 64-key chunk per unit
    C = min(SMS, prefix_steps + p["units"])
    want_tree = prefix_steps <= 32 * C or (p["units"] <= C and p["replicas"] >= 2)
    assert p["tree_in_prefix"] == int(want_tree)
    assert p["max_steps"] == prefix_steps + (p["units"] if want_tree else 0)
    # the merge alone (tree on the prefix pass) gives each warp several rows
    # when one row per warp would need more CTAs than 6 per SM
    rows = min(M, 128)
    per_cta = 4 // p["merge_warps_per_row"]
    ctas = p["units"] * -(-rows // per_cta)
    want_rpw = max(1, -(-ctas // (SMS * 6))) if want_tree else 1
    assert p["merge_rows_per_warp"] == want_rpw
    assert 1 <= p["n_ctas"] <= min(SMS, max(1, p["max_steps"]))
    if p["row_blocks"] == 1:
        assert p["replicas"] * M <= 128 or p["replicas"] == 1
        assert p["replicas"] in (1, 2, 4)
    else:
        assert p["replicas"] == 1
    assert p["merge_warps_per_row"] in (1, 2, 4)
    lib = ta.load()
    assert p["workspace_bytes"] == lib.tree_attn_workspace_size_ctas(B, Hq, Hkv, d, T, P,
                                                                      p["n_ctas"])
    # the selector never needs more scratch than the size callers allocate by
    assert p["workspace_bytes"] <= lib.tree_attn_workspace_size_ctas(B, Hq, Hkv, d, T, P, SMS)


def test_plan_rejects_bad_shapes():
    with pytest.raises(ta.TreeAttnError):
        ta.plan(1, 6, 4, 128, 4, 64, 4, SMS)
    with pytest.raises(ta.TreeAttnError):
        ta.plan(1, 8, 2, 128, 4, 64, 0, SMS)
