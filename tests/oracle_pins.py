"""Pins that tie the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and raises
``AssertionError`` when the oracle disagrees with the fact it checks.  The
same functions run against the real oracle (tests/test_oracle_pins.py) and
against copies of the C source with a planted mistake
(tests/test_oracle_mutants.py), where at least one pin must fail.

Facts used (none of them is the oracle's own formula retyped):

* Tree mask: node i attends to itself and its ancestors ("tree mask",
  pith.science review of 2508.08192, "What carries the argument").  Checked
  by enumerating root-to-node paths with a depth-first walk over child lists,
  for every valid parent array up to T = 7.
* Attention: a dense explicit-mask attention (the one-mask-over-every-key
  form the same section contrasts split attention with) evaluated by
  ``torch.nn.functional.scaled_dot_product_attention`` in float64 over K/V
  gathered into contiguous arrays; its LSE by ``torch.logsumexp``.
* Closed forms: q = 0 gives lse = ln(number of attended keys) and out = the
  mean of the attended values; constant values give out = that constant.
* Merge: attention over disjoint key chunks merged by log-sum-exp equals the
  single pass (merge_attentions, verdict record supporting_citations).
* Paging: renumbering the physical pages and rewriting the block table leaves
  the result bit-identical.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

from workloads import Config, make_workload

# Small shapes that still exercise GQA (G = 3), several pages, a ragged last
# page and an empty prefix.
PIN_CFG = Config("pin", B=3, Hq=6, Hkv=2, d=16, L=(0, 40), page=8, T=7, tree="random",
                 max_depth=4, max_branch=3, seed=11)
PIN_SEQ_LENS = [0, 13, 40]


def pin_workload(seed=11, **kw):
    kw.setdefault("seq_lens", PIN_SEQ_LENS)
    return make_workload(PIN_CFG, seed=seed, **kw)


# ---------------------------------------------------------------------------
# tree mask
# ---------------------------------------------------------------------------
def paths_mask(parents):
    """Ancestor-or-self bits by a depth-first walk from each root down."""
    T = len(parents)
    children = [[] for _ in range(T)]
    roots = []
    for i, p in enumerate(parents):
        (roots if p == -1 else children[p]).append(i)
    expect = [0] * T
    stack = [(r, 1 << r) for r in roots]
    while stack:
        node, bits = stack.pop()
        expect[node] = bits
        for ch in children[node]:
            stack.append((ch, bits | (1 << ch)))
    return expect


def all_parent_arrays(T):
    """Every topological parent array of length T (node i picks -1 or j < i)."""
    return itertools.product(*[range(-1, i) for i in range(T)])


def pin_mask_bruteforce(orc, max_T=7):
    for T in range(1, max_T + 1):
        for parents in all_parent_arrays(T):
            got = [int(x) for x in orc.tree_mask(list(parents))]
            want = paths_mask(list(parents))
            assert got == want, (parents, got, want)


# ---------------------------------------------------------------------------
# attention through a dense explicit mask (torch SDPA, float64)
# ---------------------------------------------------------------------------
def _bf16_to_f64(t):
    return t.to(torch.float64)


def dense_reference(wl, mask):
    """(out [B][T][Hq][d], lse [B][T][Hq]) from SDPA over gathered K/V."""
    c = wl.cfg
    G = c.Hq // c.Hkv
    out = torch.zeros(c.B, c.T, c.Hq, c.d, dtype=torch.float64)
    lse = torch.zeros(c.B, c.T, c.Hq, dtype=torch.float64)
    kp = _bf16_to_f64(wl.k_pages)   # [NP][Hkv][P][d]
    vp = _bf16_to_f64(wl.v_pages)
    allowed_tree = torch.tensor([[(int(mask[i]) >> j) & 1 for j in range(c.T)]
                                 for i in range(c.T)], dtype=torch.bool)
    for b in range(c.B):
        L = int(wl.seq_lens[b])
        pos = torch.arange(L)
        pages = wl.block_table[b, (pos // c.page)].long()
        slots = pos % c.page
        k_pre = kp[pages, :, slots, :]                        # [L][Hkv][d]
        v_pre = vp[pages, :, slots, :]
        k_all = torch.cat([k_pre, _bf16_to_f64(wl.tree_k[b])], 0)   # [L+T][Hkv][d]
        v_all = torch.cat([v_pre, _bf16_to_f64(wl.tree_v[b])], 0)
        k_h = k_all.permute(1, 0, 2).repeat_interleave(G, dim=0)    # [Hq][L+T][d]
        v_h = v_all.permute(1, 0, 2).repeat_interleave(G, dim=0)
        q_h = _bf16_to_f64(wl.q[b]).permute(1, 0, 2)                # [Hq][T][d]
        allowed = torch.cat([torch.ones(c.T, L, dtype=torch.bool), allowed_tree], 1)
        o = torch.nn.functional.scaled_dot_product_attention(
            q_h, k_h, v_h, attn_mask=allowed, scale=wl.scale)
        s = torch.matmul(q_h, k_h.transpose(1, 2)) * wl.scale
        s = s.masked_fill(~allowed, -math.inf)
        out[b] = o.permute(1, 0, 2)
        lse[b] = torch.logsumexp(s, dim=-1).permute(1, 0)
    return out.numpy(), lse.numpy()


def pin_dense_random_tree(orc, seed=11):
    wl = pin_workload(seed)
    mask = paths_mask(wl.parents.tolist())
    got_o, got_l = orc.verify(wl, mask)
    ref_o, ref_l = dense_reference(wl, mask)
    np.testing.assert_allclose(got_o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_l, ref_l, rtol=0, atol=1e-12)


def pin_dense_special_trees(orc):
    """Chain (causal), forest (prefix + self) and T = 1 (paged decode)."""
    T = PIN_CFG.T
    for parents in (list(range(-1, T - 1)), [-1] * T):
        wl = pin_workload(12, parents=torch.tensor(parents, dtype=torch.int32))
        mask = paths_mask(parents)
        got_o, got_l = orc.verify(wl, mask)
        ref_o, ref_l = dense_reference(wl, mask)
        np.testing.assert_allclose(got_o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(got_l, ref_l, rtol=0, atol=1e-12)
    cfg1 = Config("pin1", B=2, Hq=4, Hkv=2, d=16, L=(0, 40), page=8, T=1, tree="chain", seed=13)
    wl = make_workload(cfg1, seq_lens=[17, 32])
    got_o, got_l = orc.verify(wl, [1])
    ref_o, ref_l = dense_reference(wl, [1])
    np.testing.assert_allclose(got_o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_l, ref_l, rtol=0, atol=1e-12)


def chain_causal_reference(wl):
    """Chain tree: token i sits at position L_b + i of one causal sequence.

    Textbook causal attention in NumPy over the contiguous sequence
    [prefix ; tree], written independently of the tree mask.
    """
    c = wl.cfg
    G = c.Hq // c.Hkv
    out = np.zeros((c.B, c.T, c.Hq, c.d))
    lse = np.zeros((c.B, c.T, c.Hq))
    kp = wl.k_pages.to(torch.float64).numpy()
    vp = wl.v_pages.to(torch.float64).numpy()
    for b in range(c.B):
        L = int(wl.seq_lens[b])
        seq_k, seq_v = [], []
        for p in range(L):
            page = int(wl.block_table[b, p // c.page])
            seq_k.append(kp[page, :, p % c.page, :])
            seq_v.append(vp[page, :, p % c.page, :])
        for j in range(c.T):
            seq_k.append(wl.tree_k[b, j].to(torch.float64).numpy())
            seq_v.append(wl.tree_v[b, j].to(torch.float64).numpy())
        K = np.stack(seq_k)   # [L+T][Hkv][d]
        V = np.stack(seq_v)
        for i in range(c.T):
            last = L + i      # causal: keys 0..last
            for h in range(c.Hq):
                qv = wl.q[b, i, h].to(torch.float64).numpy()
                s = K[: last + 1, h // G, :] @ qv * wl.scale
                top = s.max()
                e = np.exp(s - top)
                out[b, i, h] = (e[:, None] * V[: last + 1, h // G, :]).sum(0) / e.sum()
                lse[b, i, h] = top + math.log(e.sum())
    return out, lse


def pin_chain_is_causal(orc):
    T = PIN_CFG.T
    parents = list(range(-1, T - 1))
    wl = pin_workload(14, parents=torch.tensor(parents, dtype=torch.int32))
    got_o, got_l = orc.verify(wl, orc.tree_mask(parents))
    ref_o, ref_l = chain_causal_reference(wl)
    np.testing.assert_allclose(got_o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_l, ref_l, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def _attended_values(wl, mask, b, i, hk):
    c = wl.cfg
    rows = []
    for p in range(int(wl.seq_lens[b])):
        page = int(wl.block_table[b, p // c.page])
        rows.append(wl.v_pages[page, hk, p % c.page].to(torch.float64).numpy())
    for j in range(c.T):
        if (int(mask[i]) >> j) & 1:
            rows.append(wl.tree_v[b, j, hk].to(torch.float64).numpy())
    return np.stack(rows)


def pin_zero_query_closed_form(orc):
    wl = pin_workload(15, q_zero=True)
    c = wl.cfg
    G = c.Hq // c.Hkv
    mask = paths_mask(wl.parents.tolist())
    got_o, got_l = orc.verify(wl, mask)
    for b in range(c.B):
        for i in range(c.T):
            n = int(wl.seq_lens[b]) + bin(int(mask[i])).count("1")
            for h in range(c.Hq):
                assert abs(got_l[b, i, h] - math.log(n)) <= 1e-12, (b, i, h)
                want = _attended_values(wl, mask, b, i, h // G).mean(0)
                np.testing.assert_allclose(got_o[b, i, h], want, rtol=0, atol=1e-12)


def pin_constant_values(orc):
    wl = pin_workload(16)
    const = torch.linspace(-2, 2, wl.cfg.d).to(torch.bfloat16)
    wl.v_pages[:] = const
    wl.tree_v[:] = const
    mask = paths_mask(wl.parents.tolist())
    got_o, _ = orc.verify(wl, mask)
    want = const.to(torch.float64).numpy()
    assert np.abs(got_o - want).max() <= 1e-12


# ---------------------------------------------------------------------------
# merge over disjoint chunks
# ---------------------------------------------------------------------------
def pin_split_merge(orc, seed=17):
    wl = pin_workload(seed)
    c = wl.cfg
    mask = orc.tree_mask(wl.parents.tolist())
    rng = np.random.default_rng(seed)
    for b in range(c.B):
        L = int(wl.seq_lens[b])
        rows = np.array([(b, i, h) for i in range(c.T) for h in range(c.Hq)], dtype=np.int32)
        full_o, full_l = orc.verify_rows(wl, mask, rows)
        cuts = sorted(set([0, L] + list(rng.integers(0, L + 1, size=3))))
        outs, lses = [], []
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            o, l = orc.chunk_rows(wl, mask, rows, lo, hi, use_tree=False)
            outs.append(o)
            lses.append(l)
        o, l = orc.chunk_rows(wl, mask, rows, 0, 0, use_tree=True)
        outs.append(o)
        lses.append(l)
        m_o, m_l = orc.merge(np.stack(outs), np.stack(lses))
        np.testing.assert_allclose(m_o, full_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(m_l, full_l, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# paging
# ---------------------------------------------------------------------------
def pin_page_renumbering(orc, seed=18):
    wl = pin_workload(seed, extra_pages=3)
    mask = paths_mask(wl.parents.tolist())
    o1, l1 = orc.verify(wl, mask)
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(wl.num_pages, generator=g)      # new id of old page
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(wl.num_pages)
    wl.k_pages = wl.k_pages[inv].contiguous()
    wl.v_pages = wl.v_pages[inv].contiguous()
    bt = wl.block_table.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    wl.block_table = bt
    o2, l2 = orc.verify(wl, mask)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------------------
# one pass under an explicit mask (the naive form split attention replaces)
# ---------------------------------------------------------------------------
def _paged_tree_workload(seed):
    return pin_workload(seed, tree_in_cache=True)


def pin_onepass_equals_split(orc, dense_mod=None):
    """With the tree in the cache, one pass under the explicit mask equals
    split tree attention (the identity the pages' two-pass design rests on)."""
    if dense_mod is None:
        import oracle.dense as dense_mod
    for seed, per_seq in ((19, False), (20, True)):
        wl = pin_workload(seed, tree_in_cache=True, per_sequence_trees=per_seq)
        c = wl.cfg
        cols = 64 * ((max(wl.seq_lens.tolist()) + c.T + 63) // 64)
        if per_seq:
            masks = np.stack([paths_mask(wl.parents[b].tolist()) for b in range(c.B)])
        else:
            masks = paths_mask(wl.parents.tolist())
        dense, key_lens = dense_mod.dense_mask(masks, wl.seq_lens.numpy(), c.T, cols)
        assert np.array_equal(key_lens, wl.seq_lens.numpy() + c.T)
        from oracle import all_rows
        rows = all_rows(c.B, c.T, c.Hq)
        got_o, got_l = orc.dense_rows(wl, key_lens, dense, rows)
        for b in range(c.B):
            sb = wl.sequence(b)
            mb = masks[b] if per_seq else masks
            ref_o, ref_l = dense_reference(sb, mb)
            sel = rows[:, 0] == b
            np.testing.assert_allclose(got_o[sel], ref_o.reshape(-1, c.d), rtol=0, atol=1e-12)
            np.testing.assert_allclose(got_l[sel], ref_l.reshape(-1), rtol=0, atol=1e-12)


def pin_onepass_random_mask(orc, seed=21):
    """An arbitrary explicit mask (some rows fully hidden) against a NumPy
    textbook softmax over K/V gathered position by position."""
    wl = _paged_tree_workload(seed)
    c = wl.cfg
    rng = np.random.default_rng(seed)
    key_lens = wl.seq_lens.numpy() + c.T
    cols = int(key_lens.max()) + 5
    dense = (rng.random((c.B, c.T, cols)) < 0.5).astype(np.uint8)
    dense[1, 2, :] = 0                       # a row that sees nothing
    from oracle import all_rows
    rows = all_rows(c.B, c.T, c.Hq)
    got_o, got_l = orc.dense_rows(wl, key_lens, dense, rows)
    kp = wl.k_pages.to(torch.float64).numpy()
    vp = wl.v_pages.to(torch.float64).numpy()
    qf = wl.q.to(torch.float64).numpy()
    G = c.Hq // c.Hkv
    for r, (b, i, h) in enumerate(rows):
        ps = [p for p in range(int(key_lens[b])) if dense[b, i, p]]
        if not ps:
            assert got_l[r] == -math.inf and not got_o[r].any()
            continue
        pages = [int(wl.block_table[b, p // c.page]) for p in ps]
        K = np.stack([kp[pg, h // G, p % c.page] for pg, p in zip(pages, ps)])
        V = np.stack([vp[pg, h // G, p % c.page] for pg, p in zip(pages, ps)])
        sc = K @ qf[b, i, h] * wl.scale
        e = np.exp(sc - sc.max())
        np.testing.assert_allclose(got_o[r], (e / e.sum()) @ V, rtol=0, atol=1e-12)
        assert abs(got_l[r] - (sc.max() + math.log(e.sum()))) < 1e-12


def pin_onepass_single_key(orc, seed=22):
    """One visible key: out is that key's value exactly, lse its score."""
    wl = _paged_tree_workload(seed)
    c = wl.cfg
    key_lens = wl.seq_lens.numpy() + c.T
    cols = int(key_lens.max())
    dense = np.zeros((c.B, c.T, cols), dtype=np.uint8)
    pick = {}
    for b in range(c.B):
        for i in range(c.T):
            p = (7 * b + 3 * i) % int(key_lens[b])
            dense[b, i, p] = 1
            pick[(b, i)] = p
    from oracle import all_rows
    rows = all_rows(c.B, c.T, c.Hq)
    got_o, got_l = orc.dense_rows(wl, key_lens, dense, rows)
    G = c.Hq // c.Hkv
    for r, (b, i, h) in enumerate(rows):
        p = pick[(b, i)]
        pg = int(wl.block_table[b, p // c.page])
        v = wl.v_pages[pg, h // G, p % c.page].to(torch.float64).numpy()
        k = wl.k_pages[pg, h // G, p % c.page].to(torch.float64).numpy()
        assert np.array_equal(got_o[r], v)
        assert abs(got_l[r] - wl.scale * float(k @ wl.q[b, i, h].to(torch.float64).numpy())) \
            < 1e-12


ALL_PINS = [
    pin_mask_bruteforce,
    pin_dense_random_tree,
    pin_dense_special_trees,
    pin_chain_is_causal,
    pin_zero_query_closed_form,
    pin_constant_values,
    pin_split_merge,
    pin_page_renumbering,
    pin_onepass_equals_split,
    pin_onepass_random_mask,
    pin_onepass_single_key,
]
