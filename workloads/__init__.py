"""Seeded synthetic inputs for split tree attention.

This module only draws random numbers and lays them out; it holds none of the
attention, mask or merge arithmetic. Both the fp64 oracle (``oracle/``) and the
CUDA path (``speculative_decoding_tree_split_gb300``) take their inputs from
here, so that the two sides see the same bits.

Workload shapes follow the Llama-shaped verification layers that the review
pages of "Efficient Speculative Decoding for Llama at Scale: Challenges and
Solutions" (arXiv 2508.08192) describe: an EAGLE draft tree of ``T`` tokens
verified against a paged KV cache (the pith.science review's Referee Report
summary counts paged, persistent KV handling among what tree attention needs).
The pages print no
tensor shapes; the five shapes below are the stated synthetic stand-ins.

Recipe (all draws come from one ``torch.Generator('cpu')`` seeded per config):

1. ``seq_lens``: ``torch.randint(lo, hi + 1)`` per sequence (inclusive range;
   not page aligned).
2. Tree: node 0 is the root (parent -1).  Node ``i`` picks its parent uniformly
   among earlier nodes whose depth is below ``max_depth`` and whose child count
   is below ``max_branch`` (depth counts nodes on the root path, root = 1).
   ``chain`` trees use ``parent[i] = i - 1``.
3. Physical pages: a random permutation of ``[0, num_pages)`` with
   ``num_pages = sum_b ceil(L_b / P)``, handed out to the sequences' logical
   pages in order, so the block-table walk is non contiguous.  Unused block
   table slots hold -1.
4. ``q``, ``k_pages``, ``v_pages``, ``tree_k``, ``tree_v``: i.i.d. N(0, 1) in
   fp32, rounded to bf16 (round to nearest even, torch's conversion).

Two layout variants (both off by default, so the default draws are unchanged):

* ``per_sequence_trees``: step 2 runs once per sequence, giving ``parents``
  of shape [B][T] (one draft tree per sequence).
* ``tree_in_cache``: the tree tokens live in the paged cache, padded after
  the prefix: each sequence's pages cover ``L_b + T`` positions and token
  ``j``'s K/V (the same ``tree_k`` / ``tree_v`` draws) is written at logical
  position ``L_b + j``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

__all__ = [
    "Config",
    "CONFIGS",
    "Workload",
    "random_tree",
    "chain_tree",
    "make_workload",
    "bf16_bits",
]


@dataclasses.dataclass(frozen=True)
class Config:
    """One verification-layer shape.

    ``L`` is a fixed prefix length, or ``(lo, hi)`` for per-sequence lengths
    drawn uniformly (inclusive).  ``tree`` is ``"chain"`` or ``"random"``.
    """

    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    L: object
    page: int
    T: int
    tree: str = "random"
    max_depth: int = 4
    max_branch: int = 3
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def M(self) -> int:
        return self.T * self.G

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} d={self.d} "
                f"L={self.L} page={self.page} T={self.T} tree={self.tree}")


# The five shapes: a tiny parity case, three Llama-3.x verification layers and
# one Llama-4-Maverick-shaped layer (GQA group of 5).  The 70B case's
# branching is not fixed by its description; 3 is taken.
CONFIGS: Dict[str, Config] = {
    "tiny": Config("tiny", B=2, Hq=4, Hkv=1, d=64, L=128, page=16, T=4,
                   tree="random", max_depth=4, max_branch=3, seed=0),
    "llama8b": Config("llama8b", B=1, Hq=32, Hkv=8, d=128, L=8192, page=64, T=12,
                      tree="random", max_depth=4, max_branch=3, seed=1),
    "llama70b": Config("llama70b", B=16, Hq=64, Hkv=8, d=128, L=(1024, 8192), page=64,
                       T=8, tree="random", max_depth=3, max_branch=3, seed=2),
    "chain": Config("chain", B=64, Hq=32, Hkv=8, d=128, L=(512, 16384), page=64, T=4,
                    tree="chain", seed=3),
    "maverick": Config("maverick", B=4, Hq=40, Hkv=8, d=128, L=32768, page=64, T=16,
                       tree="random", max_depth=4, max_branch=4, seed=4),
}


def chain_tree(T: int) -> torch.Tensor:
    """Parent array of a chain: ``parent[i] = i - 1``."""
    return torch.arange(-1, T - 1, dtype=torch.int32)


def random_tree(T: int, max_depth: int, max_branch: int,
                gen: torch.Generator) -> torch.Tensor:
    """Seeded random draft tree as a topological parent array (step 2 above)."""
    if T < 1:
        raise ValueError("T must be >= 1")
    parents = [-1]
    depth = [1]
    children = [0]
    for i in range(1, T):
        eligible = [j for j in range(i) if depth[j] < max_depth and children[j] < max_branch]
        if not eligible:
            raise ValueError(f"no eligible parent for node {i}: tree limits too tight for T={T}")
        pick = int(torch.randint(len(eligible), (1,), generator=gen).item())
        p = eligible[pick]
        parents.append(p)
        depth.append(depth[p] + 1)
        children.append(0)
        children[p] += 1
    return torch.tensor(parents, dtype=torch.int32)


def bf16_bits(t: torch.Tensor):
    """The raw bf16 bit patterns of a bf16 tensor as a numpy uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


@dataclasses.dataclass
class Workload:
    """All inputs of one ``tree_attn_verify`` call, as CPU tensors."""

    cfg: Config
    parents: torch.Tensor        # int32 [T], or [B][T] with per-sequence trees
    seq_lens: torch.Tensor       # int32 [B]
    block_table: torch.Tensor    # int32 [B][max_pages_per_seq]
    q: torch.Tensor              # bf16 [B][T][Hq][d]
    k_pages: torch.Tensor        # bf16 [num_pages][Hkv][P][d]
    v_pages: torch.Tensor        # bf16 [num_pages][Hkv][P][d]
    tree_k: torch.Tensor         # bf16 [B][T][Hkv][d]
    tree_v: torch.Tensor         # bf16 [B][T][Hkv][d]
    scale: float
    tree_in_cache: bool = False  # tree K/V also written at positions L_b + j

    def sequence(self, b: int) -> "Workload":
        """Sequence ``b`` alone, as a B = 1 workload with its own tree (the
        pages are shared; the block table row is kept)."""
        c = dataclasses.replace(self.cfg, B=1)
        par = self.parents[b] if self.parents.dim() == 2 else self.parents
        return Workload(cfg=c, parents=par.clone(), seq_lens=self.seq_lens[b:b + 1].clone(),
                        block_table=self.block_table[b:b + 1].clone(), q=self.q[b:b + 1],
                        k_pages=self.k_pages, v_pages=self.v_pages,
                        tree_k=self.tree_k[b:b + 1], tree_v=self.tree_v[b:b + 1],
                        scale=self.scale, tree_in_cache=self.tree_in_cache)

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def kv_bytes(self) -> int:
        """Prefix K+V bytes one call must read (the committed tokens only)."""
        c = self.cfg
        return int(self.seq_lens.to(torch.int64).sum().item()) * c.Hkv * c.d * 2 * 2


def _randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    # Drawn in fp32 chunks to bound peak host memory, then rounded to bf16.
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16)
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def make_workload(cfg: Config, seed: Optional[int] = None, *,
                  seq_lens: Optional[List[int]] = None,
                  parents: Optional[torch.Tensor] = None,
                  max_pages_per_seq: Optional[int] = None,
                  extra_pages: int = 0,
                  q_zero: bool = False,
                  per_sequence_trees: bool = False,
                  tree_in_cache: bool = False,
                  tree_room: bool = False) -> Workload:
    """Build the seeded inputs of ``cfg`` (recipe in the module docstring).

    ``seq_lens`` / ``parents`` override the drawn values (edge-case tests);
    ``max_pages_per_seq`` widens the block table; ``extra_pages`` adds unused
    physical pages; ``q_zero`` zeroes the queries (closed-form tests);
    ``per_sequence_trees`` / ``tree_in_cache`` select the layout variants;
    ``tree_room`` maps pages for ``L_b + T`` positions without writing the
    tree there (room for committing an accepted path).
    """
    gen = torch.Generator("cpu")
    gen.manual_seed(cfg.seed if seed is None else seed)
    B, P = cfg.B, cfg.page

    if seq_lens is None:
        if isinstance(cfg.L, tuple):
            lo, hi = cfg.L
            sl = torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64)
        else:
            sl = torch.full((B,), int(cfg.L), dtype=torch.int64)
    else:
        assert len(seq_lens) == B
        sl = torch.tensor(seq_lens, dtype=torch.int64)
    seq_lens_t = sl.to(torch.int32)

    def draw_tree() -> torch.Tensor:
        if cfg.tree == "chain":
            return chain_tree(cfg.T)
        return random_tree(cfg.T, cfg.max_depth, cfg.max_branch, gen)

    if parents is not None:
        parents_t = parents.to(torch.int32).clone()
    elif per_sequence_trees:
        parents_t = torch.stack([draw_tree() for _ in range(B)])
    else:
        parents_t = draw_tree()

    span = cfg.T if (tree_in_cache or tree_room) else 0
    pages_per = [(int(x) + span + P - 1) // P for x in sl.tolist()]
    used_pages = sum(pages_per)
    num_pages = used_pages + extra_pages
    width = max(pages_per + [1])
    if max_pages_per_seq is not None:
        assert max_pages_per_seq >= width
        width = max_pages_per_seq
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32) if num_pages else \
        torch.empty(0, dtype=torch.int32)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        n = pages_per[b]
        bt[b, :n] = perm[pos:pos + n]
        pos += n

    Hq, Hkv, d, T = cfg.Hq, cfg.Hkv, cfg.d, cfg.T
    q = _randn_bf16((B, T, Hq, d), gen)
    if q_zero:
        q.zero_()
    k_pages = _randn_bf16((num_pages, Hkv, P, d), gen)
    v_pages = _randn_bf16((num_pages, Hkv, P, d), gen)
    tree_k = _randn_bf16((B, T, Hkv, d), gen)
    tree_v = _randn_bf16((B, T, Hkv, d), gen)
    if tree_in_cache:
        for b in range(B):
            for j in range(T):
                pos = int(sl[b]) + j
                page = int(bt[b, pos // P])
                k_pages[page, :, pos % P] = tree_k[b, j]
                v_pages[page, :, pos % P] = tree_v[b, j]
    return Workload(cfg=cfg, parents=parents_t, seq_lens=seq_lens_t, block_table=bt,
                    q=q, k_pages=k_pages, v_pages=v_pages, tree_k=tree_k, tree_v=tree_v,
                    scale=1.0 / math.sqrt(d), tree_in_cache=tree_in_cache)
