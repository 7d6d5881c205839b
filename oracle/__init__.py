"""fp64 CPU oracle for split tree attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import this package.  The product path (the C-ABI library and
its Python binding) never touches it, and it shares no code with them: the
arithmetic lives in ``tree_attn_oracle.c`` (plain C, double precision, OpenMP
over query rows), compiled here with gcc.

Pins (what ties the oracle to something other than itself) live in
``tests/test_oracle_pins.py``:

* mask: brute-force root-to-node path enumeration over every valid parent
  array with T <= 7, plus networkx ancestor sets on random trees up to T = 64;
* attention: q = 0 closed form (lse = ln n, out = mean of attended values),
  constant-value invariance, chain tree == causal attention (torch SDPA and a
  NumPy textbook softmax on gathered contiguous K/V), T = 1 == paged decode,
  forest == prefix + self, empty prefix == tree-only attention;
* merge: split + merge over random disjoint chunks == single pass (1e-12);
* mutation checks: planted mistakes in a copy of the C source fail a pin.

* one-pass attention under an explicit mask (``dense_rows``) and the
  explicit mask itself (``dense_mask``): equal to the split definition on the
  same inputs (1e-12), a single visible key returns that key's value, and a
  random mask against a NumPy textbook softmax.

Parity unpinned: none of the value-producing functions is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "tree_attn_oracle.c")
_DEFAULT_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()


def compile_oracle(source: str = SOURCE, out_path: str = _DEFAULT_SO,
                   extra_flags: Sequence[str] = ()) -> str:
    """Compile the C oracle into a shared object (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", *extra_flags,
           source, "-o", out_path + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out_path + ".tmp", out_path)
    return out_path


def _fresh(so: str, src: str) -> bool:
    return os.path.exists(so) and os.path.getmtime(so) >= os.path.getmtime(src)


_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def _ptr(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        lib.oracle_tree_mask.argtypes = [_i32p, ctypes.c_int, _u64p]
        lib.oracle_tree_mask.restype = ctypes.c_int
        common = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p, _u16p, _u16p, _u64p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_double, _i32p, ctypes.c_long]
        lib.oracle_verify_rows.argtypes = common + [_f64p, _f64p, ctypes.c_int]
        lib.oracle_verify_rows.restype = ctypes.c_int
        lib.oracle_chunk_rows.argtypes = common + [ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                                   _f64p, _f64p]
        lib.oracle_chunk_rows.restype = ctypes.c_int
        lib.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_int, _f64p, _f64p,
                                     _f64p, _f64p]
        lib.oracle_merge.restype = None
        lib.oracle_dense_rows.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p,
                                          _u8p, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double, _i32p, ctypes.c_long,
                                          _f64p, _f64p]
        lib.oracle_dense_rows.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = so_path

    # ---- tree mask -------------------------------------------------------
    def tree_mask(self, parents) -> np.ndarray:
        """uint64 ancestor-or-self mask per node; raises on a bad parent array."""
        p = np.ascontiguousarray(np.asarray(parents, dtype=np.int32))
        T = int(p.shape[0])
        m = np.zeros(max(T, 1), dtype=np.uint64)
        rc = self.lib.oracle_tree_mask(_ptr(p, _i32p), T, _ptr(m, _u64p))
        if rc != 0:
            raise ValueError(f"oracle_tree_mask rejected the parent array (code {rc})")
        return m[:T]

    # ---- attention -------------------------------------------------------
    @staticmethod
    def _arrays(wl, mask):
        from workloads import bf16_bits
        c = wl.cfg
        arrs = dict(
            q=bf16_bits(wl.q), k=bf16_bits(wl.k_pages), v=bf16_bits(wl.v_pages),
            bt=np.ascontiguousarray(wl.block_table.numpy().astype(np.int32)),
            sl=np.ascontiguousarray(wl.seq_lens.numpy().astype(np.int32)),
            tk=bf16_bits(wl.tree_k), tv=bf16_bits(wl.tree_v),
            mask=np.ascontiguousarray(np.asarray(mask, dtype=np.uint64)),
        )
        dims = (c.B, c.Hq, c.Hkv, c.d, c.T, c.page, wl.num_pages)
        return arrs, dims

    def _common_args(self, wl, mask, rows):
        a, (B, Hq, Hkv, d, T, P, NP) = self._arrays(wl, mask)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        args = [_ptr(a["q"], _u16p), _ptr(a["k"], _u16p), _ptr(a["v"], _u16p),
                _ptr(a["bt"], _i32p), wl.max_pages_per_seq, _ptr(a["sl"], _i32p),
                _ptr(a["tk"], _u16p), _ptr(a["tv"], _u16p), _ptr(a["mask"], _u64p),
                B, Hq, Hkv, d, T, P, NP, float(wl.scale), _ptr(rows, _i32p), rows.shape[0]]
        return args, a, rows, d

    def verify_rows(self, wl, mask, rows, threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """(out [n][d], lse [n]) in float64 for rows (b, i, h)."""
        args, keep, rows, d = self._common_args(wl, mask, rows)
        n = rows.shape[0]
        out = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = self.lib.oracle_verify_rows(*args, _ptr(out, _f64p), _ptr(lse, _f64p), int(threads))
        if rc != 0:
            raise ValueError(f"oracle_verify_rows failed (code {rc})")
        return out, lse

    def verify(self, wl, mask, threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """Every row: out [B][T][Hq][d], lse [B][T][Hq] in float64."""
        c = wl.cfg
        rows = all_rows(c.B, c.T, c.Hq)
        out, lse = self.verify_rows(wl, mask, rows, threads)
        return out.reshape(c.B, c.T, c.Hq, c.d), lse.reshape(c.B, c.T, c.Hq)

    def chunk_rows(self, wl, mask, rows, p_begin: int, p_end: int, use_tree: bool):
        args, keep, rows, d = self._common_args(wl, mask, rows)
        n = rows.shape[0]
        out = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = self.lib.oracle_chunk_rows(*args, int(p_begin), int(p_end), int(bool(use_tree)),
                                        _ptr(out, _f64p), _ptr(lse, _f64p))
        if rc != 0:
            raise ValueError(f"oracle_chunk_rows failed (code {rc})")
        return out, lse

    def merge(self, outs: np.ndarray, lses: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """merge_attentions: outs [C][n][d], lses [C][n] -> (out [n][d], lse [n])."""
        outs = np.ascontiguousarray(outs, dtype=np.float64)
        lses = np.ascontiguousarray(lses, dtype=np.float64)
        C, n, d = outs.shape
        out = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        self.lib.oracle_merge(C, n, d, _ptr(outs, _f64p), _ptr(lses, _f64p),
                              _ptr(out, _f64p), _ptr(lse, _f64p))
        return out, lse

    # ---- one pass under an explicit mask (the naive form) -----------------
    def dense_rows(self, wl, key_lens, dense, rows) -> Tuple[np.ndarray, np.ndarray]:
        """(out [n][d], lse [n]) in float64: row (b, i, h) attends cache
        position p < key_lens[b] where dense[b][i][p] != 0."""
        from workloads import bf16_bits
        c = wl.cfg
        q, k, v = bf16_bits(wl.q), bf16_bits(wl.k_pages), bf16_bits(wl.v_pages)
        bt = np.ascontiguousarray(wl.block_table.numpy().astype(np.int32))
        kl = np.ascontiguousarray(np.asarray(key_lens, dtype=np.int32))
        dm = np.ascontiguousarray(np.asarray(dense, dtype=np.uint8))
        assert dm.shape[:2] == (c.B, c.T)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        n = rows.shape[0]
        out = np.zeros((n, c.d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = self.lib.oracle_dense_rows(
            _ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), _ptr(bt, _i32p),
            wl.max_pages_per_seq, _ptr(kl, _i32p), _ptr(dm, _u8p), dm.shape[2], c.B, c.Hq, c.Hkv,
            c.d, c.T, c.page, wl.num_pages, float(wl.scale), _ptr(rows, _i32p), n,
            _ptr(out, _f64p), _ptr(lse, _f64p))
        if rc != 0:
            raise ValueError(f"oracle_dense_rows failed (code {rc})")
        return out, lse

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


def all_rows(B: int, T: int, Hq: int) -> np.ndarray:
    """Every (b, i, h) triple in [B][T][Hq] order."""
    b, i, h = np.meshgrid(np.arange(B), np.arange(T), np.arange(Hq), indexing="ij")
    return np.stack([b.ravel(), i.ravel(), h.ravel()], axis=1).astype(np.int32)


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from ``tree_attn_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            if not _fresh(_DEFAULT_SO, SOURCE):
                compile_oracle()
            _default = Oracle(_DEFAULT_SO)
        return _default


def tree_mask(parents) -> np.ndarray:
    return get().tree_mask(parents)


def verify(wl, mask, threads: int = 0):
    return get().verify(wl, mask, threads)


def verify_rows(wl, mask, rows, threads: int = 0):
    return get().verify_rows(wl, mask, rows, threads)
