"""The C ABI library: loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_tree_split_gb300 as ta

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    ta.build()
    return ta.load()


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            names += re.findall(r"TREE_ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tree_mask_build", "tree_attn_workspace_size", "tree_attn_verify"):
        assert n in names
    assert set(names) == set(ta.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert ta.version() == 10200


def test_only_declared_symbols_are_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ta.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions())


# Fake, never-dereferenced device addresses: the host checks below return
# before any CUDA call.
A16 = 0x10000


def _verify(lib, **kw):
    args = dict(q=A16, k=A16, v=A16, bt=A16, maxp=4, sl=A16, tk=A16, tv=A16, mask=A16, out=A16,
                lse=A16, B=2, Hq=8, Hkv=2, d=128, T=4, P=64, num_pages=8, scale=0.1, ws=A16,
                ws_bytes=1 << 30, status=None, stream=None)
    args.update(kw)
    return lib.tree_attn_verify_ctas(
        args["q"], args["k"], args["v"], args["bt"], args["maxp"], args["sl"], args["tk"],
        args["tv"], args["mask"], args["out"], args["lse"], args["B"], args["Hq"], args["Hkv"],
        args["d"], args["T"], args["P"], args["num_pages"], args["scale"], args["ws"],
        args["ws_bytes"], args["status"], args["stream"], 8)


@pytest.mark.parametrize("kw", [dict(T=0), dict(T=65), dict(Hq=6, Hkv=4), dict(d=96),
                                dict(P=48), dict(maxp=0), dict(num_pages=0),
                                dict(num_pages=1 << 24, Hkv=8, P=64), dict(scale=float("nan"))])
def test_verify_rejects_bad_shapes(lib, kw):
    assert _verify(lib, **kw) == -2


@pytest.mark.parametrize("name", ["q", "k", "v", "bt", "sl", "tk", "tv", "mask", "out", "lse"])
def test_verify_rejects_null(lib, name):
    assert _verify(lib, **{name: None}) == -1


@pytest.mark.parametrize("name,addr", [("q", A16 + 8), ("k", A16 + 2), ("out", A16 + 4),
                                       ("mask", A16 + 4), ("lse", A16 + 2), ("bt", A16 + 1),
                                       ("status", A16 + 2)])
def test_verify_rejects_misaligned(lib, name, addr):
    assert _verify(lib, **{name: addr}) == -3


def test_verify_rejects_small_workspace(lib):
    need = lib.tree_attn_workspace_size_ctas(2, 8, 2, 128, 4, 64, 8)
    assert need > 0
    assert _verify(lib, ws_bytes=need - 1) == -4
    assert _verify(lib, ws=None) == -4
    assert _verify(lib, ws=A16 + 16) == -4


def test_empty_batch_enqueues_nothing(lib):
    assert _verify(lib, B=0, q=None) == 0


def test_workspace_size_formula(lib):
    # slots = units + CTAs; slot = (2*128 + 128*d) floats; rounded to 256 B
    for (B, Hq, Hkv, d, T, C) in [(1, 32, 8, 128, 12, 152), (64, 32, 8, 128, 4, 152),
                                  (2, 4, 1, 64, 4, 7), (1, 8, 1, 128, 64, 10)]:
        G = Hq // Hkv
        RB = (T * G + 127) // 128
        slots = B * Hkv * RB + C
        want = slots * (2 * 128 + 128 * d) * 4
        want = (want + 255) // 256 * 256
        assert lib.tree_attn_workspace_size_ctas(B, Hq, Hkv, d, T, 64, C) == want
    assert lib.tree_attn_workspace_size_ctas(1, 8, 3, 128, 4, 64, 8) == 0


def test_mask_build_host_checks(lib):
    assert lib.tree_mask_build(None, 4, A16, None, None) == -1
    assert lib.tree_mask_build(A16, 0, A16, None, None) == -2
    assert lib.tree_mask_build(A16, 65, A16, None, None) == -2
    assert lib.tree_mask_build(A16, 4, A16 + 4, None, None) == -3


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        ta.mask_build(torch.tensor([-1, 0], dtype=torch.int32))


def _paged_tree(lib, mask_stride=0, **kw):
    args = dict(q=A16, k=A16, v=A16, bt=A16, maxp=4, sl=A16, mask=A16, out=A16, lse=A16, B=2,
                Hq=8, Hkv=2, d=128, T=4, P=64, num_pages=8, scale=0.1)
    args.update(kw)
    return lib.tree_attn_verify_paged_tree(
        args["q"], args["k"], args["v"], args["bt"], args["maxp"], args["sl"], args["mask"],
        mask_stride, args["out"], args["lse"], args["B"], args["Hq"], args["Hkv"], args["d"],
        args["T"], args["P"], args["num_pages"], args["scale"], A16, 1 << 30, None, None)


def test_paged_tree_host_checks(lib):
    # mask stride must be 0 (one tree) or T (one tree per sequence)
    for stride in (1, 3, 5, -4):
        assert _paged_tree(lib, mask_stride=stride) == -2
    assert _paged_tree(lib, mask_stride=4, d=96) == -2
    for name in ("q", "k", "v", "bt", "sl", "mask", "out", "lse"):
        assert _paged_tree(lib, **{name: None}) == -1
    assert _paged_tree(lib, k=A16 + 2) == -3
    assert _paged_tree(lib, B=0, q=None) == 0


def test_batched_entry_host_checks(lib):
    a = A16
    verify = lib.tree_attn_verify_batched
    base = [a, a, a, a, 4, a, a, a, a, a, a, 2, 8, 2, 128, 4, 64, 8, 0.1, a, 1 << 30, None, None]
    assert verify(*base[:8], None, *base[9:]) == -1       # masks
    bad_t = list(base)
    bad_t[15] = 65
    assert verify(*bad_t) == -2
    assert lib.tree_mask_build_batched(a, 4, -1, a, None, None) == -2
    assert lib.tree_mask_build_batched(None, 4, 2, a, None, None) == -1
    assert lib.tree_mask_build_batched(a, 4, 2, a + 4, None, None) == -3
    assert lib.tree_mask_build_batched(a, 4, 0, a, None, None) == 0


def test_greedy_accept_host_checks(lib):
    a = A16
    f = lib.tree_greedy_accept
    assert f(a, 0, a, a, 2, 0, a, a, a, None) == -2          # T = 0
    assert f(a, 0, a, a, 2, 65, a, a, a, None) == -2         # T > 64
    assert f(a, 3, a, a, 2, 4, a, a, a, None) == -2          # stride neither 0 nor T
    assert f(a, 0, a, a, -1, 4, a, a, a, None) == -2
    assert f(a, 0, a, a, 0, 4, None, None, None, None) == 0  # empty batch
    for k in range(6):
        args = [a, 0, a, a, 2, 4, a, a, a, None]
        args[[0, 2, 3, 6, 7, 8][k]] = None
        assert f(*args) == -1
    assert f(a + 4, 0, a, a, 2, 4, a, a, a, None) == -3
    assert f(a, 0, a + 2, a, 2, 4, a, a, a, None) == -3


def _commit(lib, **kw):
    args = dict(k=A16, v=A16, bt=A16, maxp=4, sl=A16, tk=A16, tv=A16, path=A16, n=A16,
                sl_out=A16 + 256, B=2, Hkv=2, d=128, T=4, P=64, num_pages=8, status=None)
    args.update(kw)
    return lib.tree_kv_commit(args["k"], args["v"], args["bt"], args["maxp"], args["sl"],
                              args["tk"], args["tv"], args["path"], args["n"], args["sl_out"],
                              args["B"], args["Hkv"], args["d"], args["T"], args["P"],
                              args["num_pages"], args["status"], None)


def test_kv_commit_host_checks(lib):
    for kw in (dict(d=96), dict(T=0), dict(T=65), dict(P=48), dict(maxp=0), dict(num_pages=0),
               dict(Hkv=0), dict(sl_out=A16)):          # seq_lens_out aliasing seq_lens
        assert _commit(lib, **kw) == -2, kw
    for name in ("k", "v", "bt", "sl", "path", "n"):
        assert _commit(lib, **{name: None}) == -1, name
    assert _commit(lib, tk=None) == -1                 # tree_k / tree_v: both or neither
    assert _commit(lib, k=A16 + 8) == -3
    assert _commit(lib, tk=A16 + 8) == -3
    assert _commit(lib, B=0, k=None) == 0


def test_dense_entries_host_checks(lib):
    a = A16
    f = lib.tree_dense_mask_build
    assert f(a, 0, a, 2, 4, 15, a, a, None, None) == -2      # cols not a multiple of 16
    assert f(a, 3, a, 2, 4, 64, a, a, None, None) == -2      # stride neither 0 nor T
    assert f(a, 0, a, 2, 65, 64, a, a, None, None) == -2
    assert f(None, 0, a, 2, 4, 64, a, a, None, None) == -1
    assert f(a, 0, a, 2, 4, 64, a + 8, a, None, None) == -3  # dense rows need 16 B alignment
    assert f(a, 0, a, 0, 4, 64, None, None, None, None) == 0
    v = lib.tree_attn_verify_dense
    base = [a, a, a, a, 4, a, a, 64, a, a, 2, 8, 2, 128, 4, 64, 8, 0.1, a, 1 << 30, None, None]
    args = list(base)
    args[6] = None
    assert v(*args) == -1
    args = list(base)
    args[7] = 40
    assert v(*args) == -2
    args = list(base)
    args[6] = a + 4
    assert v(*args) == -3


def test_verify_tree_host_checks(lib):
    a = A16
    f = lib.tree_attn_verify_tree
    base = [a, a, a, a, 4, a, a, a, a, 0, None, a, a, 2, 8, 2, 128, 4, 64, 8, 0.1, a, 1 << 30,
            None, None]
    args = list(base)
    args[8] = None
    assert f(*args) == -1          # parents
    args = list(base)
    args[9] = 3
    assert f(*args) == -2          # stride neither 0 nor T
    args = list(base)
    args[8] = a + 2
    assert f(*args) == -3
    args = list(base)
    args[10] = a + 4
    assert f(*args) == -3          # mask_out alignment


def test_plan_info_layout_matches_the_header(tmp_path):
    # The ctypes mirror of tree_attn_plan_info must have the C struct's size
    # and field offsets (a field added on one side only would shift the rest).
    from speculative_decoding_tree_split_gb300._lib import PlanInfo
    fields = [name for name, _ in PlanInfo._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "tree_attn.h"',
             'int main(void) {', '  printf("%zu\\n", sizeof(tree_attn_plan_info));']
    lines += [f'  printf("%zu\\n", offsetof(tree_attn_plan_info, {f}));' for f in fields]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(PlanInfo)] + [getattr(PlanInfo, f).offset for f in fields]
    assert got == want


def test_binding_argument_counts_match_the_header(lib):
    # Every prototype's parameter count equals the ctypes argtypes the binding
    # declares for it (a parameter added on one side only would misalign the call).
    text = ""
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text += open(os.path.join(HEADER_DIR, f)).read()
    protos = re.findall(r"TREE_ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)\s*;", text)
    assert len(protos) == len(declared_functions())
    for name, params in protos:
        params = " ".join(params.split())
        n = 0 if params in ("", "void") else params.count(",") + 1
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None, name
        assert len(argtypes) == n, (name, len(argtypes), n)


def test_wait_limit_setting_is_host_only_and_restorable(lib):
    # no CUDA call is made: this runs on a machine without a GPU
    assert ta.set_wait_limit_ns(5000) == ta.DEFAULT_WAIT_NS
    assert ta.set_wait_limit_ns(7) == 5000
    assert ta.set_wait_limit_ns(0) == 7          # 0 restores the default
    assert ta.set_wait_limit_ns(0) == ta.DEFAULT_WAIT_NS
