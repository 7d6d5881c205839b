"""Host-side parts of bench.py on the CPU: the max-over-ranks reduction with
two gloo ranks, and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
    q.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == [2.0, 10.0] and results[1] == [2.0, 10.0]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.0]) == [3.5, 1.0]


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert key in line
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_kernel_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    # The ncu traffic record is keyed by this hash: a comment or whitespace
    # edit must keep it, any code edit must change it.
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(ROOT, "speculative_decoding_tree_split_gb300", "csrc")
    dst = tmp_path / "speculative_decoding_tree_split_gb300" / "csrc"
    dst.mkdir(parents=True)
    texts = {}
    for name in ("kernels.cu", "prefix_early.cu", "layout.h", "ptx.cuh"):
        with open(os.path.join(src, name), encoding="utf-8") as f:
            texts[name] = f.read()

    def sha_with(layout_text):
        for name, text in texts.items():
            (dst / name).write_text(layout_text if name == "layout.h" else text, encoding="utf-8")
        monkeypatch.setattr(bench, "_ROOT", str(tmp_path))
        return bench.kernel_source_sha()

    base = sha_with(texts["layout.h"])
    commented = texts["layout.h"] + "\n// a new comment\n/* and a\n   block comment */\n\n   \n"
    assert sha_with(commented) == base
    code = texts["layout.h"].replace("constexpr int kTreeInPrefixMaxSteps = 32;",
                                     "constexpr int kTreeInPrefixMaxSteps = 33;")
    assert code != texts["layout.h"]
    assert sha_with(code) != base
