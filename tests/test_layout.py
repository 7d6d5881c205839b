"""Work partition and descriptor helpers of csrc/layout.h, compiled with g++
on the CPU (tests/native/layout_check.cpp)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layout_helpers(tmp_path):
    exe = os.path.join(tmp_path, "layout_check")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I",
                    os.path.join(ROOT, "speculative_decoding_tree_split_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "native", "layout_check.cpp"), "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
