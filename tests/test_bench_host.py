"""Host logic of bench.py that needs no GPU: the kernel hash that ties an ncu summary under
profiles/ to the kernel source it was taken on, and the traffic figure scaled from it."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comment_edits_leave_the_code_unchanged():
    code = "int f(int x) {\n  return x + 1;  // add one\n}\n"
    commented = "/* a new note\n   over two lines */\nint f(int x) {\n  // why\n  return x + 1;\n}\n"
    assert bench.strip_comments(code) == bench.strip_comments(commented)
    assert bench.strip_comments(code) != bench.strip_comments(code.replace("+ 1", "+ 2"))


def test_kernel_hash_covers_every_attention_source_and_the_build_options(monkeypatch):
    base = bench.kernel_sha()
    assert re.fullmatch(r"[0-9a-f]{16}", base)
    monkeypatch.setenv("PDA_NVCC_DEFINES", "PDA_ATTN_WARPS=8")
    assert bench.kernel_sha() != base
    monkeypatch.delenv("PDA_NVCC_DEFINES")
    assert bench.kernel_sha() == base
    for p in bench.ATTN_SOURCES:
        assert os.path.exists(os.path.join(ROOT, p)), p


def test_headline_traffic_scales_the_profiled_ratio_when_the_hash_matches():
    path = os.path.join(ROOT, "profiles", "attn_partial_gqa_skew_b256.md")
    text = open(path).read()
    sha = re.search(r"kernel_sha:\s*([0-9a-f]+)", text).group(1)
    ratio = float(re.search(r"dram_traffic_ratio:\s*([0-9.]+)", text).group(1))
    got = bench.profiled_traffic("gqa_skew_b256", 10**9)
    if sha == bench.kernel_sha():
        assert got == int(round(ratio * 10**9))
    else:  # a summary of another kernel gives no traffic figure
        assert got is None
    assert bench.profiled_traffic("no_such_workload", 10**9) is None
