"""Host logic of bench.py that needs no GPU: the hash that decides whether a profiled DRAM traffic
still applies covers the kernels' code, not their comments."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_only_ignores_comments_and_blank_lines():
    a = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    b = "// f adds one\nint f(int x) {\n\n    /* the sum */ return x + 1;\n}\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_every_kernel_source_exists_and_the_traffic_record_names_known_kernels():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "semi_ar_draft_gb300", "csrc", f)), (kernel, f)
        assert len(bench.source_hash(kernel)) == 16
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        tr = json.load(f)
    assert set(tr) <= set(bench.KERNEL_SOURCES)
    for rec in tr.values():
        assert rec["dram_bytes_per_launch"] > 0 and len(rec["source_hash"]) == 16
