"""The bench's roofline reads per-launch DRAM traffic and instruction
counts from committed ncu summaries.  Each combination of workload, method
variant and error storage launches its own kernel instantiation, so each
has its own summary, and a figure is used only when the summary was taken
on the current kernel source."""
import os

import bench


def test_each_kernel_instantiation_has_its_own_summary():
    names = {bench.profile_summary("large", v, e) for v in ("lamb", "adam") for e in ("f32", "bf16")}
    assert len(names) == 4
    assert bench.profile_summary("large") == os.path.join("profiles", "compress_kernel_large.md")


def test_a_missing_summary_gives_no_figure():
    traffic, why = bench.profiled_traffic("no_such_workload", "adam", "bf16")
    assert traffic is None and "compress_kernel_no_such_workload_adam_bf16err.md" in why
    assert bench.profiled_instructions("no_such_workload") is None


def test_committed_summaries_name_a_kernel_source():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for f in os.listdir(os.path.join(root, "profiles")):
        if f.startswith("compress_kernel_"):
            text = open(os.path.join(root, "profiles", f)).read()
            assert "source_sha:" in text, f


def test_code_hash_ignores_comments_and_layout_only():
    a = 'int f(int x) {  // one\n  return x + 1; /* two */ }\nconst char* s = "a // b";\n'
    b = 'int f(int x) { return x + 1; }\n/* moved */ const char* s = "a // b";'
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens('s = "a // b";') == 's = "a // b";'       # literals are kept whole
    assert bench.code_tokens("c = '/'; d = a / b;") == "c = '/'; d = a / b;"
    assert bench.code_tokens(a) != bench.code_tokens(a.replace("x + 1", "x + 2"))
    assert bench.code_tokens(a) != bench.code_tokens(a.replace('"a // b"', '"a  // b"'))
