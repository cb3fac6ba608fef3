"""Host-side pieces of bench.py: the comment-blind source hash that keys profiles/traffic.txt."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_c_comments_keeps_code_and_literals():
    src = ('int a = 1; // trailing\n/* block\n   comment */ const char *s = "x // y /* z */";\n'
           "char q = '\"'; char e = '\\\\';   int   b = 2;\n")
    assert bench.strip_c_comments(src) == (
        'int a = 1; const char *s = "x // y /* z */"; char q = \'"\'; char e = \'\\\\\'; int b = 2;')


def test_strip_c_comments_ignores_comment_and_layout_edits_only():
    a = "__global__ void k(int *p) { p[0] = 1; }  // one\n"
    b = "// header\n__global__ void k(int *p)\n{\n    p[0] = 1;   /* same code */\n}\n"
    c = "__global__ void k(int *p) { p[0] = 2; }\n"
    assert bench.strip_c_comments(a) == bench.strip_c_comments(b)
    assert bench.strip_c_comments(a) != bench.strip_c_comments(c)


def test_traffic_lines_name_existing_sources():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    lines = [ln.split() for ln in open(path) if ln.startswith("kernel=")]
    assert lines
    for parts in lines:
        kv = dict(p.split("=", 1) for p in parts)
        assert set(kv) == {"kernel", "file", "src_sha", "dram_bytes_per_launch", "workload"}
        assert os.path.exists(os.path.join(ROOT, "rl_infra_gb300", "csrc", kv["file"]))
        assert len(kv["src_sha"]) == 16 and int(kv["src_sha"], 16) >= 0
        assert float(kv["dram_bytes_per_launch"]) > 0
