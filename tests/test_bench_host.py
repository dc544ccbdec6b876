"""Host logic of bench.py that needs no GPU: the traffic record is keyed on a
hash of the kernel's source with its comments removed, so a comment-only edit
keeps it and any code edit drops it."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comments_and_blank_lines_are_removed():
    src = 'int a; // one\n\n/* two\n three */ int b;\n   \nint c; /* four */ int d;\n'
    assert bench.strip_comments(src) == 'int a;\n  int b;\nint c;   int d;'


def test_literals_survive():
    src = 'const char* u = "x//y/*z*/"; char c = \'/\'; char q = \'"\'; // gone\nasm("mov.u32 %0, 1;");\n'
    out = bench.strip_comments(src)
    assert '"x//y/*z*/"' in out and "'/'" in out and "'\"'" in out and 'asm("mov.u32 %0, 1;");' in out
    assert "gone" not in out


def test_escaped_quotes_inside_a_literal():
    src = 'const char* s = "a\\"//b"; // c\n'
    assert bench.strip_comments(src) == 'const char* s = "a\\"//b";'


def test_comment_edits_keep_the_code_and_code_edits_change_it():
    base = "// header\nint f(int x) {  // body\n  return x + 1;\n}\n"
    reworded = "// a different header\n\nint f(int x) {  /* other words */\n  return x + 1;\n}\n"
    changed = "// header\nint f(int x) {  // body\n  return x + 2;\n}\n"
    assert bench.strip_comments(base) == bench.strip_comments(reworded)
    assert bench.strip_comments(base) != bench.strip_comments(changed)


def test_the_committed_record_is_well_formed():
    # (whether it still matches the source is the bench's own check: a
    # record taken on other code reads as null)
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["decode_tc_kernel"]
    assert len(rec["source_hash"]) == 16
    # at least the decode point's algorithmic bytes, at most a few percent more
    assert 13_041_620 <= rec["dram_bytes_per_launch"] <= 1.2 * 13_041_620
    assert rec["dram_bytes_per_launch"] == rec["dram_read"] + rec["dram_write"]
