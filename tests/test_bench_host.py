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


def test_the_committed_record_matches_the_committed_kernel():
    # the decode kernel's DRAM bytes were captured on this source
    assert bench.traffic_record("decode_tc_kernel") is not None
