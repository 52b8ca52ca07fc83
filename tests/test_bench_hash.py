"""The benchmark's record of which device code an ncu capture was taken on: comments and
layout do not count, code (including string literals) does.  (A record whose code changed
is reported as null traffic by bench.py, not as a failure.)"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_text_drops_comments_and_layout_only():
    src = 'a = "x // y";  // note\nb /* c */ = \'/\';\n/* d\n   e */ f(1,\n  2);'
    assert bench.code_text(src) == 'a = "x // y"; b = \'/\'; f(1, 2);'
    assert bench.code_text('s = "q\\" // still in the string"; // gone') == 's = "q\\" // still in the string";'
    assert bench.code_text("x = 1; // a\n") == bench.code_text("x  =  1;")
    assert bench.code_text("x = 1;") != bench.code_text("x = 2;")

