"""The profile digest covers code, not comments or layout: a comment edit keeps a captured
profile's traffic valid, any code edit voids it."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comments_and_layout_do_not_count():
    a = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    b = "/* header */\nint f(int x)\n{\n  // a comment\n  return x + 1;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_count():
    a = "int f(int x) { return x + 1; }"
    assert bench._code_only(a) != bench._code_only(a.replace("+ 1", "+ 2"))
    assert bench._code_only(a) != bench._code_only(a.replace("int x", "long x"))


def test_literals_are_kept_verbatim():
    s = 'const char *p = "a // not a comment /* nor this */"; char q = \'"\';'
    assert bench._code_only(s) == s
    esc = 'asm("mov.b32 %0, %1;\\n\\t" : "=r"(a) : "r"(b)); // tail'
    assert bench._code_only(esc) == 'asm("mov.b32 %0, %1;\\n\\t" : "=r"(a) : "r"(b));'


def test_digest_is_stable():
    assert bench.kernel_source_digest() == bench.kernel_source_digest()
    assert len(bench.kernel_source_digest()) == 16
