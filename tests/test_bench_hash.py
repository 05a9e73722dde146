"""The key under which bench.py looks up committed ncu traffic figures: the library's source code,
with comments and layout ignored (no GPU needed)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_comments_and_layout_do_not_change_the_code():
    a = 'int f(int x) {  // doubles x\n  return 2 * x; /* the\n block */ }\nconst char* s = "a//b";'
    b = 'int f(int x) {\n  // another comment\n  return 2 * x;\n}\nconst char* s = "a//b";'
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_and_literals_are_kept():
    base = bench._code_only("int y = 2 * x;")
    assert bench._code_only("int y = 3 * x;") != base
    assert "\"a//b\"" in bench._code_only('const char* s = "a//b"; // tail')
    assert "'/'" in bench._code_only("char c = '/'; /* x */")


def test_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash() and len(h) == 16
