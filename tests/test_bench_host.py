"""Host-side checks of bench.py's helpers (no GPU): the code stamp that gates
the committed ncu traffic figure, and the parsing of that stamp."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines():
    src = 'int a = 1;  // one\n\n/* block\n comment */ int b = 2;\nconst char* s = "// not a comment";\n'
    assert bench.code_only(src) == 'int a = 1;\n int b = 2;\nconst char* s = "// not a comment";'


def test_code_stamp_ignores_comments_but_not_code():
    base = "__device__ int f(int x) {\n  return x + 1;\n}\n"
    commented = "// f adds one\n__device__ int f(int x) {  // the argument\n\n  return x + 1;  /* plus one */\n}\n"
    changed = "__device__ int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_only(base) == bench.code_only(commented)
    assert bench.code_only(base) != bench.code_only(changed)


def test_profiled_traffic_matches_current_source():
    """The committed fused-step summary carries the stamp of the current decode
    kernel code, so the bench reports its measured traffic."""
    t = bench.profiled_traffic()
    assert t is not None and 270_000_000 < t < 290_000_000
