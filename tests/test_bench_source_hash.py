"""bench.py keys the committed ncu counters by a hash of the kernel sources' code: a comment
or layout change keeps the counters valid, a change to the code makes them stale."""
from __future__ import annotations

import bench

_SRC = """// header comment
#pragma once
/* block
   comment */
__device__ int f(int a) {   // trailing comment
  return a + 1;
}
"""


def test_comments_and_layout_do_not_change_the_code():
    reworded = _SRC.replace("header comment", "another header").replace(
        "trailing comment", "says something else")
    relaid = _SRC.replace("  return a + 1;", "\treturn   a + 1;\n\n")
    assert bench._code_only(reworded) == bench._code_only(_SRC)
    assert bench._code_only(relaid) == bench._code_only(_SRC)
    assert "comment" not in bench._code_only(_SRC)


def test_code_changes_are_seen():
    assert bench._code_only(_SRC.replace("a + 1", "a + 2")) != bench._code_only(_SRC)
    assert bench._code_only(_SRC.replace("#pragma once", "")) != bench._code_only(_SRC)


def test_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
