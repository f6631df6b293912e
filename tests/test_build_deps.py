"""The build's staleness check sees every file the library is compiled from: a change to any
source or header (the .cu, every kernel header it includes, the public header) makes
up_to_date() false, so build() never loads a library built from older sources."""
from __future__ import annotations

import os
import re

import pytest

from fp8_quant_row_gb300 import _build


def included_files(path, seen=None):
    """Transitive closure of the quoted #include files of a source, resolved in its own
    directory and the public include directory."""
    seen = set() if seen is None else seen
    path = os.path.abspath(path)
    if path in seen:
        return seen
    seen.add(path)
    for name in re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(path).read(), flags=re.M):
        for d in (os.path.dirname(path), _build.INCLUDE):
            cand = os.path.join(d, name)
            if os.path.exists(cand):
                included_files(cand, seen)
                break
        else:
            raise AssertionError(f"{path}: #include \"{name}\" not found")
    return seen


def test_every_included_file_is_a_dependency():
    deps = {os.path.abspath(d) for d in _build.deps()}
    for src in _build.SOURCES:
        missing = included_files(src) - deps
        assert not missing, f"not in the build's dependency list: {sorted(missing)}"


def test_touching_any_dependency_makes_the_library_stale(monkeypatch):
    _build.build()
    assert _build.up_to_date()
    lib_time = os.path.getmtime(_build.LIB)
    real = os.path.getmtime
    for dep in _build.deps():
        monkeypatch.setattr(os.path, "getmtime",
                            lambda p, dep=dep: lib_time + 1.0 if p == dep else real(p))
        assert not _build.up_to_date(), f"a change to {os.path.basename(dep)} went unnoticed"
    monkeypatch.setattr(os.path, "getmtime", real)
    assert _build.up_to_date()
