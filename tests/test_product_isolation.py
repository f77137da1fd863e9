"""The product path stands apart from the oracle and has no fallback: the package and its
CUDA sources never import, include or load anything under oracle/, and the binding raises
when librepstep.so is missing instead of computing anything another way."""
import os
import re

import pytest

from bitwise_reproducible_step_gb300 import repstep as rs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bitwise_reproducible_step_gb300")


def _sources():
    for d, _, files in os.walk(PKG):
        if "__pycache__" in d:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                yield os.path.join(d, f)
    for f in os.listdir(os.path.join(ROOT, "include")):
        yield os.path.join(ROOT, "include", f)


def test_package_never_imports_the_oracle():
    bad = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|#\s*include\s+[\"<][^\">]*oracle)"
                     r"|liboracle|oracle\.c\b", re.M)
    for path in _sources():
        text = open(path, encoding="utf-8").read()
        m = bad.search(text)
        assert m is None, f"{os.path.relpath(path, ROOT)}: {m.group(0)!r}"


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(rs, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "librepstep.so"))
    monkeypatch.setattr(rs, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        rs.lib()
    with pytest.raises(RuntimeError, match="missing"):
        rs.Repstep(4096)
