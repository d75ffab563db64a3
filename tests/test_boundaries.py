"""Static checks of the split between the product path and its test infrastructure.

The library and its binding must not reach the float64 oracle or the input
generators (the oracle is test infrastructure; a product path routed through
it, or any CPU fallback, would make the parity tests meaningless), and the
binding must fail loudly when the compiled library is missing.
"""

import ast
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "checkpoint_input_replay_gb300")


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_package_imports_neither_oracle_nor_workloads():
    for f in os.listdir(PKG):
        if f.endswith(".py"):
            bad = _imports(os.path.join(PKG, f)) & {"oracle", "workloads", "tests", "numpy"}
            assert not bad, (f, bad)


def test_cuda_sources_do_not_mention_the_oracle():
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(csrc, f)).read().lower()
            assert "oracle" not in text, f


def test_oracle_says_it_is_test_infrastructure():
    head = open(os.path.join(ROOT, "oracle", "__init__.py")).read(400)
    assert "TEST INFRASTRUCTURE ONLY" in head


def test_missing_library_fails_loudly(monkeypatch):
    from checkpoint_input_replay_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB", os.path.join(ROOT, "no_such_dir", "libreplayssm.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()
