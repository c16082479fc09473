"""The product path has no fallback: without libhb.so the binding raises
instead of computing anything, and no module of the package imports the
oracle (only tests, smoke() and the bench's CPU legs may)."""
import ast
import os

import pytest

from _hbutil import ROOT, host_batch, lib

PKG = os.path.join(ROOT, "chunked_prefill_decode_gb300")


def test_binding_fails_loudly_without_the_library(monkeypatch):
    hb = lib()
    b, ql, cl = host_batch(hb, [(1, 40), (5, 9)])
    monkeypatch.setattr(hb, "_lib", None)
    monkeypatch.setattr(hb, "_LIB_PATH", os.path.join(ROOT, "no-such-dir", "libhb.so"))
    with pytest.raises(RuntimeError, match="missing"):
        hb.load()
    with pytest.raises(RuntimeError, match="missing"):
        hb.hb_plan_sizes(b, ql, cl, 152)
    with pytest.raises(RuntimeError, match="missing"):
        hb.Builder(8, 16, 10, 4)


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def test_package_never_imports_the_oracle():
    seen = 0
    for name in sorted(os.listdir(PKG)):
        if not name.endswith(".py"):
            continue
        seen += 1
        for mod in _imports(os.path.join(PKG, name)):
            assert not mod.split(".")[0] == "oracle", f"{name} imports {mod}"
    assert seen >= 5
