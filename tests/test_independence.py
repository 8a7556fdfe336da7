"""Structure checks: the product and the oracle share no code, and the product
has no fallback path.

  * nothing under turboquant_paged_kv_gb300/ (Python or CUDA/C++ sources)
    imports, includes or names the oracle package;
  * nothing under oracle/ imports the product;
  * the binding raises ImportError when libtq.so is missing instead of
    computing anything itself.
"""

import ast
import importlib
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "turboquant_paged_kv_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d or "_lib" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imported_modules(path):
    tree = ast.parse(open(path, encoding="utf-8").read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield (node.module or "") if node.level == 0 else "." * node.level + (node.module or "")


def test_product_python_never_imports_the_oracle():
    files = list(_files(PKG, (".py",)))
    assert files
    for path in files:
        for mod in _imported_modules(path):
            assert not mod.split(".")[0] in ("oracle", "parity", "workloads"), (path, mod)


def test_product_native_sources_never_name_the_oracle():
    files = list(_files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".cpp", ".h"))) + \
        list(_files(os.path.join(ROOT, "include"), (".h",)))
    assert files
    for path in files:
        text = open(path, encoding="utf-8").read()
        assert "oracle" not in text.lower(), path


def test_oracle_never_imports_the_product():
    files = list(_files(ORACLE, (".py",)))
    assert files
    for path in files:
        for mod in _imported_modules(path):
            assert mod.split(".")[0] != "turboquant_paged_kv_gb300", (path, mod)


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    abi = importlib.import_module("turboquant_paged_kv_gb300._abi")
    monkeypatch.setattr(abi, "_LIB_PATH", str(tmp_path / "missing" / "libtq.so"))
    monkeypatch.setattr(abi, "_lib", None)
    with pytest.raises(ImportError):
        abi.load()
    import turboquant_paged_kv_gb300 as tq
    with pytest.raises(ImportError):
        tq.tq_build_codebook(128, 4)
