"""Structural rules of the boundary between the product and the oracle,
checked on the sources (CPU only):

* the product (the package and its CUDA sources) never imports, includes or
  reads anything under oracle/, and the oracle never imports the product;
* the one module both sides share, the seeded input generator, holds none of
  the method's arithmetic;
* the binding has no fallback: without libcfc.so every call raises.
"""

import ast
import os
import re

import pytest

import recurrent_cell_gb300 as cfc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "recurrent_cell_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for dirpath, _, names in os.walk(top):
        if "__pycache__" in dirpath or "_build" in dirpath:
            continue
        for n in sorted(names):
            if n.endswith(exts):
                yield os.path.join(dirpath, n)


def _imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def _code_strings(path):
    """String constants of a module other than its docstrings."""
    tree = ast.parse(open(path).read(), path)
    docs = set()
    for node in ast.walk(tree):
        if isinstance(node, (ast.Module, ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)) and node.body:
            first = node.body[0]
            if isinstance(first, ast.Expr) and isinstance(first.value, ast.Constant):
                docs.add(id(first.value))
    for node in ast.walk(tree):
        if isinstance(node, ast.Constant) and isinstance(node.value, str) and id(node) not in docs:
            yield node.value


def test_product_python_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        for mod in _imported_modules(path):
            assert not mod.split(".")[0] == "oracle", f"{path} imports {mod}"
        for text in _code_strings(path):
            assert "oracle" not in text, f"{path} refers to the oracle in code: {text!r}"


def test_product_cuda_sources_never_include_the_oracle():
    for path in list(_files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h"))) + \
            list(_files(os.path.join(ROOT, "include"), (".h",))):
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert "oracle" not in inc, f"{path} includes {inc}"


def test_oracle_never_imports_the_product():
    for path in _files(ORACLE, (".py",)):
        for mod in _imported_modules(path):
            assert mod.split(".")[0] not in ("recurrent_cell_gb300", "torch"), f"{path} imports {mod}"


def test_shared_input_generator_holds_no_cell_arithmetic():
    """workloads.py draws and rounds inputs; it must not evaluate the cell
    (no tanh, sigmoid, exponentials, GELU or contractions)."""
    src = open(os.path.join(PKG, "workloads.py")).read()
    code = "\n".join(line.split("#", 1)[0] for line in src.splitlines())
    for name in ("tanh", "np.exp", "sigmoid", "erf", "einsum", "matmul", " @ ", ".dot("):
        assert name not in code, f"workloads.py uses {name!r}"


def test_binding_raises_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(cfc, "_lib", None)
    monkeypatch.setattr(cfc, "LIB_PATH", str(tmp_path / "missing_libcfc.so"))
    with pytest.raises(RuntimeError, match="libcfc.so not found"):
        cfc.load_library(str(tmp_path / "missing_libcfc.so"))
