"""The CUDA path and the oracle stay apart (no GPU).

* nothing in the package or the headers imports, includes or names a path
  of the oracle;
* the oracle imports only the standard library and numpy;
* the seeded input generator imports neither side;
* outside tests/, only the benchmark's CPU-oracle sample and smoke() import
  the oracle;
* the binding fails loudly when the library is missing (no CPU path).
"""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_denoising_gb300")


def _files(top, exts):
    for d, _, fs in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _imports(path):
    """(module, enclosing top-level function or None) of every import."""
    tree = ast.parse(open(path).read())
    out = []

    def visit(node, fn):
        for ch in ast.iter_child_nodes(node):
            f = fn
            if isinstance(ch, (ast.FunctionDef, ast.AsyncFunctionDef)) and fn is None:
                f = ch.name
            if isinstance(ch, ast.Import):
                out.extend((a.name, f) for a in ch.names)
            elif isinstance(ch, ast.ImportFrom):
                out.append(((("." * ch.level) + (ch.module or "")), f))
            visit(ch, f)

    visit(tree, None)
    return out


def test_product_code_does_not_reach_the_oracle():
    pat = re.compile(r"import\s+oracle|from\s+oracle|oracle/|dinfer_oracle|#\s*include\s*[<\"].*oracle")
    bad = []
    for p in list(_files(PKG, (".py", ".cu", ".cuh", ".h", ".c", ".cpp"))) + list(
            _files(os.path.join(ROOT, "include"), (".h",))):
        for i, line in enumerate(open(p, errors="replace"), 1):
            if pat.search(line):
                bad.append(f"{os.path.relpath(p, ROOT)}:{i}: {line.strip()}")
    assert not bad, bad


def test_oracle_imports_only_numpy_and_the_standard_library():
    allowed = {"__future__", "dataclasses", "typing", "numpy", "math"}
    for p in _files(os.path.join(ROOT, "oracle"), (".py",)):
        mods = {m.split(".")[0] for m, _ in _imports(p)}
        assert mods <= allowed, (p, mods - allowed)


def test_input_generator_imports_neither_side():
    mods = {m for m, _ in _imports(os.path.join(PKG, "inputs.py"))}
    assert not any(m.startswith(("oracle", ".dinfer", "block_denoising_gb300.dinfer", ".build")) for m in mods), mods


def test_oracle_is_imported_only_by_its_allowed_callers():
    allowed = {"bench.py": {"oracle_sample"}, "__graft_entry__.py": {"smoke"}}
    for name, fns in allowed.items():
        users = {fn for m, fn in _imports(os.path.join(ROOT, name)) if m.split(".")[0] == "oracle"}
        assert users <= fns, (name, users)
    for p in _files(PKG, (".py",)):
        assert not any(m.split(".")[0] == "oracle" for m, _ in _imports(p)), p


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from block_denoising_gb300 import dinfer
    monkeypatch.setattr(dinfer, "_lib", None)
    monkeypatch.setattr(dinfer, "LIB_PATH", str(tmp_path / "libdinfer.so"))
    with pytest.raises(RuntimeError, match="missing"):
        dinfer.lib()
