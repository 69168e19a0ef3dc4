"""Structural invariants of the repository (CPU only).

* The oracle and the CUDA path share no code: nothing in the package (Python,
  CUDA, headers) refers to ``oracle``, nothing in ``oracle/`` refers to the
  package or its sources, and the seeded input generators in ``synth/`` import
  neither.
* bench.py reaches the oracle only inside its CPU legs (no module-level import).
* Nothing committed refers to the scratch folder.
* The product path fails loudly without the compiled library: no fallback.
"""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "speculative_decode_verify_sdv_gb300"


def files_under(sub, exts):
    out = []
    for dirpath, dirnames, names in os.walk(os.path.join(ROOT, sub)):
        dirnames[:] = [d for d in dirnames if d not in ("__pycache__",)]
        out += [os.path.join(dirpath, n) for n in names if n.endswith(exts)]
    return sorted(out)


def python_imports(path):
    tree = ast.parse(open(path).read(), path)
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            mods.add(node.module.split(".")[0])
    return mods


def test_package_never_reaches_the_oracle():
    for path in files_under(PKG, (".py",)):
        assert "oracle" not in python_imports(path), path
    for path in files_under(PKG, (".cu", ".cuh", ".h")) + files_under("include", (".h",)):
        includes = re.findall(r'#include\s*[<"]([^>"]+)[>"]', open(path).read())
        assert not any("oracle" in inc for inc in includes), path


def test_oracle_never_reaches_the_package():
    for path in files_under("oracle", (".py",)):
        mods = python_imports(path)
        assert PKG not in mods and "bench" not in mods, path
        text = open(path).read()
        assert "csrc" not in text and "libsdv" not in text, path
    cpp = files_under("oracle", (".c", ".h", ".cpp", ".hpp"))
    assert cpp, "the oracle's C++ sources are missing"
    for path in cpp:
        text = open(path).read()
        assert "sdv_kernels" not in text and "sdv_device" not in text and "sdv.h" not in text, path
        # standard headers only: nothing of the CUDA path, no CUDA, no BLAS
        for inc in re.findall(r'#include\s*([<"][^>"]+[>"])', text):
            assert inc.startswith("<"), (path, inc)
            assert not any(b in inc for b in ("cuda", "cublas", "cblas", "mkl", "immintrin", "arm_neon")), (path, inc)


def test_generators_import_neither_side():
    for path in files_under("synth", (".py",)):
        mods = python_imports(path)
        assert "oracle" not in mods and PKG not in mods, path


def test_bench_imports_the_oracle_only_inside_its_cpu_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    for node in tree.body:  # module level only
        if isinstance(node, ast.Import):
            assert not any(a.name.split(".")[0] == "oracle" for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            assert (node.module or "").split(".")[0] != "oracle"


def test_nothing_committed_refers_to_the_scratch_folder():
    pattern = re.compile(r"(^|[^A-Za-z0-9])_work/")
    roots = [PKG, "oracle", "synth", "tests", "include"]
    paths = [os.path.join(ROOT, f) for f in ("bench.py", "__graft_entry__.py")]
    for sub in roots:
        paths += files_under(sub, (".py", ".cu", ".cuh", ".h", ".c", ".txt"))
    here = os.path.abspath(__file__)
    for path in paths:
        if os.path.abspath(path) == here:
            continue
        assert not pattern.search(open(path, errors="replace").read()), path


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from speculative_decode_verify_sdv_gb300 import sdv
    monkeypatch.setattr(sdv, "_lib", None)
    monkeypatch.setattr(sdv, "LIB_PATH", str(tmp_path / "libsdv.so"))
    with pytest.raises(RuntimeError, match="libsdv.so not found"):
        sdv.load()
    with pytest.raises(RuntimeError):
        sdv.sdv_version()
