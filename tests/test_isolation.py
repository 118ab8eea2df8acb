"""The library never reaches the oracle, and the two share no code.

The CUDA path is checked against the oracle only if it does not use it: the
package's modules must import without pulling in anything under oracle/,
and no source file of the package (Python or CUDA) or header may name it.
The oracle, in turn, imports nothing from the package. bench.py may use the
oracle only for its CPU timing legs, inside functions.
"""

from __future__ import annotations

import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "adaptive_sparse_paged_gb300")


def test_package_import_does_not_load_the_oracle():
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import adaptive_sparse_paged_gb300, adaptive_sparse_paged_gb300.binding, "
            "adaptive_sparse_paged_gb300.step, adaptive_sparse_paged_gb300.synth, "
            "adaptive_sparse_paged_gb300.diagnostics, adaptive_sparse_paged_gb300.build\n"
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]\n"
            "assert not bad, bad\n" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _sources(top, exts):
    for d, _, files in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_no_product_source_names_the_oracle():
    for path in list(_sources(PKG, (".py", ".cu", ".cuh", ".h"))) + \
            list(_sources(os.path.join(ROOT, "include"), (".h",))):
        text = open(path).read()
        if path.endswith(".py"):
            tree = ast.parse(text)
            for node in ast.walk(tree):
                if isinstance(node, ast.Import):
                    assert not any(a.name.split(".")[0] == "oracle" for a in node.names), path
                if isinstance(node, ast.ImportFrom) and node.module:
                    assert node.module.split(".")[0] != "oracle", path
        else:
            assert "oracle" not in text.lower(), path


def test_oracle_imports_nothing_from_the_package():
    for path in _sources(os.path.join(ROOT, "oracle"), (".py",)):
        tree = ast.parse(open(path).read())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom) and node.module:
                names = [node.module]
            for n in names:
                assert not n.startswith(("adaptive_sparse_paged_gb300", "torch")), (path, n)


def test_bench_imports_the_oracle_only_inside_functions():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    for node in tree.body:  # module level
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            mod = node.module if isinstance(node, ast.ImportFrom) else node.names[0].name
            assert not (mod or "").startswith("oracle")


def test_missing_library_fails_loudly(tmp_path):
    """Without libasp.so every call raises: there is no CPU fallback."""
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import torch\n"
            "from adaptive_sparse_paged_gb300 import binding as B\n"
            "B.LIB_PATH = %r\n"
            "try:\n"
            "    B.load_library(B.LIB_PATH)\n"
            "except RuntimeError as e:\n"
            "    assert 'libasp.so not found' in str(e), e\n"
            "else:\n"
            "    raise SystemExit('loaded a library that does not exist')\n"
            % (ROOT, str(tmp_path / "libasp.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr + r.stdout
