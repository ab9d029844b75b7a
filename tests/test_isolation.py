"""The product path never reaches the oracle, and fails loudly without its CUDA library.

The oracle is test infrastructure: only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may load it.  The library's binding must raise (not fall back)
when libmita.so is missing, and the CUDA sources share nothing with the oracle.
"""
import ast
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_top_landmark_gb300")


def _python_files(folder):
    for base, _, files in os.walk(folder):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def test_product_package_never_imports_the_oracle():
    for path in _python_files(PKG):
        tree = ast.parse(open(path).read(), path)
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            assert not any(n == "oracle" or n.startswith("oracle.") for n in names), path


def test_cuda_sources_share_nothing_with_the_oracle():
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "oracle" not in text.lower() or f.endswith(".md"), f
    oracle_src = open(os.path.join(ROOT, "oracle", "mita_oracle.cpp")).read()
    assert "#include \"" not in oracle_src          # no header of the CUDA library


def test_oracle_imports_nothing_from_the_product():
    for path in _python_files(os.path.join(ROOT, "oracle")):
        assert "sparse_top_landmark_gb300" not in open(path).read(), path


def test_binding_raises_when_the_library_is_missing(monkeypatch, tmp_path):
    from sparse_top_landmark_gb300 import mita
    monkeypatch.setattr(mita, "_lib", None)
    monkeypatch.setattr(mita, "LIB_PATH", str(tmp_path / "libmita.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        mita.load()
