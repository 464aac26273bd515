"""The product path fails loudly without its CUDA library and never reaches
the oracle: the binding raises when libtoktier.so is missing (no CPU
fallback), no Python module of the package imports the oracle, and no
native source of the package includes anything from it."""
import ast
import os
import re

import numpy as np
import pytest

from exact_bpe_tokenization_gb300 import binding

PKG = os.path.dirname(os.path.abspath(binding.__file__))


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libtoktier.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()
    merges = np.zeros((0, 2), dtype=np.int32)
    vb = np.arange(256, dtype=np.uint8)
    vo = np.arange(257, dtype=np.int64)
    with pytest.raises(RuntimeError, match="not built"):
        binding.Tokenizer(merges, vb, vo, binding.TT_FAMILY_CL100K_STYLE)


def _python_files():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def test_package_never_imports_the_oracle():
    files = list(_python_files())
    assert any(f.endswith("binding.py") for f in files)
    for path in files:
        with open(path) as fh:
            tree = ast.parse(fh.read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            else:
                continue
            assert not any(n.split(".")[0] == "oracle" for n in names), (path, names)


def test_native_sources_include_nothing_from_the_oracle():
    seen = 0
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".cu", ".cuh", ".h", ".c", ".cpp")):
                with open(os.path.join(dirpath, f)) as fh:
                    for line in fh:
                        m = re.match(r'\s*#\s*include\s*[<"]([^>"]+)[>"]', line)
                        if m:
                            seen += 1
                            assert "oracle" not in m.group(1), (f, line)
    assert seen > 0
