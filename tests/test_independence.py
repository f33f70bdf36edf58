"""Static checks that keep the checker and the product apart (CPU only).

The CPU oracle is test infrastructure: the GPU library and its Python binding
must neither import, include nor link it, and the oracle must not use the
GPU sources, so that agreement between the two means something. The binding
must also refuse to run without its CUDA library rather than fall back to
anything else.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "hyper_connection_rank_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def files(top, exts):
    for d, _, fs in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_product_never_uses_the_oracle():
    for p in files(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        text = open(p).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f"{p} imports the oracle"
        assert not re.search(r"import_module\(\s*['\"]oracle", text), f"{p} imports the oracle"
        assert "hc_oracle" not in text, f"{p} names the oracle library"
    for p in files(os.path.join(ROOT, "include"), (".h",)):
        assert "oracle" not in open(p).read().lower().replace("oracles", ""), f"{p} refers to the oracle"


def test_oracle_never_uses_the_product():
    for p in files(ORACLE, (".py", ".cpp", ".h")):
        text = open(p).read()
        assert "hyper_connection_rank_gb300" not in text, f"{p} uses the GPU package"
        assert not re.search(r'#\s*include\s*[<"][^>"]*(hc_lowrank_mix|hc_row_ops|hc_common|hc_internal)',
                             text), f"{p} includes a GPU header"
        assert "libhc_lowrank_mix" not in text, f"{p} loads the GPU library"


def test_binding_refuses_to_run_without_its_library(tmp_path):
    from hyper_connection_rank_gb300 import _binding as B
    saved = B._lib
    B._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            B.load_library(str(tmp_path / "missing.so"))
    finally:
        B._lib = saved
