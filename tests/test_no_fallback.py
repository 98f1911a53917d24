"""The product path has no CPU fallback, checked on the CPU.

Without libdattn.so every entry point of the binding raises before computing anything, and
no module of the package (Python, CUDA or C) refers to the oracle, so the oracle cannot
stand in for a kernel.
"""
import ast
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import split_kv_decode_distattention_gb300 as dattn  # noqa: E402

PKG = os.path.join(ROOT, "split_kv_decode_distattention_gb300")
# an import or include of the oracle, its library or source file, a call of one of its C
# functions, or its folder named in a path string (prose mentioning the oracle is fine)
REF = re.compile(r"^\s*(import|from)\s+oracle\b|#\s*include\s*[<\"][^>\"]*oracle|dattn_oracle|"
                 r"\borc_\w+\s*\(|[\"'][^\"'\n]*\boracle[/\\\\\"']", re.M)


def test_a_missing_library_raises(tmp_path, monkeypatch):
    missing = str(tmp_path / "libdattn.so")
    with pytest.raises(dattn.DattnError, match="missing"):
        dattn.load_library(missing)
    monkeypatch.setattr(dattn, "_lib", None)
    monkeypatch.setattr(dattn, "_LIB_PATH", missing)
    for call in (dattn.dattn_version, lambda: dattn.dattn_status_string(0),
                 lambda: dattn.dattn_workspace_size(8, 32, 8, 128),
                 lambda: dattn.dattn_auto_splits(1024),
                 lambda: dattn.dattn_split_owner(3, 10, 2)):
        with pytest.raises(dattn.DattnError, match="missing"):
            call()


def test_no_package_source_refers_to_the_oracle():
    hits = []
    for dirpath, _, files in os.walk(PKG):
        if "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                if REF.search(text):
                    hits.append(os.path.relpath(os.path.join(dirpath, f), ROOT))
    assert hits == []


def test_bench_imports_the_oracle_only_in_its_cpu_baseline_and_reference_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read())
    allowed = {"oracle_sample", "dequantized", "time_oracle", "sparse_oracle_sample",
               "cpu_baseline_sparse", "cpu_baseline", "run_reference", "prefill_cpu_baseline",
               "SparseOracleStep"}

    def imports_oracle(node):
        return any(isinstance(n, (ast.Import, ast.ImportFrom)) and
                   any((a.name.split(".")[0] == "oracle") for a in n.names) or
                   (isinstance(n, ast.ImportFrom) and (n.module or "").split(".")[0] == "oracle")
                   for n in ast.walk(node))

    for node in tree.body:
        if isinstance(node, (ast.FunctionDef, ast.ClassDef)):
            if imports_oracle(node):
                assert node.name in allowed, f"bench.{node.name} imports the oracle"
        else:
            assert not imports_oracle(node), "bench.py imports the oracle at module level"
