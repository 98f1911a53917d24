"""The Python binding's marshalling checked against include/dattn.h, on the CPU.

The binding declares every entry point's argument and result types and mirrors the
header's structs as ctypes structures. A drift between the two passes arguments in the
wrong registers or reads struct fields at the wrong offsets, so this test pins them:
- gcc compiles a small C program against the header (as plain C, the boundary's language)
  and prints every struct field's offset and size and each struct's size, which must equal
  the ctypes layout field by field;
- each struct's fields, in declaration order, must be the binding's fields;
- each prototype's parameter kinds (pointer, struct pointer, int32, int64, float, size_t)
  and result kind must be the binding's, entry point by entry point.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dattn.h")

import sys  # noqa: E402
sys.path.insert(0, ROOT)
import split_kv_decode_distattention_gb300 as dattn  # noqa: E402

STRUCTS = {"dattn_kv_layout": dattn._Layout, "dattn_sparse": dattn._Sparse,
           "dattn_prefill_sparse": dattn._PrefillSparse}
SCALARS = {"int32_t": "i32", "dattn_status_t": "i32", "int64_t": "i64", "float": "f32",
           "size_t": "size"}


def _header_text():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return "\n".join(ln for ln in src.splitlines() if not ln.lstrip().startswith("#"))


def _kind(decl: str, is_result: bool = False):
    """Kind of one C parameter or result type (the parameter's name is dropped)."""
    decl = " ".join(decl.replace("*", " * ").split())
    words = [w for w in decl.split() if w not in ("const", "struct")]
    if "*" in words:
        base = words[0]
        if base in STRUCTS:
            return ("struct", base)
        if is_result and base == "char":
            return "str"
        return "ptr"
    if words == ["void"]:
        return None
    assert words[0] in SCALARS, f"unmapped C type in {decl!r}"
    return SCALARS[words[0]]


def _header_prototypes():
    text = _header_text()
    protos = {}
    for stmt in text.split(";"):
        stmt = re.split(r"[{}]", stmt)[-1].strip()
        m = re.match(r"^(.*?)\b(dattn_\w+)\s*\((.*)\)$", stmt, flags=re.S)
        if not m or stmt.startswith("typedef"):
            continue
        res, name, params = m.group(1), m.group(2), m.group(3).strip()
        kinds = [] if params in ("", "void") else [
            _kind(re.sub(r"\b\w+\s*$", "", p.strip()) if not p.strip().endswith("*") else p)
            for p in params.split(",")]
        protos[name] = (_kind(res, is_result=True), kinds)
    return protos


def _ctypes_kind(t):
    if t is None:
        return None
    if t is ctypes.c_char_p:
        return "str"
    if t is ctypes.c_void_p:
        return "ptr"
    for cname, cls in STRUCTS.items():
        if t is ctypes.POINTER(cls):
            return ("struct", cname)
    if isinstance(t, type) and issubclass(t, ctypes._Pointer):
        return "ptr"
    table = {ctypes.c_int32: "i32", ctypes.c_int64: "i64", ctypes.c_float: "f32",
             ctypes.c_size_t: "size"}
    assert t in table, f"unmapped ctypes type {t}"
    return table[t]


def _header_struct_fields(name):
    text = _header_text()
    m = re.search(r"typedef\s+struct\s+" + name + r"\s*\{(.*?)\}\s*" + name + r"\s*;", text,
                  flags=re.S)
    assert m, f"struct {name} not found in the header"
    return [re.findall(r"\w+", f)[-1] for f in m.group(1).split(";") if f.strip()]


def test_every_declared_entry_point_has_a_binding_of_the_same_kinds():
    protos = _header_prototypes()
    assert len(protos) >= 14
    assert set(protos) == set(dattn._SIGS), (
        f"declared only: {set(protos) - set(dattn._SIGS)}, "
        f"bound only: {set(dattn._SIGS) - set(protos)}")
    for name, (res, params) in protos.items():
        bres, bparams = dattn._SIGS[name]
        assert _ctypes_kind(bres) == res, f"{name}: result"
        got = [_ctypes_kind(t) for t in bparams]
        assert len(got) == len(params), f"{name}: {len(got)} arguments bound, {len(params)} declared"
        for i, (g, w) in enumerate(zip(got, params)):
            assert g == w, f"{name}: argument {i} bound as {g}, declared as {w}"


def test_struct_fields_follow_the_header_in_order():
    for cname, cls in STRUCTS.items():
        assert [f for f, _ in cls._fields_] == _header_struct_fields(cname), cname


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_struct_layouts_equal_the_c_compilers(tmp_path):
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "dattn.h"',
             "int main(void) {"]
    for cname, cls in STRUCTS.items():
        lines.append(f'printf("{cname} . %zu %zu\\n", (size_t)0, sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu %zu\\n", offsetof({cname}, {f}), '
                         f"sizeof((({cname} *)0)->{f}));")
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for ln in out.split("\n"):
        if ln:
            s, f, off, size = ln.split()
            got[(s, f)] = (int(off), int(size))
    for cname, cls in STRUCTS.items():
        assert got[(cname, ".")][1] == ctypes.sizeof(cls), f"sizeof {cname}"
        for f, t in cls._fields_:
            assert got[(cname, f)] == (getattr(cls, f).offset, ctypes.sizeof(t)), f"{cname}.{f}"


def test_constants_equal_the_headers_defines():
    defines = dict(re.findall(r"^#define\s+DATTN_(\w+)\s+(0x[0-9a-fA-F]+|\d+)", open(HEADER).read(),
                              flags=re.M))
    defines = {k: int(v, 0) for k, v in defines.items()}
    assert {k: v for k, v in defines.items() if k.startswith("DEVERR_")} == {
        "DEVERR_" + k: v for k, v in dattn.DEVERR.items()}
    for k in ("HEAD_DENSE", "HEAD_RETRIEVAL", "HEAD_STREAMING", "KV_BF16", "KV_FP8_E4M3",
              "KV_INT4", "KV_MIXED"):
        assert getattr(dattn, k) == defines[k], k
    assert {k for k in defines if k.startswith(("HEAD_", "KV_"))} == {
        "HEAD_DENSE", "HEAD_RETRIEVAL", "HEAD_STREAMING", "KV_BF16", "KV_FP8_E4M3", "KV_INT4",
        "KV_MIXED"}
