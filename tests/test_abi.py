"""The C-ABI library builds and exports every function include/hs.h declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

import dsa_sparse_mla_gb300 as hs
from dsa_sparse_mla_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "hs.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:hs_status|int|const char\*)\s+(hs_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("hs_indexer_scores", "hs_topk", "hs_sparse_mla_fwd", "hs_hisparse_resolve", "hs_indexer_topk"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert hs.hs_abi_version() == 7
    hs.load()
    for code, name in enumerate(["HS_OK", "HS_ERR_INVALID", "HS_ERR_UNSUPPORTED", "HS_ERR_CUDA",
                                 "HS_ERR_DEVICE_FLAG", "HS_ERR_TIMEOUT"]):
        assert hs.load().hs_status_str(code).decode() == name


def test_invalid_arguments_rejected_before_any_device_work(lib):
    """Host-side checks fail with HS_ERR_INVALID and a message, without touching a GPU."""
    L = hs.load()
    st = L.hs_topk(None, 10, None, 1, 0, None, None, None)          # k = 0
    assert st == 1 and b"k must be" in L.hs_last_error()
    a = hs._IndexerArgs()
    a.T, a.B, a.Hi, a.Di = 4, 1, 12, 128                              # Hi = 12
    assert L.hs_indexer_scores(ctypes.byref(a), None) == 1 and b"Hi" in L.hs_last_error()
    assert L.hs_indexer_topk(ctypes.byref(a), 2048, None, None) == 1 and b"Hi" in L.hs_last_error()
    a.Hi = 64
    assert L.hs_indexer_topk(ctypes.byref(a), 0, None, None) == 1 and b"k must be" in L.hs_last_error()
    m = hs._MlaArgs()
    m.T, m.H, m.k = 1, 0, 1
    assert L.hs_sparse_mla_fwd(ctypes.byref(m), None) == 1
    m.H, m.err_flag, m.q, m.kv_pool, m.idx, m.out, m.R = 1, 16, 16, 16, 16, 16, 1
    m.idx_row, m.idx_rows = 16, 0                                     # shared rows, but none
    assert L.hs_sparse_mla_fwd(ctypes.byref(m), None) == 1 and b"idx_rows" in L.hs_last_error()
    m.idx_row, m.token_kvlen = None, 16                               # a causal limit without a block table
    assert L.hs_sparse_mla_fwd(ctypes.byref(m), None) == 1 and b"token_kvlen needs" in L.hs_last_error()
    m.token_kvlen, m.R = None, 2 ** 31                                # the gather keeps rows as int32
    assert L.hs_sparse_mla_fwd(ctypes.byref(m), None) == 1 and b"R must be" in L.hs_last_error()
    m.R = 1
    n = ctypes.c_uint64(0)
    assert L.hs_sparse_mla_workspace_size(0, ctypes.byref(n)) == 1 and b"H must be" in L.hs_last_error()
    r = hs._ResolveArgs()
    r.B, r.k, r.S, r.step = 1, 9, 8, 0                                # k > S
    assert L.hs_hisparse_resolve(ctypes.byref(r), None) == 1
    r.k, r.S = 8, 9000                                                # S too large
    assert L.hs_hisparse_resolve(ctypes.byref(r), None) == 1
    ap = hs._AppendArgs()
    ap.T, ap.B = 4, 1
    ap.err_flag = 16
    assert L.hs_kv_append(ctypes.byref(ap), None) == 1 and b"nothing to append" in L.hs_last_error()
    ap.index_key, ap.Di = 16, 32
    ap.token_req, ap.token_pos, ap.block_table, ap.bt_stride = 16, 16, 16, 1
    assert L.hs_kv_append(ctypes.byref(ap), None) == 1 and b"Di must be" in L.hs_last_error()
    oa = hs._OffloadArgs()
    oa.n, oa.L, oa.B, oa.err_flag = 3, 1, 1, 16
    assert L.hs_kv_offload(ctypes.byref(oa), None) == 1 and b"NULL" in L.hs_last_error()
    assert L.hs_hisparse_touch_host(-1, None, None, None, None, None) == 1
    assert L.hs_hisparse_touch_host(2, None, None, None, ctypes.c_void_p(16), None) == 1
    assert b"NULL" in L.hs_last_error()


def test_calls_without_library_fail_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(hs, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(hs, "_lib", None)
    with pytest.raises(hs.HSError):
        hs.load()


_STRUCTS = {"hs_indexer_args": "_IndexerArgs", "hs_mla_args": "_MlaArgs", "hs_resolve_args": "_ResolveArgs",
            "hs_kv_append_args": "_AppendArgs", "hs_kv_offload_args": "_OffloadArgs"}


def _struct_fields(text, name):
    """Field names of `typedef struct { ... } name;` in declaration order."""
    m = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + r"\s*;", text)
    assert m, name
    body = re.sub(r"/\*.*?\*/", "", m.group(1), flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "const int32_t* a, *b" / "int32_t T, H, k" -> names after the type
        first, *rest = [d.strip() for d in decl.split(",")]
        fields.append(re.findall(r"(\w+)\s*$", first)[0])
        fields += [re.findall(r"(\w+)\s*$", r)[0] for r in rest]
    return fields


def test_argument_structs_match_the_binding(tmp_path):
    """Every args struct of include/hs.h has the binding's field names, order, offsets and size
    (offsets from the C compiler itself)."""
    import subprocess
    with open(os.path.join(ROOT, "include", "hs.h")) as f:
        text = f.read()
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "hs.h"', "int main(void) {"]
    fields = {}
    for cname in _STRUCTS:
        fields[cname] = _struct_fields(text, cname)
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for fld in fields[cname]:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, fld, cname, fld))
    lines += ["return 0;", "}"]
    src, exe = tmp_path / "layout.c", tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for ln in out:
        if ln:
            parts = ln.split()
            got[(parts[0], parts[1])] = int(parts[2])
    for cname, pyname in _STRUCTS.items():
        cls = getattr(hs, pyname)
        assert [f[0] for f in cls._fields_] == fields[cname], cname
        assert ctypes.sizeof(cls) == got[(cname, "size")], cname
        for fld in fields[cname]:
            assert getattr(cls, fld).offset == got[(cname, fld)], (cname, fld)
