"""The C-ABI library builds, loads and exports every symbol its header declares, and the binding
agrees with every declared signature (CPU only)."""
import ctypes
import os
import re

import pytest

from tests.helpers import ROOT

HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from moe_expert_offload_router_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("moe_router_topk", "moe_slot_ensure", "moe_copy_missing", "moe_expert_forward",
              "moe_ladder_classify", "moe_group_pairs", "moe_cache_create"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls(lib):
    lib.moe_fp4_expert_bytes.restype = ctypes.c_size_t
    lib.moe_int2_expert_bytes.restype = ctypes.c_size_t
    lib.moe_fp8_expert_bytes.restype = ctypes.c_size_t
    assert lib.moe_fp4_expert_bytes(4096, 2048) == 13369344
    assert lib.moe_int2_expert_bytes(4096, 2048) == 7077888
    assert lib.moe_fp8_expert_bytes(4096, 2048) == 25198592
    assert lib.moe_fp4_expert_bytes(4096, 2047) == 0
    assert lib.moe_version() >= 1


def test_binding_names_match_header(lib):
    from moe_expert_offload_router_gb300 import _lib as L
    for n in _declared():
        if n in ("moe_cache_create", "moe_cache_destroy", "moe_cache_reset", "moe_cache_state",
                 "moe_cache_export", "moe_cache_import", "moe_last_error"):
            continue   # wrapped by the moe_cache class / error path
        assert hasattr(L, n), n


def test_oracle_not_imported_by_product_code():
    pkg = os.path.join(ROOT, "moe_expert_offload_router_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f


def _prototypes():
    """(return type, name, [parameter types]) of every function the header declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = []
    for ret, name, params in re.findall(r"([A-Za-z_][A-Za-z0-9_ \*]*?)\b(moe_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;",
                                        src, flags=re.S):
        ps = [" ".join(p.split()) for p in params.split(",")]
        ps = [] if ps == ["void"] else [re.sub(r"\s*\b[A-Za-z_][A-Za-z0-9_]*$", "", p) if not p.endswith("*")
                                        else p for p in ps]
        out.append((" ".join(ret.split()), name, ps))
    return out


def _c_class(t):
    """The ctypes class a C parameter or return type of the header must be bound as."""
    t = t.replace("const ", "").strip()
    if t.endswith("*") or t in ("cudaStream_t", "cudaEvent_t"):
        return "pointer"
    return {"int": ctypes.c_int, "int32_t": ctypes.c_int, "moe_status": ctypes.c_int,
            "size_t": ctypes.c_size_t, "uint64_t": ctypes.c_uint64, "int64_t": ctypes.c_int64,
            "float": ctypes.c_float, "double": ctypes.c_double}[t]


def _is_pointer(ct):
    return ct in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(ct, type) and issubclass(ct, ctypes._Pointer))


def test_binding_signatures_match_header(lib):
    # a parameter added, dropped or retyped on one side only is undefined
    # behaviour at the call: every declared function's binding must agree in
    # arity and in the class of every parameter and of the result
    from moe_expert_offload_router_gb300 import _lib as L
    protos = _prototypes()
    assert len(protos) == len(_declared())
    for ret, name, params in protos:
        assert name in L._SIGS, name
        res, args = L._SIGS[name]
        assert len(args) == len(params), (name, params, args)
        for p, a in zip(params, args):
            want = _c_class(p)
            if want == "pointer":
                assert _is_pointer(a), (name, p, a)
            else:
                assert a is want or ctypes.sizeof(a) == ctypes.sizeof(want) and a._type_ == want._type_, \
                    (name, p, a)
        want = _c_class(ret)
        if want == "pointer":
            assert _is_pointer(res), (name, ret, res)
        else:
            assert res is want or ctypes.sizeof(res) == ctypes.sizeof(want), (name, ret, res)


def test_views_struct_matches_header(lib):
    # moe_expert_views crosses the boundary by pointer: field order, types and
    # offsets of the ctypes mirror must be the header's
    from moe_expert_offload_router_gb300 import _lib as L
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef\s+struct\s*\w*\s*\{([^}]*)\}\s*moe_expert_views\s*;", src, flags=re.S).group(1)
    fields = []
    for decl in body.split(";"):
        decl = " ".join(decl.split())
        if decl:   # "int H, I" declares two fields of the base type
            first, *more = decl.split(",")
            typ, name = re.match(r"(.*?)\s*\b([A-Za-z_][A-Za-z0-9_]*)$", first.strip()).groups()
            fields.append((name, typ))
            base = typ.rstrip("* ")
            for d in more:
                d = d.strip()
                fields.append((d.lstrip("* "), base + "*" * d.count("*")))
    mirror = L.moe_expert_views._fields_
    assert [n for n, _ in fields] == [n for n, _ in mirror]
    for (name, typ), (_, ct) in zip(fields, mirror):
        want = _c_class(typ)
        if want == "pointer":
            assert _is_pointer(ct), (name, typ, ct)
        else:
            assert ct is want, (name, typ, ct)


def test_header_comments_name_only_defined_constants():
    # a status or constant named in the documentation must exist in the header
    src = open(HEADER).read()
    comments = " ".join(re.findall(r"/\*.*?\*/", src, flags=re.S))
    code = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    used = set(re.findall(r"\bMOE_[A-Z0-9_]+\b", comments))
    defined = set(re.findall(r"#define\s+(MOE_[A-Z0-9_]+)", code)) | \
        set(re.findall(r"\b(MOE_[A-Z0-9_]+)\s*(?:=|,|\})", code))
    assert used and not used - defined, sorted(used - defined)


def _header_constants():
    code = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    vals = {}
    for body in re.findall(r"enum\s*\w*\s*\{([^}]*)\}", code, flags=re.S):
        cur = -1
        for item in (i.strip() for i in body.split(",")):
            if item:
                name, expr = re.match(r"(MOE_[A-Z0-9_]+)\s*(?:=\s*(.+))?$", item).groups()
                cur = int(eval(expr, {}, dict(vals))) if expr else cur + 1
                vals[name] = cur
    for m in re.finditer(r"#define\s+(MOE_[A-Z0-9_]+)\s+\(?(-?\d+)\)?", code):
        vals[m.group(1)] = int(m.group(2))
    return vals


def test_binding_constants_match_header(lib):
    from moe_expert_offload_router_gb300 import _lib as L
    vals = _header_constants()
    assert len(vals) > 20
    for name, v in vals.items():
        assert hasattr(L, name), name
        assert getattr(L, name) == v, (name, getattr(L, name), v)
    assert L.KERNEL_NAMES and len(L.KERNEL_NAMES) == vals["MOE_K_COUNT"]


def test_plain_c_program_uses_the_header(tmp_path):
    # the boundary is a C ABI: a C99 program compiled by gcc against the header
    # links against the library and gets the declared results from the calls
    # that need no GPU
    import shutil
    import subprocess
    from moe_expert_offload_router_gb300 import build
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    so = build.build()
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    exe = str(tmp_path / "abi_consumer")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), "-isystem", cuda_inc,
                    os.path.join(ROOT, "tests", "c", "abi_consumer.c"), "-o", exe,
                    "-L", os.path.dirname(so), "-l:" + os.path.basename(so),
                    "-Wl,-rpath," + os.path.dirname(so)], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
