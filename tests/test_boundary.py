"""The C-ABI library loads and exports every symbol include/nt.h declares, and
rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "nt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:nt_status|const char\*|int)\s+(nt_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("nt_ctx_create", "nt_gemv_q", "nt_rmsnorm", "nt_rope", "nt_attn_decode", "nt_swiglu"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from block_quantized_gemv_nt_gb300 import nt
    lib = ctypes.CDLL(nt.library_path())
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_declared()) <= set(nt.EXPORTED)


def test_geometry_and_null_context():
    from block_quantized_gemv_nt_gb300 import nt
    assert [nt.nt_block_bytes(f) for f in range(7)] == [34, 18, 144, 176, 210, 64, 128]
    assert [nt.nt_block_elems(f) for f in range(7)] == [32, 32, 256, 256, 256, 32, 32]
    assert nt.nt_block_bytes(9) == 0
    L = nt.lib()
    assert L.nt_gemv_q(None, 0, None, None, None, 1, 32, None, None) == nt.NT_ERR_INVALID_ARG
    assert L.nt_ctx_sync(None) == nt.NT_ERR_INVALID_ARG
    assert L.nt_ctx_destroy(None) == nt.NT_ERR_INVALID_ARG


def test_no_gpu_context_fails_loudly():
    import torch
    from block_quantized_gemv_nt_gb300 import nt
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(nt.NtError):
        nt.Context(0)


def test_every_context_call_refuses_a_null_context():
    """Each entry point that takes a context checks it first: with a NULL
    context (and every other argument zero or NULL) it returns
    NT_ERR_INVALID_ARG without touching CUDA, so this runs without a GPU."""
    from block_quantized_gemv_nt_gb300 import nt
    no_ctx = {"nt_ctx_create", "nt_last_error", "nt_block_bytes", "nt_block_elems", "nt_attn_decode_static",
              "nt_layer_blob_layout", "nt_plan_residency", "nt_debug_stall_waits", "nt_debug_file_refuse_in_place"}
    L = nt.lib()
    checked = 0
    for name in nt.EXPORTED:
        if name in no_ctx:
            continue
        f = getattr(L, name)
        args = [0.0 if t is ctypes.c_float else (0 if t in (ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                                          ctypes.c_uint64, ctypes.c_size_t) else None)
                for t in f.argtypes]
        assert f(*args) == nt.NT_ERR_INVALID_ARG, name
        checked += 1
    assert checked >= 25


# the allocation-free attention: a form the pages have no counterpart for, so
# its comment says that instead of citing a passage
NO_PASSAGE = {"nt_attn_decode_static"}


def test_every_declaration_cites_a_passage():
    """Each entry point's comment in include/nt.h names the page passage it
    serves (one of the tags the header's preamble defines), except the ones
    the pages have no counterpart for, whose comment says so."""
    src = open(os.path.join(ROOT, "include", "nt.h")).read()
    decls = list(re.finditer(r"(/\*(?:(?!\*/).)*\*/)\s*((?:typedef[^;]*;\s*)?)(?:nt_status|const char\*|int)\s+(nt_\w+)\s*\(",
                             src, flags=re.S))
    missing = [m.group(3) for m in decls
               if m.group(3) not in NO_PASSAGE and not re.search(r"\[(about|code|feat|cache|road)\]", m.group(1))]
    assert not missing, missing
    for m in decls:
        if m.group(3) in NO_PASSAGE:
            assert "no counterpart" in m.group(1), m.group(3)


def _prototypes():
    """name -> (return type, [parameter types]) of every function nt.h declares."""
    src = open(os.path.join(ROOT, "include", "nt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    protos = {}
    for m in re.finditer(r"^\s*(nt_status|const char\*|int)\s+(nt_\w+)\s*\(([^;]*?)\)\s*;", src, flags=re.M | re.S):
        params = [p.strip() for p in " ".join(m.group(3).split()).split(",") if p.strip()]
        if params == ["void"]:
            params = []
        types = []
        for p in params:
            p = re.sub(r"\[\s*\d*\s*\]$", "*", p)              # an array parameter is a pointer
            p = re.sub(r"\s*\b\w+\s*(\*?)$", r"\1", p)        # drop the parameter's name
            types.append(" ".join(p.replace("*", " * ").split()))
        protos[m.group(2)] = (m.group(1), types)
    return protos


def _ctype_of(c_type: str):
    """The ctypes classes a C parameter type may be bound as."""
    if "*" in c_type:
        return "pointer"
    base = c_type.replace("const ", "").strip()
    return {"int": ctypes.c_int, "int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "uint64_t": ctypes.c_uint64,
            "size_t": ctypes.c_size_t, "float": ctypes.c_float}[base]


def test_binding_matches_header_prototypes():
    """The ctypes binding declares every entry point with the header's
    parameter count and types (pointers as pointers, each integer and float
    width as itself) and its return type: a mismatch would pass arguments
    in the wrong registers."""
    from block_quantized_gemv_nt_gb300 import nt
    lib = nt.lib()
    protos = _prototypes()
    assert set(protos) == set(_declared())
    for name, (ret, params) in protos.items():
        f = getattr(lib, name)
        assert f.argtypes is not None, name
        assert len(f.argtypes) == len(params), (name, params, f.argtypes)
        for c_type, py in zip(params, f.argtypes):
            want = _ctype_of(c_type)
            if want == "pointer":
                assert py in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(py, ctypes._Pointer), (name, c_type, py)
            else:
                assert py is want, (name, c_type, py)
        assert f.restype is (ctypes.c_char_p if ret == "const char*" else ctypes.c_int), name
