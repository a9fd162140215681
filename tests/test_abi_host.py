"""CPU-side checks of the C ABI: the library builds, loads and exports every
symbol include/spec_attn.h declares, and host-side validation rejects bad
problems before touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_attn.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return sa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(spec_attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_symbols():
    assert sorted(sa.EXPORTED_SYMBOLS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sa.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    assert sa.spec_attn_version() == 100
    for st in (0, -1, -2, -3, -4, -5):
        assert sa.status_string(st) and sa.status_string(st) != "unknown status"
    assert sa.status_string(12345) == "unknown status"


def _problem(**over):
    base = dict(num_reqs=1, total_q_rows=4, max_w=4, num_q_heads=4, num_kv_heads=1, head_dim=64,
                page_size=16, num_pages=17, block_table_stride=17, mask_mode=0, kv_dtype=0,
                sm_scale=0.0, max_seq_len=260, force_splits=0, kernel_variant=0)
    base.update(over)
    return base


@pytest.mark.parametrize("over,status", [
    (dict(max_w=17), sa.SPEC_ATTN_E_UNSUPPORTED),            # W > 16 fails loudly
    (dict(head_dim=96), sa.SPEC_ATTN_E_UNSUPPORTED),
    (dict(page_size=48), sa.SPEC_ATTN_E_UNSUPPORTED),
    (dict(page_size=128), sa.SPEC_ATTN_E_UNSUPPORTED),
    (dict(window_left=-1), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(window_left=8, mask_mode=1), sa.SPEC_ATTN_E_INVALID_ARG),         # the window is causal-only
    (dict(kv_page_stride=1024), sa.SPEC_ATTN_E_INVALID_ARG),                # below the dense page (2048 B)
    (dict(kv_page_stride=2056), sa.SPEC_ATTN_E_INVALID_ARG),                # not a multiple of 16
    (dict(kv_dtype=1, scale_page_stride=32), sa.SPEC_ATTN_E_INVALID_ARG),   # below 16 keys x 4 scale bytes
    (dict(kv_dtype=1, kv_page_stride=520), sa.SPEC_ATTN_E_INVALID_ARG),     # codes: dense 512 B, not x16
    (dict(dense_block_kv=2), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(dense_block_kv=1, w_invariant=1), sa.SPEC_ATTN_E_INVALID_ARG),     # exactness is a cache-only rule
    (dict(dense_block_kv=1, kv_dtype=1), sa.SPEC_ATTN_E_UNSUPPORTED),       # the block operand is bf16
    (dict(early_metadata=2), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(early_context_kv=2, early_metadata=1), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(early_context_kv=1), sa.SPEC_ATTN_E_INVALID_ARG),                 # needs early_metadata
    (dict(test_stall=1), sa.SPEC_ATTN_E_INVALID_ARG),                       # the stall hook needs TCGEN05
    (dict(num_q_heads=34, num_kv_heads=2), sa.SPEC_ATTN_E_UNSUPPORTED),  # group 17
    (dict(num_q_heads=6, num_kv_heads=4), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(max_w=0), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(mask_mode=2), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(kv_dtype=3), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(block_table_stride=16), sa.SPEC_ATTN_E_INVALID_ARG),  # 260 keys need 17 pages
    (dict(block_table_stride=2 ** 26, page_size=64), sa.SPEC_ATTN_E_UNSUPPORTED),   # 2^32 keys a row
    (dict(max_seq_len=2 ** 31), sa.SPEC_ATTN_E_UNSUPPORTED),
    (dict(sm_scale=-1.0), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(kernel_variant=7), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(num_reqs=-1), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(w_invariant=2), sa.SPEC_ATTN_E_INVALID_ARG),
    (dict(w_invariant=1, fixed_keys_per_split=100), sa.SPEC_ATTN_E_INVALID_ARG),   # not a multiple of 64
    (dict(w_invariant=1, fixed_keys_per_split=-64), sa.SPEC_ATTN_E_INVALID_ARG),
])
def test_plan_rejects_bad_problems_on_the_host(lib, over, status):
    pr = sa.spec_attn_problem(**_problem(**over))
    handle = ctypes.c_void_p()
    st = lib.spec_attn_plan_create(ctypes.byref(pr), None, None, ctypes.byref(handle), None)
    assert st == status
    assert not handle.value


def test_plan_checks_host_windows_and_lengths(lib):
    import numpy as np
    pr = sa.spec_attn_problem(**_problem(num_reqs=2, total_q_rows=8))
    handle = ctypes.c_void_p()
    qi = np.array([0, 4, 21], dtype=np.int32)   # second window 17 rows
    st = lib.spec_attn_plan_create(ctypes.byref(pr), None, qi.ctypes.data_as(ctypes.c_void_p),
                                   ctypes.byref(handle), None)
    assert st == sa.SPEC_ATTN_E_UNSUPPORTED
    qi = np.array([0, 4, 8], dtype=np.int32)
    sl = np.array([260, 3], dtype=np.int32)     # seq_len below its window
    st = lib.spec_attn_plan_create(ctypes.byref(pr), sl.ctypes.data_as(ctypes.c_void_p),
                                   qi.ctypes.data_as(ctypes.c_void_p), ctypes.byref(handle), None)
    assert st == sa.SPEC_ATTN_E_INVALID_ARG
    sl = np.array([261, 100], dtype=np.int32)   # above max_seq_len
    st = lib.spec_attn_plan_create(ctypes.byref(pr), sl.ctypes.data_as(ctypes.c_void_p),
                                   qi.ctypes.data_as(ctypes.c_void_p), ctypes.byref(handle), None)
    assert st == sa.SPEC_ATTN_E_INVALID_ARG


def test_null_arguments(lib):
    assert lib.spec_attn_plan_create(None, None, None, None, None) == sa.SPEC_ATTN_E_INVALID_ARG
    assert lib.spec_attn_plan_get_info(None, None) == sa.SPEC_ATTN_E_INVALID_ARG
    assert lib.spec_attn_reset_device_status(None, None) == sa.SPEC_ATTN_E_INVALID_ARG
    assert lib.spec_attn_check_device_status(None, None, None) == sa.SPEC_ATTN_E_INVALID_ARG
    assert lib.spec_attn_append_kv(*([None] * 7), ctypes.c_float(1.0), ctypes.c_float(1.0),
                                   *([None] * 4), 0, None) == sa.SPEC_ATTN_E_INVALID_ARG
    assert lib.spec_attn_run_append(*([None] * 8), ctypes.c_float(1.0), ctypes.c_float(1.0),
                                    *([None] * 6), 0, None) == sa.SPEC_ATTN_E_INVALID_ARG
    assert lib.spec_attn_run_dense_block(*([None] * 13), 0, None) == sa.SPEC_ATTN_E_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        sa.load_library(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("cstruct,pystruct", [("spec_attn_problem", sa.spec_attn_problem),
                                              ("spec_attn_plan_info", sa.spec_attn_plan_info)])
def test_binding_structs_match_the_header_layout(tmp_path, cstruct, pystruct):
    """The ctypes mirrors of the header's structs have the C compiler's size
    and every field at the C compiler's offset (a field added to one side
    only, or in another order, fails here)."""
    names = [f[0] for f in pystruct._fields_]
    lines = [f'printf("size %zu\\n", sizeof({cstruct}));']
    lines += [f'printf("{n} %zu\\n", offsetof({cstruct}, {n}));' for n in names]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "spec_attn.h"\nint main(void) {\n    '
                   + "\n    ".join(lines) + "\n    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(pystruct)
    for n in names:
        assert int(out[n]) == getattr(pystruct, n).offset, n
    # and the C struct has no field the binding lacks
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct " + cstruct + r"\s*\{(.*?)\}\s*" + cstruct + ";", text, flags=re.S).group(1)
    c_fields = []
    for stmt in body.split(";"):
        if stmt.strip():   # "<type> a" or "<type> a, b, c" (the header's types are one word)
            c_fields += [d.strip() for d in stmt.split(None, 1)[1].split(",")]
    assert c_fields == names


def _header_prototypes():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\*?\s+\*?(spec_attn_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M | re.S):
        params = [p.strip() for p in m.group(2).split(",")]
        protos[m.group(1)] = [] if params == ["void"] else params
    return protos


def _kind(param):
    """Argument class of a C parameter: pointer, size_t, 32-bit int or float."""
    if "*" in param or param.startswith("spec_attn_stream_t"):
        return "ptr"
    t = param.split()[0]
    return {"size_t": "size", "int": "i32", "int32_t": "i32", "uint32_t": "i32", "float": "f32"}[t]


def _ctypes_kind(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    return {ctypes.c_size_t: "size", ctypes.c_int32: "i32", ctypes.c_uint32: "i32", ctypes.c_float: "f32"}[t]


def test_binding_argtypes_match_the_header_prototypes(lib):
    """Every entry point's ctypes argtypes have the header's parameter count and,
    position by position, its argument class (a missing or extra pointer
    shifts every later argument: caught here, without a GPU)."""
    protos = _header_prototypes()
    assert sorted(protos) == declared_functions()
    for name, params in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert [_kind(p) for p in params] == [_ctypes_kind(t) for t in fn.argtypes], name
