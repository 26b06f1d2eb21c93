"""The C ABI library loads and exports every entry point include/treespec.h declares (no GPU needed).

Also checks host-side argument validation, which runs before any CUDA call,
and that the C structs match their ctypes mirrors in size.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treespec.h")
PKG = os.path.join(ROOT, "speculative_decoding_tree_forward_gb300")
LIB = os.path.join(PKG, "libtreespec.so")


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(LIB)


def _declared():
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^TS_API\s+[\w\s\*]+?\b(\w+)\(", text, flags=re.M)


def setup_module(module):
    if not os.path.exists(LIB):
        import importlib.util
        spec = importlib.util.spec_from_file_location("ts_build", os.path.join(PKG, "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


def test_header_declares_the_boundary():
    names = set(_declared())
    for required in ("tree_attn_forward", "tree_attn_workspace_size", "tree_accept_greedy", "tree_cache_compact",
                     "ts_status_string", "ts_read_device_error", "tree_build_mask"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_symbol():
    with open(os.path.join(PKG, "__init__.py")) as f:
        src = f.read()
    for n in _declared():
        assert f'"{n}"' in src, n


def test_status_strings(lib):
    lib.ts_status_string.restype = ctypes.c_char_p
    for code in range(5):
        assert lib.ts_status_string(code).startswith(b"TS_")
    assert lib.ts_version() >= 1


def test_host_validation_without_gpu(lib):
    lib.tree_attn_workspace_size.restype = ctypes.c_size_t
    lib.tree_attn_forward.restype = ctypes.c_int
    assert lib.tree_attn_workspace_size(None) == 0
    assert lib.tree_attn_forward(None, None, 0, None) == 1          # TS_ERR_INVALID_ARG
    lib.tree_accept_greedy.restype = ctypes.c_int
    assert lib.tree_accept_greedy(None, None, 0, None) == 1
    lib.tree_cache_compact.restype = ctypes.c_int
    assert lib.tree_cache_compact(None, None, 0, None) == 1
    lib.ts_read_device_error.restype = ctypes.c_int
    assert lib.ts_read_device_error(None, None, 0, None) == 1


def test_struct_layouts_match_header():
    """Every field of every ctypes mirror sits at the offset the C declaration
    gives it, and every struct has the C size (checked by compiling the header)."""
    import subprocess
    import tempfile
    import torch  # noqa: F401
    import speculative_decoding_tree_forward_gb300 as ts
    mirrors = {"ts_attn_args": ts.AttnArgs, "ts_accept_args": ts.AcceptArgs, "ts_compact_args": ts.CompactArgs,
               "ts_sample_args": ts.SampleArgs, "ts_expand_args": ts.ExpandArgs, "ts_select_args": ts.SelectArgs}
    lines, expect = [], []
    for cname, py in mirrors.items():
        lines.append(f'  printf("%zu\\n", sizeof({cname}));')
        expect.append(ctypes.sizeof(py))
        for field, _ in py._fields_:
            lines.append(f'  printf("%zu\\n", offsetof({cname}, {field}));')
            expect.append(getattr(py, field).offset)
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"treespec.h\"\nint main(void) {\n" + "\n".join(lines) + \
          "\n  return 0;\n}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        with open(c, "w") as f:
            f.write(src)
        r = subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe],
                           capture_output=True, text=True)
        if r.returncode != 0:
            pytest.skip("no C compiler: " + r.stderr[:200])
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True).stdout.split()]
    assert got == expect


def test_empty_batches_and_null_arguments_are_rejected_on_the_host(lib):
    """Validation happens before any CUDA call: an empty batch or a null
    pointer returns TS_ERR_INVALID_ARG with no GPU present."""
    import torch  # noqa: F401
    import speculative_decoding_tree_forward_gb300 as ts
    for name in ("tree_accept_sample", "tree_expand", "tree_select_subtree"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        assert f(None, None, 0, None) == 1, name
    for name in ("tree_accept_sample_workspace_size", "tree_expand_workspace_size", "tree_select_workspace_size",
                 "tree_accept_workspace_size", "tree_compact_workspace_size"):
        f = getattr(lib, name)
        f.restype = ctypes.c_size_t
        assert f(None) == 0, name
    lib.tree_build_mask.restype = ctypes.c_int
    assert lib.tree_build_mask(None, None, 1, 16, None, None, None, 0, None) == 1
    a = ts.AttnArgs(num_requests=0, num_q_heads=8, num_kv_heads=2, head_dim=64, n_tree_max=16, n_query=16,
                    max_kv_len=256)
    assert lib.tree_attn_forward(ctypes.byref(a), None, 0, None) == 1
    assert lib.tree_attn_workspace_size(ctypes.byref(a)) == 0
    acc = ts.AcceptArgs(num_requests=0, n_tree_max=16, vocab=100)
    assert lib.tree_accept_greedy(ctypes.byref(acc), None, 0, None) == 1
    cmp_ = ts.CompactArgs(num_requests=0, n_tree_max=16, num_layers=1, num_kv_heads=2, head_dim=64, elem_bytes=2)
    assert lib.tree_cache_compact(ctypes.byref(cmp_), None, 0, None) == 1
