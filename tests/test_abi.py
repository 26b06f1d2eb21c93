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
    """Field order/size of the ctypes mirrors equals the C declarations (checked by compiling the header)."""
    import subprocess
    import tempfile
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "treespec.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(ts_attn_args), offsetof(ts_attn_args, num_ctas),
         sizeof(ts_accept_args), offsetof(ts_accept_args, verified_len),
         sizeof(ts_compact_args), offsetof(ts_compact_args, src_rows));
  return 0;
}
'''
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
    import torch  # noqa: F401
    import speculative_decoding_tree_forward_gb300 as ts
    assert got == [ctypes.sizeof(ts.AttnArgs), ts.AttnArgs.num_ctas.offset, ctypes.sizeof(ts.AcceptArgs),
                   ts.AcceptArgs.verified_len.offset, ctypes.sizeof(ts.CompactArgs), ts.CompactArgs.src_rows.offset]
