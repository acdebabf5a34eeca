"""The C ABI loads without a GPU, exports every entry point include/moe.h
declares, and the binding's ctypes structs match the header's layout.  No
compute call runs here (only the host-side sizing and argument checks)."""
import ctypes
import os
import re
import subprocess

import pytest

import combine_counting_sort_gb300 as moe
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from combine_counting_sort_gb300 import _build
    _build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|void)\s+(moe_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(names) == set(moe.EXPORTS)


def test_status_strings(lib):
    assert moe.status_string(0) == "MOE_OK"
    assert moe.status_string(5) == "MOE_ERR_TIMEOUT"
    assert moe.status_string(99) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("T,k,E,G", [(128, 2, 8, 2), (2048, 8, 256, 8), (8192, 8, 256, 8), (1, 1, 1, 1),
                                     (16384, 8, 256, 8), (1000, 32, 1024, 4)])
def test_layout_sizes_match_oracle_capacity(lib, T, k, E, G):
    s = moe.moe_layout_sizes(T, k, E, G)
    assert s.pairs == T * k
    assert s.max_tiles == oracle.max_tiles(T, k, E, 128)
    assert s.rowmap_len == s.max_tiles * 128
    assert s.layout_ws_bytes > 0 and s.stage1_ws_bytes > 0


@pytest.mark.parametrize("args", [(0, 2, 8, 2), (128, 0, 8, 2), (128, 9, 8, 2), (128, 2, 8, 3),
                                  (128, 2, 2048, 2), (128, 2, 8, 2, 64), (1 << 21, 1, 8, 1), (128, 33, 64, 1)])
def test_layout_sizes_rejects_bad_shapes(lib, args):
    out = moe.LayoutSizes()
    T, k, E, G = args[:4]
    bm = args[4] if len(args) > 4 else 128
    assert lib.moe_layout_sizes(T, k, E, G, bm, ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG


def test_null_arguments_are_rejected_on_host(lib):
    # every compute entry point checks its pointers before touching the device
    L = moe.LayoutC()
    assert lib.moe_route_layout(None, None, ctypes.byref(L), None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_quant(None, 256, ctypes.byref(L), None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_gemm1(None, None, None, None, 512, 256, ctypes.byref(L), None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, 256, ctypes.byref(L), None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_router_topk(None, 4, 8, 2, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_weights(None, 1, 128, 128, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dequant_rows(None, None, 256, ctypes.byref(L), None, None) == moe.MOE_ERR_INVALID_ARG
    opts = moe.stage1_opts()
    assert lib.moe_stage1(None, 256, ctypes.byref(L), None, None, 512, ctypes.byref(opts), None, None, None,
                          None, 0, None, None) == moe.MOE_ERR_INVALID_ARG


PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "moe.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(moe_layout_t), offsetof(moe_layout_t, count),
         offsetof(moe_layout_t, token_order), sizeof(moe_layout_sizes_t), sizeof(moe_stage1_opts_t),
         offsetof(moe_stage1_opts_t, timeout_ns));
  return 0;
}
"""


def test_ctypes_structs_match_header(tmp_path):
    src = tmp_path / "probe.c"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(moe.LayoutC), moe.LayoutC.count.offset, moe.LayoutC.token_order.offset,
            ctypes.sizeof(moe.LayoutSizes), ctypes.sizeof(moe.Stage1Opts), moe.Stage1Opts.timeout_ns.offset]
    assert got == want
