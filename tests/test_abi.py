"""The C ABI loads without a GPU, exports every entry point include/moe.h
declares, and the binding's ctypes structs match the header's layout.  No
compute call runs here (only the host-side sizing and argument checks)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

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


def test_binding_refuses_wrong_shapes_before_any_device_call(lib):
    # The C entry points take bare pointers; the binding checks every tensor's
    # shape against the layout and the other operands first (CPU tensors here:
    # a shape error comes before the device check, a right shape reaches it).
    T, k, E, G, H, N = 40, 2, 8, 2, 256, 512
    R = T * k
    L = moe.Layout(T, k, E, G, device="cpu")
    st = torch.zeros(1, dtype=torch.int32)
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    x = torch.zeros(T, H, dtype=bf)
    A, As = torch.zeros(R, H, dtype=u8), torch.zeros(H // 128, R, dtype=f32)
    W, Ws = torch.zeros(E, N, H, dtype=u8), torch.zeros(E, N // 128, H // 128, dtype=f32)
    Y, out = torch.zeros(R, N, dtype=bf), torch.zeros(T, N, dtype=bf)
    bad = [
        lambda: moe.moe_route_layout(torch.zeros(T, k + 1, dtype=torch.int32), torch.zeros(T, k), L, st),
        lambda: moe.moe_route_layout_noalloc(torch.zeros(T, k, dtype=torch.int32), torch.zeros(T - 1, k), L, st),
        lambda: moe.moe_dispatch_quant(torch.zeros(T + 1, H, dtype=bf), L, A, As, st),
        lambda: moe.moe_dispatch_quant(x, L, A[:-1], As, st),
        lambda: moe.moe_dispatch_quant(x, L, A, As[:, :-1], st),
        lambda: moe.moe_grouped_gemm1(A, As, W[:-1], Ws[:-1], L, Y, st),
        lambda: moe.moe_grouped_gemm1(A, As, W, Ws[:, :-1], L, Y, st),
        lambda: moe.moe_grouped_gemm1(A, As, W, Ws, L, Y[:-1], st),
        lambda: moe.moe_combine(Y, L, out[:-1], st),
        lambda: moe.moe_combine(Y[:-1], L, out, st),
        lambda: moe.moe_stage1(x, L, W, Ws, A, As, Y[:, :-128], torch.zeros(16, dtype=u8), st),
        lambda: moe.moe_router_topk(torch.zeros(T, E), k, torch.zeros(T, k + 1, dtype=torch.int32),
                                    torch.zeros(T, k + 1)),
        lambda: moe.moe_quant_weights(torch.zeros(E, N, H, dtype=bf), W[:, :-1], Ws),
        lambda: moe.moe_dequant_rows(A, As, L, torch.zeros(R, H + 128, dtype=bf)),
        lambda: moe.moe_combine(Y, L, out, torch.zeros(0, dtype=torch.int32)),
    ]
    for call in bad:
        with pytest.raises(ValueError, match="shape|dimensions|status"):
            call()
    # right shapes pass the shape checks and stop at the device check
    with pytest.raises(ValueError, match="CUDA tensor"):
        moe.moe_grouped_gemm1(A, As, W, Ws, L, Y, st)
    with pytest.raises(ValueError, match="CUDA tensor"):
        moe.moe_combine(Y, L, out, st)
