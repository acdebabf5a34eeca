"""moe_route_layout_noalloc, the layout entry point for callers that cannot
allocate device memory (for example a plugin inside a framework whose memory
pool owns the whole device, or a latency-critical path that must not hit the
device-wide synchronisation a cudaMalloc can cause): its scratch is a fixed
array inside the library, so the caller passes only inputs and outputs.

Checked through the C ABI against moe_route_layout (which takes a caller
workspace) on two calls in a row, with a different shape between them so that
anything left in the shared array by the previous call would show up.  The
layout tables are integer data: the comparison is bit-exact.  This file is
collected last and builds the library itself, so it runs the same alone in a
fresh process or after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import combine_counting_sort_gb300 as moe
import oracle
from combine_counting_sort_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from combine_counting_sort_gb300 import _build
    _build.build()
    moe.lib()


def routed(cfg):
    logits = inputs.make_logits(cfg.T, cfg.E, cfg.zipf, cfg.seed).numpy()
    ids, w = oracle.router_topk(logits, cfg.k)
    return torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()


def layout_with_workspace(cfg, ids, w):
    L = moe.Layout(cfg.T, cfg.k, cfg.E, cfg.G)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_route_layout(ids, w, L, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return L.numpy()


def layout_noalloc_via_abi(cfg, ids, w):
    """Call the C entry point directly (ctypes), tables poisoned beforehand."""
    L = moe.Layout(cfg.T, cfg.k, cfg.E, cfg.G)
    for t in L.t.values():
        t.fill_(-3)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_route_layout_noalloc(
        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.byref(L.c),
        ctypes.c_void_p(st.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == moe.MOE_OK, moe.status_string(rc)
    torch.cuda.synchronize()
    assert st.item() == 0, moe.status_string(st.item())
    return L.numpy()


def assert_same(got, want):
    for name in want:
        assert np.array_equal(got[name].view(np.uint32), want[name].view(np.uint32)), name


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    big = inputs.CONFIGS["t8192_zipf1.2"]
    small = inputs.CONFIGS["tiny"]
    ids_b, w_b = routed(big)
    ids_s, w_s = routed(small)
    want_b = layout_with_workspace(big, ids_b, w_b)
    want_s = layout_with_workspace(small, ids_s, w_s)
    # call 1: the large skewed workload; call 2: a different, small shape
    assert_same(layout_noalloc_via_abi(big, ids_b, w_b), want_b)
    assert_same(layout_noalloc_via_abi(small, ids_s, w_s), want_s)
    # and again in the other order: the array keeps the last call's contents
    assert_same(layout_noalloc_via_abi(big, ids_b, w_b), want_b)
    assert_same(layout_noalloc_via_abi(big, ids_b, w_b), want_b)


def test_noalloc_rejects_more_experts_than_its_scratch_holds():
    T, k, E, G = 64, 4, 512, 4
    L = moe.Layout(T, k, E, G)
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T, k, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_route_layout_noalloc(
        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.byref(L.c),
        ctypes.c_void_p(st.data_ptr()), None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
