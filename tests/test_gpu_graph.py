"""The whole step (routing layout, fused stage1, combine) captured into one CUDA
graph and replayed gives the same bytes as the eager calls: the calls do no
host synchronisation and keep every count on the device."""
import numpy as np
import pytest
import torch

import combine_counting_sort_gb300 as moe
from combine_counting_sort_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.build()


def test_step_replays_from_a_cuda_graph():
    cfg = inputs.MoEConfig("graph", T=600, H=512, E=32, G=4, k=4, N=512, zipf=1.2, seed=12)
    ids, w = gu.routed(cfg)
    dev = "cuda"
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed).to(dev)
    ids_d, w_d = torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device=dev)
    Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device=dev)
    Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device=dev)
    moe.moe_quant_weights(W, Wq, Ws)
    R = cfg.T * cfg.k
    L = moe.Layout(cfg.T, cfg.k, cfg.E, cfg.G, device=dev)
    A = torch.empty(R, cfg.H, dtype=torch.uint8, device=dev)
    As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device=dev)
    Y = torch.empty(R, cfg.N, dtype=torch.bfloat16, device=dev)
    out = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(int(L.sizes.stage1_ws_bytes), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    opts = moe.stage1_opts(comm_sms=8)

    def step():
        moe.moe_route_layout(ids_d, w_d, L, status)
        moe.moe_stage1(x, L, Wq, Ws, A, As, Y, ws, status, opts)
        moe.moe_combine(Y, L, out, status)

    step()
    torch.cuda.synchronize()
    assert status.item() == 0
    want_out, want_y = out.clone(), Y.clone()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (out, Y):
        t.fill_(float("nan"))
    for t in L.t.values():
        t.fill_(-7)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(out.view(torch.int16), want_out.view(torch.int16))
    assert torch.equal(Y.view(torch.int16), want_y.view(torch.int16))


def test_variant_paths_replay_from_a_cuda_graph():
    # the no-plan layout, GEMM1 with the combine overlapped, the send runs with
    # the gathered GEMM1 and the MXFP8 dispatch + GEMM1, captured together into
    # one graph: replays give the eager bytes (the no-plan layout's order-free
    # tables; everything downstream is independent of its row order, so the
    # captured calls use the counting-sort layout)
    cfg = inputs.MoEConfig("graph2", T=300, H=512, E=16, G=4, k=4, N=512, zipf=1.1, seed=21)
    ids, w = gu.routed(cfg)
    dev = "cuda"
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed).to(dev)
    ids_d, w_d = torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device=dev)
    Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device=dev)
    Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device=dev)
    moe.moe_quant_weights(W, Wq, Ws)
    Wq_mx = torch.empty_like(Wq)
    W_sf = torch.empty(moe.mx_sf_w_shape(cfg.E, cfg.N, cfg.H), dtype=torch.uint8, device=dev)
    moe.moe_quant_weights_mx(W, Wq_mx, W_sf)
    R = cfg.T * cfg.k
    L = moe.Layout(cfg.T, cfg.k, cfg.E, cfg.G, device=dev)
    Lnp = moe.Layout(cfg.T, cfg.k, cfg.E, cfg.G, device=dev)
    runs = moe.SendRuns(L)
    A = torch.empty(R, cfg.H, dtype=torch.uint8, device=dev)
    As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device=dev)
    Y = torch.empty(R, cfg.N, dtype=torch.bfloat16, device=dev)
    out = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device=dev)
    ws_gc = torch.empty(int(L.sizes.gemm_combine_ws_bytes), dtype=torch.uint8, device=dev)
    A_send = torch.empty(runs.max_rows, cfg.H, dtype=torch.uint8, device=dev)
    As_send = torch.empty(cfg.H // 128, runs.max_rows, dtype=torch.float32, device=dev)
    Yg = torch.empty_like(Y)
    A_mx = torch.empty_like(A)
    A_sf = torch.empty(moe.mx_sf_a_shape(L, cfg.H), dtype=torch.uint8, device=dev)
    Y_mx = torch.empty_like(Y)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        moe.moe_route_layout_noplan(ids_d, w_d, Lnp, status)
        moe.moe_route_layout(ids_d, w_d, L, status)
        moe.moe_dispatch_quant(x, L, A, As, status)
        moe.moe_grouped_gemm1_combine(A, As, Wq, Ws, L, Y, out, ws_gc, status)
        moe.moe_send_layout(ids_d, L, runs, status)
        moe.moe_dispatch_quant_runs(x, L, runs, A_send, As_send, status)
        moe.moe_grouped_gemm1_gather(A_send, As_send, Wq, Ws, L, runs, Yg, status)
        moe.moe_dispatch_quant_mx(x, L, A_mx, A_sf, status)
        moe.moe_grouped_gemm1_mx(A_mx, A_sf, Wq_mx, W_sf, L, Y_mx, status)

    step()
    torch.cuda.synchronize()
    assert status.item() == 0
    order_free = ["count", "expert_offset", "expert_tile_offset", "rowmap", "tile_rows", "num_tiles"]
    want = {n: t.clone() for n, t in (("out", out), ("Y", Y), ("Yg", Yg), ("Y_mx", Y_mx), ("A_send", A_send))}
    want_np = {n: Lnp[n].clone() for n in order_free}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (out, Y, Yg, Y_mx):
        t.fill_(float("nan"))
    A_send.fill_(0xEE)
    for t in list(Lnp.t.values()) + list(L.t.values()):
        t.fill_(-7)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert status.item() == 0
    for n, t in (("out", out), ("Y", Y), ("Yg", Yg), ("Y_mx", Y_mx)):
        assert torch.equal(t.view(torch.int16), want[n].view(torch.int16)), n
    n_send = int(runs["run_offset"][-1].item())
    assert torch.equal(A_send[:n_send], want["A_send"][:n_send])
    for n in order_free:
        assert torch.equal(Lnp[n], want_np[n]), n
