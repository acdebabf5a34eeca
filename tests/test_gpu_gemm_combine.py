"""GPU parity of moe_grouped_gemm1_combine (GEMM1 with the combine overlapped,
gated per token) against the unfused calls and the oracle.

Its Y and out must be bit-for-bit what moe_grouped_gemm1 followed by
moe_combine write (same arithmetic, same order), on small shapes, ragged and
skewed routing, invalid ids and the benchmark's full-size workload; out must be
within the stated tolerance of the oracle's combine of the oracle's GEMM1.  A
token that never completes (the last tile withheld by lowering num_tiles on the
device, so nothing ever stores its rows) ends the call with MOE_ERR_TIMEOUT,
and the next call on the same context is clean."""
import numpy as np
import pytest
import torch

import combine_counting_sort_gb300 as moe
import oracle
from combine_counting_sort_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.build()


def prepare(cfg, ids=None, w=None, W=None):
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed).cuda()
    if ids is None:
        ids, w = gu.routed(cfg)
    L, st = gu.gpu_layout(ids, w, cfg.E, cfg.G)
    R = cfg.T * cfg.k
    A = torch.empty(R, cfg.H, dtype=torch.uint8, device="cuda")
    As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device="cuda")
    moe.moe_dispatch_quant(x, L, A, As, st)
    if W is None:
        W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device="cuda")
    Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W, Wq, Ws)
    torch.cuda.synchronize()
    return dict(x=x, ids=ids, w=w, L=L, A=A, As=As, W=W, Wq=Wq, Ws=Ws, R=R, layout_status=st.item())


def run_both(cfg, p):
    L, R = p["L"], p["R"]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y0 = torch.full((R, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    out0 = torch.full((cfg.T, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm1(p["A"], p["As"], p["Wq"], p["Ws"], L, Y0, st)
    moe.moe_combine(Y0, L, out0, st)
    Y1 = torch.full_like(Y0, float("nan"))
    out1 = torch.full_like(out0, float("nan"))
    ws = torch.full((int(L.sizes.gemm_combine_ws_bytes),), 0x5A, dtype=torch.uint8, device="cuda")  # poisoned
    moe.moe_grouped_gemm1_combine(p["A"], p["As"], p["Wq"], p["Ws"], L, Y1, out1, ws, st)
    torch.cuda.synchronize()
    return st.item(), (Y0, out0), (Y1, out1)


@pytest.mark.parametrize("T,H,E,G,k,N,skew", [
    (128, 256, 8, 2, 2, 512, None),     # the tiny shapes
    (300, 512, 16, 4, 4, 512, 1.3),     # ragged tails, empty experts
    (1, 256, 4, 2, 1, 256, None),       # a single token
    (700, 1024, 8, 2, 2, 1024, 2.0),    # heavy skew
    (2000, 512, 64, 8, 8, 768, 1.2),    # more tokens than combining warps
])
def test_gemm_combine_bit_identical_to_unfused(T, H, E, G, k, N, skew):
    cfg = inputs.MoEConfig("gc", T=T, H=H, E=E, G=G, k=k, N=N, zipf=skew, seed=6)
    p = prepare(cfg)
    st, (Y0, out0), (Y1, out1) = run_both(cfg, p)
    assert st == 0, moe.status_string(st)
    assert torch.equal(Y1.view(torch.int16), Y0.view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))


def test_gemm_combine_tiny_matches_oracle():
    cfg = inputs.CONFIGS["tiny"]
    p = prepare(cfg, W=inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed).cuda())
    st, _, (Y1, out1) = run_both(cfg, p)
    assert st == 0
    ref = oracle.route_layout(p["ids"], p["w"], cfg.E, cfg.G)
    q, s = oracle.quantize_rows(inputs.bf16_bits(p["x"]))
    A, As = oracle.dispatch(q, s, ref["pair_row"], cfg.k)
    Wq, Ws = oracle.quantize_weights(inputs.bf16_bits(p["W"]))
    Y = oracle.grouped_gemm1(A, As, Wq, Ws, ref["expert_offset"])
    want = oracle.combine(Y, ref["pair_row"], p["w"])
    gu.assert_close_bf16(gu.bits(out1), want, "gemm1_combine")


def test_gemm_combine_invalid_ids_give_the_unfused_output():
    cfg = inputs.MoEConfig("gc_bad", T=200, H=256, E=8, G=2, k=2, N=256, seed=2)
    ids, w = gu.routed(cfg)
    ids = ids.copy()
    ids[5, 0] = -1               # one invalid pair
    ids[9, :] = cfg.E + 3        # a token with no valid pair at all: out = 0
    p = prepare(cfg, ids=ids, w=w)
    assert p["layout_status"] == moe.MOE_ERR_EXPERT_ID      # reported by the layout
    st, (Y0, out0), (Y1, out1) = run_both(cfg, p)
    assert st == 0
    valid = p["L"]["expert_offset"][-1].item()
    assert torch.equal(Y1[:valid].view(torch.int16), Y0[:valid].view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
    assert torch.all(out1[9].float() == 0)


def test_gemm_combine_full_size_bench_workload():
    cfg = inputs.CONFIGS["t8192_zipf1.2"]
    p = prepare(cfg)
    st, (Y0, out0), (Y1, out1) = run_both(cfg, p)
    assert st == 0
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
    assert torch.equal(Y1.view(torch.int16), Y0.view(torch.int16))


def test_gemm_combine_times_out_on_a_token_that_never_completes_then_recovers():
    cfg = inputs.MoEConfig("gc_stall", T=256, H=256, E=8, G=2, k=2, N=256, seed=8)
    p = prepare(cfg)
    L = p["L"]
    nt = L["num_tiles"].item()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = torch.empty(p["R"], cfg.N, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(int(L.sizes.gemm_combine_ws_bytes), dtype=torch.uint8, device="cuda")
    L["num_tiles"].fill_(nt - 1)          # the last tile is never computed: its tokens never complete
    moe.moe_grouped_gemm1_combine(p["A"], p["As"], p["Wq"], p["Ws"], L, Y, out, ws, st)
    torch.cuda.synchronize()
    assert st.item() == moe.MOE_ERR_TIMEOUT
    # the context is usable: the full call now succeeds and matches the unfused path
    L["num_tiles"].fill_(nt)
    st.zero_()
    st2, (Y0, out0), (Y1, out1) = run_both(cfg, p)
    assert st2 == 0
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
