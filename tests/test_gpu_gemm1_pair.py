"""GPU parity of moe_grouped_gemm1_pair (GEMM1 on CTA pairs, M = 256 MMAs over
two SMs) against the oracle (stated tolerance) and against the single-CTA
moe_grouped_gemm1, whose Y it must reproduce bit for bit: both fold the same
fp32 partials of 128 x 256 x 128 products in the same order.  Shapes cover
experts with odd and even M-tile counts (the odd CTA of the last pair has no
rows), single-row experts, empty experts, a single token and the full-size
workloads; rows past the valid range stay untouched."""
import numpy as np
import pytest
import torch

import combine_counting_sort_gb300 as moe
from combine_counting_sort_gb300 import inputs
from tests import gpu_util as gu
from tests.test_gpu_gemm1 import oracle_rows_expected, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.build()


def both(cfg, W_dev, ids=None, w=None):
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed)
    if ids is None:
        ids, w = gu.routed(cfg)
    L, status = gu.gpu_layout(ids, w, cfg.E, cfg.G)
    R = cfg.T * cfg.k
    A = torch.empty(R, cfg.H, dtype=torch.uint8, device="cuda")
    As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, status)
    Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W_dev, Wq, Ws)
    Y1 = torch.full((R + 128, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.full_like(Y1, float("nan"))
    moe.moe_grouped_gemm1(A, As, Wq, Ws, L, Y1[:R], status)
    moe.moe_grouped_gemm1(A, As, Wq, Ws, L, Y2[:R], status, pair=True)
    torch.cuda.synchronize()
    return dict(ids=ids, w=w, L=L, Y1=Y1, Y2=Y2, R=R, Wq=Wq, status=status.item())


def test_pair_tiny_matches_oracle_and_single():
    cfg = inputs.CONFIGS["tiny"]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed).cuda()
    r = both(cfg, W)
    assert r["status"] == 0, moe.status_string(r["status"])
    R = r["R"]
    want, _, _ = oracle_rows_expected(cfg, W, r["ids"], r["w"], np.arange(R))
    gu.assert_close_bf16(gu.bits(r["Y2"])[:R], want, "gemm1_pair")
    assert torch.equal(r["Y2"].view(torch.int16)[:R], r["Y1"].view(torch.int16)[:R])
    assert torch.isnan(r["Y2"][R:].float()).all()


@pytest.mark.parametrize("T,H,E,G,k,N,skew", [
    (300, 512, 16, 4, 4, 512, 1.3),     # ragged tails, empty experts, 1- and 3-tile experts
    (1, 256, 4, 2, 1, 256, None),       # a single row: one pair, odd CTA empty
    (129, 384, 2, 1, 2, 768, None),     # 2 tiles per expert: one full pair each
    (700, 1024, 8, 2, 2, 1024, 2.0),    # heavy skew: one expert > 5 tiles
    (1500, 256, 3, 1, 1, 256, 1.1),     # odd and even tile counts side by side
    (2000, 512, 64, 8, 8, 768, 1.2),    # more pair units than resident clusters
])
def test_pair_small_bit_identical_to_single(T, H, E, G, k, N, skew):
    cfg = inputs.MoEConfig("pair", T=T, H=H, E=E, G=G, k=k, N=N, zipf=skew, seed=4)
    W = inputs.make_weights(E, N, H, seed=4).cuda()
    r = both(cfg, W)
    assert r["status"] == 0, moe.status_string(r["status"])
    R = r["R"]
    assert torch.equal(r["Y2"].view(torch.int16)[:R], r["Y1"].view(torch.int16)[:R])
    assert torch.isnan(r["Y2"][R:].float()).all()
    want, _, _ = oracle_rows_expected(cfg, W, r["ids"], r["w"], np.arange(R))
    gu.assert_close_bf16(gu.bits(r["Y2"])[:R], want, "gemm1_pair")


@pytest.mark.parametrize("name", ["t2048_uniform", "t8192_zipf1.2", "stage1_t16384_zipf1.0"])
def test_pair_full_size(name):
    cfg = inputs.CONFIGS[name]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device="cuda")
    r = both(cfg, W)
    assert r["status"] == 0, moe.status_string(r["status"])
    R = r["R"]
    assert torch.equal(r["Y2"].view(torch.int16)[:R], r["Y1"].view(torch.int16)[:R])
    assert torch.isnan(r["Y2"][R:].float()).all()
    rows = sample_rows(dict(L=r["L"]), n_experts=4)
    want, _, _ = oracle_rows_expected(cfg, W, r["ids"], r["w"], rows)
    gu.assert_close_bf16(gu.bits(r["Y2"])[rows], want, "gemm1_pair")
