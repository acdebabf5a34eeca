"""GPU parity of the tcgen05 grouped GEMM1 against the oracle (stated
tolerance), on small problems computed in full and on the full-size
workloads through sampled rows; rows outside the valid range stay untouched."""
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


def run_stage1_unfused(cfg, W_dev, ids=None, w=None):
    """Layout -> dispatch -> weight quant -> GEMM1 on the GPU; returns host copies."""
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
    Y = torch.full((R + 128, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")  # poison + guard rows
    moe.moe_grouped_gemm1(A, As, Wq, Ws, L, Y[:R], status)
    torch.cuda.synchronize()
    assert status.item() == 0, moe.status_string(status.item())
    return dict(ids=ids, w=w, L=L, A=A, As=As, Wq=Wq, Ws=Ws, Y=Y, R=R)


def check_rows(r, rows):
    L = r["L"]
    eo = L["expert_offset"].cpu().numpy()
    experts = np.unique(oracle.row_experts(eo, r["R"])[rows])
    Wq = {int(e): r["Wq"][e].cpu().numpy() for e in experts}
    Ws = {int(e): r["Ws"][e].cpu().numpy() for e in experts}
    # the oracle takes full weight arrays; give it only the experts that are used
    E, N, H = r["Wq"].shape
    Wq_full = np.zeros((E, N, H), np.uint8) if E * N * H <= (1 << 28) else None
    A, As = r["A"].cpu().numpy(), r["As"].cpu().numpy()
    got = gu.bits(r["Y"])[rows]
    if Wq_full is not None:
        Ws_full = np.zeros((E, N // 128, H // 128), np.float32)
        for e in experts:
            Wq_full[e], Ws_full[e] = Wq[int(e)], Ws[int(e)]
        want = oracle.grouped_gemm1(A, As, Wq_full, Ws_full, eo, rows)
    else:
        rexp = oracle.row_experts(eo, r["R"])[rows]
        want = np.zeros((len(rows), N), np.uint16)
        for e in experts:
            sel = np.nonzero(rexp == e)[0]
            a = oracle.dequantize_rows(A, As, rows[sel])
            b = oracle.dequantize_weights(Wq[int(e)], Ws[int(e)])
            want[sel] = oracle.f64_to_bf16(a @ b.T)
    return gu.assert_close_bf16(got, want, "gemm1")


def test_gemm1_tiny_full():
    cfg = inputs.CONFIGS["tiny"]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed).cuda()
    r = run_stage1_unfused(cfg, W)
    R = r["R"]
    check_rows(r, np.arange(R))
    assert torch.isnan(r["Y"][R:].float()).all()          # guard rows untouched
    # weights quantised on the GPU are the oracle's bits
    q, s = oracle.quantize_weights(inputs.bf16_bits(W))
    assert np.array_equal(r["Wq"].cpu().numpy(), q)


@pytest.mark.parametrize("T,H,E,G,k,N,skew", [
    (300, 512, 16, 4, 4, 512, 1.3),     # several tiles per popular expert, ragged tails, empty experts
    (1, 256, 4, 2, 1, 256, None),       # a single row
    (129, 384, 2, 1, 2, 768, None),     # every token to both experts: 2 tiles of 128 + 1 row each
    (700, 1024, 8, 2, 2, 1024, 2.0),    # heavy skew: one expert > 5 tiles
])
def test_gemm1_small_full(T, H, E, G, k, N, skew):
    cfg = inputs.MoEConfig("small", T=T, H=H, E=E, G=G, k=k, N=N, zipf=skew, seed=3)
    W = inputs.make_weights(E, N, H, seed=3).cuda()
    r = run_stage1_unfused(cfg, W)
    check_rows(r, np.arange(r["R"]))
    assert torch.isnan(r["Y"][r["R"]:].float()).all()


def sample_rows(r, n_experts=10, seed=0):
    """First and last row of every tile of a few experts (largest, smallest, random) plus random rows."""
    L = r["L"]
    eo = L["expert_offset"].cpu().numpy()
    cnt = np.diff(eo)
    nz = np.nonzero(cnt)[0]
    rng = np.random.default_rng(seed)
    pick = set([int(nz[np.argmax(cnt[nz])]), int(nz[np.argmin(cnt[nz])])])
    pick |= set(int(e) for e in rng.choice(nz, size=min(n_experts, len(nz)), replace=False))
    rows = []
    for e in sorted(pick):
        for b in range(eo[e], eo[e + 1], 128):
            rows += [b, min(b + 127, eo[e + 1] - 1)]
        rows += list(rng.integers(eo[e], eo[e + 1], size=4))
    return np.unique(np.array(rows, dtype=np.int64))


@pytest.mark.parametrize("name", ["t2048_uniform", "t8192_zipf1.2", "stage1_t16384_zipf1.0"])
def test_gemm1_full_size_sampled(name):
    cfg = inputs.CONFIGS[name]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device="cuda")
    r = run_stage1_unfused(cfg, W)
    rows = sample_rows(r)
    check_rows(r, rows)
    assert torch.isnan(r["Y"][r["R"]:].float()).all()
    # the sampled experts' weights quantised on the GPU are the oracle's bits
    e = int(oracle.row_experts(r["L"]["expert_offset"].cpu().numpy(), r["R"])[rows[0]])
    q, s = oracle.quantize_weights(inputs.bf16_bits(W[e:e + 1]))
    assert np.array_equal(r["Wq"][e:e + 1].cpu().numpy(), q)
    # every valid row was written (no NaN left from the poison)
    assert not torch.isnan(r["Y"][: r["R"]].float()).any()
