"""GPU parity of the tcgen05 grouped GEMM1 against the oracle (stated
tolerance), on small problems computed in full and on the full-size
workloads through sampled rows; rows outside the valid range stay untouched.
Every expected value comes from the oracle's own layout, quantisers and
matmul on the seeded inputs: no operand is read back from the device."""
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


def oracle_rows_expected(cfg, W, ids, w, rows):
    """Expected GEMM1 output of dense rows ``rows``, from the oracle alone: the
    oracle's layout, its quantiser on the tokens those rows hold (row r of the
    dispatch buffer holds the codes and scales of token row_pair[r] // k, the
    dispatch's definition) and its weight quantiser on the experts they use.
    Nothing the CUDA path produced enters.  Also returns the oracle's weight
    codes of those experts."""
    ref = oracle.route_layout(ids, w, cfg.E, cfg.G)
    R = cfg.T * cfg.k
    rexp = oracle.row_experts(ref["expert_offset"], R)[rows]
    toks = ref["row_pair"][rows].astype(np.int64) // cfg.k
    q, s = oracle.quantize_rows(inputs.bf16_bits(inputs.make_x(cfg.T, cfg.H, cfg.seed)[torch.as_tensor(toks)]))
    want = np.zeros((len(rows), cfg.N), np.uint16)
    wq = {}
    for e in np.unique(rexp):
        sel = np.nonzero(rexp == e)[0]
        Wq_e, Ws_e = oracle.quantize_weights(inputs.bf16_bits(W[int(e):int(e) + 1]))
        wq[int(e)] = Wq_e[0]
        a = oracle.dequantize_rows(q[sel], np.ascontiguousarray(s[sel].T), np.arange(len(sel)))
        b = oracle.dequantize_weights(Wq_e[0], Ws_e[0])
        want[sel] = oracle.f64_to_bf16(a @ b.T)
    return want, wq, ref


def test_gemm1_tiny_full():
    cfg = inputs.CONFIGS["tiny"]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed).cuda()
    r = run_stage1_unfused(cfg, W)
    R = r["R"]
    want, _, _ = oracle_rows_expected(cfg, W, r["ids"], r["w"], np.arange(R))
    gu.assert_close_bf16(gu.bits(r["Y"])[:R], want, "gemm1")
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
    want, _, _ = oracle_rows_expected(cfg, W, r["ids"], r["w"], np.arange(r["R"]))
    gu.assert_close_bf16(gu.bits(r["Y"])[: r["R"]], want, "gemm1")
    assert torch.isnan(r["Y"][r["R"]:].float()).all()


@pytest.mark.parametrize("H,N", [(512, 512), (256, 768)])
def test_gemm1_few_row_tiles_full(H, N):
    """Tiles of 1..32 valid rows run transposed (W as the M = 128 operand, the
    tile's rows as N = 32), tiles of 33 and more as usual: expert sizes around
    every boundary (1, 31, 32, 33 rows; 128 + 32, 128 + 33 rows, whose last
    tile is short), every row checked against the oracle."""
    counts = gu.FEW_ROW_COUNTS
    ids, w = gu.routing_with_counts(counts, seed=5)
    cfg = inputs.MoEConfig("few_rows", T=len(ids), H=H, E=len(counts), G=4, k=1, N=N, zipf=None, seed=5)
    W = inputs.make_weights(cfg.E, N, H, seed=5).cuda()
    r = run_stage1_unfused(cfg, W, ids, w)
    want, _, _ = oracle_rows_expected(cfg, W, ids, w, np.arange(r["R"]))
    gu.assert_close_bf16(gu.bits(r["Y"])[: r["R"]], want, "gemm1")
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
    rows = sample_rows(r, n_experts=6)
    want, wq, ref = oracle_rows_expected(cfg, W, r["ids"], r["w"], rows)
    # the device layout is the oracle's (so the sampled rows name the same pairs)
    assert np.array_equal(r["L"]["row_pair"].cpu().numpy(), ref["row_pair"])
    gu.assert_close_bf16(gu.bits(r["Y"])[rows], want, "gemm1")
    assert torch.isnan(r["Y"][r["R"]:].float()).all()
    # the sampled experts' weights quantised on the GPU are the oracle's bits
    for e, q in wq.items():
        assert np.array_equal(r["Wq"][e].cpu().numpy(), q), e
    # every valid row was written (no NaN left from the poison)
    assert not torch.isnan(r["Y"][: r["R"]].float()).any()
