"""GPU parity of the MXFP8 variant (e8m0 scales per 32 values, block-scaled
tcgen05 GEMM1) against the oracle: codes and e8m0 scales bit-exact (read back
through the documented scale-factor layouts), GEMM1 within the stated
tolerance.  Every expected value comes from the oracle's layout, MX quantisers
and fp64 matmul on the seeded inputs; no operand is read back from the device
to build an expected value."""
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


def run_mx(cfg, W_dev, x=None, ids=None, w=None, gemm=True):
    """Layout -> MX dispatch -> MX weight quant -> MX GEMM1 on the GPU."""
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed) if x is None else x
    if ids is None:
        ids, w = gu.routed(cfg)
    L, status = gu.gpu_layout(ids, w, cfg.E, cfg.G)
    R = cfg.T * cfg.k
    A = torch.empty(R, cfg.H, dtype=torch.uint8, device="cuda")
    A_sf = torch.full(moe.mx_sf_a_shape(L, cfg.H), 0xFF, dtype=torch.uint8, device="cuda")
    moe.moe_dispatch_quant_mx(x.cuda(), L, A, A_sf, status)
    out = dict(x=x, ids=ids, w=w, L=L, A=A, A_sf=A_sf, R=R, status=status)
    if W_dev is not None:
        Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device="cuda")
        W_sf = torch.empty(moe.mx_sf_w_shape(cfg.E, cfg.N, cfg.H), dtype=torch.uint8, device="cuda")
        moe.moe_quant_weights_mx(W_dev, Wq, W_sf)
        out.update(Wq=Wq, W_sf=W_sf)
        if gemm:
            Y = torch.full((R + 128, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")  # poison + guard
            moe.moe_grouped_gemm1_mx(A, A_sf, Wq, W_sf, L, Y[:R], status)
            out["Y"] = Y
    torch.cuda.synchronize()
    assert status.item() == 0, moe.status_string(status.item())
    return out


def check_dispatch(r, cfg, tokens=None):
    """Codes and e8m0 scales of the rows of ``tokens`` (default all) against the oracle."""
    ref = oracle.route_layout(r["ids"], r["w"], cfg.E, cfg.G)
    toks = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    q, s = oracle.quantize_rows_mx(inputs.bf16_bits(r["x"][torch.as_tensor(toks)]))
    rows = ref["pair_row"].reshape(cfg.T, cfg.k)[toks]              # [n, k]
    A = r["A"].cpu().numpy()
    A_sf = r["A_sf"].cpu().numpy()
    for j in range(cfg.k):
        assert np.array_equal(A[rows[:, j]], q), f"codes of slot {j}"
        assert np.array_equal(gu.sf_a_rows(A_sf, ref, rows[:, j]), s), f"e8m0 scales of slot {j}"
    return ref


def expected_gemm(cfg, x, W, ref, rows):
    """Oracle GEMM1 (MX) of dense rows ``rows`` from the oracle's own operands."""
    R = cfg.T * cfg.k
    rexp = oracle.row_experts(ref["expert_offset"], R)[rows]
    toks = ref["row_pair"][rows].astype(np.int64) // cfg.k
    q, s = oracle.quantize_rows_mx(inputs.bf16_bits(x[torch.as_tensor(toks)]))
    want = np.zeros((len(rows), cfg.N), np.uint16)
    wq = {}
    for e in np.unique(rexp):
        sel = np.nonzero(rexp == e)[0]
        Wq_e, Ws_e = oracle.quantize_weights_mx(inputs.bf16_bits(W[int(e):int(e) + 1]))
        wq[int(e)] = (Wq_e[0], Ws_e[0])
        a = oracle.dequantize_mx(q[sel], s[sel])
        b = oracle.dequantize_mx(Wq_e[0], Ws_e[0])
        want[sel] = oracle.f64_to_bf16(a @ b.T)
    return want, wq


def test_mx_tiny_every_output():
    cfg = inputs.CONFIGS["tiny"]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed).cuda()
    r = run_mx(cfg, W)
    ref = check_dispatch(r, cfg)
    R = r["R"]
    # weights: codes and scales of every row of every expert
    Wq_ref, Ws_ref = oracle.quantize_weights_mx(inputs.bf16_bits(W))
    assert np.array_equal(r["Wq"].cpu().numpy(), Wq_ref)
    W_sf = r["W_sf"].cpu().numpy()
    for e in range(cfg.E):
        assert np.array_equal(gu.sf_w_rows(W_sf, e, np.arange(cfg.N)), Ws_ref[e]), e
    # GEMM1 in full
    A_ref, As_ref = oracle.dispatch_mx(*oracle.quantize_rows_mx(inputs.bf16_bits(r["x"])), ref["pair_row"], cfg.k)
    want = oracle.grouped_gemm1_mx(A_ref, As_ref, Wq_ref, Ws_ref, ref["expert_offset"])
    gu.assert_close_bf16(gu.bits(r["Y"])[:R], want, "gemm1_mx")
    assert torch.isnan(r["Y"][R:].float()).all()


def test_mx_quantiser_codes_across_the_bf16_range():
    # blocks whose amax runs over every bf16 exponent (subnormal to near the
    # top), boundaries 1.75 * 2**j and one ulp above, zero blocks, and blocks of
    # e4m3 rounding midpoints under amax 448 (ties to even)
    rng = np.random.default_rng(7)
    H = 4096
    T = 64
    blocks = []
    for ebits in range(0, 0xFF):
        amax_bits = (ebits << 7) | int(rng.integers(0, 128))
        blocks.append(amax_bits)
    vals = np.zeros((T * H // 32, 32), np.float64)
    nb = vals.shape[0]
    amax = oracle.bf16_to_f32(np.array(blocks * (nb // len(blocks) + 1), np.uint16)[:nb]).astype(np.float64)
    vals[:, 0] = amax
    vals[:, 1:] = amax[:, None] * rng.uniform(-1, 1, size=(nb, 31))
    grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2
    for b in range(0, 64):                                      # midpoint blocks
        vals[b, 0] = 448.0
        vals[b, 1:] = mids[(np.arange(31) + 31 * b) % len(mids)] * np.where(np.arange(31) % 2, -1, 1)
    for b in range(64, 128):                                    # boundaries 1.75 * 2**j, one ulp above
        j = b - 96
        vals[b, 0] = 1.75 * 2.0 ** j * (1 + (b % 2) * 2.0 ** -7)
        vals[b, 1:] = 1.75 * 2.0 ** j * rng.uniform(-1, 1, size=31)
    vals[128:160] = 0.0                                         # zero blocks
    x_bits = oracle.f64_to_bf16(vals.reshape(T, H))
    cfg = inputs.MoEConfig("mxsweep", T=T, H=H, E=4, G=2, k=2, N=256, seed=1)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16)
    r = run_mx(cfg, None, x=x)
    check_dispatch(r, cfg)


@pytest.mark.parametrize("T,H,E,G,k,N,skew", [
    (300, 512, 16, 4, 4, 512, 1.3),     # several tiles per popular expert, ragged tails, empty experts
    (1, 256, 4, 2, 1, 256, None),       # a single row
    (129, 384, 2, 1, 2, 768, None),     # every token to both experts: 2 tiles of 128 + 1 row each
    (700, 1024, 8, 2, 2, 1024, 2.0),    # heavy skew: one expert > 5 tiles
])
def test_mx_small_full(T, H, E, G, k, N, skew):
    cfg = inputs.MoEConfig("small", T=T, H=H, E=E, G=G, k=k, N=N, zipf=skew, seed=3)
    W = inputs.make_weights(E, N, H, seed=3).cuda()
    r = run_mx(cfg, W)
    ref = check_dispatch(r, cfg)
    want, _ = expected_gemm(cfg, r["x"], W, ref, np.arange(r["R"]))
    gu.assert_close_bf16(gu.bits(r["Y"])[: r["R"]], want, "gemm1_mx")
    assert torch.isnan(r["Y"][r["R"]:].float()).all()


def test_mx_few_row_tiles_full():
    """Tiles of 1..32 valid rows run transposed (W's halves as the M = 128
    operands with W's scale atoms, the tile's rows as N = 32 with A's), the
    others as usual: expert sizes around every boundary, every row checked."""
    ids, w = gu.routing_with_counts(gu.FEW_ROW_COUNTS, seed=5)
    cfg = inputs.MoEConfig("few_rows", T=len(ids), H=512, E=len(gu.FEW_ROW_COUNTS), G=4, k=1, N=512, zipf=None,
                           seed=5)
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, seed=5).cuda()
    r = run_mx(cfg, W, ids=ids, w=w)
    ref = check_dispatch(r, cfg)
    want, _ = expected_gemm(cfg, r["x"], W, ref, np.arange(r["R"]))
    gu.assert_close_bf16(gu.bits(r["Y"])[: r["R"]], want, "gemm1_mx")
    assert torch.isnan(r["Y"][r["R"]:].float()).all()


def sample_rows(eo, n_experts=6, seed=0):
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


@pytest.mark.parametrize("name", ["t2048_uniform", "t8192_zipf1.2"])
def test_mx_full_size_sampled(name):
    cfg = inputs.CONFIGS[name]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device="cuda")
    r = run_mx(cfg, W)
    rng = np.random.default_rng(5)
    ref = check_dispatch(r, cfg, tokens=rng.choice(cfg.T, 256, replace=False))
    rows = sample_rows(ref["expert_offset"])
    want, wq = expected_gemm(cfg, r["x"], W, ref, rows)
    gu.assert_close_bf16(gu.bits(r["Y"])[rows], want, "gemm1_mx")
    W_sf = r["W_sf"].cpu().numpy()
    for e, (q, s) in wq.items():
        assert np.array_equal(r["Wq"][e].cpu().numpy(), q), e
        assert np.array_equal(gu.sf_w_rows(W_sf, e, np.arange(cfg.N)), s), e
    assert torch.isnan(r["Y"][r["R"]:].float()).all()
    assert not torch.isnan(r["Y"][: r["R"]].float()).any()
