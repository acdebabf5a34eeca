"""GPU parity of the FP8 dispatch (bit-exact codes and scales), the weight
quantiser (bit-exact), the identity expert (bit-exact) and the combine
(stated tolerance) against the oracle."""
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


def dispatch_on_gpu(cfg, x):
    ids, w = gu.routed(cfg)
    L, status = gu.gpu_layout(ids, w, cfg.E, cfg.G)
    R = cfg.T * cfg.k
    A = torch.full((R, cfg.H), 0x7F, dtype=torch.uint8, device="cuda")           # poison (NaN code)
    As = torch.full((cfg.H // 128, R), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return ids, w, L, A, As


@pytest.mark.parametrize("name", ["tiny", "t2048_uniform", "t8192_zipf1.2"])
def test_dispatch_matches_oracle_bit_exact(name):
    cfg = inputs.CONFIGS[name]
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed)
    ids, w, L, A, As = dispatch_on_gpu(cfg, x)
    q, s = oracle.quantize_rows(inputs.bf16_bits(x))
    A_ref, As_ref = oracle.dispatch(q, s, L["pair_row"].cpu().numpy(), cfg.k)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_ref.view(np.uint32))


@pytest.mark.parametrize("T,H,E,G,k", [
    (64, 1152, 4, 2, 1),      # one row per token; H not a multiple of 512 (ragged rounds)
    (200, 640, 16, 4, 5),     # k not a multiple of 8
    (300, 1152, 32, 8, 12),   # block scales stored in two groups of 8 rows
    (130, 384, 64, 8, 32),    # the largest k: four groups of 8 rows
    (8300, 256, 24, 4, 12),   # the large-batch dispatch (4 rounds per slice), k > 8
])
def test_dispatch_k_and_widths_bit_exact(T, H, E, G, k):
    rng = np.random.default_rng(T + k)
    x = inputs.make_x(T, H, seed=k)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[3, k // 2] = -1                      # a skipped pair: its row is absent
    w = np.full((T, k), 1.0 / k, np.float32)
    L, status = gu.gpu_layout(ids, w, E, G)
    assert status.item() == moe.MOE_ERR_EXPERT_ID
    R = T * k
    A = torch.full((R, H), 0x7F, dtype=torch.uint8, device="cuda")
    As = torch.full((H // 128, R), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    q, s = oracle.quantize_rows(inputs.bf16_bits(x))
    pair_row = L["pair_row"].cpu().numpy()
    valid = int(L["expert_offset"][-1].item())
    A_ref, As_ref = oracle.dispatch(q, s, pair_row, k)
    assert np.array_equal(A.cpu().numpy()[:valid], A_ref[:valid])
    assert np.array_equal(As.cpu().numpy()[:, :valid].view(np.uint32), As_ref[:, :valid].view(np.uint32))
    # rows past the valid ones (the skipped pair's) were never written
    assert np.all(A.cpu().numpy()[valid:] == 0x7F)
    assert np.isnan(As.cpu().numpy()[:, valid:]).all()


def test_dispatch_special_blocks_bit_exact():
    # zero blocks, constant blocks, signed zeros, exact grid values, subnormal-range values, ragged T
    T, H, E, G, k = 45, 640, 6, 3, 3
    rng = np.random.default_rng(5)
    xv = rng.standard_normal((T, H))
    xv[0] = 0.0
    xv[1, :128] = -0.0
    xv[2, 128:256] = 3.0
    xv[3] *= 1e-30
    xv[4, :127] = oracle.e4m3_decode(np.arange(127, dtype=np.uint8)) * 2.0 ** -5
    xv[5] *= 1e4
    xb = oracle.f64_to_bf16(xv)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = np.full((T, k), 1.0 / k, np.float32)
    L, status = gu.gpu_layout(ids, w, E, G)
    R = T * k
    A = torch.empty((R, H), dtype=torch.uint8, device="cuda")
    As = torch.empty((H // 128, R), dtype=torch.float32, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, status)
    torch.cuda.synchronize()
    q, s = oracle.quantize_rows(xb)
    A_ref, As_ref = oracle.dispatch(q, s, L["pair_row"].cpu().numpy(), k)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_ref.view(np.uint32))


@pytest.mark.parametrize("E,N,H", [(2, 256, 384), (3, 512, 1024)])
def test_weight_quant_bit_exact(E, N, H):
    W = inputs.make_weights(E, N, H, seed=2)
    Wq = torch.empty(E, N, H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(E, N // 128, H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W.cuda(), Wq, Ws)
    torch.cuda.synchronize()
    q, s = oracle.quantize_weights(inputs.bf16_bits(W))
    assert np.array_equal(Wq.cpu().numpy(), q)
    assert np.array_equal(Ws.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_weight_quant_tiny_blocks_bit_exact():
    # blocks whose scale amax/448 is an fp32 subnormal (and bf16 subnormal weights)
    E, N, H = 2, 256, 256
    W = inputs.make_weights(E, N, H, seed=6).float()
    W[0] *= 2.0 ** -118
    W[1, :128] *= 2.0 ** -124
    W[1, 128:] *= 2.0 ** -128
    W = W.to(torch.bfloat16)
    Wq = torch.empty(E, N, H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(E, N // 128, H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W.cuda(), Wq, Ws)
    torch.cuda.synchronize()
    q, s = oracle.quantize_weights(inputs.bf16_bits(W))
    assert np.array_equal(Wq.cpu().numpy(), q)
    assert np.array_equal(Ws.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_identity_expert_bit_exact():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed)
    ids, w, L, A, As = dispatch_on_gpu(cfg, x)
    Y = torch.empty(cfg.T * cfg.k, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dequant_rows(A, As, L, Y)
    torch.cuda.synchronize()
    R = cfg.T * cfg.k
    assert np.array_equal(gu.bits(Y), oracle.identity_expert(A.cpu().numpy(), As.cpu().numpy(), np.arange(R)))


@pytest.mark.parametrize("name", ["tiny", "bw_t2048"])
def test_dispatch_identity_combine(name):
    cfg = inputs.CONFIGS[name]
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed)
    ids, w, L, A, As = dispatch_on_gpu(cfg, x)
    R = cfg.T * cfg.k
    Y = torch.empty(R, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dequant_rows(A, As, L, Y)
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_combine(Y, L, out, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Y_ref = oracle.identity_expert(A.cpu().numpy(), As.cpu().numpy(), np.arange(R))
    assert np.array_equal(gu.bits(Y), Y_ref)
    ref = oracle.combine(Y_ref, L["pair_row"].cpu().numpy(), w)
    gu.assert_close_bf16(gu.bits(out), ref, "combine")
    # the invariant: weights summing to one bring back the dequantised input
    q, s = oracle.quantize_rows(inputs.bf16_bits(x))
    deq = (oracle.e4m3_decode(q).reshape(cfg.T, -1, 128) * s.astype(np.float64)[:, :, None]).reshape(cfg.T, -1)
    gu.assert_close_bf16(gu.bits(out), oracle.f64_to_bf16(deq), "dispatch->identity->combine")


@pytest.mark.parametrize("T,k,D", [(1, 1, 8), (33, 3, 200), (257, 8, 4096), (100, 12, 1032)])
def test_combine_random_matches_oracle(T, k, D):
    rng = np.random.default_rng(T * k)
    E = max(k, 16)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    L, status = gu.gpu_layout(ids, w, E, 1)
    Yb = oracle.f64_to_bf16(rng.standard_normal((T * k, D)))
    Y = torch.from_numpy(Yb.view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(Y, L, out, status)
    torch.cuda.synchronize()
    ref = oracle.combine(Yb, L["pair_row"].cpu().numpy(), w)
    gu.assert_close_bf16(gu.bits(out), ref, "combine")
    # one-hot weights: an exact gather
    onehot = np.zeros_like(w)
    onehot[np.arange(T), np.arange(T) % k] = 1.0
    L2, _ = gu.gpu_layout(ids, onehot, E, 1)
    moe.moe_combine(Y, L2, out, status)
    torch.cuda.synchronize()
    assert np.array_equal(gu.bits(out), oracle.combine(Yb, L2["pair_row"].cpu().numpy(), onehot))


def test_dispatch_every_bf16_quotient_bit_exact():
    # For block maxima a (random bf16 values plus awkward ones), quantise every
    # bf16 value |x| <= a in blocks whose maximum is a: every quotient x/scale the
    # format can produce, including those closest to the e4m3 rounding midpoints.
    rng = np.random.default_rng(11)
    amaxes = list(oracle.bf16_to_f32(rng.integers(0x3C00, 0x4600, 24).astype(np.uint16)))
    amaxes += [1.0, 3.0, 448.0, 0.1, 7.0 / 3.0, 1e-3, 1e4]
    # tiny blocks: scale amax/448 below the fp32 normal range (subnormal scales,
    # bf16 subnormal inputs), where RN(1/scale) overflows or loses precision
    amaxes += [2.0 ** -110, 2.0 ** -118, 2.0 ** -120, 2.0 ** -126, 2.0 ** -130, 2.0 ** -133]
    # either side of scale 2^-80 (block maxima near 448 * 2^-80), where the
    # quantiser switches between the fma-corrected quotient and the division,
    # and random maxima over the whole bf16 normal range
    amaxes += [2.0 ** -69, 2.0 ** -70, 448.0 * 2.0 ** -80, 2.0 ** -71.3, 2.0 ** -72, 2.0 ** -90, 2.0 ** -100]
    amaxes += list(oracle.bf16_to_f32(rng.integers(0x0080, 0x7F00, 16).astype(np.uint16)))
    blocks = []
    for a in amaxes:
        ab = oracle.f64_to_bf16(np.array([a]))[0]
        a = float(oracle.bf16_to_f32(np.array([ab]))[0])
        pos = np.arange(0, int(ab) + 1, dtype=np.uint32).astype(np.uint16)      # every bf16 in [0, a]
        vals = np.concatenate([pos, pos | np.uint16(0x8000)])
        rng.shuffle(vals)
        per = 127
        nblk = (len(vals) + per - 1) // per
        vals = np.concatenate([vals, np.zeros(nblk * per - len(vals), np.uint16)]).reshape(nblk, per)
        blocks.append(np.concatenate([np.full((nblk, 1), ab, np.uint16), vals], axis=1))   # max = a
    allb = np.concatenate(blocks)
    H, k, E, G = 1024, 1, 4, 1
    per_tok = H // 128
    T = (len(allb) + per_tok - 1) // per_tok
    allb = np.concatenate([allb, np.zeros((T * per_tok - len(allb), 128), np.uint16)])
    xb = allb.reshape(T, H)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    ids = (np.arange(T) % E).astype(np.int32)[:, None]
    w = np.ones((T, k), np.float32)
    L, status = gu.gpu_layout(ids, w, E, G)
    R = T * k
    A = torch.empty((R, H), dtype=torch.uint8, device="cuda")
    As = torch.empty((H // 128, R), dtype=torch.float32, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, status)
    torch.cuda.synchronize()
    q, s = oracle.quantize_rows(xb)
    A_ref, As_ref = oracle.dispatch(q, s, L["pair_row"].cpu().numpy(), k)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_ref.view(np.uint32))


@pytest.mark.parametrize("name", ["bw_t4096", "bw_t8192", "bw_t16384", "stage1_t16384_zipf1.0"])
def test_dispatch_identity_combine_full_size_sampled(name):
    # The bandwidth sweep's sizes and the T=16384 workload, run in full on the
    # device as the benchmark launches them, checked on sampled tokens (the
    # first, the last and 254 random ones): their k rows of codes, scales and
    # identity-expert outputs bit-exact, their combined output within the
    # tolerance, and the dequantised-input invariant.
    cfg = inputs.CONFIGS[name]
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed)
    ids, w, L, A, As = dispatch_on_gpu(cfg, x)
    R, k = cfg.T * cfg.k, cfg.k
    Y = torch.empty(R, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dequant_rows(A, As, L, Y)
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_combine(Y, L, out, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    rng = np.random.default_rng(cfg.T)
    toks = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, 254, replace=False)]))
    S = len(toks)
    rows = torch.from_numpy(L["pair_row"].cpu().numpy().reshape(cfg.T, k)[toks].reshape(-1).astype(np.int64)).cuda()
    q, s = oracle.quantize_rows(inputs.bf16_bits(x)[toks])
    A_s, As_s = A.index_select(0, rows).cpu().numpy(), As.index_select(1, rows).cpu().numpy()
    assert np.array_equal(A_s, np.repeat(q, k, axis=0))                       # row t*k + j holds token t
    assert np.array_equal(As_s.view(np.uint32), np.repeat(s.T, k, axis=1).view(np.uint32))
    Y_ref = oracle.identity_expert(A_s, As_s, np.arange(S * k))
    assert np.array_equal(gu.bits(Y.index_select(0, rows)), Y_ref)
    got = gu.bits(out[torch.from_numpy(toks).cuda()])
    gu.assert_close_bf16(got, oracle.combine(Y_ref, np.arange(S * k), w[toks]), "combine")
    deq = (oracle.e4m3_decode(q).reshape(S, -1, 128) * s.astype(np.float64)[:, :, None]).reshape(S, -1)
    gu.assert_close_bf16(got, oracle.f64_to_bf16(deq), "dispatch->identity->combine")
