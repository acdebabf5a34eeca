"""Pins for the oracle's quantiser, dispatch, GEMM1 and combine.

Quantiser: error bounds of round-to-nearest on the e4m3 grid, closed-form
blocks (zero, constant, a block that is exactly the e4m3 grid times a power of
two).  GEMM1: entries recomputed as exactly-rounded sums (math.fsum of exact
products), the identity-weight special case, per-expert scaling.  Combine:
one-hot weights reduce it to a gather; the identity expert with weights summing
to one reproduces the dequantised input (the dispatch -> identity -> combine
invariant).  Also a few planted mistakes, each of which one of these pins must
catch."""
import math

import numpy as np
import pytest

import oracle
from combine_counting_sort_gb300 import inputs


def rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return oracle.f64_to_bf16(v.astype(np.float64))


# ---------------------------------------------------------------- quantiser

def test_quant_error_bound_and_extremes():
    x = rand_bf16((64, 1024), 11)
    q, s = oracle.quantize_rows(x)
    xv = oracle.bf16_to_f32(x).astype(np.float64).reshape(64, 8, 128)
    dq = oracle.e4m3_decode(q).reshape(64, 8, 128) * s.astype(np.float64)[:, :, None]
    # round to nearest on the e4m3 grid: |x/s - q| <= half the grid step at |x/s|
    # (step 2**-9 below 2**-6, else 2**(floor(log2|v|) - 3)), plus the fp32 division's rounding
    v = np.abs(xv) / s.astype(np.float64)[:, :, None]
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(v, 1e-300))), -6) - 3)
    err = np.abs(xv - dq) / s.astype(np.float64)[:, :, None]
    assert np.all(err <= step / 2 * (1 + 1e-6) + v * 2.0 ** -23)
    # the block's largest magnitude maps to +-448
    am = np.abs(xv).argmax(axis=2)
    codes = np.take_along_axis(q.reshape(64, 8, 128), am[:, :, None], 2)[:, :, 0]
    assert np.all((codes == 0x7E) | (codes == 0xFE))
    assert np.array_equal(s, (np.abs(xv).max(axis=2) / 448.0).astype(np.float32)) or \
        np.array_equal(s, (np.abs(oracle.bf16_to_f32(x).reshape(64, 8, 128)).max(axis=2) / np.float32(448)))


def test_quant_special_blocks():
    H = 512
    x = np.zeros((3, H), np.float64)
    x[1, :128] = -2.5                          # constant block
    grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))   # 127 grid values, max 448
    x[2, 128:255] = grid * 2.0 ** -3           # the e4m3 grid times a power of two
    x[2, 255] = -grid[5] * 2.0 ** -3
    q, s = oracle.quantize_rows(oracle.f64_to_bf16(x))
    assert np.all(s[0] == 0) and np.all(q[0] == 0)                      # all-zero row
    assert s[1, 0] == np.float32(2.5 / 448) and np.all(q[1, :128] == 0xFE)
    assert s[1, 1] == 0 and np.all(q[1, 128:] == 0)
    assert s[2, 1] == np.float32(2.0 ** -3)                            # 448 * 2**-3 / 448 exactly
    assert np.array_equal(q[2, 128:255], np.arange(0, 0x7F, dtype=np.uint8))
    assert q[2, 255] == (5 | 0x80)


def test_quant_tiny_blocks_with_subnormal_scales():
    # amax/448 below the fp32 normal range: the scale is the single rounding of
    # the exact quotient (float64 division, then one rounding to float32, which
    # is correct rounding for a quotient of float32 operands, subnormal results
    # included), and every code is the e4m3 rounding of the single-rounded
    # quotient x/scale computed the same way.  A flush-to-zero or a reciprocal
    # shortcut fails here.
    x = rand_bf16((4, 512), 13)
    xv = oracle.bf16_to_f32(x).astype(np.float64)
    xv[0] *= 2.0 ** -118
    xv[1] *= 2.0 ** -124
    xv[2] *= 2.0 ** -128
    xv[3, :128] = 2.0 ** -133                  # bf16's smallest subnormal, constant block
    xb = oracle.f64_to_bf16(xv)
    q, s = oracle.quantize_rows(xb)
    xf = oracle.bf16_to_f32(xb).astype(np.float64).reshape(4, 4, 128)
    amax = np.abs(xf).max(axis=2)
    s_ref = (amax / 448.0).astype(np.float32)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.any((s_ref > 0) & (s_ref < np.float32(2.0 ** -126)))    # the case is exercised
    sd = s_ref.astype(np.float64)[:, :, None]
    with np.errstate(invalid="ignore", divide="ignore"):
        v = np.where(sd > 0, xf / sd, 0.0).astype(np.float32)
    assert np.array_equal(q.reshape(4, 4, 128), oracle.e4m3_encode(v))
    assert np.all(q[3, :128] == 0x7E)


def _brute_e4m3(v: "Fraction") -> int:
    """e4m3 code of an exact rational by direct search: the nearest of the 127
    non-negative grid values (3 mantissa bits, exponent bias 7, subnormal step
    2**-9), ties to the even code, magnitudes above 448 saturated; sign from v."""
    from fractions import Fraction
    grid = [Fraction(8 + m, 8) * Fraction(2) ** (e - 7) if e else Fraction(m, 512)
            for e in range(16) for m in range(8)][:127]
    a = min(abs(v), Fraction(448))
    best = min(range(127), key=lambda c: (abs(grid[c] - a), c & 1))
    return best | (0x80 if v < 0 else 0)


def _fp32_of(v: "Fraction") -> "Fraction":
    """Round an exact rational to the nearest fp32 value (ties to even), by
    integer arithmetic on the 24-bit significand (normal range)."""
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    sign, a = (-1 if v < 0 else 1), abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    scaled = a / Fraction(2) ** (e - 23)                   # in [2**23, 2**24)
    n, rem = divmod(scaled.numerator, scaled.denominator)
    twice = 2 * rem
    if twice > scaled.denominator or (twice == scaled.denominator and n & 1):
        n += 1
    return sign * Fraction(n) * Fraction(2) ** (e - 23)


def test_quant_codes_are_the_e4m3_rounding_of_the_ieee_quotient():
    # For a few block maxima, every bf16 value of [-amax, amax] in one block
    # each: the code must be the e4m3 rounding of RN_fp32(x / scale) with
    # scale = RN_fp32(amax / 448), here computed in exact rational arithmetic
    # with a brute-force nearest-code search for the values whose quotient lies
    # near an e4m3 rounding boundary, and for the rest through float64 (a
    # quotient of fp32 operands rounded once to float64 and again to float32 is
    # rounded correctly).  A reciprocal shortcut x * RN(1/scale) fails.
    from fractions import Fraction
    rng = np.random.default_rng(17)
    amaxes = [7.0 / 3.0, 0.1, 13.7, 1e4, 3.0, 1.0]
    amaxes += list(oracle.bf16_to_f32(rng.integers(0x3C00, 0x4600, 16).astype(np.uint16)).astype(np.float64))
    bad_shortcut, checked = 0, 0
    for a in amaxes:
        ab = oracle.f64_to_bf16(np.array([a]))[0]
        pos = np.arange(0, int(ab) + 1, dtype=np.uint32).astype(np.uint16)
        vals = np.concatenate([pos, pos | np.uint16(0x8000)])
        nb = (len(vals) + 126) // 127
        blocks = np.concatenate([vals, np.zeros(nb * 127 - len(vals), np.uint16)]).reshape(nb, 127)
        xb = np.concatenate([np.full((nb, 1), ab, np.uint16), blocks], axis=1).reshape(1, -1)
        q, s = oracle.quantize_rows(xb)
        scale = np.float32(s[0, 0])
        assert np.all(s == scale)
        assert Fraction(float(scale)) == _fp32_of(Fraction(float(oracle.bf16_to_f32(np.array([ab]))[0])) / 448)
        xf = oracle.bf16_to_f32(xb[0])
        quot = (xf.astype(np.float64) / np.float64(scale)).astype(np.float32)
        assert np.array_equal(q[0], oracle.e4m3_encode(quot))
        # the delicate values: quotients within 2**-20 (relative) of an e4m3 midpoint
        grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
        mids = (grid[1:] + grid[:-1]) / 2
        aq = np.abs(xf.astype(np.float64) / float(scale))
        near = np.nonzero(np.min(np.abs(aq[:, None] - mids[None, :]) / np.maximum(mids[None, :], 1e-30), axis=1)
                          < 2.0 ** -20)[0]
        for i in near[:400]:
            exact = _fp32_of(Fraction(float(xf[i])) / Fraction(float(scale)))
            assert q[0, i] == _brute_e4m3(exact), (a, i)
            checked += 1
        short = oracle.e4m3_encode((xf * (np.float32(1) / scale)).astype(np.float32))
        bad_shortcut += int(np.count_nonzero(short != q[0]))
    assert checked >= 100            # quotients at or next to a rounding midpoint were checked exactly
    assert bad_shortcut > 0          # the pin tells the IEEE quotient from the reciprocal shortcut


def test_dispatch_places_every_copy():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.bf16_bits(inputs.make_x(cfg.T, cfg.H))
    ids, w = oracle.router_topk(inputs.make_logits(cfg.T, cfg.E).numpy(), cfg.k)
    L = oracle.route_layout(ids, w, cfg.E, cfg.G)
    q, s = oracle.quantize_rows(x)
    A, As = oracle.dispatch(q, s, L["pair_row"], cfg.k)
    for r in range(cfg.T * cfg.k):
        t = L["row_pair"][r] // cfg.k
        assert np.array_equal(A[r], q[t]) and np.array_equal(As[:, r], s[t])


def test_weight_quant_blocks():
    w = rand_bf16((2, 256, 384), 12, scale=0.05)
    q, s = oracle.quantize_weights(w)
    assert s.shape == (2, 2, 3)
    wv = oracle.bf16_to_f32(w).astype(np.float64)
    for e in range(2):
        for nb in range(2):
            for kb in range(3):
                blk = wv[e, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
                assert s[e, nb, kb] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448))
    dq = oracle.dequantize_weights(q[1], s[1])
    assert np.max(np.abs(dq - wv[1])) <= np.max(s) * 16 + 1e-12


# ---------------------------------------------------------------- GEMM1

def small_problem(T=24, H=256, E=4, G=2, k=2, N=256, seed=5):
    x = rand_bf16((T, H), seed)
    logits = np.random.default_rng(seed + 1).standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.router_topk(logits, k)
    L = oracle.route_layout(ids, w, E, G)
    q, s = oracle.quantize_rows(x)
    A, As = oracle.dispatch(q, s, L["pair_row"], k)
    Wq, Ws = oracle.quantize_weights(rand_bf16((E, N, H), seed + 2, scale=1 / 16))
    return x, ids, w, L, A, As, Wq, Ws


def fsum_entry(A, As, Wq, Ws, e, r, n):
    a = oracle.dequantize_rows(A, As, [r])[0]
    b = oracle.dequantize_weights(Wq[e], Ws[e])[n]
    return math.fsum(float(u) * float(v) for u, v in zip(a, b))   # products exact in fp64


def test_gemm1_entries_are_correctly_rounded_sums():
    x, ids, w, L, A, As, Wq, Ws = small_problem()
    Y = oracle.grouped_gemm1(A, As, Wq, Ws, L["expert_offset"])
    rexp = oracle.row_experts(L["expert_offset"], A.shape[0])
    rng = np.random.default_rng(0)
    for r, n in zip(rng.integers(0, A.shape[0], 60), rng.integers(0, Wq.shape[1], 60)):
        want = oracle.f64_to_bf16(np.array([fsum_entry(A, As, Wq, Ws, rexp[r], r, n)]))[0]
        assert Y[r, n] == want, (r, n)


def test_gemm1_identity_weights_return_dequantised_rows():
    x, ids, w, L, A, As, Wq, Ws = small_problem(N=256)
    E, N, H = Wq.shape
    eye = np.zeros((E, N, H), np.float64)
    for e in range(E):
        eye[e] = np.eye(N, H) * 448.0              # code 0x7E on the diagonal
    Iq, Is = oracle.quantize_weights(oracle.f64_to_bf16(eye))
    # diagonal 128x128 blocks have amax 448 (scale 1); the others are all zero (scale 0)
    assert np.array_equal(Is, np.broadcast_to(np.eye(N // 128, H // 128, dtype=np.float32), Is.shape))
    Y = oracle.grouped_gemm1(A, As, Iq, Is, L["expert_offset"])
    want = oracle.f64_to_bf16(oracle.dequantize_rows(A, As, np.arange(A.shape[0])) * 448.0)
    assert np.array_equal(Y, want)


def test_gemm1_uses_each_rows_own_expert():
    x, ids, w, L, A, As, Wq, Ws = small_problem()
    E = Wq.shape[0]
    Ws2 = Ws * np.exp2(np.arange(E, dtype=np.float32))[:, None, None]   # expert e scaled by 2**e
    Y1 = oracle.bf16_to_f32(oracle.grouped_gemm1(A, As, Wq, Ws, L["expert_offset"]))
    Y2 = oracle.bf16_to_f32(oracle.grouped_gemm1(A, As, Wq, Ws2, L["expert_offset"]))
    rexp = oracle.row_experts(L["expert_offset"], A.shape[0])
    assert np.array_equal(Y2, Y1 * np.exp2(rexp.astype(np.float32))[:, None])


def test_gemm1_row_subset_matches_full():
    x, ids, w, L, A, As, Wq, Ws = small_problem()
    Y = oracle.grouped_gemm1(A, As, Wq, Ws, L["expert_offset"])
    rows = np.array([0, 5, 17, 40, 47])
    assert np.array_equal(oracle.grouped_gemm1(A, As, Wq, Ws, L["expert_offset"], rows), Y[rows])


# ---------------------------------------------------------------- combine

def test_combine_one_hot_is_a_gather():
    x, ids, w, L, A, As, Wq, Ws = small_problem()
    Y = oracle.grouped_gemm1(A, As, Wq, Ws, L["expert_offset"])
    T, k = ids.shape
    onehot = np.zeros((T, k), np.float32)
    pick = np.arange(T) % k
    onehot[np.arange(T), pick] = 1.0
    out = oracle.combine(Y, L["pair_row"], onehot)
    assert np.array_equal(out, Y[L["pair_row"].reshape(T, k)[np.arange(T), pick]])


def test_combine_entries_are_correctly_rounded_sums():
    x, ids, w, L, A, As, Wq, Ws = small_problem()
    Y = oracle.grouped_gemm1(A, As, Wq, Ws, L["expert_offset"])
    out = oracle.combine(Y, L["pair_row"], w)
    T, k = ids.shape
    Yf = oracle.bf16_to_f32(Y)
    for t in range(0, T, 5):
        for c in range(0, Y.shape[1], 37):
            s = math.fsum(float(w[t, j]) * float(Yf[L["pair_row"][t * k + j], c]) for j in range(k))
            assert out[t, c] == oracle.f64_to_bf16(np.array([s]))[0]


def test_dispatch_identity_combine_reproduces_dequantised_input():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.bf16_bits(inputs.make_x(cfg.T, cfg.H))
    ids, w = oracle.router_topk(inputs.make_logits(cfg.T, cfg.E).numpy(), cfg.k)
    L = oracle.route_layout(ids, w, cfg.E, cfg.G)
    q, s = oracle.quantize_rows(x)
    A, As = oracle.dispatch(q, s, L["pair_row"], cfg.k)
    Y = oracle.identity_expert(A, As, np.arange(cfg.T * cfg.k))
    out = oracle.bf16_to_f32(oracle.combine(Y, L["pair_row"], w)).astype(np.float64)
    deq = (oracle.e4m3_decode(q).reshape(cfg.T, -1, 128) * s.astype(np.float64)[:, :, None]).reshape(cfg.T, -1)
    # two bf16 roundings (identity expert, combine) and sum(w) = 1 within fp32: <= ~2**-8 relative
    assert np.all(np.abs(out - deq) <= np.abs(deq) * 2.0 ** -7 + 1e-30)
    # and against the original input: the e4m3 error dominates (relative 2**-4 of the block scale * 448)
    xv = oracle.bf16_to_f32(x).astype(np.float64)
    assert np.max(np.abs(out - xv)) <= np.max(s) * 16


# ---------------------------------------------------------------- planted mistakes

def test_planted_transposed_weight_is_caught():
    x, ids, w, L, A, As, Wq, Ws = small_problem(H=256, N=256)
    bad = oracle.grouped_gemm1(A, As, np.ascontiguousarray(Wq.transpose(0, 2, 1)), Ws,
                               L["expert_offset"])
    r, n = 3, 7
    rexp = oracle.row_experts(L["expert_offset"], A.shape[0])
    want = oracle.f64_to_bf16(np.array([fsum_entry(A, As, Wq, Ws, rexp[r], r, n)]))[0]
    assert bad[r, n] != want


def test_planted_unstable_sort_is_caught():
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 5, size=(30, 3)).astype(np.int32)
    flat = ids.reshape(-1)
    p = np.arange(flat.size)
    bad_row_pair = np.lexsort((-p, flat))       # same keys, equal keys in reverse order
    brute = sorted(range(flat.size), key=lambda q: (flat[q], q))
    assert list(oracle.route_layout(ids, np.zeros(ids.shape, np.float32), 5, 1, 4)["row_pair"]) == brute
    assert list(bad_row_pair) != brute


def test_planted_wrong_first_expert_is_caught():
    # a token order built on the LAST expert instead of the first breaks the landed-prefix property
    rng = np.random.default_rng(4)
    ids = rng.integers(0, 8, size=(64, 3)).astype(np.int32)
    L = oracle.route_layout(ids, np.zeros(ids.shape, np.float32), 8, 2)
    wrong = np.argsort(ids.max(axis=1), kind="stable")
    pos = np.empty(64, np.int64)
    pos[wrong] = np.arange(64)
    broken = any(np.any(pos[np.nonzero((ids == e).any(axis=1))[0]] >= L["ready_tokens"][e]) for e in range(8))
    assert broken
