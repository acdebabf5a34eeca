"""Pins for the oracle's MXFP8 variant (e8m0 power-of-two scales per 32 values).

Each pin checks the oracle against something other than itself:

* the scale exponent against its definition (the smallest X with
  448 * 2**X >= amax, clamped to the e8m0 range), searched upward one integer
  at a time in exact arithmetic, over every finite non-negative bf16 value;
* e8m0 codes against torch's own float8_e8m0fnu encoding of the same powers
  of two (a library routine);
* quantised blocks against the rounding error bound of the e4m3 grid, the
  "no saturation" property the rule is chosen for, and the tightness of the
  power of two (the block maximum lands in (224, 448]);
* closed-form blocks (zero, exactly 448 * 2**j, the e4m3 grid times a power of
  two, one ulp above a boundary) and the independence of neighbouring blocks;
* GEMM1 entries against correctly rounded sums of the exact products
  (math.fsum), identity weights returning the dequantised rows;
* planted mistakes (the OCP floor rule, 128-value blocks, a dropped scale)
  that one of these pins must catch.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return oracle.f64_to_bf16(v.astype(np.float64))


def all_finite_nonneg_bf16() -> np.ndarray:
    """Every finite non-negative bf16 value, as float64 (0x0000 .. 0x7F7F)."""
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    return oracle.bf16_to_f32(bits).astype(np.float64)


def scale_exponent_by_search(a: float) -> int:
    """The definition, searched: the smallest integer X >= -127 with
    448 * 2**X >= a (math.ldexp is exact), and at most 127."""
    X = -127
    while 448.0 * math.ldexp(1.0, X) < a:
        X += 1
    return min(X, 127)


# ---------------------------------------------------------------- scale exponent

def check_scale_exponent(fn):
    a = all_finite_nonneg_bf16()
    X = fn(a).astype(np.int64)
    assert X.min() >= -127 and X.max() <= 127
    up = 448.0 * np.ldexp(1.0, X)                  # exact in fp64
    down = 448.0 * np.ldexp(1.0, X - 1)
    assert np.all(up >= a), "scale too small: a value would exceed 448"
    assert np.all((X == -127) | (down < a)), "not the smallest power of two"
    # a sample against the one-at-a-time search of the definition
    rng = np.random.default_rng(0)
    for i in rng.choice(len(a), 400, replace=False):
        assert X[i] == scale_exponent_by_search(a[i]), a[i]


def test_scale_exponent_is_its_definition_over_every_bf16_value():
    check_scale_exponent(oracle.mx_scale_exponent)
    # a few by hand: 448 -> 0, just above 448 -> 1, 1.75 -> -8, 1.76 -> -7, 0 -> -127
    X = oracle.mx_scale_exponent(np.array([448.0, 449.0, 1.75, 1.7578125, 0.0]))
    assert list(X) == [0, 1, -8, -7, -127]


def test_e8m0_codes_match_torch_encoding():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu")
    X = np.arange(-127, 128)
    t = torch.from_numpy(np.ldexp(1.0, X).astype(np.float32)).to(torch.float8_e8m0fnu)
    assert np.array_equal(t.view(torch.uint8).numpy().astype(np.int64), X + 127)
    back = torch.from_numpy((X + 127).astype(np.uint8)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(back, oracle.e8m0_decode((X + 127).astype(np.uint8)))


# ---------------------------------------------------------------- quantiser

def check_mx_quantiser(quantize):
    x = rand_bf16((48, 512), 21, scale=3.0)
    x[5, 64:96] = 0                                       # a zero block
    q, s = quantize(x)
    assert q.shape == (48, 512) and s.shape == (48, 16)
    xv = oracle.bf16_to_f32(x).astype(np.float64).reshape(48, 16, 32)
    sc = oracle.e8m0_decode(s)                            # 2**X
    v = np.abs(xv) / sc[:, :, None]                       # exact
    amax = v.max(axis=2)
    nz = np.abs(xv).max(axis=2) > 0
    # no value is pushed past 448, and the power of two is the tightest one
    assert np.all(amax <= 448.0)
    assert np.all(amax[nz] > 224.0)
    # round to nearest on the e4m3 grid (exact quotient: no division error)
    dq = oracle.e4m3_decode(q).reshape(48, 16, 32) * sc[:, :, None]
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(v, 1e-300))), -6) - 3)
    assert np.all(np.abs(xv - dq) / sc[:, :, None] <= step / 2)
    assert np.all(q.reshape(48, 16, 32)[5, 2] == 0) and s[5, 2] == 0


def test_mx_quantiser_bounds():
    check_mx_quantiser(oracle.quantize_rows_mx)


def test_mx_quantiser_closed_form_blocks():
    H = 256
    x = np.zeros((2, H), np.float64)
    x[0, 0:32] = 448.0 * 2.0 ** -5                        # exactly 448 * 2**-5: X = -5, code 448
    grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    x[0, 32:64] = grid[np.linspace(0, 126, 32).astype(int)] * 2.0 ** 3   # grid * 2**3, max 448 * 8
    x[0, 64:96] = -1.0                                    # 1 -> X = -8, code of 256
    x[0, 96] = 448.0 * (1 + 2.0 ** -7)                    # one bf16 ulp above 448 -> X = 1
    x[1, 128:160] = 2.0 ** -130                           # tiny block: clamped at X = -127
    q, s = oracle.quantize_rows_mx(oracle.f64_to_bf16(x))
    X = s.astype(np.int64) - 127
    assert X[0, 0] == -5 and np.all(q[0, 0:32] == 0x7E)
    assert X[0, 1] == 3 and np.array_equal(q[0, 32:64], np.linspace(0, 126, 32).astype(np.uint8))
    assert X[0, 2] == -8 and np.all(q[0, 64:96] == (0x78 | 0x80))   # 256 = 1.0 * 2**8: code 0x78
    assert X[0, 3] == 1 and q[0, 96] == 0x76                        # bf16 452, /2 = 226 -> 224 = 0x76
    assert X[1, 4] == -127 and np.all(q[1, 128:160] == oracle.e4m3_encode(np.float32(2.0 ** -3)))
    # untouched blocks: X = -127 and zero codes
    assert X[1, 0] == -127 and np.all(q[1, :32] == 0)


def test_mx_blocks_are_independent_32_value_blocks():
    # one large value per 32-block changes that block's scale only
    x = np.ones((1, 256), np.float64)
    x[0, 37] = 1000.0
    q, s = oracle.quantize_rows_mx(oracle.f64_to_bf16(x))
    X = s[0].astype(np.int64) - 127
    assert X[1] == oracle.mx_scale_exponent(np.array([1000.0]))[0]
    assert np.all(np.delete(X, 1) == -8)


def test_mx_weight_quantiser_is_per_row_and_32_block():
    w = rand_bf16((2, 4, 128), 5)
    q, s = oracle.quantize_weights_mx(w)
    assert s.shape == (2, 4, 4)
    for e in range(2):
        qr, sr = oracle.quantize_rows_mx(w[e])
        assert np.array_equal(q[e], qr) and np.array_equal(s[e], sr)


def test_dispatch_mx_places_every_copy():
    x = rand_bf16((10, 64), 8)
    q, s = oracle.quantize_rows_mx(x)
    rng = np.random.default_rng(1)
    pair_row = rng.permutation(30).astype(np.int32)
    A, S = oracle.dispatch_mx(q, s, pair_row, 3)
    for p in range(30):
        assert np.array_equal(A[pair_row[p]], q[p // 3]) and np.array_equal(S[pair_row[p]], s[p // 3])


# ---------------------------------------------------------------- GEMM1 (MX)

def mx_problem(T=20, H=128, E=3, N=64, k=2, seed=0):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = np.full((T, k), 1.0 / k, np.float32)
    L = oracle.route_layout(ids, w, E, 1, 8)
    x = rand_bf16((T, H), seed + 1)
    q, s = oracle.quantize_rows_mx(x)
    A, As = oracle.dispatch_mx(q, s, L["pair_row"], k)
    W = rand_bf16((E, N, H), seed + 2, scale=1.0 / math.sqrt(H))
    Wq, Ws = oracle.quantize_weights_mx(W)
    return L, A, As, Wq, Ws


def fsum_entry(A, As, Wq, Ws, e, r, n):
    a = oracle.dequantize_mx(A[r], As[r])
    b = oracle.dequantize_mx(Wq[e, n], Ws[e, n])
    return math.fsum(float(u) * float(v) for u, v in zip(a, b))   # products exact in fp64


def test_gemm1_mx_entries_are_correctly_rounded_sums():
    L, A, As, Wq, Ws = mx_problem()
    Y = oracle.grouped_gemm1_mx(A, As, Wq, Ws, L["expert_offset"])
    rexp = oracle.row_experts(L["expert_offset"], A.shape[0])
    rng = np.random.default_rng(2)
    for _ in range(60):
        r, n = int(rng.integers(A.shape[0])), int(rng.integers(Wq.shape[1]))
        want = oracle.f64_to_bf16(np.array([fsum_entry(A, As, Wq, Ws, rexp[r], r, n)]))[0]
        assert Y[r, n] == want, (r, n)


def test_gemm1_mx_identity_weights_return_dequantised_rows():
    L, A, As, _, _ = mx_problem(H=128, N=128)
    E = 3
    eye = np.broadcast_to(np.eye(128), (E, 128, 128))
    Wq, Ws = oracle.quantize_weights_mx(oracle.f64_to_bf16(eye))
    # row n holds its single 1 in block n // 32 (amax 1 -> X = -8); its other blocks are zero (X = -127)
    blk = np.arange(128) // 32
    assert np.all(Ws[:, np.arange(128), blk] == 127 - 8)
    assert np.count_nonzero(Ws) == E * 128
    Y = oracle.grouped_gemm1_mx(A, As, Wq, Ws, L["expert_offset"])
    # e4m3 values times powers of two are exact in bf16 (3 mantissa bits of 7)
    assert np.array_equal(Y, oracle.f64_to_bf16(oracle.dequantize_mx(A, As)))


# ---------------------------------------------------------------- planted mistakes

def test_planted_ocp_floor_rule_is_caught():
    # the OCP "floor(log2 amax) - 8" exponent lets values reach (448, 512) and saturate
    def floor_rule(a):
        a = np.asarray(a, np.float64)
        _, e = np.frexp(a)
        return np.clip(np.where(a > 0, e - 1 - 8, -127), -127, 127)
    with pytest.raises(AssertionError):
        check_scale_exponent(floor_rule)


def test_planted_128_value_blocks_are_caught():
    def per128(x_bits):
        x = oracle.bf16_to_f32(x_bits)
        T, H = x.shape
        blocks = x.reshape(T, H // 128, 128)
        X = oracle.mx_scale_exponent(np.abs(blocks).max(axis=2))
        q = oracle.e4m3_encode((blocks * np.ldexp(1.0, -X)[:, :, None]).astype(np.float32))
        return q.reshape(T, H), np.repeat((X + 127).astype(np.uint8), 4, axis=1)
    with pytest.raises(AssertionError):
        check_mx_quantiser(per128)


def test_planted_dropped_weight_scale_is_caught():
    L, A, As, Wq, Ws = mx_problem(seed=4)
    bad = oracle.grouped_gemm1_mx(A, As, Wq, np.full_like(Ws, 127), L["expert_offset"])
    rexp = oracle.row_experts(L["expert_offset"], A.shape[0])
    r, n = 3, 5
    want = oracle.f64_to_bf16(np.array([fsum_entry(A, As, Wq, Ws, rexp[r], r, n)]))[0]
    assert bad[r, n] != want
