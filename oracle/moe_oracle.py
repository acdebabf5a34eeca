"""CPU oracle for the MoE stage1 (routing layout, FP8 quant + dispatch, GEMM1) and combine.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the CUDA path computes.  Only the test suite, the smoke check
and the CPU-baseline leg of the benchmark may import it; the product path never
does, and it shares no code, table or constant generator with the CUDA sources.

Sources (web pages, cited by title and section):

* [mori] "poc(cco): MegaMoE stage1 dispatch over SDMA" (mori PR #1): section
  "How it works now" (counting sort by (destination, first expert); quantise
  each token once and store it to every run it is in; GEMM1 reads A rows
  through a rowmap), the recv_layout commit message (receiver counts routes
  per expert, pads each expert to the sort block of 128 rows and writes the
  expert-major tables rowmap / srcmap_em / wts_em / tile tables).
* [mojo] "EPDispatchKernel" (Mojo ep_comm API page): parameters
  ``ep_final_layout`` (each routed row written straight to its final
  contiguous per-expert row) and ``n_local_experts = n_experts // n_ranks``
  (logical groups are contiguous expert ranges).
* [tilepipe] "TilePipe: MoE Communication and Overlap Kernels with CuteDSL",
  section "Overlap" (per-tile semaphores, expert-major GEMM order).

Precision.  The pages fix the activation quantiser's arithmetic only through
the recipe "fp32 per-128-element block scale = amax / 448, e4m3 codes", so the
quantiser runs in fp32 exactly as stated (the code is an integer decided by
floating point, and both sides decide it in fp32).  Everything else here (the
router softmax, the dequantised matmul, the weighted combine) is computed in
fp64 and rounded once to the output format; the pages leave that precision
open.

Readings where the pages are silent:

* top-k ties go to the lower expert id; a token's slots are ordered by
  descending probability;
* logical group g holds experts [g*E/G, (g+1)*E/G), so the sort key
  (group, expert) orders like the expert id, and within an expert rows follow
  ascending (token, slot);
* a token's "first expert" is the smallest expert id among its k routes;
* a block whose amax is 0 gets scale 0 and all-zero codes;
* e4m3 conversion rounds to nearest even and saturates to +-448;
* weight scales are per 128x128 block (n-block x k-block);
* tiles past ``num_tiles`` hold tile_expert = -1, tile_row_begin = T*k,
  tile_rows = 0, and every rowmap slot not holding a row holds -1.

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
brute force, closed forms, invariants or library routines; none is unpinned
(the MXFP8 functions at the end by ``tests/test_oracle_mx.py``).
"""
from __future__ import annotations

import numpy as np

BLOCK = 128          # quantisation block along the hidden dimension
E4M3_MAX = 448.0     # largest finite e4m3 magnitude


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (bf16 is the top half of an fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _round_to_grid(a: np.ndarray, mant_bits: int, min_exp: int) -> np.ndarray:
    """Round non-negative fp64 values ``a`` to the nearest point of a binary
    floating-point grid with ``mant_bits`` stored mantissa bits and smallest
    normal exponent ``min_exp``; ties go to the even neighbour.

    The spacing of the grid around ``a`` is 2**(max(floor(log2 a), min_exp) - mant_bits);
    below 2**min_exp the spacing stays at the subnormal step.  Dividing by a
    power of two is exact, and ``np.rint`` rounds half to even."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a > 0
    _, e = np.frexp(a[nz])                 # a = m * 2**e with m in [0.5, 1)
    exp = np.maximum(e - 1, min_exp)       # floor(log2 a), clamped to the normal range
    quantum = np.ldexp(1.0, exp - mant_bits)
    out[nz] = np.rint(a[nz] / quantum) * quantum
    return out


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """Values -> bfloat16 bit patterns, one rounding to nearest even (no double
    rounding through fp32).  bf16: 8 exponent bits (bias 127), 7 mantissa bits.
    Finite inputs whose rounded magnitude exceeds the largest bf16 become inf."""
    v = np.asarray(v, dtype=np.float64)
    mag = _round_to_grid(np.abs(v), 7, -126)
    mag = np.where(mag > 3.3895313892515355e38, np.inf, mag)   # (2 - 2**-7) * 2**127
    signed = np.where(np.signbit(v), -mag, mag)
    # every rounded magnitude is exactly representable in fp32; bf16 is its top half
    return (signed.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ("fn" variant) code -> value, from the format's definition:
    sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is
    subnormal (m * 2**-9); S.1111.111 is NaN; there are no infinities."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


# The 127 non-negative finite e4m3 values, in code order 0x00..0x7E (strictly increasing).
_E4M3_POS = e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float32 values -> e4m3 codes: round to nearest even on the e4m3 grid
    (3 mantissa bits, smallest normal 2**-6, subnormal step 2**-9), saturating
    magnitudes above 448 to 448.  The sign is carried from the sign bit, so -0
    and negative values that round to zero give 0x80."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    r = _round_to_grid(a, 3, -6)
    r = np.minimum(r, E4M3_MAX)            # satfinite
    code = np.searchsorted(_E4M3_POS, r).astype(np.uint8)
    assert np.array_equal(_E4M3_POS[code], r), "rounded value off the e4m3 grid"
    return np.where(np.signbit(v), code | np.uint8(0x80), code).astype(np.uint8)


# --------------------------------------------------------------------------
# Router (input preparation; the layout starts from its top-k pairs)
# --------------------------------------------------------------------------

def router_topk(logits: np.ndarray, k: int):
    """Softmax over each token's E logits (fp64, max subtracted), the k largest
    probabilities (ties: lower expert id first), slots in descending order, and
    weights renormalised to sum to one over the selected k.

    Returns (topk_ids int32 [T, k], topk_w float32 [T, k])."""
    logits = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = logits.shape
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    expert = np.arange(E)
    for t in range(T):
        order = np.lexsort((expert, -p[t]))      # primary key: -p, then expert id
        sel = order[:k]
        ids[t] = sel
        w[t] = (p[t, sel] / p[t, sel].sum()).astype(np.float32)
    return ids, w


# --------------------------------------------------------------------------
# Routing layout: stable counting sort by (group, expert)
# --------------------------------------------------------------------------

def max_tiles(T: int, k: int, E: int, block_m: int = BLOCK) -> int:
    """Capacity of the tile tables: sum_e ceil(count_e / BM) <= (T*k + E*(BM-1)) / BM
    (each expert pads to the sort block, the recv_layout commit's "up to
    epr * 128 rows past the routes"), and never more tiles than routed pairs."""
    return min(T * k, (T * k + E * (block_m - 1)) // block_m)


def route_layout(topk_ids: np.ndarray, topk_w: np.ndarray, E: int, G: int, block_m: int = BLOCK):
    """Expert-major layout of the T*k (token, slot) pairs ([mori] "How it works
    now": counting sort; recv_layout commit: per-expert counts, padding to the
    sort block, expert-major tables; [mojo] ep_final_layout: each pair's row is
    its final row in one dense per-expert range).

    Pair p = t*k + j goes to dense row ``pair_row[p]``; rows are ordered by the
    key (group, expert) and, within a key, by p (a stable sort).  Returns a dict
    of int32 / float32 arrays (names as in the C ABI)."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    assert ids.min() >= 0 and ids.max() < E, "expert id out of range"
    assert E % G == 0
    epg = E // G                              # experts per logical group ([mojo] n_local_experts)
    flat = ids.reshape(-1)
    group = flat // epg
    key = group * E + flat                    # (group, expert), lexicographic
    row_pair = np.argsort(key, kind="stable")
    pair_row = np.empty_like(row_pair)
    pair_row[row_pair] = np.arange(T * k)

    count = np.bincount(flat, minlength=E)
    expert_offset = np.concatenate([[0], np.cumsum(count)])
    tiles = (count + block_m - 1) // block_m
    expert_tile_offset = np.concatenate([[0], np.cumsum(tiles)])
    group_offset = expert_offset[np.arange(G + 1) * epg]
    num_tiles = int(expert_tile_offset[E])

    first = ids.min(axis=1)                   # each token's first (smallest) expert
    fcount = np.bincount(first, minlength=E)
    token_order = np.argsort(first, kind="stable")
    ready_tokens = np.cumsum(fcount)

    cap = max_tiles(T, k, E, block_m)
    assert num_tiles <= cap
    tile_expert = np.full(cap, -1, np.int64)
    tile_row_begin = np.full(cap, T * k, np.int64)
    tile_rows = np.zeros(cap, np.int64)
    rowmap = np.full(cap * block_m, -1, np.int64)
    for e in range(E):
        for i in range(tiles[e]):
            m = expert_tile_offset[e] + i
            begin = expert_offset[e] + i * block_m
            rows = min(block_m, count[e] - i * block_m)
            tile_expert[m] = e
            tile_row_begin[m] = begin
            tile_rows[m] = rows
            rowmap[m * block_m: m * block_m + rows] = begin + np.arange(rows)

    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return {
        "count": i32(count),
        "expert_offset": i32(expert_offset),
        "expert_tile_offset": i32(expert_tile_offset),
        "group_offset": i32(group_offset),
        "ready_tokens": i32(ready_tokens),
        "pair_row": i32(pair_row),
        "row_pair": i32(row_pair),
        "row_weight": np.asarray(topk_w, dtype=np.float32).reshape(-1)[row_pair],
        "rowmap": i32(rowmap),
        "tile_expert": i32(tile_expert),
        "tile_row_begin": i32(tile_row_begin),
        "tile_rows": i32(tile_rows),
        "num_tiles": np.array([num_tiles], dtype=np.int32),
        "token_order": i32(token_order),
        "max_tiles": cap,
    }


# --------------------------------------------------------------------------
# FP8 quantisation and dispatch
# --------------------------------------------------------------------------

def quantize_rows(x_bits: np.ndarray):
    """Per token and per 128-element block along H: amax = max |x|,
    scale = amax / 448 (fp32), code = e4m3(x / scale) (fp32 division, then
    round to nearest even, saturating).  A block with amax 0 gets scale 0 and
    zero codes.  ([mori] "How it works now": each token is quantised once.)

    x_bits: bf16 bit patterns [T, H].  Returns (q uint8 [T, H], scale f32 [T, H/128])."""
    x = bf16_to_f32(x_bits)
    T, H = x.shape
    assert H % BLOCK == 0
    xb = x.reshape(T, H // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=2)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    v = (xb / safe[:, :, None]).astype(np.float32)
    q = e4m3_encode(v)
    q = np.where((scale > 0)[:, :, None], q, np.uint8(0))
    return q.reshape(T, H).astype(np.uint8), scale


def dispatch(q: np.ndarray, scale: np.ndarray, pair_row: np.ndarray, k: int):
    """Scatter: token t's codes and scales go to each of its k rows
    ``pair_row[t*k + j]`` ([mori] "How it works now": the quant writes each row
    once to every run it is in).

    Returns (A uint8 [T*k, H], A_scale f32 [H/128, T*k]); the scale tensor is
    stored block-major so that one block's scales for consecutive rows are
    contiguous."""
    T, H = q.shape
    R = T * k
    A = np.zeros((R, H), dtype=np.uint8)
    A_scale = np.zeros((H // BLOCK, R), dtype=np.float32)
    rows = np.asarray(pair_row, dtype=np.int64).reshape(T, k)
    for j in range(k):
        A[rows[:, j]] = q
        A_scale[:, rows[:, j]] = scale.T
    return A, A_scale


def quantize_weights(w_bits: np.ndarray):
    """Expert weights bf16 [E, N, H] -> (codes uint8 [E, N, H], scale f32
    [E, N/128, H/128]), one scale per 128 (n) x 128 (k) block, with the same
    amax / 448 rule as the activations."""
    w = bf16_to_f32(w_bits)
    E, N, H = w.shape
    assert N % BLOCK == 0 and H % BLOCK == 0
    wb = w.reshape(E, N // BLOCK, BLOCK, H // BLOCK, BLOCK)
    amax = np.abs(wb).max(axis=(2, 4))
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    v = (wb / safe[:, :, None, :, None]).astype(np.float32)
    q = e4m3_encode(v)
    q = np.where((scale > 0)[:, :, None, :, None], q, np.uint8(0))
    return q.reshape(E, N, H).astype(np.uint8), scale


def dequantize_rows(A: np.ndarray, A_scale: np.ndarray, rows) -> np.ndarray:
    """Dense rows of the dispatch buffer back to values: q * scale (fp64, exact)."""
    rows = np.asarray(rows, dtype=np.int64)
    H = A.shape[1]
    vals = e4m3_decode(A[rows]).reshape(len(rows), H // BLOCK, BLOCK)
    return (vals * A_scale[:, rows].T.astype(np.float64)[:, :, None]).reshape(len(rows), H)


def dequantize_weights(Wq_e: np.ndarray, Ws_e: np.ndarray) -> np.ndarray:
    """One expert's weight codes [N, H] and scales [N/128, H/128] -> fp64 values."""
    N, H = Wq_e.shape
    vals = e4m3_decode(Wq_e).reshape(N // BLOCK, BLOCK, H // BLOCK, BLOCK)
    return (vals * Ws_e.astype(np.float64)[:, None, :, None]).reshape(N, H)


def identity_expert(A: np.ndarray, A_scale: np.ndarray, rows) -> np.ndarray:
    """The identity expert used by the bandwidth sweep: Y = bf16(q * scale)."""
    return f64_to_bf16(dequantize_rows(A, A_scale, rows))


# --------------------------------------------------------------------------
# GEMM1 and combine
# --------------------------------------------------------------------------

def row_experts(expert_offset: np.ndarray, R: int) -> np.ndarray:
    """Expert of every dense row, from the exclusive prefix of expert counts."""
    eo = np.asarray(expert_offset, dtype=np.int64)
    return np.searchsorted(eo, np.arange(R), side="right") - 1


def grouped_gemm1(A, A_scale, Wq, W_scale, expert_offset, rows=None):
    """Y[r, n] = bf16( sum_k deq(A)[r, k] * deq(W_e)[n, k] ) for each dense row r
    of expert e, in fp64 ([mori] "What": GEMM1 reads its A rows in place through
    the rowmap; the expert of a row follows from the expert-major offsets).

    ``rows``: dense row indices to compute (default all).  Returns bf16 bit
    patterns [len(rows), N]."""
    R = A.shape[0]
    rows = np.arange(R) if rows is None else np.asarray(rows, dtype=np.int64)
    N = Wq.shape[1]
    rexp = row_experts(expert_offset, R)[rows]
    out = np.zeros((len(rows), N), dtype=np.uint16)
    for e in np.unique(rexp):
        sel = np.nonzero(rexp == e)[0]
        a = dequantize_rows(A, A_scale, rows[sel])
        w = dequantize_weights(Wq[e], W_scale[e])
        out[sel] = f64_to_bf16(a @ w.T)
    return out


def combine(Y_bits: np.ndarray, pair_row: np.ndarray, topk_w: np.ndarray, tokens=None):
    """out[t] = bf16( sum_{j=0}^{k-1} w[t, j] * Y[pair_row[t*k + j]] ) in fp64,
    slots in ascending order: the weighted gather of each token's k expert
    outputs back into token order ([tilepipe] "Communication Kernels" names the
    combine as the counterpart of the dispatch; the router weighting and the
    fp64 accumulation in slot order are this oracle's reading).

    Returns bf16 bit patterns [len(tokens), D]."""
    w = np.asarray(topk_w, dtype=np.float32)
    T, k = w.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    rows = np.asarray(pair_row, dtype=np.int64).reshape(T, k)[tokens]
    acc = np.zeros((len(tokens), Y_bits.shape[1]), dtype=np.float64)
    for j in range(k):
        acc += w[tokens, j].astype(np.float64)[:, None] * bf16_to_f32(Y_bits[rows[:, j]]).astype(np.float64)
    return f64_to_bf16(acc)


# --------------------------------------------------------------------------
# Per-(token, group) send runs (the next step of the path: no CUDA kernel reads
# these yet; the dense dispatch above is what the kernels compute)
# --------------------------------------------------------------------------

def group_runs(topk_ids: np.ndarray, E: int, G: int, row_pair: np.ndarray):
    """One send row per (token, logical group) that the token routes into,
    the rows of group g forming run g ([mori] "What": the sender quantises each
    token once into a send buffer grouped by destination; "How it works now":
    a counting sort by (destination, first expert) places every token's row
    so that a landed prefix of a run is a prefix of experts).  Within run g
    rows follow (the token's smallest expert id in g, token).  GEMM1 would read
    dense expert-major row r (pair p = row_pair[r] of token t = p // k, expert
    e) from send row ``send_row[t, e // (E/G)]``: ``gather_row[r]``.

    Returns a dict: run_offset [G+1]; send_token [S] (token of each send row);
    send_row [T, G] (-1 where the token has no route into g); run_ready [E]
    (for expert e of group g, the end of the run prefix that holds every token
    routed to e); gather_row [T*k]."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    assert E % G == 0
    epg = E // G
    grp = ids // epg
    send_row = np.full((T, G), -1, np.int64)
    run_offset = np.zeros(G + 1, np.int64)
    run_ready = np.zeros(E, np.int64)
    send_token = []
    for g in range(G):
        in_g = grp == g
        toks = np.nonzero(in_g.any(axis=1))[0]
        first = np.where(in_g, ids, E).min(axis=1)[toks]       # smallest expert of g per token
        order = toks[np.argsort(first, kind="stable")]
        run_offset[g + 1] = run_offset[g] + len(order)
        send_row[order, g] = run_offset[g] + np.arange(len(order))
        send_token.append(order)
        run_ready[g * epg:(g + 1) * epg] = run_offset[g] + np.cumsum(np.bincount(first - g * epg, minlength=epg))
    rp = np.asarray(row_pair, dtype=np.int64)
    gather_row = send_row[rp // k, ids.reshape(-1)[rp] // epg]
    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return {"run_offset": i32(run_offset), "send_token": i32(np.concatenate(send_token)),
            "send_row": i32(send_row), "run_ready": i32(run_ready), "gather_row": i32(gather_row)}


def dispatch_runs(q: np.ndarray, scale: np.ndarray, send_token: np.ndarray):
    """The send buffer: each send row holds its token's codes once, scales
    block-major as in ``dispatch`` (A_send [S, H], A_send_scale [H/128, S])."""
    st = np.asarray(send_token, dtype=np.int64)
    return q[st].copy(), np.ascontiguousarray(scale[st].T)


# --------------------------------------------------------------------------
# MXFP8 variant: e8m0 (power-of-two) scales per 32 values
# --------------------------------------------------------------------------
#
# [mori] (the stage1 page's first commit: "GEMM1 reads its A rows and e8m0
# scales through a rowmap"; the quant-LDS commit packs "the e8m0 scales four
# per dword") quantises with power-of-two scales.  The pages do not state the
# block size or how the power of two is chosen.  Readings:
#   * the block is 32 consecutive values along the reduction dimension (the
#     OCP microscaling block; the tensor core's block-scaled FP8 MMA consumes
#     one scale per 32 values), for activations and for each weight row alike;
#   * the scale is the fp32 recipe's amax / 448 rounded UP to a power of two,
#     2**X with X the smallest integer such that 448 * 2**X >= amax (so no
#     value is pushed past 448 by the scale), clamped to the e8m0 range
#     [-127, 127]; an all-zero block gets X = -127;
#   * e8m0 code = X + 127 (0xFF, NaN, is never produced); codes of the values
#     are e4m3(x / 2**X), round to nearest even, saturating.

MX_BLOCK = 32
E8M0_MIN_EXP, E8M0_MAX_EXP = -127, 127


def mx_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer X with 448 * 2**X >= amax, clamped to [-127, 127]
    (amax == 0 gives -127).  Exact: amax = m * 2**e with m in [0.5, 1)
    (frexp), so 448 * 2**X = 0.875 * 2**(X + 9) >= m * 2**e holds for
    X = e - 9 when m <= 0.875 and needs X = e - 8 otherwise."""
    a = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(a)
    X = np.where(m <= 0.875, e - 9, e - 8).astype(np.int64)
    X = np.where(a > 0, X, E8M0_MIN_EXP)
    return np.clip(X, E8M0_MIN_EXP, E8M0_MAX_EXP)


def e8m0_decode(codes: np.ndarray) -> np.ndarray:
    """e8m0 code -> 2**(code - 127) (fp64); code 0xFF is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def _mx_quantize_blocks(vals: np.ndarray):
    """vals [..., nb, 32] float32 -> (codes uint8 same shape, e8m0 uint8 [..., nb])."""
    amax = np.abs(vals).max(axis=-1)
    X = mx_scale_exponent(amax)
    scaled = (vals.astype(np.float64) * np.ldexp(1.0, -X)[..., None]).astype(np.float32)   # exact
    return e4m3_encode(scaled), (X + 127).astype(np.uint8)


def quantize_rows_mx(x_bits: np.ndarray):
    """Per token and per 32-value block along H: X from the block's amax as
    above, code = e4m3(x / 2**X).  x_bits: bf16 [T, H] -> (q uint8 [T, H],
    e8m0 uint8 [T, H/32])."""
    x = bf16_to_f32(x_bits)
    T, H = x.shape
    assert H % MX_BLOCK == 0
    q, s = _mx_quantize_blocks(x.reshape(T, H // MX_BLOCK, MX_BLOCK))
    return q.reshape(T, H), s


def quantize_weights_mx(w_bits: np.ndarray):
    """Expert weights bf16 [E, N, H] -> (codes uint8 [E, N, H], e8m0 uint8
    [E, N, H/32]): one scale per weight row n and 32-value block along K."""
    w = bf16_to_f32(w_bits)
    E, N, H = w.shape
    assert H % MX_BLOCK == 0
    q, s = _mx_quantize_blocks(w.reshape(E, N, H // MX_BLOCK, MX_BLOCK))
    return q.reshape(E, N, H), s


def dequantize_mx(q: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    """codes [..., H] and e8m0 scales [..., H/32] -> fp64 values (exact)."""
    vals = e4m3_decode(q)
    sh = vals.shape
    v = vals.reshape(sh[:-1] + (sh[-1] // MX_BLOCK, MX_BLOCK)) * e8m0_decode(e8m0)[..., None]
    return v.reshape(sh)


def dispatch_mx(q: np.ndarray, e8m0: np.ndarray, pair_row: np.ndarray, k: int):
    """The dispatch of the MX variant: token t's codes and e8m0 scales go to
    each of its k dense rows pair_row[t*k + j], as in ``dispatch``.
    Returns (A uint8 [T*k, H], A_e8m0 uint8 [T*k, H/32])."""
    T, H = q.shape
    R = T * k
    A = np.zeros((R, H), dtype=np.uint8)
    S = np.zeros((R, H // MX_BLOCK), dtype=np.uint8)
    rows = np.asarray(pair_row, dtype=np.int64).reshape(T, k)
    for j in range(k):
        A[rows[:, j]] = q
        S[rows[:, j]] = e8m0
    return A, S


def grouped_gemm1_mx(A, A_e8m0, Wq, W_e8m0, expert_offset, rows=None):
    """Y[r, n] = bf16( sum_k deq(A)[r, k] * deq(W_e)[n, k] ) in fp64 for each
    dense row r of expert e, with the MX scales (every product is exact)."""
    R = A.shape[0]
    rows = np.arange(R) if rows is None else np.asarray(rows, dtype=np.int64)
    N = Wq.shape[1]
    rexp = row_experts(expert_offset, R)[rows]
    out = np.zeros((len(rows), N), dtype=np.uint16)
    for e in np.unique(rexp):
        sel = np.nonzero(rexp == e)[0]
        a = dequantize_mx(A[rows[sel]], A_e8m0[rows[sel]])
        w = dequantize_mx(Wq[e], W_e8m0[e])
        out[sel] = f64_to_bf16(a @ w.T)
    return out
