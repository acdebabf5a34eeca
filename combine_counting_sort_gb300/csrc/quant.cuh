// quant.cuh: per-token FP8 quantise-once + scatter, shared by the dispatch
// kernel and the producer role of the fused stage1 kernel.
//
// ("How it works now" and the quant-once commit of the mori stage1 page: a
// token's bf16 row is read and quantised once and stored to its row in every
// run it belongs to.)  One warp per token.  A lane owns 16 consecutive values
// (two 16-byte loads), so a 128-value quantisation block is 8 lanes and a warp
// round covers 512 values; the block amax is a 3-step xor-shuffle reduction.
// The 16 codes of a lane are one 16-byte store, so a warp's store covers 512
// contiguous bytes of the destination row: fully coalesced with no
// shared-memory staging.  (The page's LDS swizzle fixes a lane layout that
// wrote two 16-byte pieces 32 bytes apart; this layout never has that problem.)
#pragma once

#include "common.cuh"

namespace moe {

MOE_DEV void unpack16(const uint4& a, const uint4& b, float (&f)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) { f[2 * i] = bf16_lo(w[i]); f[2 * i + 1] = bf16_hi(w[i]); }
}

// 16 values of one quantisation block (this lane's share) -> 16 e4m3 codes:
// code = e4m3_rn_satfinite(RN(x / scale)) with the IEEE fp32 quotient; scale 0
// -> codes 0.
//
// Fast path: v' = RN(x * RN(1/scale)).  Both roundings are relative errors of
// at most 2^-24, so v' is within 3 fp32 ulps of the exact quotient RN(x/scale),
// and both lie on the same side of every e4m3 rounding boundary unless v' is
// within 4 ulps of one.  In the e4m3 normal range those boundaries (midpoints
// between adjacent codes) are exactly the fp32 values whose low 20 mantissa
// bits are 0x80000; binade edges are codes, not boundaries.  So v' gives the
// same code as the quotient unless its low 20 bits lie in a window around
// 0x80000 or it lies below 2^-6 (the e4m3 subnormal range); a lane holding any
// such value recomputes its 16 values with the IEEE division, and so does a
// lane whose scale is below the fp32 normal range (where RN(1/scale) is not
// within 2^-24, or overflows).
//
// The window test is ((bits(v') + 4) & 0xFFFF0) == 0x80000, i.e. low 20 bits
// in [0x80000 - 4, 0x80000 + 11], a superset of the +-4 needed; it is folded
// into a running minimum of ((bits + 4) & 0xFFFF0) ^ 0x80000 (zero = hit), and
// the subnormal test into a running minimum of |v'|, so the fast path costs
// five instructions per value.
MOE_DEV uint4 quant16(const float (&f)[16], float scale) {
  uint32_t p[4] = {0u, 0u, 0u, 0u};
  if (scale > 0.0f) {
    const float inv = __frcp_rn(scale);
    float v[16];
    uint32_t near_mid = 0xFFFFFFFFu;
    float min_abs = INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = __fmul_rn(f[i], inv);
      near_mid = min(near_mid, ((__float_as_uint(v[i]) + 4u) & 0xFFFF0u) ^ 0x80000u);
      min_abs = fminf(min_abs, fabsf(v[i]));
    }
    if (near_mid == 0u || min_abs < 0x1p-6f || scale < 0x1p-126f) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __fdiv_rn(f[i], scale);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = e4m3x2(v[4 * i + 0], v[4 * i + 1]);
      const uint32_t hi = e4m3x2(v[4 * i + 2], v[4 * i + 3]);
      p[i] = lo | (hi << 16);
    }
  }
  return make_uint4(p[0], p[1], p[2], p[3]);
}

// amax over the 8 lanes of a quantisation block (lanes 8g..8g+7)
MOE_DEV float block_amax8(const float (&f)[16]) {
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(f[i]));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
  return am;
}

// One slice [c0, c0 + 512*ROUNDS) of token t (the mori page's --split: a
// token's hidden dimension shared by several warps): all 2*ROUNDS 16-byte
// loads of the lane are issued before any arithmetic, so each warp keeps
// ROUNDS KB of the row in flight; then the 512-column rounds are quantised
// and stored to the token's k rows.  `myrow` as in quant_scatter_token.
template <int ROUNDS>
MOE_DEV void quant_scatter_slice(const uint16_t* __restrict__ x, int H, int t, int c0, int k, long long R,
                                 int myrow, uint8_t* __restrict__ A, float* __restrict__ A_scale) {
  const int lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4 raw[2 * ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int col = c0 + r * 512 + lane * 16;
    raw[2 * r] = make_uint4(0, 0, 0, 0);
    raw[2 * r + 1] = raw[2 * r];
    if (col < H) {
      raw[2 * r] = __ldcs(xr + col / 8);
      raw[2 * r + 1] = __ldcs(xr + col / 8 + 1);
    }
  }
  uint4 q[ROUNDS];
  float sc[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    float f[16];
    unpack16(raw[2 * r], raw[2 * r + 1], f);
    sc[r] = __fdiv_rn(block_amax8(f), 448.0f);
    q[r] = quant16(f, sc[r]);
  }
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, myrow, j);
    if (row < 0) continue;
    uint8_t* arow = A + (size_t)row * H;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int col = c0 + r * 512 + lane * 16;
      if (col < H) {
        *reinterpret_cast<uint4*>(arow + col) = q[r];
        if ((lane & 7) == 0) A_scale[(size_t)(col / kQBlock) * R + row] = sc[r];
      }
    }
  }
}

// Quantise token t once (scale = amax/448 per 128 values) and store codes and
// scales to each of its k rows; `myrow` is pair_row[t*k + lane] for lanes < k
// (-1 elsewhere / for skipped pairs).  Whole warp, converged.
MOE_DEV void quant_scatter_token(const uint16_t* __restrict__ x, int H, int t, int k, long long R, int myrow,
                                 uint8_t* __restrict__ A, float* __restrict__ A_scale) {
  const int lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  for (int c0 = 0; c0 < H; c0 += 1024) {
    // two rounds of 512 values in flight
    const int colA = c0 + lane * 16, colB = colA + 512;
    const bool actA = colA < H, actB = colB < H;
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, b0 = a0, b1 = a0;
    if (actA) { a0 = __ldcs(xr + colA / 8); a1 = __ldcs(xr + colA / 8 + 1); }
    if (actB) { b0 = __ldcs(xr + colB / 8); b1 = __ldcs(xr + colB / 8 + 1); }
    float fa[16], fb[16];
    unpack16(a0, a1, fa);
    unpack16(b0, b1, fb);
    const float sA = __fdiv_rn(block_amax8(fa), 448.0f);
    const float sB = __fdiv_rn(block_amax8(fb), 448.0f);
    const uint4 qA = quant16(fa, sA);
    const uint4 qB = quant16(fb, sB);
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, myrow, j);
      if (r < 0) continue;
      uint8_t* arow = A + (size_t)r * H;
      if (actA) {
        *reinterpret_cast<uint4*>(arow + colA) = qA;
        if ((lane & 7) == 0) A_scale[(size_t)(colA / kQBlock) * R + r] = sA;
      }
      if (actB) {
        *reinterpret_cast<uint4*>(arow + colB) = qB;
        if ((lane & 7) == 0) A_scale[(size_t)(colB / kQBlock) * R + r] = sB;
      }
    }
  }
}

}  // namespace moe
