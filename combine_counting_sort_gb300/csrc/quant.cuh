// quant.cuh: per-token FP8 quantise-once + scatter, shared by the dispatch
// kernel and the producer role of the fused stage1 kernel.
//
// ("How it works now" and the quant-once commit of the mori stage1 page: a
// token's bf16 row is read and quantised once and stored to its row in every
// run it belongs to.)  A warp quantises a slice of 512 x ROUNDS columns of one
// token at a time (the dispatch kernel splits a token's row into slices over
// several warps; a fused-stage1 producer warp walks whole tokens).  A lane owns 16 consecutive values
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
// at most 2^-24, so v' is within 3 * 2^-24 (relative) of the exact quotient
// q = RN(x/scale).  The e4m3 rounding (nearest-even, saturating) is monotonic,
// so if it maps the bracket lo = RN(v' * (1 - 2^-21)) and hi = RN(v' *
// (1 + 2^-21)) to the same code, q (inside the bracket: 2^-21 - 2^-24 >
// 3 * 2^-24) has that code too.  Where v' is an fp32 subnormal the bounds do
// not hold, but there |q| < 2^-10 as well and both round to the signed zero of
// their (exact) sign.
//
// A value whose bracket straddles a rounding boundary takes the IEEE division,
// and so does every value of a lane whose scale is below the fp32 normal range
// (RN(1/scale) not within 2^-24, or overflowing).  With bf16 inputs straddling
// is common (q often lands exactly on a midpoint between two codes: ~0.5% of
// values, so most warps hold one somewhere in a 16-value round), so only the
// flagged values are divided: the warp loops while any lane has one left,
// each lane taking its next flagged value (selected from the 16 by compare
// and select, so nothing is indexed dynamically).  Whole warp, converged.
MOE_DEV uint4 quant16(const float (&f)[16], float scale) {
  constexpr float kBelow = 1.0f - 0x1p-21f, kAbove = 1.0f + 0x1p-21f;
  uint32_t p[4] = {0u, 0u, 0u, 0u};
  uint32_t need = 0u;   // bit j: value j takes the IEEE division
  if (scale > 0.0f) {
    const float inv = __frcp_rn(scale);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __fmul_rn(f[4 * i + j], inv);
      const uint32_t below = e4m3x2(__fmul_rn(v[0], kBelow), __fmul_rn(v[1], kBelow)) |
                             ((uint32_t)e4m3x2(__fmul_rn(v[2], kBelow), __fmul_rn(v[3], kBelow)) << 16);
      const uint32_t above = e4m3x2(__fmul_rn(v[0], kAbove), __fmul_rn(v[1], kAbove)) |
                             ((uint32_t)e4m3x2(__fmul_rn(v[2], kAbove), __fmul_rn(v[3], kAbove)) << 16);
      // one bit per differing byte: bytes 0..3 -> bits 0..3 (the multiply gathers them into bits 24..27)
      const uint32_t bytes = __vcmpne4(below, above) & 0x01010101u;
      need |= ((bytes * 0x01020408u) >> 24) << (4 * i);
      p[i] = below;
    }
    if (scale < 0x1p-126f) need = 0xFFFFu;
  }
  while (__any_sync(0xffffffffu, need != 0u)) {
    if (need != 0u) {
      const int j = __ffs(need) - 1;
      need &= need - 1u;
      float xj = f[0];
#pragma unroll
      for (int k = 1; k < 16; ++k) xj = j == k ? f[k] : xj;
      const uint32_t c = e4m3x2(__fdiv_rn(xj, scale), 0.0f) & 0xFFu;
      const int w = j >> 2, sh = (j & 3) * 8;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (w == k) p[k] = (p[k] & ~(0xFFu << sh)) | (c << sh);
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
// and stored to the token's k rows.  `myrow` is pair_row[t*k + lane] for
// lanes < k (-1 elsewhere / for skipped pairs).  Whole warp, converged.
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

// As quant_scatter_slice, but the codes go to shared memory (the row's bytes
// [c0, c0 + 512*ROUNDS) at row_s + c0, 16 bytes per lane per round) for bulk
// copies to the token's rows; the block scales still go to every row directly.
template <int ROUNDS>
MOE_DEV void quant_stage_slice(const uint16_t* __restrict__ x, int H, int t, int c0, int k, long long R,
                               int myrow, float* __restrict__ A_scale, uint32_t row_s) {
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
  float sc[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    float f[16];
    unpack16(raw[2 * r], raw[2 * r + 1], f);
    sc[r] = __fdiv_rn(block_amax8(f), 448.0f);
    const uint4 q = quant16(f, sc[r]);
    const int col = c0 + r * 512 + lane * 16;
    if (col < H)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row_s + (uint32_t)col), "r"(q.x), "r"(q.y),
                   "r"(q.z), "r"(q.w)
                   : "memory");
  }
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, myrow, j);
    if (row < 0) continue;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int col = c0 + r * 512 + lane * 16;
      if (col < H && (lane & 7) == 0) A_scale[(size_t)(col / kQBlock) * R + row] = sc[r];
    }
  }
}

}  // namespace moe
