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
// The quotient by one fused-multiply-add correction of the reciprocal product
// (Markstein's division step, as given for FMA machines in "Computation of
// elementary functions on the IBM RISC System/6000 processor", 1990, and in
// the Handbook of Floating-Point Arithmetic, division chapter): with
// r = RN(1/scale), q0 = RN(x r), rem = RN(x - q0 scale) (one fma),
// q = RN(q0 + rem r) (one fma); x = +-0 keeps its own sign.  q is not always
// the correctly rounded fp32 quotient, but its e4m3 code is: for every bf16
// block maximum a with scale = RN(a / 448) >= 2^-80 and every bf16 x with
// |x| <= a, the code of q equals the code of the IEEE quotient (all 1.06e9
// pairs compared on the GPU against the IEEE division).  Below 2^-80 (the
// residual can fall under the fp32 normal range) and for a non-finite scale
// the lane divides instead (rare: block maxima under 2^-71).  No branch on the
// values, so a warp stays converged.
MOE_DEV uint4 quant16(const float (&f)[16], float scale) {
  uint32_t p[4] = {0u, 0u, 0u, 0u};
  if (scale >= 0x1p-80f && scale <= 0x1.fffffep127f) {
    const float inv = __frcp_rn(scale);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = f[4 * i + j];
        const float q0 = __fmul_rn(x, inv);
        const float rem = __fmaf_rn(-q0, scale, x);
        const float q = __fmaf_rn(rem, inv, q0);
        v[j] = x == 0.0f ? x : q;
      }
      p[i] = e4m3x2(v[0], v[1]) | ((uint32_t)e4m3x2(v[2], v[3]) << 16);
    }
  } else if (scale > 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[i] = e4m3x2(__fdiv_rn(f[4 * i], scale), __fdiv_rn(f[4 * i + 1], scale)) |
             ((uint32_t)e4m3x2(__fdiv_rn(f[4 * i + 2], scale), __fdiv_rn(f[4 * i + 3], scale)) << 16);
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

// The slice's block scales to the token's k rows with every lane storing: a
// round's 4 scales sit in lanes 0, 8, 16, 24 (sc[r]); lane l takes row
// l / 4 (of each group of 8 rows) and block l % 4 of every round, so one
// store instruction covers 8 rows x 4 blocks instead of 4 lanes' worth.
template <int ROUNDS>
MOE_DEV void store_block_scales(const float (&sc)[ROUNDS], int H, int c0, int k, long long R, int myrow,
                                float* __restrict__ A_scale) {
  const int lane = threadIdx.x & 31;
  const int part = lane & 3;
  float v[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) v[r] = __shfl_sync(0xffffffffu, sc[r], 8 * part);
  for (int jb = 0; jb < k; jb += 8) {
    const int j = jb + (lane >> 2);
    const int row = __shfl_sync(0xffffffffu, myrow, j & 31);
    if (j < k && row >= 0) {
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        const int col = c0 + r * 512 + part * kQBlock;
        if (col < H) A_scale[(size_t)(col / kQBlock) * R + row] = v[r];
      }
    }
  }
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
  store_block_scales<ROUNDS>(sc, H, c0, k, R, myrow, A_scale);
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, myrow, j);
    if (row < 0) continue;
    uint8_t* arow = A + (size_t)row * H;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int col = c0 + r * 512 + lane * 16;
      if (col < H) *reinterpret_cast<uint4*>(arow + col) = q[r];
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
  store_block_scales<ROUNDS>(sc, H, c0, k, R, myrow, A_scale);
}

}  // namespace moe
