// mx.cu: the MXFP8 variant of the path: e8m0 (power-of-two) scales per 32
// values, applied by the tensor core itself.
//
// The mori stage1 page quantises with e8m0 scales (first commit: "GEMM1 reads
// its A rows and e8m0 scales through a rowmap"; quant-LDS commit: the e8m0
// scales packed four per 32-bit word) and feeds them to a block-scaled GEMM.
// On sm_103a the block-scaled FP8 MMA (tcgen05.mma kind::mxf8f6f4
// .block_scale) multiplies every 32-value K chunk of A and B by a power of two
// taken from tensor memory, so GEMM1 needs no promotion on the CUDA cores.
//
// Scale rule (the pages give none): 2**X with X the smallest integer such that
// 448 * 2**X >= amax of the 32-value block (the fp32 recipe's amax / 448
// rounded up to a power of two), clamped to [-127, 127]; e8m0 code = X + 127;
// values are coded e4m3(x * 2**-X), which is exact before the e4m3 rounding,
// so no division is needed.  For a finite amax with biased exponent ea > 0
// and mantissa field mf, X = ea - 135 + (mf > 0x600000): amax <= 1.75 * 2**(ea-127)
// keeps X = ea - 135, anything above needs one more; amax below the fp32
// normal range (or zero) gives X = -127.
//
// Scale-factor layouts in HBM, MMA-ready: the scales of one 128-row (or
// 128-column) block over one 128-value K block are one 512-byte atom, the
// tensor memory image that a 32x128b.warpx4 tcgen05.cp expands: byte
// (i % 32) * 16 + (i / 32) * 4 + j holds row i's scale of the j-th 32-value
// chunk.
//   A_sf  [max_tiles][H/128][512]: atom of (M-tile m, K block kb); row i is
//         tile slot i (dense row tile_row_begin[m] + i).  Slots past the
//         tile's rows are never written.
//   W_sf  [E][H/128][N/128][512]: atom of (expert e, K block kb, 128-row
//         block nb of the weight's N rows), so the two atoms of a 256-wide
//         N-block are one contiguous 1 KB copy.
#include "gemm1.cuh"
#include "quant.cuh"
#include "tmem_drain.cuh"
#include "host_util.h"

namespace moe {

MOE_DEV uint32_t sf_atom_offset(int i) { return (uint32_t)((i & 31) * 16 + (i >> 5) * 4); }

// 16 values of one lane (half of a 32-value block: lanes 2b and 2b+1 hold
// block b) -> 16 e4m3 codes and the block's e8m0 code.  Whole warp, converged.
MOE_DEV uint4 mx_quant16(const float (&f)[16], uint32_t& e8m0) {
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(f[i]));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  const uint32_t b = __float_as_uint(am);
  const int ea = (int)(b >> 23);
  int X = -127;
  if (ea != 0) X = max(ea - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0), -127);
  e8m0 = (uint32_t)(X + 127);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2**-X (X <= 120 for finite bf16)
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = (uint32_t)e4m3x2(__fmul_rn(f[4 * i], inv), __fmul_rn(f[4 * i + 1], inv)) |
           ((uint32_t)e4m3x2(__fmul_rn(f[4 * i + 2], inv), __fmul_rn(f[4 * i + 3], inv)) << 16);
  return make_uint4(p[0], p[1], p[2], p[3]);
}

// The four e8m0 codes of the 128-value K block that lanes 8c..8c+7 cover, one
// byte per 32-value chunk in chunk order, valid in lane 8c.
MOE_DEV uint32_t mx_pack_kblock(uint32_t e8m0) {
  const uint32_t s1 = __shfl_down_sync(0xffffffffu, e8m0, 2);
  const uint32_t s2 = __shfl_down_sync(0xffffffffu, e8m0, 4);
  const uint32_t s3 = __shfl_down_sync(0xffffffffu, e8m0, 6);
  return e8m0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// One slice [c0, c0 + 512*ROUNDS) of token t: all loads first, then per
// 512-value round the codes (one 16-byte store per lane per destination row)
// and the scale words (lane 8c stores the 4 codes of K block c of the round).
// Lane j < k holds its row (`myrow`) and the byte offset of that row's slot in
// its tile's first scale atom (`mysf`).
template <int ROUNDS>
MOE_DEV void mx_quant_scatter_slice(const uint16_t* __restrict__ x, int H, int t, int c0, int k, int myrow,
                                    long long mysf, uint8_t* __restrict__ A, uint8_t* __restrict__ A_sf) {
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
  uint32_t word[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    float f[16];
    unpack16(raw[2 * r], raw[2 * r + 1], f);
    uint32_t e8;
    q[r] = mx_quant16(f, e8);
    word[r] = mx_pack_kblock(e8);
  }
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, myrow, j);
    const long long sf = __shfl_sync(0xffffffffu, mysf, j);
    if (row < 0) continue;
    uint8_t* arow = A + (size_t)row * H;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int col = c0 + r * 512 + lane * 16;
      if (col < H) {
        *reinterpret_cast<uint4*>(arow + col) = q[r];
        if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(A_sf + sf + (long long)(col / 128) * 512) = word[r];
      }
    }
  }
}

constexpr int kMxQuantWarps = 8;
constexpr int kMxMaxE = 1024;

// Tile slot of dense row `row`: the expert from the offsets (largest e with
// eoff[e] <= row), then its tile and the slot within the tile.  Returns the
// byte offset of the slot in the tile's first scale atom, or -1 for row < 0.
MOE_DEV long long row_sf_offset(int row, const int* s_eoff, const int* s_toff, int E, int KB) {
  if (row < 0) return -1;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_eoff[mid] <= row) lo = mid; else hi = mid;
  }
  const int rel = row - s_eoff[lo];
  const long long m = (long long)s_toff[lo] + rel / kBlockM;
  return m * KB * 512 + sf_atom_offset(rel % kBlockM);
}

// One warp per (token, column range) item, as the fp32-scale dispatch.
template <int ROUNDS>
__global__ void __launch_bounds__(kMxQuantWarps * 32) dispatch_quant_mx_kernel(
    const uint16_t* __restrict__ x, int H, LayoutDev L, int splits, uint8_t* __restrict__ A,
    uint8_t* __restrict__ A_sf) {
  __shared__ int s_eoff[kMxMaxE + 1];
  __shared__ int s_toff[kMxMaxE + 1];
  for (int e = threadIdx.x; e <= L.E; e += blockDim.x) {
    s_eoff[e] = L.expert_offset[e];
    s_toff[e] = L.expert_tile_offset[e];
  }
  __syncthreads();
  constexpr int kSliceCols = 512 * ROUNDS;
  const int lane = threadIdx.x & 31;
  const int T = L.T, k = L.k, KB = H / 128;
  const int chunks = (H + kSliceCols - 1) / kSliceCols;
  const int per = (chunks + splits - 1) / splits;
  const long long items = (long long)T * splits;
  for (long long w = (long long)blockIdx.x * kMxQuantWarps + (threadIdx.x >> 5); w < items;
       w += (long long)gridDim.x * kMxQuantWarps) {
    const int t = (int)(w / splits), sp = (int)(w % splits);
    const int myrow = lane < k ? L.pair_row[(size_t)t * k + lane] : -1;
    const long long mysf = row_sf_offset(myrow, s_eoff, s_toff, L.E, KB);
    const int cend = min(chunks, (sp + 1) * per);
    for (int c = sp * per; c < cend; ++c)
      mx_quant_scatter_slice<ROUNDS>(x, H, t, c * kSliceCols, k, myrow, mysf, A, A_sf);
  }
}

// One warp per weight row (e, n): codes in place, scale words into W_sf.
__global__ void __launch_bounds__(256) quant_weights_mx_kernel(const uint16_t* __restrict__ W, int E, int N, int H,
                                                               uint8_t* __restrict__ Wq, uint8_t* __restrict__ W_sf) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)E * N;
  const int KB = H / 128, NB = N / 128;
  for (long long rw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); rw < rows; rw += (long long)gridDim.x * 8) {
    const int e = (int)(rw / N), n = (int)(rw % N);
    const uint4* src = reinterpret_cast<const uint4*>(W + (size_t)rw * H);
    uint8_t* dst = Wq + (size_t)rw * H;
    const long long sf_row = (long long)(n / 128) * 512 + sf_atom_offset(n % 128);
    for (int c0 = 0; c0 < H; c0 += 512) {
      const int col = c0 + lane * 16;
      uint4 a = make_uint4(0, 0, 0, 0), b = a;
      if (col < H) {
        a = __ldcs(src + col / 8);
        b = __ldcs(src + col / 8 + 1);
      }
      float f[16];
      unpack16(a, b, f);
      uint32_t e8;
      const uint4 q = mx_quant16(f, e8);
      const uint32_t word = mx_pack_kblock(e8);
      if (col < H) {
        *reinterpret_cast<uint4*>(dst + col) = q;
        if ((lane & 7) == 0)
          *reinterpret_cast<uint32_t*>(W_sf + ((long long)e * KB + col / 128) * NB * 512 + sf_row) = word;
      }
    }
  }
}

// ---------------------------------------------------------------- block-scaled GEMM1
//
// Persistent, one CTA per SM, 384 threads, the unit order and the unit ring of
// the fp32-scale GEMM1 (gemm1.cuh).  Per CTA:
//   warp 0       claims units and streams each K block into a 4-stage ring:
//                A (2-D TMA, 128 rows x 128 values) and W (3-D TMA, 256 rows x
//                128 values), 128-byte swizzled, plus the K block's two scale
//                atoms of W and one of A by bulk copies, all on one mbarrier.
//   warp 2       per K block copies the stage's three scale atoms into the
//                stage's 12 tensor-memory columns (tcgen05.cp 32x128b.warpx4)
//                and commits them to the stage's scale-ready barrier.
//   warp 1       per K block waits for the stage's operands and scales and
//                issues 4 block-scaled MMAs (M128 N256 K32; the 32-value
//                chunk kk of the K block takes byte kk of each scale column),
//                all accumulating into one 256-column fp32 accumulator for the
//                whole K = H; a commit per K block hands the stage back, one
//                per unit hands the accumulator to the epilogue.  One thread
//                issues a tcgen05 instruction about every 90 cycles and four
//                MMAs of a K block take ~512 tensor cycles, so the copies run
//                in their own warp, not between the MMAs.
//   warps 4..11  epilogue: each thread drains its row's 128 columns of the
//                accumulator into registers, hands the accumulator back to
//                the MMA warp at once, and stores the valid rows as bf16.
// Tensor memory: accumulator in columns [0, 256), scale factors of stage s in
// [256 + 12 s, 256 + 12 s + 12): A's atom in 4 columns, W's two in 8.

constexpr uint32_t kMxSfaBytes = 512, kMxSfbBytes = 1024;
constexpr uint32_t kMxSfStageBytes = kMxSfaBytes + kMxSfbBytes;
constexpr uint32_t kMxTmemSf = 256;
constexpr uint32_t kMxSfCols = 12;
constexpr size_t kMxSmemBytes = 1024 + (size_t)kGemmStages * kStageBytes + (size_t)kGemmStages * kMxSfStageBytes +
                                ((sizeof(GemmShared) + 127) & ~size_t(127)) + 8 * kGemmStages;
static_assert(kMxSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kMxTmemSf + kGemmStages * kMxSfCols <= kTmemCols, "tensor memory budget");

// Instruction descriptor of kind::mxf8f6f4 with e8m0 scales: A and B e4m3
// (bits 7-9, 10-12 = 0), K-major, N >> 3 in bits 17-22, scale type UE8M0
// (bit 23), M >> 4 in bits 24-28; the scale byte of B in bits 4-5 and of A in
// bits 29-30 are set per MMA.
constexpr uint32_t idesc_mxf8_e4m3(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kMxIdesc = idesc_mxf8_e4m3(kGemmBM, kGemmBN);
// Transposed units (tiles of at most kSwapRows rows): W's two 128-row halves
// as M = 128 operands with W's scale atoms, the tile's rows as N = 32 with
// A's atom (rows 0..31 of an atom sit in lanes 0..31, as the N = 32 operand's
// scale factors are read); the accumulator of W half h in columns
// [h * kSwapRows, +kSwapRows).
constexpr uint32_t kMxIdescSwap = idesc_mxf8_e4m3(kGemmBM, kSwapRows);

MOE_DEV void umma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                       uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Shared-memory descriptor of one 512-byte scale atom: 32 rows of 16 bytes,
// no swizzle (8-row core matrices 128 bytes apart).
MOE_DEV uint64_t sf_atom_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
         ((uint64_t)1 << 46);
}

MOE_DEV void tmem_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}

// Bulk copy global -> shared, completing `bytes` on mbarrier `bar`.
MOE_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}

struct MxParams {
  const uint8_t* A_sf;   // [max_tiles][H/128][512]
  const uint8_t* W_sf;   // [E][H/128][N/128][512]
  LayoutDev L;
  int N, H;
  uint16_t* Y;           // [R][N]
  int32_t* status;
  uint64_t timeout_ns;
};

struct MxSmem {
  uint8_t* stages;       // kGemmStages x (A | W), 1024-aligned
  uint8_t* sf;           // kGemmStages x (A atom | W atoms)
  GemmShared* sh;
  uint64_t* sfready;     // kGemmStages: the stage's scales are in tensor memory
};

MOE_DEV MxSmem mx_smem(uint8_t* raw) {
  const uint32_t s = smem_u32(raw);
  const uint32_t pad = (1024u - (s & 1023u)) & 1023u;
  MxSmem g;
  g.stages = raw + pad;
  g.sf = g.stages + (size_t)kGemmStages * kStageBytes;
  g.sh = reinterpret_cast<GemmShared*>(g.sf + (size_t)kGemmStages * kMxSfStageBytes);
  g.sfready = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(g.sh) + ((sizeof(GemmShared) + 127) & ~size_t(127)));
  return g;
}

// Scale-copy warp (all 32 lanes, converged; one elected lane issues): for every
// K block of every unit, in the MMA warp's order, copy the stage's scale atoms
// into its tensor-memory columns once the stage is full.
MOE_DEV void mx_sf_loop(const MxSmem& S, int KB, int units_here, int32_t* status, uint64_t tmo) {
  GemmShared* sh = S.sh;
  const uint32_t tmem = sh->tmem_base;
  uint32_t it = 0;
  bool ok = true;
  for (int j = 0; j < units_here && ok; ++j) {
    for (int kb = 0; kb < KB; ++kb) {
      const int s = (int)(it % kGemmStages);
      const uint32_t ph = (it / kGemmStages) & 1u;
      if (!mbar_wait(smem_u32(&sh->full[s]), ph, &sh->abort_flag, status, tmo)) { ok = false; break; }
      tc_fence_after();
      if (elect_one()) {
        const uint32_t sf0 = smem_u32(S.sf + (size_t)s * kMxSfStageBytes);
        const uint32_t tsf = tmem + kMxTmemSf + (uint32_t)s * kMxSfCols;
        tmem_cp_sf_atom(tsf, sf_atom_desc(sf0));
        tmem_cp_sf_atom(tsf + 4, sf_atom_desc(sf0 + kMxSfaBytes));
        tmem_cp_sf_atom(tsf + 8, sf_atom_desc(sf0 + kMxSfaBytes + 512));
        umma_commit(smem_u32(&S.sfready[s]));
      }
      __syncwarp();
      ++it;
    }
  }
  // no copy may be in flight when tensor memory is freed: the last commit
  // covers every copy this thread issued (bounded wait, abort flag ignored)
  if (it > 0) {
    int dummy_abort = 0;
    mbar_wait(smem_u32(&S.sfready[(it - 1) % kGemmStages]), ((it - 1) / kGemmStages) & 1u, &dummy_abort, nullptr, tmo);
  }
}

// A tile of at most 32 (64) valid rows loads only that many A rows (the
// 32- and 64-row maps of `tmA_short`): rows past the tile's end feed output
// rows that are never stored.
MOE_DEV bool mx_produce_unit(const MxSmem& S, const CUtensorMap* tmA, const CUtensorMap* tmW, const MxParams& p,
                             const Unit& u, int KB, uint32_t& it, const CUtensorMap* tmA_short) {
  GemmShared* sh = S.sh;
  const CUtensorMap* mapA = tmA;
  uint32_t a_bytes = kATileBytes;
  if (u.rows <= 64) {
    mapA = u.rows <= 32 ? tmA_short : tmA_short + 1;
    a_bytes = (u.rows <= 32 ? 32u : 64u) * kGemmBK;
  }
  const int NB = p.N / 128;
  const uint8_t* sfa = p.A_sf + (size_t)u.m * KB * kMxSfaBytes;
  const uint8_t* sfb = p.W_sf + ((size_t)u.e * KB * NB + (size_t)u.nb * 2) * 512;
  for (int kb = 0; kb < KB; ++kb) {
    const int s = (int)(it % kGemmStages);
    const uint32_t ph = (it / kGemmStages) & 1u;
    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, &sh->abort_flag, p.status, p.timeout_ns)) return false;
    if (elect_one()) {
      const uint32_t full = smem_u32(&sh->full[s]);
      mbar_arrive_expect_tx(full, a_bytes + kBTileBytes + kMxSfStageBytes);
      const uint32_t dstA = smem_u32(S.stages + (size_t)s * kStageBytes);
      tma_load_2d(dstA, mapA, kb * kGemmBK, u.row0, full);
      tma_load_3d(dstA + kATileBytes, tmW, kb * kGemmBK, u.nb * kGemmBN, u.e, full);
      const uint32_t dsf = smem_u32(S.sf + (size_t)s * kMxSfStageBytes);
      bulk_load(dsf, sfa + (size_t)kb * kMxSfaBytes, kMxSfaBytes, full);
      bulk_load(dsf + kMxSfaBytes, sfb + (size_t)kb * NB * 512, kMxSfbBytes, full);
    }
    __syncwarp();
    ++it;
  }
  return true;
}

MOE_DEV void mx_mma_loop(const MxSmem& S, int KB, int32_t* status, uint64_t tmo) {
  GemmShared* sh = S.sh;
  const uint32_t tmem = sh->tmem_base;
  uint32_t it = 0;
  bool issued = false;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, status, tmo))
      break;
    const int m = sh->unit[slot].x;
    const bool swap = sh->unit_rows[slot] <= kSwapRows;
    __syncwarp();
    if (elect_one()) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (m < 0) break;
    // the epilogue has drained the accumulator of the previous unit
    if (!mbar_wait(smem_u32(&sh->tempty[0]), ((uint32_t)j & 1u) ^ 1u, &sh->abort_flag, status, tmo)) break;
    tc_fence_after();
    bool ok = true;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = (int)(it % kGemmStages);
      const uint32_t ph = (it / kGemmStages) & 1u;
      ok = mbar_wait(smem_u32(&sh->full[s]), ph, &sh->abort_flag, status, tmo) &&
           mbar_wait(smem_u32(&S.sfready[s]), ph, &sh->abort_flag, status, tmo);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(S.stages + (size_t)s * kStageBytes);
      const uint32_t b0 = a0 + kATileBytes;
      const uint32_t tsf = tmem + kMxTmemSf + (uint32_t)s * kMxSfCols;
      if (elect_one()) {
        if (swap) {
#pragma unroll
          for (int k4 = 0; k4 < kGemmBK / 32; ++k4)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              umma_mxf8(tmem + h * kSwapRows, sw128_kmajor_desc(b0 + h * (kBTileBytes / 2) + k4 * 32),
                        sw128_kmajor_desc(a0 + k4 * 32), kMxIdescSwap | ((uint32_t)k4 << 4) | ((uint32_t)k4 << 29),
                        tsf + 4 + 4 * h, tsf, (kb > 0 || k4 > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int k4 = 0; k4 < kGemmBK / 32; ++k4)
            umma_mxf8(tmem, sw128_kmajor_desc(a0 + k4 * 32), sw128_kmajor_desc(b0 + k4 * 32),
                      kMxIdesc | ((uint32_t)k4 << 4) | ((uint32_t)k4 << 29), tsf, tsf + 4,
                      (kb > 0 || k4 > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&sh->empty[s]));   // the stage is free once these MMAs are done
      }
      __syncwarp();
      issued = true;
      ++it;
    }
    if (!ok) break;
    if (elect_one()) umma_commit(smem_u32(&sh->tfull[0]));
    __syncwarp();
  }
  if (issued) {   // no MMA may be in flight when TMEM is freed
    int dummy_abort = 0;
    if (elect_one()) umma_commit(smem_u32(&sh->drain));
    __syncwarp();
    mbar_wait(smem_u32(&sh->drain), 0u, &dummy_abort, nullptr, tmo);
  }
}

MOE_DEV void mx_epilogue_loop(const MxSmem& S, const MxParams& p) {
  GemmShared* sh = S.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                 // TMEM lane quarter this warp may access
  const int h = (warp - kEpiWarp0) >> 2;  // column half: [h*128, h*128+128)
  const int r_in_tile = q * 32 + lane;
  const uint32_t tmem = sh->tmem_base;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, p.status,
                   p.timeout_ns))
      return;
    const int4 un = sh->unit[slot];
    const int rows = sh->unit_rows[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (un.x < 0) return;
    if (!mbar_wait(smem_u32(&sh->tfull[0]), (uint32_t)j & 1u, &sh->abort_flag, p.status, p.timeout_ns)) return;
    tc_fence_after();
    if (rows <= kSwapRows) {
      // transposed unit: this thread's W row of half h, one column per token;
      // stored as one output column (a warp covers 32 consecutive columns)
      float v[32];
      tmem_drain32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kSwapRows), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[0]));
      uint16_t* yc = p.Y + (size_t)un.w * p.N + (size_t)un.y * kGemmBN + h * 128 + q * 32 + lane;
#pragma unroll
      for (int t = 0; t < kSwapRows; ++t)
        if (t < rows) yc[(size_t)t * p.N] = __bfloat16_as_ushort(__float2bfloat16_rn(v[t]));
      continue;
    }
    float acc[128];
    tmem_drain128(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128), acc);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[0]));
    if (r_in_tile < rows) {
      uint4* dst = reinterpret_cast<uint4*>(p.Y + (size_t)(un.w + r_in_tile) * p.N + (size_t)un.y * kGemmBN + h * 128);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        dst[c] = make_uint4(pack_bf16x2(acc[8 * c], acc[8 * c + 1]), pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3]),
                            pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5]), pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]));
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm1_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                            const __grid_constant__ ShortMaps tmS, const __grid_constant__ MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  const MxSmem S = mx_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
  }
  {
    GemmSmem g;
    g.stages = S.stages;
    g.sh = S.sh;
    g.out_stage = nullptr;
    if (threadIdx.x == 0) {
      for (int i = 0; i < kGemmStages; ++i) mbar_init(smem_u32(&S.sfready[i]), 1);
    }
    gemm_setup(g);   // (its fence and barrier also publish the sfready inits)
  }
  const int nbn = p.N / kGemmBN;
  const int KB = p.H / kGemmBK;
  const int units = p.L.num_tiles[0] * nbn;
  if (warp < kEpiWarp0) {
    regs_dealloc<kRegsControl>();
    if (warp == 0) {
      uint32_t it = 0;
      int j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
        const Unit x = unit_of(p.L, u, nbn);
        ok = publish_unit(S.sh, j, x, p.status, p.timeout_ns) && mx_produce_unit(S, &tmA, &tmW, p, x, KB, it, tmS.m);
      }
      if (ok) {
        Unit end = {-1, 0, 0, 0, 0};
        publish_unit(S.sh, j, end, p.status, p.timeout_ns);
      }
      // wait (bounded) for the last fills in flight before leaving
      int dummy_abort = 0;
      const uint32_t first = it > (uint32_t)kGemmStages ? it - kGemmStages : 0u;
      for (uint32_t i = first; i < it; ++i)
        mbar_wait(smem_u32(&S.sh->full[i % kGemmStages]), (i / kGemmStages) & 1u, &dummy_abort, nullptr,
                  p.timeout_ns);
    } else if (warp == 1) {
      mx_mma_loop(S, KB, p.status, p.timeout_ns);
    } else if (warp == 2) {
      const int here = units > (int)blockIdx.x ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
      mx_sf_loop(S, KB, here, p.status, p.timeout_ns);
    }
  } else {
    regs_alloc<kRegsEpilogue>();
    mx_epilogue_loop(S, p);
  }
  {
    GemmSmem g;
    g.stages = S.stages;
    g.sh = S.sh;
    g.out_stage = nullptr;
    gemm_teardown(g);
  }
}

}  // namespace moe

using namespace moe;

static int mx_check_layout_h(const moe_layout_t* L, int H) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (L->E > kMxMaxE) return MOE_ERR_INVALID_ARG;
  if (H < 128 || H % 128 != 0 || H > 32768) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

extern "C" int moe_dispatch_quant_mx(const uint16_t* x, int H, const moe_layout_t* L, uint8_t* A, uint8_t* A_sf,
                                     int32_t* status, moe_stream_t stream) {
  (void)status;
  int rc = mx_check_layout_h(L, H);
  if (rc) return rc;
  if (!x || !A || !A_sf) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(A) || !aligned16(A_sf)) return MOE_ERR_INVALID_ARG;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const bool small = L->T < 8192;
  const int cols = small ? 1024 : 2048;
  const int chunks = (H + cols - 1) / cols;
  const long long want = (long long)nsm * 64;
  const int splits = small ? chunks : (int)std::max(1LL, std::min((long long)chunks, (want + L->T - 1) / L->T));
  const long long items = (long long)L->T * splits;
  const int blocks = (int)std::max(1LL, std::min((items + kMxQuantWarps - 1) / kMxQuantWarps, (long long)nsm * 16));
  if (small)
    dispatch_quant_mx_kernel<2><<<blocks, kMxQuantWarps * 32, 0, (cudaStream_t)stream>>>(x, H, to_dev(L), splits, A, A_sf);
  else
    dispatch_quant_mx_kernel<4><<<blocks, kMxQuantWarps * 32, 0, (cudaStream_t)stream>>>(x, H, to_dev(L), splits, A, A_sf);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_quant_weights_mx(const uint16_t* W, int E, int N, int H, uint8_t* Wq, uint8_t* W_sf,
                                    moe_stream_t stream) {
  if (!W || !Wq || !W_sf) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 65535 || N < 128 || N % 128 || H < 128 || H % 128 || N > 32768 || H > 32768)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(Wq) || !aligned16(W_sf)) return MOE_ERR_INVALID_ARG;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const long long rows = (long long)E * N;
  const int blocks = (int)std::max(1LL, std::min((rows + 7) / 8, (long long)nsm * 32));
  quant_weights_mx_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(W, E, N, H, Wq, W_sf);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_grouped_gemm1_mx(const uint8_t* A, const uint8_t* A_sf, const uint8_t* W, const uint8_t* W_sf,
                                    int N, int H, const moe_layout_t* L, uint16_t* Y, int32_t* status,
                                    moe_stream_t stream) {
  int rc = mx_check_layout_h(L, H);
  if (rc) return rc;
  if (!A || !A_sf || !W || !W_sf || !Y) return MOE_ERR_INVALID_ARG;
  if (N < kGemmBN || N % kGemmBN != 0 || N > 32768) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(Y) || !aligned16(A_sf) || !aligned16(W_sf))
    return MOE_ERR_INVALID_ARG;
  if (!device_has_tcgen05()) return MOE_ERR_UNSUPPORTED;
  const long long R = (long long)L->T * L->k;
  CUtensorMap tmA, tmW;
  {
    const uint64_t dA[2] = {(uint64_t)H, (uint64_t)R};
    const uint64_t sA[1] = {(uint64_t)H};
    const uint32_t bA[2] = {kGemmBK, kGemmBM};
    const uint64_t dW[3] = {(uint64_t)H, (uint64_t)N, (uint64_t)L->E};
    const uint64_t sW[2] = {(uint64_t)H, (uint64_t)N * H};
    const uint32_t bW[3] = {kGemmBK, kGemmBN, 1};
    if (!encode_u8_map(&tmA, A, 2, dA, sA, bA)) return MOE_ERR_CUDA;
    if (!encode_u8_map(&tmW, W, 3, dW, sW, bW)) return MOE_ERR_CUDA;
  }
  ShortMaps tmS;
  for (int i = 0; i < 2; ++i) {
    const uint64_t dA[2] = {(uint64_t)H, (uint64_t)R};
    const uint64_t sA[1] = {(uint64_t)H};
    const uint32_t bA[2] = {kGemmBK, i == 0 ? 32u : 64u};
    if (!encode_u8_map(&tmS.m[i], A, 2, dA, sA, bA)) return MOE_ERR_CUDA;
  }
  MxParams p;
  p.A_sf = A_sf;
  p.W_sf = W_sf;
  p.L = to_dev(L);
  p.N = N;
  p.H = H;
  p.Y = Y;
  p.status = status;
  p.timeout_ns = 2000000000ull;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const long long max_units = (long long)L->max_tiles * (N / kGemmBN);
  const int grid = (int)std::max(1LL, std::min((long long)nsm, max_units));
  static const bool split_ok = register_split_fits(grouped_gemm1_mx_kernel);
  if (!split_ok) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(grouped_gemm1_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kMxSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  grouped_gemm1_mx_kernel<<<grid, kGemmThreads, kMxSmemBytes, (cudaStream_t)stream>>>(tmA, tmW, tmS, p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
