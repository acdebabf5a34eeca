// gemm1.cuh: the GEMM1 consumer pipeline (TMA producer thread, tcgen05 MMA
// thread, promotion/epilogue warps) shared by moe_grouped_gemm1 and the fused
// moe_stage1 kernel.
//
// GEMM1 of the mori stage1 page ("What": GEMM1 reads its A rows in place
// through a rowmap; "How it works now": tiles in a static order gated per tile,
// or in readiness order).  Work unit = (M-tile m, N-block nb): 128 dense rows
// of one expert times 256 output columns, the full K = H.
//
// Per CTA (one per SM, 384 threads = 3 warpgroups):
//   warp 0           (converged; one elected lane issues) claims units,
//                    publishes them through a shared-memory ring, and streams
//                    the K-blocks (128 FP8 values of K) of A (2-D TMA, rows
//                    [row0, row0+128) of the dense buffer, the rowmap's first
//                    slot of the tile) and of W (3-D TMA, rows [nb*256, +256)
//                    of expert e) into a 4-stage ring, 128-byte swizzled.
//   warp 1           (converged; one elected lane issues) 4 tcgen05.mma (K=32
//                    each, M=128, N=256, e4m3 x e4m3 -> fp32) per K-block into
//                    one of two TMEM partial buffers (2 x 256 columns), one
//                    commit to the smem stage's empty barrier (the stage goes
//                    back to the TMA thread as soon as the MMAs that read it
//                    are done) and one to that buffer's partial-ready barrier;
//                    a tile of at most kSwapRows rows runs transposed instead
//                    (8 MMAs of M=128, N=32 per K-block: W's two halves times
//                    the tile's rows, see kSwapRows).
//   warps 2, 3       idle (they complete warpgroup 0, whose registers go to
//                    the promotion warpgroups: setmaxnreg 40 / 232), or, with
//                    A gathered row by row, copying half of each A tile.
//   warps 4..11      promotion: each thread owns one row (TMEM lane) and 128
//                    columns; per K-block it loads the fp32 partial and folds it
//                    into register accumulators with the two block scales,
//                    acc += partial * (sa[row, kb] * sb[e, n/128, kb]), the two
//                    scales fetched ahead by cp.async; after the last K-block it
//                    rounds to bf16 and stores the valid rows (a transposed
//                    tile: one W row's 32 token columns per thread, each with
//                    its token's scale, stored as one output column).
//
// fp32 block scales per 128 values are not a tensor-core mode (the hardware
// block-scaled kinds take power-of-two scales per 32), so the scales are
// applied in software on the CUDA cores, one FMA per accumulator per K-block,
// overlapped with the next K-block's MMAs through the two TMEM buffers.
#pragma once

#include "common.cuh"
#include "tmem_fold.cuh"

namespace moe {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 128;
constexpr int kGemmStages = 4;
// CTA pairs (M = 256 over two SMs): a stage holds this CTA's 128 rows of A and
// its 128 of the unit's 256 W rows, 32 KiB, so six fit where four single-CTA
// stages do.
constexpr int kPairStages = 6;
constexpr int kGemmMaxStages = 6;
constexpr int kScaleAhead = 4;   // K-blocks of block scales the promotion warps fetch ahead
constexpr int kGemmThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;                          // first promotion warp (warpgroups 1 and 2)
// Register split: launched at 168 per thread (65536 / 384, rounded down to 8);
// warpgroup 0 gives back to 40, the two promotion warpgroups take 232
// (128 accumulators + 64 in-flight TMEM values + loop state, no spill):
// 128 x 40 + 256 x 232 = 64512 = 384 x 168.
constexpr uint32_t kRegsControl = 40;
constexpr uint32_t kRegsEpilogue = 232;
static_assert(128 * kRegsControl + 256 * kRegsEpilogue <= 168u * kGemmThreads, "register split exceeds launch");

// setmaxnreg.inc draws on the registers the CTA was launched with (threads x
// the kernel's per-thread count), not on the SM's register file, and waits
// until they are free: host side, refuse the launch when the compiled kernel
// holds fewer than the split needs, instead of launching a kernel that would
// never get past its register re-allocation.
template <typename Kernel>
inline bool register_split_fits(Kernel kernel) {
  cudaFuncAttributes a;
  if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess) return false;
  return 128u * kRegsControl + (uint32_t)(kGemmThreads - 128) * kRegsEpilogue <=
         (uint32_t)a.numRegs * (uint32_t)kGemmThreads;
}
constexpr int kUnitRing = 4;
constexpr uint32_t kATileBytes = kGemmBM * kGemmBK;   // 16 KiB
constexpr uint32_t kBTileBytes = kGemmBN * kGemmBK;   // 32 KiB
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 512;                   // two fp32 partial buffers of 256 columns
constexpr uint32_t kIdesc = idesc_f8_e4m3_f32(kGemmBM, kGemmBN);
// Transposed units: a tile of at most kSwapRows valid rows is computed as
// Y^T = W A^T, the unit's 256 W rows as two M = 128 operands and its rows as
// one N = kSwapRows operand (the 32-row A box), so the tensor core reads 8 KB
// of A per K-block instead of 16 and the promotion warps fold 32 columns per
// thread instead of 128.  The partial of W half h sits at TMEM columns
// [h * kSwapRows, +kSwapRows) of the K-block's buffer, lane = W row.
constexpr int kSwapRows = 32;
constexpr uint32_t kIdescSwap = idesc_f8_e4m3_f32(kGemmBM, kSwapRows);

struct GemmShared {
  uint64_t full[kGemmMaxStages];
  uint64_t empty[kGemmMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t ufull[kUnitRing];
  uint64_t uempty[kUnitRing];
  uint64_t stored[kUnitRing];   // the epilogue warps have stored the unit's Y rows (fused combine)
  uint64_t drain;
  int4 unit[kUnitRing];     // {m (-1: end), nb, expert, row0}
  int unit_rows[kUnitRing];
  uint32_t tmem_base;
  int abort_flag;
};

// Output staging: 4 KB per promotion warp (32 rows x 64 bf16 columns, 16-byte
// chunks XOR-swizzled by row) so that the Y store goes out in full 128-byte
// row segments.
constexpr uint32_t kOutStageBytes = 32 * 64 * 2;
constexpr size_t kGemmSmemBytes =
    1024 + (size_t)kGemmStages * kStageBytes + ((sizeof(GemmShared) + 127) & ~size_t(127)) +
    (size_t)kEpiWarps * kOutStageBytes;
static_assert(kScaleAhead * 256 <= kOutStageBytes, "scale ring fits the staging tile");
static_assert(kGemmSmemBytes <= 232448, "shared memory budget of one CTA");

struct GemmParams {
  const float* A_scale;   // [H/128][R]
  const float* W_scale;   // [E][N/128][H/128]
  LayoutDev L;
  int N, H;
  long long R;            // rows of A (the stride of A_scale): T*k, or the send-run capacity
  uint16_t* Y;            // [T*k][N]
  int32_t* status;
  uint64_t timeout_ns;
  const int32_t* gather_row;   // [T*k] row of A holding dense row r (gathered A), or null (A dense)
};

// Shared-memory carve-up: 1024-aligned stage buffers, then the barriers.
struct GemmSmem {
  uint8_t* stages;
  GemmShared* sh;
  uint8_t* out_stage;   // kEpiWarps x kOutStageBytes
};

MOE_DEV GemmSmem gemm_smem(uint8_t* raw) {
  const uint32_t s = smem_u32(raw);
  const uint32_t pad = (1024u - (s & 1023u)) & 1023u;
  GemmSmem g;
  g.stages = raw + pad;
  g.sh = reinterpret_cast<GemmShared*>(g.stages + (size_t)kGemmStages * kStageBytes);
  g.out_stage = reinterpret_cast<uint8_t*>(g.sh) + ((sizeof(GemmShared) + 127) & ~size_t(127));
  return g;
}

// Barrier init + TMEM allocation (whole CTA calls this).  `extra_unit_consumers`
// warps besides the MMA warp and the epilogue warps read every unit from the
// ring (and arrive on its empty barrier).
MOE_DEV void gemm_setup(const GemmSmem& S, int extra_unit_consumers = 0, int stage_fillers = 1) {
  GemmShared* sh = S.sh;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(smem_u32(&sh->full[s]), stage_fillers);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_u32(&sh->tfull[p]), 1);
      mbar_init(smem_u32(&sh->tempty[p]), kEpiWarps);
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(smem_u32(&sh->ufull[i]), 1);
      mbar_init(smem_u32(&sh->uempty[i]), 1 + kEpiWarps + extra_unit_consumers);
      mbar_init(smem_u32(&sh->stored[i]), kEpiWarps);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

MOE_DEV void gemm_teardown(const GemmSmem& S) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(S.sh->tmem_base, kTmemCols);
  }
}

// A maps with boxes 32 and 64 rows high, for tiles with that few rows (dense A).
struct ShortMaps {
  CUtensorMap m[2];
};

// A unit handed from the producer thread to the MMA thread and the epilogue warps.
struct Unit {
  int m, nb, e, row0, rows;
};

// Producer warp (all 32 lanes, converged; one elected lane writes and issues):
// publish unit j (m < 0 = end of work) into the ring.
MOE_DEV bool publish_unit(GemmShared* sh, int j, const Unit& u, int32_t* status, uint64_t tmo) {
  const int slot = j % kUnitRing;
  const uint32_t ph = (uint32_t)(j / kUnitRing) & 1u;
  if (!mbar_wait(smem_u32(&sh->uempty[slot]), ph ^ 1u, &sh->abort_flag, status, tmo)) return false;
  if (elect_one()) {
    sh->unit[slot] = make_int4(u.m, u.nb, u.e, u.row0);
    sh->unit_rows[slot] = u.rows;
    mbar_arrive(smem_u32(&sh->ufull[slot]));
  }
  __syncwarp();
  return true;
}

// Producer warp: stream the K-blocks of one unit into the stage ring.  `it`
// counts stage fills.  With `tmA_short` (maps whose boxes are 32 and 64 rows
// high), a tile of at most 32 (64) valid rows loads only that many A rows:
// the MMA still reads all 128 rows of the stage, but rows past the tile's
// end only feed output rows that are never stored, so whatever the stage
// held there before does not matter, and the short box saves shared-memory
// and L2 traffic on the experts with few rows.
MOE_DEV bool produce_unit(const GemmSmem& S, const CUtensorMap* tmA, const CUtensorMap* tmW,
                          const Unit& u, int KB, uint32_t& it, int32_t* status, uint64_t tmo,
                          const CUtensorMap* tmA_short = nullptr) {
  GemmShared* sh = S.sh;
  const CUtensorMap* mapA = tmA;
  uint32_t a_bytes = kATileBytes;
  if (tmA_short != nullptr && u.rows <= 64) {
    mapA = u.rows <= 32 ? tmA_short : tmA_short + 1;
    a_bytes = (u.rows <= 32 ? 32u : 64u) * kGemmBK;
  }
  for (int kb = 0; kb < KB; ++kb) {
    const int s = (int)(it % kGemmStages);
    const uint32_t ph = (it / kGemmStages) & 1u;
    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, &sh->abort_flag, status, tmo)) return false;
    if (elect_one()) {
      const uint32_t full = smem_u32(&sh->full[s]);
      mbar_arrive_expect_tx(full, a_bytes + kBTileBytes);
      const uint32_t dstA = smem_u32(S.stages + (size_t)s * kStageBytes);
      tma_load_2d(dstA, mapA, kb * kGemmBK, u.row0, full);
      tma_load_3d(dstA + kATileBytes, tmW, kb * kGemmBK, u.nb * kGemmBN, u.e, full);
    }
    __syncwarp();
    ++it;
  }
  return true;
}

// 16-byte asynchronous copy global -> shared (zero-filled, nothing read, when
// src_bytes == 0).
MOE_DEV void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(src_bytes)
               : "memory");
}

// Gathered A (per-(token, group) send runs): dense row row0 + i of a unit is
// row gather[row0 + i] of A.  A row slice of a K-block is 128 bytes, and two
// engines fetch them side by side: the TMA warp gathers tile rows [0, 64)
// with tile::gather4 (16 lanes, four rows each, the tensor map's box one row
// high; the copy engine swizzles each row by its shared-memory address), and
// warps 2 and 3 copy rows [64, 128) 16 bytes at a time with cp.async into the
// same 128-byte-swizzled layout (16-byte chunk c of row r at
// r*128 + (c ^ (r & 7)) * 16).  Either engine alone moves too few rows per
// K-block (the copy engine takes tens of cycles per row request, the
// load/store path a few tens of bytes per clock).  A stage's full barrier
// counts the TMA warp's arrival with W's and the gathered rows' bytes, plus
// one arrival from the gather warp that filled its other half: warp 2 fills
// the even stages of the CTA's sequence, warp 3 the odd ones, each waiting
// for its own copies, making them visible to the tensor core
// (fence.proxy.async) and arriving before it moves on.
constexpr int kGatherTmaRows = 64;
constexpr int kGatherCopyRows = kGemmBM - kGatherTmaRows;
static_assert(kGatherTmaRows % 4 == 0 && kGatherTmaRows / 4 <= 32 && kGatherCopyRows % 32 == 0,
              "gather split: whole gather4 lanes, whole warps of copied rows");

// TMA gather of four rows of a 2-D tensor map whose box is one row high: the
// rows land at dst as four consecutive 128-byte rows.
MOE_DEV void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2, int y3,
                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}

// TMA warp, gathered A: W tile plus tile rows [0, kGatherTmaRows) (slots past
// the unit's rows repeat its first row; their products are never stored); a
// unit of at most kSwapRows rows (run transposed) gathers rows [0, kSwapRows)
// only.
MOE_DEV bool produce_unit_gather(const GemmSmem& S, const CUtensorMap* tmA, const CUtensorMap* tmW,
                                 const int32_t* __restrict__ gather, const Unit& u, int KB, uint32_t& it,
                                 int32_t* status, uint64_t tmo) {
  GemmShared* sh = S.sh;
  const int lane = threadIdx.x & 31;
  const int first = gather[u.row0];
  const int grows = u.rows <= kSwapRows ? kSwapRows : kGatherTmaRows;   // rows gathered by TMA
  int r4[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int slot = 4 * (lane % (kGatherTmaRows / 4)) + q;
    r4[q] = slot < u.rows ? gather[u.row0 + slot] : first;
  }
  for (int kb = 0; kb < KB; ++kb) {
    const int s = (int)(it % kGemmStages);
    const uint32_t ph = (it / kGemmStages) & 1u;
    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, &sh->abort_flag, status, tmo)) return false;
    const uint32_t full = smem_u32(&sh->full[s]);
    const uint32_t dstA = smem_u32(S.stages + (size_t)s * kStageBytes);
    if (elect_one()) {
      mbar_arrive_expect_tx(full, kBTileBytes + (uint32_t)grows * kGemmBK);
      tma_load_3d(dstA + kATileBytes, tmW, kb * kGemmBK, u.nb * kGemmBN, u.e, full);
    }
    __syncwarp();
    if (lane < grows / 4)
      tma_gather4(dstA + 512u * (uint32_t)lane, tmA, kb * kGemmBK, r4[0], r4[1], r4[2], r4[3], full);
    __syncwarp();
    ++it;
  }
  return true;
}

// Gather warps (2 and 3): lane l copies tile rows kGatherTmaRows + l + 32 m of
// the K-blocks of its parity.  Reads every unit from the ring like the MMA and
// epilogue warps.  A unit run transposed reads only rows [0, kSwapRows), all
// gathered by the TMA warp: the gather warp copies nothing and only arrives.
MOE_DEV void gather_a_loop(const GemmSmem& S, const uint8_t* __restrict__ A, const int32_t* __restrict__ gather,
                           int H, int KB, int32_t* status, uint64_t tmo) {
  constexpr int kM = kGatherCopyRows / 32;
  GemmShared* sh = S.sh;
  const int lane = threadIdx.x & 31;
  const uint32_t par = (((int)threadIdx.x >> 5) - 2) & 1u;
  uint32_t it = 0;
  bool ok = true;
  for (int j = 0; ok; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, status, tmo)) break;
    const int4 un = sh->unit[slot];
    const int rows = sh->unit_rows[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (un.x < 0) break;
    const uint8_t* src[kM];
    uint32_t nbytes[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      const int r = kGatherTmaRows + lane + 32 * m;
      src[m] = A + (size_t)(r < rows ? gather[un.w + r] : 0) * H;
      nbytes[m] = r < rows ? 16u : 0u;
    }
    const bool copy = rows > kSwapRows;
    for (int kb = 0; kb < KB; ++kb, ++it) {
      if ((it & 1u) != par) continue;
      const int s = (int)(it % kGemmStages);
      const uint32_t ph = (it / kGemmStages) & 1u;
      if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, &sh->abort_flag, status, tmo)) { ok = false; break; }
      if (!copy) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->full[s]));
        continue;
      }
      const uint32_t dst = smem_u32(S.stages + (size_t)s * kStageBytes);
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        const int r = kGatherTmaRows + lane + 32 * m;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          cp_async16(dst + (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4), src[m] + kb * kGemmBK + c * 16,
                     nbytes[m]);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->full[s]));
    }
  }
  cp_async_wait<0>();
}

// Before leaving, wait (bounded, ignoring the abort flag) for the last fills in flight.
MOE_DEV void drain_fills(const GemmSmem& S, uint32_t it, uint64_t tmo) {
  int dummy_abort = 0;
  const uint32_t first = it > (uint32_t)kGemmStages ? it - kGemmStages : 0u;
  for (uint32_t i = first; i < it; ++i)
    mbar_wait(smem_u32(&S.sh->full[i % kGemmStages]), (i / kGemmStages) & 1u, &dummy_abort, nullptr, tmo);
}

// MMA warp (all 32 lanes run the loop; one elected lane issues the tcgen05
// instructions, so descriptors and addresses stay warp-uniform): consume units
// until the end marker.  kCommitRelease: a commit after the K-block's MMAs
// hands its smem stage back (the standalone GEMM1 kernels); otherwise the
// first promotion warp does when it sees the partial (epilogue_loop's
// kReleaseStage; the fused kernels, where that measured faster).  kSwap: units
// of at most kSwapRows rows run transposed (the producer loads their A rows
// as the 32-row box).
template <bool kCommitRelease = true, bool kSwap = false>
MOE_DEV void mma_loop(const GemmSmem& S, int KB, int32_t* status, uint64_t tmo) {
  GemmShared* sh = S.sh;
  const uint32_t tmem = sh->tmem_base;
  uint32_t it = 0, pit = 0;
  bool issued = false;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, status, tmo))
      break;
    const int m = sh->unit[slot].x;
    const bool swap = kSwap && sh->unit_rows[slot] <= kSwapRows;
    __syncwarp();
    if (elect_one()) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (m < 0) break;
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
      const uint32_t p = pit & 1u, pph = (pit >> 1) & 1u;
      const int s = (int)(it % kGemmStages);
      const uint32_t ph = (it / kGemmStages) & 1u;
      ok = mbar_wait(smem_u32(&sh->tempty[p]), pph ^ 1u, &sh->abort_flag, status, tmo) &&
           mbar_wait(smem_u32(&sh->full[s]), ph, &sh->abort_flag, status, tmo);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(S.stages + (size_t)s * kStageBytes);
      const uint32_t b0 = a0 + kATileBytes;
      if (elect_one()) {
        if (swap) {
#pragma unroll
          for (int k4 = 0; k4 < kGemmBK / 32; ++k4)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              umma_f8f6f4(tmem + p * kGemmBN + h * kSwapRows,
                          sw128_kmajor_desc(b0 + h * (kBTileBytes / 2) + k4 * 32), sw128_kmajor_desc(a0 + k4 * 32),
                          kIdescSwap, k4 > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int k4 = 0; k4 < kGemmBK / 32; ++k4)
            umma_f8f6f4(tmem + p * kGemmBN, sw128_kmajor_desc(a0 + k4 * 32), sw128_kmajor_desc(b0 + k4 * 32),
                        kIdesc, k4 > 0 ? 1u : 0u);
        }
        // the stage is free once these MMAs are done; the partial is ready then too
        if (kCommitRelease) umma_commit(smem_u32(&sh->empty[s]));
        umma_commit(smem_u32(&sh->tfull[p]));
      }
      __syncwarp();
      issued = true;
      ++it;
      ++pit;
    }
    if (!ok) break;
  }
  if (issued) {   // no MMA may be in flight when TMEM is freed
    int dummy_abort = 0;
    if (elect_one()) umma_commit(smem_u32(&sh->drain));
    __syncwarp();
    mbar_wait(smem_u32(&sh->drain), 0u, &dummy_abort, nullptr, tmo);
  }
}

// The promotion warps' accumulators, one row x 128 columns per thread: plain
// fp32 values folded with fma.rn.f32, or packed pairs folded with
// fma.rn.f32x2 (bit-identical sums).
template <bool kPacked>
struct FoldAcc;

template <>
struct FoldAcc<false> {
  float v[128];
  MOE_DEV void zero() {
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = 0.0f;
  }
  MOE_DEV void fold(uint32_t taddr, float sc) { tmem_fold128(taddr, sc, v); }
  MOE_DEV uint32_t bf16x2(int c) const { return pack_bf16x2(v[c], v[c + 1]); }   // columns c, c + 1
  // transposed unit: 32 token columns with their own scales into v[0..31]
  MOE_DEV void fold_cols(uint32_t taddr, const unsigned long long (&c)[16]) { tmem_fold32(taddr, c, v); }
  MOE_DEV float col(int t) const { return v[t]; }
};

template <>
struct FoldAcc<true> {
  unsigned long long v[64];   // column 2i in the low half, 2i + 1 in the high half
  MOE_DEV void zero() {
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = 0ull;
  }
  MOE_DEV void fold(uint32_t taddr, float sc) { tmem_fold128x2(taddr, sc, v); }
  MOE_DEV uint32_t bf16x2(int c) const { return pack_bf16x2_from_pair(v[c / 2]); }   // c even
  // transposed unit: 32 token columns with their own scales into v[0..15]
  MOE_DEV void fold_cols(uint32_t taddr, const unsigned long long (&c)[16]) { tmem_fold32x2(taddr, c, v); }
  MOE_DEV float col(int t) const { return __uint_as_float((t & 1) ? (uint32_t)(v[t / 2] >> 32) : (uint32_t)v[t / 2]); }
};

// Promotion + epilogue warps (warps 4..11).  Returns when the end marker arrives.
// In the fused kernel a unit reaches the ring only after the TMA warp acquired
// its ready flag, so the A_scale reads here need no wait of their own.  With
// kSignal each warp arrives on the unit's `stored` barrier once its Y stores
// are issued (the fused combine's counting warp takes it from there).
// With kPair the CTA is one of a pair running M = 256 MMAs: a TMEM partial is
// free again once both CTAs' warps have loaded it, so every promotion warp
// reports to the even CTA's barrier.  With kReleaseStage the first promotion
// warp hands the K-block's smem stage back when it sees the partial (paired
// with mma_loop<false>).  With kSwap, units of at most kSwapRows rows arrive
// transposed (mma_loop<..., true>): each thread folds its W row's 32 token
// columns, with the 32 tokens' A scales from the warp's scale ring, and
// stores one output column.
template <bool kPacked, bool kSignal = false, bool kGather = false, bool kPair = false, bool kReleaseStage = false,
          bool kSwap = false>
MOE_DEV void epilogue_loop(const GemmSmem& S, const GemmParams& g) {
  static_assert(!kSwap || !kPair, "transposed units: one CTA");
  GemmShared* sh = S.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                 // TMEM lane quarter this warp may access
  const int h = (warp - kEpiWarp0) >> 2;  // column half: [h*128, h*128+128)
  const int r_in_tile = q * 32 + lane;
  const int KB = g.H / kGemmBK;
  const int nsb = g.N / 128;
  const uint32_t tmem = sh->tmem_base;
  uint32_t pit = 0;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, g.status,
                   g.timeout_ns))
      return;
    const int4 un = sh->unit[slot];
    const int rows = sh->unit_rows[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (un.x < 0) return;
    const int nb = un.y, e = un.z, row0 = un.w;
    const bool swap = kSwap && rows <= kSwapRows;
    // the A row whose scales this thread fetches: its own row, or in a
    // transposed unit the token of its lane (the warp shares all 32)
    const int r_scale = swap ? lane : r_in_tile;
    const bool valid = r_scale < rows;
    // Scale addresses as 32-bit element offsets from the parameter bases (no
    // 64-bit pointers live across the K loop).  Rows past the tile's end read
    // nothing (zero-filled copies) from a clamped, valid address.  With A
    // gathered, a dense row's scales sit at its row of A.
    const uint32_t sa_row =
        kGather ? (uint32_t)(valid ? g.gather_row[row0 + r_scale] : 0)
                : (uint32_t)min((long long)(row0 + r_scale), (long long)g.R - 1);
    const uint32_t sa_bytes = valid ? 4u : 0u;
    const uint32_t sb_off = (uint32_t)((e * nsb + nb * 2 + h) * KB);
    FoldAcc<kPacked> acc;
    acc.zero();
    // Block scales kScaleAhead K-blocks ahead (they come from L2): each thread
    // keeps its own ring of (sa, sb) pairs in the warp's staging tile, filled
    // by cp.async, so no register waits on a load in flight; one commit group
    // per K-block (empty past the end).  Slot i is the 256 bytes at
    // stg_s + i * 256: (sa, sb) of lane l at 8 l, or in a transposed unit the
    // 32 tokens' sa in the first 128 bytes and each lane's copy of sb after.
    uint8_t* stg = S.out_stage + (size_t)(warp - kEpiWarp0) * kOutStageBytes;
    const uint32_t stg_s = smem_u32(stg);
    const uint32_t sa_dst = stg_s + (swap ? lane * 4u : lane * 8u);
    const uint32_t sb_dst = stg_s + (swap ? 128u + lane * 4u : lane * 8u + 4u);
#pragma unroll
    for (int i = 0; i < kScaleAhead; ++i) {
      if (i < KB) {
        cp_async4(sa_dst + i * 256, g.A_scale + (size_t)i * g.R + sa_row, sa_bytes);
        cp_async4(sb_dst + i * 256, g.W_scale + sb_off + i, 4u);
      }
      cp_async_commit();
    }
    auto refill = [&](int kb, uint32_t so) {
      if (kb + kScaleAhead < KB) {
        const int kn = kb + kScaleAhead;
        cp_async4(sa_dst + so, g.A_scale + (size_t)kn * g.R + sa_row, sa_bytes);
        cp_async4(sb_dst + so, g.W_scale + sb_off + kn, 4u);
      }
      cp_async_commit();
    };
    // wait for partial p; hand the stage back (kReleaseStage)
    auto take = [&](uint32_t p, uint32_t pph) -> bool {
      if (!mbar_wait(smem_u32(&sh->tfull[p]), pph, &sh->abort_flag, g.status, g.timeout_ns)) return false;
      // the MMAs that read smem stage (pit % stages) are complete: hand the stage back to the TMA thread
      if (kReleaseStage && warp == kEpiWarp0 && lane == 0) mbar_arrive(smem_u32(&sh->empty[pit % kGemmStages]));
      tc_fence_after();
      return true;
    };
    // partial p is loaded: report it free
    auto give_back = [&](uint32_t p) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair)   // the even CTA's barrier, from either CTA
          mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&sh->tempty[p]), 0));
        else
          mbar_arrive(smem_u32(&sh->tempty[p]));
      }
    };
    if (kSwap && swap) {
      for (int kb = 0; kb < KB; ++kb) {
        const uint32_t so = (uint32_t)(kb % kScaleAhead) * 256;
        cp_async_wait<kScaleAhead - 1>();
        __syncwarp();   // every lane's copy of this K-block's scales has landed
        float sb;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sb) : "r"(sb_dst + so) : "memory");
        // column scales, token 2i in the low half of c[i]
        unsigned long long c[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float a0, a1, a2, a3;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                       : "r"(stg_s + so + i * 16)
                       : "memory");
          c[2 * i] = pack_f32x2(__fmul_rn(a0, sb), __fmul_rn(a1, sb));
          c[2 * i + 1] = pack_f32x2(__fmul_rn(a2, sb), __fmul_rn(a3, sb));
        }
        __syncwarp();   // all lanes have read the slot before any lane refills it
        refill(kb, so);
        const uint32_t p = pit & 1u, pph = (pit >> 1) & 1u;
        if (!take(p, pph)) return;
        acc.fold_cols(tmem + ((uint32_t)(q * 32) << 16) + p * kGemmBN + h * kSwapRows, c);
        give_back(p);
        ++pit;
      }
    } else {
      for (int kb = 0; kb < KB; ++kb) {
        const uint32_t so = (uint32_t)(kb % kScaleAhead) * 256;
        cp_async_wait<kScaleAhead - 1>();
        float sa, sb;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(sa), "=f"(sb) : "r"(sa_dst + so) : "memory");
        const float sc = sa * sb;
        refill(kb, so);
        const uint32_t p = pit & 1u, pph = (pit >> 1) & 1u;
        if (!take(p, pph)) return;
        acc.fold(tmem + ((uint32_t)(q * 32) << 16) + p * kGemmBN + h * 128, sc);
        give_back(p);
        ++pit;
      }
    }
    if (kSwap && swap) {
      // Y^T column: this thread's output column, one bf16 per token (a warp
      // store covers 32 consecutive columns of one row)
      cp_async_wait<0>();
      __syncwarp();
      uint16_t* yc = g.Y + (size_t)row0 * g.N + (size_t)nb * kGemmBN + h * 128 + q * 32 + lane;
#pragma unroll
      for (int t = 0; t < kSwapRows; ++t) {
        if (t < rows) yc[(size_t)t * g.N] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.col(t)));
      }
      __syncwarp();
      if (kSignal && lane == 0) mbar_arrive(smem_u32(&sh->stored[slot]));
      continue;
    }
    // bf16 output through the warp's staging tile: lane = row on the way in,
    // 8 lanes per row (4 rows per instruction) on the way out (the scale ring
    // there is drained: its last groups are empty)
    cp_async_wait<0>();
    __syncwarp();
    uint16_t* ybase = g.Y + (size_t)row0 * g.N + (size_t)nb * kGemmBN + h * 128;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int a = pass * 64 + c * 8;
        const uint32_t dst = stg_s + lane * 128 + ((c ^ (lane & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                     "r"(acc.bf16x2(a + 0)), "r"(acc.bf16x2(a + 2)), "r"(acc.bf16x2(a + 4)),
                     "r"(acc.bf16x2(a + 6))
                     : "memory");
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = i * 4 + (lane >> 3), chunk = lane & 7;
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(stg_s + row * 128 + ((chunk ^ (row & 7)) << 4))
                     : "memory");
        const int r = q * 32 + row;
        if (r < rows)
          *reinterpret_cast<uint4*>(ybase + (size_t)r * g.N + pass * 64 + chunk * 8) = v;
      }
      __syncwarp();
    }
    if (kSignal && lane == 0) mbar_arrive(smem_u32(&sh->stored[slot]));
  }
}

MOE_DEV Unit unit_of(const LayoutDev& L, int u, int nbn) {
  Unit x;
  x.m = u / nbn;
  x.nb = u % nbn;
  x.e = L.tile_expert[x.m];
  x.row0 = L.rowmap[(size_t)x.m * kGemmBM];   // the tile's rows are contiguous from its first slot
  x.rows = L.tile_rows[x.m];
  return x;
}

}  // namespace moe
