// gemm1_pair.cu: moe_grouped_gemm1 on CTA pairs (tcgen05 cta_group::2).
//
// The same GEMM1 as gemm1.cu (mori stage1 page, "What": GEMM1 reads its A
// rows in place; per-128 block scales folded on the CUDA cores), with each
// MMA spanning two SMs: a 2-CTA cluster takes a pair unit, two consecutive
// 128-row M-tiles of one expert (the odd CTA's tile empty when the expert has
// an odd tile count) against one 256-column N-block, and runs
// tcgen05.mma.cta_group::2 with M = 256, N = 256.  Each CTA loads its own 128
// A rows and 128 of the 256 W rows; the MMA reads the W halves of both SMs.
// So an SM takes in 32 KiB per K-block instead of the single-CTA kernel's 48
// KiB (A 16 + W 32) for the same 128 x 256 x 128 multiply-adds of its own.
//
// Roles per CTA (384 threads, as in gemm1.cuh):
//   warp 0     both CTAs: walk the cluster's pair units, publish this CTA's
//              half (rows, first row) to its own unit ring, and stream its A
//              rows and W half into a 6-stage ring; both CTAs' copies complete
//              on the even CTA's full barrier, whose expected bytes the even
//              CTA's producer sets for both.
//   warp 1     even CTA: 4 pair MMAs per K-block into one of two TMEM
//              partials, then two commits multicast to both CTAs: the smem
//              stage's empty barrier and the partial-ready barrier; odd CTA:
//              reads the unit ring only.
//   warps 4-11 both CTAs: fold their 128 rows' partials (gemm1.cuh
//              epilogue_loop), report the partial loaded to the even CTA,
//              store their valid rows of Y.
// The fold is the single-CTA kernel's, column for column, so Y is the same.
#include "gemm1.cuh"
#include "host_util.h"

namespace moe {

constexpr uint32_t kPairBTileBytes = (kGemmBN / 2) * kGemmBK;            // 16 KiB: this CTA's W rows
constexpr uint32_t kPairStageBytes = kATileBytes + kPairBTileBytes;       // 32 KiB
constexpr uint32_t kPairIdesc = idesc_f8_e4m3_f32(2 * kGemmBM, kGemmBN);  // M = 256, N = 256
static_assert((size_t)kPairStages * kPairStageBytes <= (size_t)kGemmStages * kStageBytes,
              "pair stages fit the single-CTA stage region");

MOE_DEV void gemm_setup_pair(const GemmSmem& S) {
  GemmShared* sh = S.sh;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);    // even CTA: its producer's expect_tx arrival
      mbar_init(smem_u32(&sh->empty[s]), 1);   // the even CTA's MMA commit, multicast
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_u32(&sh->tfull[p]), 1);
      mbar_init(smem_u32(&sh->tempty[p]), 2 * kEpiWarps);   // even CTA: both CTAs' promotion warps
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(smem_u32(&sh->ufull[i]), 1);
      mbar_init(smem_u32(&sh->uempty[i]), 1 + kEpiWarps);
      mbar_init(smem_u32(&sh->stored[i]), kEpiWarps);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync();   // the peer CTA is running (and its barriers exist) before the pair allocation
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sh->tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // TMEM allocated in both CTAs before any MMA, copy, commit or arrival crosses
  tc_fence_after();
}

// Pair units: expert e's M-tiles [expert_tile_offset[e], expert_tile_offset[e+1])
// two at a time, pair-major with the N-block inner.  The producer walks its
// cluster's units in increasing order, so a cursor over the experts finds each
// unit's expert.
struct PairCursor {
  int e = 0, base = 0;   // first pair index of expert e
};

MOE_DEV int pair_count(const LayoutDev& L, int e) {
  return (L.expert_tile_offset[e + 1] - L.expert_tile_offset[e] + 1) >> 1;
}

// Warp 0: total pair units of the layout (all lanes get it).
MOE_DEV int total_pairs(const LayoutDev& L) {
  const int lane = threadIdx.x & 31;
  int t = 0;
  for (int e0 = 0; e0 < L.E; e0 += 32) {
    const int e = e0 + lane;
    int c = e < L.E ? pair_count(L, e) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    t += c;
  }
  return t;
}

// This CTA's half of pair unit u: rows [row0, row0 + rows) of the dense
// buffer; an empty half reads rows past the end of A (zero-filled by the copy
// engine, nothing fetched) and stores nothing.
MOE_DEV Unit pair_half(const LayoutDev& L, int u, int nbn, uint32_t rank, long long R, PairCursor& c) {
  const int p = u / nbn;
  while (c.e < L.E - 1) {   // (the bound only guards against inconsistent tables)
    const int n = pair_count(L, c.e);
    if (p < c.base + n) break;
    c.base += n;
    ++c.e;
  }
  const int t = L.expert_tile_offset[c.e] + 2 * (p - c.base) + (int)rank;
  Unit x;
  x.m = p;
  x.nb = u % nbn;
  x.e = c.e;
  if (t < L.expert_tile_offset[c.e + 1]) {
    x.row0 = L.tile_row_begin[t];
    x.rows = L.tile_rows[t];
  } else {
    x.row0 = (int)min(R, (long long)0x7FFFFF00);
    x.rows = 0;
  }
  return x;
}

// Producer warp of either CTA: stream one unit's K-blocks.  `full_even` is the
// even CTA's full barrier 0 as a shared::cluster address (barrier s at + 8 s).
MOE_DEV bool produce_unit_pair(const GemmSmem& S, const CUtensorMap* tmA, const CUtensorMap* tmWh, const Unit& u,
                               int KB, uint32_t rank, uint32_t full_even, uint32_t& it, int32_t* status,
                               uint64_t tmo) {
  GemmShared* sh = S.sh;
  for (int kb = 0; kb < KB; ++kb) {
    const int s = (int)(it % kPairStages);
    const uint32_t ph = (it / kPairStages) & 1u;
    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, &sh->abort_flag, status, tmo)) return false;
    if (elect_one()) {
      if (rank == 0) mbar_arrive_expect_tx(smem_u32(&sh->full[s]), 2 * kPairStageBytes);
      const uint32_t full = full_even + 8u * (uint32_t)s;
      const uint32_t dst = smem_u32(S.stages + (size_t)s * kPairStageBytes);
      tma_load_2d_pair(dst, tmA, kb * kGemmBK, u.row0, full);
      tma_load_3d_pair(dst + kATileBytes, tmWh, kb * kGemmBK, u.nb * kGemmBN + (int)rank * (kGemmBN / 2), u.e,
                       full);
    }
    __syncwarp();
    ++it;
  }
  return true;
}

// Even CTA's MMA warp (one elected lane issues).
MOE_DEV void mma_loop_pair(const GemmSmem& S, int KB, int32_t* status, uint64_t tmo) {
  GemmShared* sh = S.sh;
  const uint32_t tmem = sh->tmem_base;
  uint32_t it = 0, pit = 0;
  bool issued = false;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, status, tmo))
      break;
    const int m = sh->unit[slot].x;
    __syncwarp();
    if (elect_one()) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (m < 0) break;
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
      const uint32_t p = pit & 1u, pph = (pit >> 1) & 1u;
      const int s = (int)(it % kPairStages);
      const uint32_t ph = (it / kPairStages) & 1u;
      ok = mbar_wait(smem_u32(&sh->tempty[p]), pph ^ 1u, &sh->abort_flag, status, tmo) &&
           mbar_wait(smem_u32(&sh->full[s]), ph, &sh->abort_flag, status, tmo);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(S.stages + (size_t)s * kPairStageBytes);
      const uint32_t b0 = a0 + kATileBytes;
      if (elect_one()) {
#pragma unroll
        for (int k4 = 0; k4 < kGemmBK / 32; ++k4)
          umma_f8f6f4_pair(tmem + p * kGemmBN, sw128_kmajor_desc(a0 + k4 * 32), sw128_kmajor_desc(b0 + k4 * 32),
                           kPairIdesc, k4 > 0 ? 1u : 0u);
        umma_commit_pair_multicast(smem_u32(&sh->empty[s]), (uint16_t)0x3);   // both CTAs' stage s
        umma_commit_pair_multicast(smem_u32(&sh->tfull[p]), (uint16_t)0x3);
      }
      __syncwarp();
      issued = true;
      ++it;
      ++pit;
    }
    if (!ok) break;
  }
  if (issued) {   // no MMA may be in flight when TMEM is freed or the odd CTA leaves
    int dummy_abort = 0;
    if (elect_one()) umma_commit_pair_multicast(smem_u32(&sh->drain), (uint16_t)0x1);
    __syncwarp();
    mbar_wait(smem_u32(&sh->drain), 0u, &dummy_abort, nullptr, tmo);
  }
}

// Odd CTA's MMA warp: keeps the unit ring's accounting (it issues nothing).
MOE_DEV void unit_reader(const GemmSmem& S, int32_t* status, uint64_t tmo) {
  GemmShared* sh = S.sh;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), (uint32_t)(j / kUnitRing) & 1u, &sh->abort_flag, status, tmo))
      break;
    const int m = sh->unit[slot].x;
    __syncwarp();
    if (elect_one()) mbar_arrive(smem_u32(&sh->uempty[slot]));
    if (m < 0) break;
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm1_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmWh,
                              const __grid_constant__ GemmParams g) {
  extern __shared__ uint8_t smem_raw[];
  const GemmSmem S = gemm_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmWh);
  }
  gemm_setup_pair(S);
  const int nbn = g.N / kGemmBN;
  const int KB = g.H / kGemmBK;
  const int cluster = (int)blockIdx.x >> 1, clusters = (int)gridDim.x >> 1;

  if (warp < kEpiWarp0) {
    regs_dealloc<kRegsControl>();
    if (warp == 0) {
      const int units = total_pairs(g.L) * nbn;
      const uint32_t full_even = mapa_shared(smem_u32(&S.sh->full[0]), 0);
      PairCursor cur;
      uint32_t it = 0;
      int j = 0;
      bool ok = true;
      for (int u = cluster; u < units && ok; u += clusters, ++j) {
        const Unit x = pair_half(g.L, u, nbn, rank, g.R, cur);
        ok = publish_unit(S.sh, j, x, g.status, g.timeout_ns) &&
             produce_unit_pair(S, &tmA, &tmWh, x, KB, rank, full_even, it, g.status, g.timeout_ns);
      }
      if (ok) {
        Unit end = {-1, 0, 0, 0, 0};
        publish_unit(S.sh, j, end, g.status, g.timeout_ns);
      }
      // the even CTA's full barriers count both CTAs' copies: once it has seen
      // them complete, nothing is in flight into either CTA
      if (rank == 0) {
        int dummy_abort = 0;
        const uint32_t first = it > (uint32_t)kPairStages ? it - kPairStages : 0u;
        for (uint32_t i = first; i < it; ++i)
          mbar_wait(smem_u32(&S.sh->full[i % kPairStages]), (i / kPairStages) & 1u, &dummy_abort, nullptr,
                    g.timeout_ns);
      }
    } else if (warp == 1) {
      if (rank == 0)
        mma_loop_pair(S, KB, g.status, g.timeout_ns);
      else
        unit_reader(S, g.status, g.timeout_ns);
    }
  } else {
    regs_alloc<kRegsEpilogue>();
    epilogue_loop<true, false, false, true>(S, g);
  }
  tc_fence_before();
  cluster_sync();   // both CTAs done: no MMA, copy, commit or arrival still aimed at either
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(S.sh->tmem_base, kTmemCols);
  }
}

}  // namespace moe

using namespace moe;

int gemm1_check_args(const uint8_t* A, const float* A_scale, const uint8_t* W, const float* W_scale, int N,
                     int H, const moe_layout_t* L, const uint16_t* Y);

extern "C" int moe_grouped_gemm1_pair(const uint8_t* A, const float* A_scale, const uint8_t* W,
                                      const float* W_scale, int N, int H, const moe_layout_t* L, uint16_t* Y,
                                      int32_t* status, moe_stream_t stream) {
  int rc = gemm1_check_args(A, A_scale, W, W_scale, N, H, L, Y);
  if (rc) return rc;
  const long long R = (long long)L->T * L->k;
  CUtensorMap tmA, tmWh;
  const uint64_t dA[2] = {(uint64_t)H, (uint64_t)R};
  const uint64_t sA[1] = {(uint64_t)H};
  const uint32_t bA[2] = {kGemmBK, kGemmBM};
  const uint64_t dW[3] = {(uint64_t)H, (uint64_t)N, (uint64_t)L->E};
  const uint64_t sW[2] = {(uint64_t)H, (uint64_t)N * H};
  const uint32_t bW[3] = {kGemmBK, kGemmBN / 2, 1};
  if (!encode_u8_map(&tmA, A, 2, dA, sA, bA)) return MOE_ERR_CUDA;
  if (!encode_u8_map(&tmWh, W, 3, dW, sW, bW)) return MOE_ERR_CUDA;
  GemmParams g;
  g.A_scale = A_scale;
  g.W_scale = W_scale;
  g.L = to_dev(L);
  g.N = N;
  g.H = H;
  g.R = R;
  g.Y = Y;
  g.status = status;
  g.timeout_ns = 2000000000ull;
  g.gather_row = nullptr;
  const int nsm = device_sm_count();
  if (nsm < 2) return MOE_ERR_UNSUPPORTED;
  static const bool split_ok = register_split_fits(grouped_gemm1_pair_kernel);
  if (!split_ok) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(grouped_gemm1_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent grid with a static share of units per cluster: as many
  // clusters as are resident at once
  static int resident = -1;
  if (resident < 0) {
    cfg.gridDim = dim3(2 * (nsm / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm1_pair_kernel, &cfg) != cudaSuccess || n < 1)
      return MOE_ERR_CUDA;
    resident = n;
  }
  const long long max_units = ((long long)L->max_tiles + L->E) / 2 * (N / kGemmBN);
  const int clusters = (int)std::max(1LL, std::min((long long)std::min(resident, nsm / 2), max_units));
  cfg.gridDim = dim3(2 * clusters);
  if (cudaLaunchKernelEx(&cfg, grouped_gemm1_pair_kernel, tmA, tmWh, g) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
