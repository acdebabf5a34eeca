// gemm1.cu: moe_grouped_gemm1, the persistent tcgen05 grouped FP8 GEMM1.
//
// Units (M-tile, N-block) in expert-major order, M-tile outer and N-block inner:
// the tile tables list an expert's M-tiles consecutively, so the ~#SM units in
// flight at any moment cover a few M-tiles of one or two experts; each A tile
// is read from HBM once and served from L2 to its N/256 N-blocks, and the
// expert's weights (N*H bytes) are read from HBM about once while its M-tiles
// run (the L2 reuse that the TilePipe page's "Overlap" section names as the
// reason for an expert-major GEMM order).  CTA c takes units c, c + grid, ...
#include "gemm1.cuh"
#include "host_util.h"

namespace moe {

// kGather: A is read row by row through g.gather_row (per-(token, group) send
// rows; half the tile rows gathered by the TMA warp, half copied by warps 2
// and 3) instead of as 128-row boxes of the dense buffer; `A` is then the
// send buffer.
template <bool kGather>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm1_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ ShortMaps tmS, const __grid_constant__ GemmParams g,
                         const uint8_t* A) {
  extern __shared__ uint8_t smem_raw[];
  const GemmSmem S = gemm_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
  }
  // gathered A: warps 2 and 3 read every unit; one of them arrives on each stage's full barrier
  gemm_setup(S, kGather ? 2 : 0, kGather ? 2 : 1);
  const int nbn = g.N / kGemmBN;
  const int KB = g.H / kGemmBK;
  const int units = g.L.num_tiles[0] * nbn;

  if (warp < kEpiWarp0) {
    regs_dealloc<kRegsControl>();
    if (warp == 0) {
      uint32_t it = 0;
      int j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
        const Unit x = unit_of(g.L, u, nbn);
        ok = publish_unit(S.sh, j, x, g.status, g.timeout_ns) &&
             (kGather ? produce_unit_gather(S, &tmA, &tmW, g.gather_row, x, KB, it, g.status, g.timeout_ns)
                      : produce_unit(S, &tmA, &tmW, x, KB, it, g.status, g.timeout_ns, tmS.m));
      }
      if (ok) {
        Unit end = {-1, 0, 0, 0, 0};
        publish_unit(S.sh, j, end, g.status, g.timeout_ns);
      }
      drain_fills(S, it, g.timeout_ns);
    } else if (warp == 1) {
      mma_loop<true, true>(S, KB, g.status, g.timeout_ns);
    } else if (kGather) {
      gather_a_loop(S, A, g.gather_row, g.H, KB, g.status, g.timeout_ns);
    }
  } else {
    regs_alloc<kRegsEpilogue>();
    epilogue_loop<true, false, kGather, false, false, true>(S, g);
  }
  gemm_teardown(S);
}

}  // namespace moe

using namespace moe;

// Tensor maps of one call: A [R, H] and W [E, N, H], both u8 with 128x128 / 256x128 boxes
// (A's box one row high when it is gathered).
static int encode_gemm_maps(const uint8_t* A, const uint8_t* W, long long R, int E, int N, int H,
                            CUtensorMap* tmA, CUtensorMap* tmW, bool gather = false) {
  const uint64_t dA[2] = {(uint64_t)H, (uint64_t)R};
  const uint64_t sA[1] = {(uint64_t)H};
  const uint32_t bA[2] = {kGemmBK, gather ? 1u : (uint32_t)kGemmBM};
  const uint64_t dW[3] = {(uint64_t)H, (uint64_t)N, (uint64_t)E};
  const uint64_t sW[2] = {(uint64_t)H, (uint64_t)N * H};
  const uint32_t bW[3] = {kGemmBK, kGemmBN, 1};
  if (!encode_u8_map(tmA, A, 2, dA, sA, bA)) return MOE_ERR_CUDA;
  if (!encode_u8_map(tmW, W, 3, dW, sW, bW)) return MOE_ERR_CUDA;
  return MOE_OK;
}

int gemm1_check_args(const uint8_t* A, const float* A_scale, const uint8_t* W, const float* W_scale, int N,
                     int H, const moe_layout_t* L, const uint16_t* Y) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!A || !A_scale || !W || !W_scale || !Y) return MOE_ERR_INVALID_ARG;
  if (N < kGemmBN || N % kGemmBN != 0 || N > 32768) return MOE_ERR_INVALID_ARG;
  if (H < kGemmBK || H % kGemmBK != 0 || H > 32768) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
  if (!device_has_tcgen05()) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

extern "C" int moe_grouped_gemm1(const uint8_t* A, const float* A_scale, const uint8_t* W,
                                 const float* W_scale, int N, int H, const moe_layout_t* L, uint16_t* Y,
                                 int32_t* status, moe_stream_t stream) {
  int rc = gemm1_check_args(A, A_scale, W, W_scale, N, H, L, Y);
  if (rc) return rc;
  const long long R = (long long)L->T * L->k;
  CUtensorMap tmA, tmW;
  rc = encode_gemm_maps(A, W, R, L->E, N, H, &tmA, &tmW);
  if (rc) return rc;
  ShortMaps tmS;
  for (int i = 0; i < 2; ++i) {
    const uint64_t dA[2] = {(uint64_t)H, (uint64_t)R};
    const uint64_t sA[1] = {(uint64_t)H};
    const uint32_t bA[2] = {kGemmBK, i == 0 ? 32u : 64u};
    if (!encode_u8_map(&tmS.m[i], A, 2, dA, sA, bA)) return MOE_ERR_CUDA;
  }
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
  if (nsm <= 0) return MOE_ERR_CUDA;
  const long long max_units = (long long)L->max_tiles * (N / kGemmBN);
  const int grid = (int)std::max(1LL, std::min((long long)nsm, max_units));
  static const bool split_ok = register_split_fits(grouped_gemm1_kernel<false>);
  if (!split_ok) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(grouped_gemm1_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  grouped_gemm1_kernel<false><<<grid, kGemmThreads, kGemmSmemBytes, (cudaStream_t)stream>>>(tmA, tmW, tmS, g, A);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_grouped_gemm1_gather(const uint8_t* A_send, const float* A_send_scale, const uint8_t* W,
                                        const float* W_scale, int N, int H, const moe_layout_t* L,
                                        const int32_t* gather_row, long long send_rows, uint16_t* Y,
                                        int32_t* status, moe_stream_t stream) {
  int rc = gemm1_check_args(A_send, A_send_scale, W, W_scale, N, H, L, Y);
  if (rc) return rc;
  if (!gather_row || send_rows < 1 || send_rows >= ((long long)1 << 31)) return MOE_ERR_INVALID_ARG;
  CUtensorMap tmA, tmW;
  rc = encode_gemm_maps(A_send, W, send_rows, L->E, N, H, &tmA, &tmW, /*gather=*/true);
  if (rc) return rc;
  GemmParams g;
  g.A_scale = A_send_scale;
  g.W_scale = W_scale;
  g.L = to_dev(L);
  g.N = N;
  g.H = H;
  g.R = send_rows;
  g.Y = Y;
  g.status = status;
  g.timeout_ns = 2000000000ull;
  g.gather_row = gather_row;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const long long max_units = (long long)L->max_tiles * (N / kGemmBN);
  const int grid = (int)std::max(1LL, std::min((long long)nsm, max_units));
  static const bool split_ok = register_split_fits(grouped_gemm1_kernel<true>);
  if (!split_ok) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(grouped_gemm1_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  ShortMaps unused;   // the gathered path loads A row by row
  unused.m[0] = tmA;
  unused.m[1] = tmA;
  grouped_gemm1_kernel<true><<<grid, kGemmThreads, kGemmSmemBytes, (cudaStream_t)stream>>>(tmA, tmW, unused, g,
                                                                                           A_send);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
