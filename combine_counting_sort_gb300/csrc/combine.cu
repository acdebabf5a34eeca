// combine.cu: weighted gather of each token's k expert outputs back into
// token order (the combine of the TilePipe page's "Communication Kernels";
// run unchanged after stage1 on the mori stage1 page).
//
// out[t, :] = bf16( sum_{j<k} w[t,j] * Y[pair_row[t*k+j], :] ), fp32 FMAs with
// the slots in ascending order.  One warp per token; a lane owns 8 columns
// (one 16-byte load per route) and keeps up to 8 routes' loads in flight
// before folding them into the accumulator in slot order.
#include "common.cuh"
#include "host_util.h"

namespace moe {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const uint16_t* __restrict__ Y,
                                                                     int D, LayoutDev L,
                                                                     uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int T = L.T, k = L.k;
  for (int t = blockIdx.x * kCombineWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kCombineWarps) {
    int myrow = -1;
    float myw = 0.0f;
    if (lane < k) {
      myrow = L.pair_row[(size_t)t * k + lane];
      if (myrow >= 0) myw = L.row_weight[myrow];
    }
    for (int c0 = 0; c0 < D; c0 += 256) {
      const int col = c0 + lane * 8;
      const bool act = col < D;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 v[8];
        float wj[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          const int r = __shfl_sync(0xffffffffu, myrow, j & 31);
          wj[jj] = __shfl_sync(0xffffffffu, myw, j & 31);
          v[jj] = make_uint4(0, 0, 0, 0);
          if (j < k && r >= 0 && act)
            v[jj] = __ldcs(reinterpret_cast<const uint4*>(Y + (size_t)r * D + col));
          else
            wj[jj] = 0.0f;
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj >= k) break;
          const uint32_t w4[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(wj[jj], bf16_lo(w4[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(wj[jj], bf16_hi(w4[i]), acc[2 * i + 1]);
          }
        }
      }
      if (act) {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(out + (size_t)t * D + col) = o;
      }
    }
  }
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine(const uint16_t* Y, int D, const moe_layout_t* L, uint16_t* out,
                           int32_t* status, moe_stream_t stream) {
  (void)status;
  int rc = check_layout(L);
  if (rc) return rc;
  if (!Y || !out) return MOE_ERR_INVALID_ARG;
  if (D < 8 || D % 8 != 0 || D > 65536) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Y) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const int blocks = std::max(1, std::min((L->T + kCombineWarps - 1) / kCombineWarps, nsm * 8));
  combine_kernel<<<blocks, kCombineWarps * 32, 0, (cudaStream_t)stream>>>(Y, D, to_dev(L), out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
