// combine.cu: weighted gather of each token's k expert outputs back into
// token order (the combine of the TilePipe page's "Communication Kernels";
// run unchanged after stage1 on the mori stage1 page).
//
// out[t, :] = bf16( sum_{j<k} w[t,j] * Y[pair_row[t*k+j], :] ), fp32 FMAs with
// the slots in ascending order.
#include "common.cuh"
#include "host_util.h"

namespace moe {

constexpr int kCombineWarps = 4;
constexpr int kCombineSlice = 2048;   // columns per work item (a token's output split across warps)

// One warp per (token, 2048-column slice); a lane owns 16 consecutive columns
// of each 512-column round and keeps the round's k rows (2 x 16 bytes each) in
// flight before folding them into the accumulator in slot order.
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const uint16_t* __restrict__ Y,
                                                                     int D, LayoutDev L,
                                                                     uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int T = L.T, k = L.k;
  const int slices = (D + kCombineSlice - 1) / kCombineSlice;
  const long long items = (long long)T * slices;
  for (long long w = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5); w < items;
       w += (long long)gridDim.x * kCombineWarps) {
    const int t = (int)(w / slices), s0 = (int)(w % slices) * kCombineSlice;
    int myrow = -1;
    float myw = 0.0f;
    if (lane < k) {
      myrow = L.pair_row[(size_t)t * k + lane];
      if (myrow >= 0) myw = L.row_weight[myrow];
    }
    const int s1 = min(D, s0 + kCombineSlice);
    for (int c0 = s0; c0 < s1; c0 += 512) {
      const int col = c0 + lane * 16;
      const bool act = col < s1;   // D % 8 == 0: a lane's 16 columns are all in or (only at D's end) half in
      const bool act2 = col + 8 < s1;
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 v[8][2];
        float wj[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          const int r = __shfl_sync(0xffffffffu, myrow, j & 31);
          wj[jj] = __shfl_sync(0xffffffffu, myw, j & 31);
          v[jj][0] = make_uint4(0, 0, 0, 0);
          v[jj][1] = v[jj][0];
          if (j < k && r >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(Y + (size_t)r * D + col);
            if (act) v[jj][0] = __ldcs(src);
            if (act2) v[jj][1] = __ldcs(src + 1);
          } else {
            wj[jj] = 0.0f;
          }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj >= k) break;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t w4[4] = {v[jj][hh].x, v[jj][hh].y, v[jj][hh].z, v[jj][hh].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[hh * 8 + 2 * i] = fmaf(wj[jj], bf16_lo(w4[i]), acc[hh * 8 + 2 * i]);
              acc[hh * 8 + 2 * i + 1] = fmaf(wj[jj], bf16_hi(w4[i]), acc[hh * 8 + 2 * i + 1]);
            }
          }
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(out + (size_t)t * D + col);
      if (act) {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        dst[0] = o;
      }
      if (act2) {
        uint4 o;
        o.x = pack_bf16x2(acc[8], acc[9]);
        o.y = pack_bf16x2(acc[10], acc[11]);
        o.z = pack_bf16x2(acc[12], acc[13]);
        o.w = pack_bf16x2(acc[14], acc[15]);
        dst[1] = o;
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
  const long long items = (long long)L->T * ((D + kCombineSlice - 1) / kCombineSlice);
  const int blocks = (int)std::max(1LL, std::min((items + kCombineWarps - 1) / kCombineWarps, (long long)nsm * 16));
  combine_kernel<<<blocks, kCombineWarps * 32, 0, (cudaStream_t)stream>>>(Y, D, to_dev(L), out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
