// quant.cu: FP8 e4m3 quantise-once + dispatch scatter, weight quantisation,
// and the identity expert.  The per-token quantise + scatter lives in
// quant.cuh (shared with the producer role of the fused stage1 kernel).
#include "quant.cuh"
#include "host_util.h"

namespace moe {

constexpr int kQuantWarps = 8;

// One warp per (token, column range) work item: a token's H columns are split
// into `splits` ranges of whole chunks of ROUNDS x 512 columns (the mori page's
// --split), as many as it takes to give every SM enough warps; each item walks
// its range chunk by chunk.  Batches below 8192 tokens use 1024-column chunks
// (more items), larger ones 2048-column chunks (4 KB of the row in flight per warp).
// `rows` holds per_token destination rows of each token (-1: none), R is the
// row count of A (the stride of A_scale): the dense layout passes pair_row, k
// and T*k; the per-(token, group) send runs pass send_row, G and their capacity.
template <int ROUNDS>
__global__ void __launch_bounds__(kQuantWarps * 32, ROUNDS == 2 ? 4 : 3) dispatch_quant_kernel(
    const uint16_t* __restrict__ x, int H, int T, const int32_t* __restrict__ rows, int per_token, long long R,
    int splits, uint8_t* __restrict__ A, float* __restrict__ A_scale) {
  constexpr int kSliceCols = 512 * ROUNDS;
  const int lane = threadIdx.x & 31;
  const int k = per_token;
  const int chunks = (H + kSliceCols - 1) / kSliceCols;
  const int per = (chunks + splits - 1) / splits;
  const long long items = (long long)T * splits;
  for (long long w = (long long)blockIdx.x * kQuantWarps + (threadIdx.x >> 5); w < items;
       w += (long long)gridDim.x * kQuantWarps) {
    const int t = (int)(w / splits), sp = (int)(w % splits);
    const int myrow = lane < k ? rows[(size_t)t * k + lane] : -1;
    const int cend = min(chunks, (sp + 1) * per);
    for (int c = sp * per; c < cend; ++c)
      quant_scatter_slice<ROUNDS>(x, H, t, c * kSliceCols, k, R, myrow, A, A_scale);
  }
}

// One CTA per 128x128 weight block: thread = (row, half) owns 64 consecutive values.
__global__ void __launch_bounds__(256) quant_weights_kernel(const uint16_t* __restrict__ W, int N,
                                                            int H, uint8_t* __restrict__ Wq,
                                                            float* __restrict__ Ws) {
  __shared__ float red[8];
  const int kb = blockIdx.x, nb = blockIdx.y, e = blockIdx.z;
  const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
  const size_t off = ((size_t)e * N + (size_t)nb * 128 + row) * H + (size_t)kb * 128 + half * 64;
  const uint4* src = reinterpret_cast<const uint4*>(W + off);
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldcs(src + i);
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w4[j])), fabsf(bf16_hi(w4[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
  __syncthreads();
  am = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) am = fmaxf(am, red[i]);
  const float scale = __fdiv_rn(am, 448.0f);
  uint4* dst = reinterpret_cast<uint4*>(Wq + off);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float f[16];
    unpack16(v[2 * c], v[2 * c + 1], f);
    dst[c] = quant16(f, scale);
  }
  if (threadIdx.x == 0) Ws[((size_t)e * (N / 128) + nb) * (H / 128) + kb] = scale;
}

// Identity expert: Y[r, :] = bf16(code * scale), one rounding of the exact product.
__global__ void __launch_bounds__(256) dequant_rows_kernel(const uint8_t* __restrict__ A,
                                                           const float* __restrict__ A_scale, int H,
                                                           LayoutDev L, uint16_t* __restrict__ Y) {
  const int lane = threadIdx.x & 31;
  const long long R = (long long)L.T * L.k;
  const int rows = L.expert_offset[L.E];
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += gridDim.x * 8) {
    for (int c0 = 0; c0 < H; c0 += 512) {
      const int col = c0 + lane * 16;
      if (col >= H) continue;
      const uint4 q = *reinterpret_cast<const uint4*>(A + (size_t)r * H + col);
      const float s = A_scale[(size_t)(col / kQBlock) * R + r];
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v0 = e4m3x2_to_float2((uint16_t)(qw[i] & 0xFFFFu));
        const float2 v1 = e4m3x2_to_float2((uint16_t)(qw[i] >> 16));
        o[2 * i] = (uint32_t)bf16_of_product(v0.x, s) | ((uint32_t)bf16_of_product(v0.y, s) << 16);
        o[2 * i + 1] = (uint32_t)bf16_of_product(v1.x, s) | ((uint32_t)bf16_of_product(v1.y, s) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(Y + (size_t)r * H + col);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

}  // namespace moe

using namespace moe;

// Launch of the quantise-once scatter over T tokens with `per_token`
// destination rows each (shared by the dense and the send-run dispatch).
int launch_dispatch(const uint16_t* x, int H, int T, const int32_t* rows, int per_token, long long R, uint8_t* A,
                    float* A_scale, cudaStream_t stream) {
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  // small batches: every 1024-column chunk is an item; large ones: split tokens
  // only as far as needed for ~64 warps per SM
  const bool small = T < 8192;
  const int cols = small ? 1024 : 2048;
  const int chunks = (H + cols - 1) / cols;
  const long long want = (long long)nsm * 64;
  const int splits = small ? chunks : (int)std::max(1LL, std::min((long long)chunks, (want + T - 1) / T));
  const long long items = (long long)T * splits;
  const int blocks = (int)std::max(1LL, std::min((items + kQuantWarps - 1) / kQuantWarps, (long long)nsm * 16));
  if (small)
    dispatch_quant_kernel<2><<<blocks, kQuantWarps * 32, 0, stream>>>(x, H, T, rows, per_token, R, splits, A, A_scale);
  else
    dispatch_quant_kernel<4><<<blocks, kQuantWarps * 32, 0, stream>>>(x, H, T, rows, per_token, R, splits, A, A_scale);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_dispatch_quant(const uint16_t* x, int H, const moe_layout_t* L, uint8_t* A,
                                  float* A_scale, int32_t* status, moe_stream_t stream) {
  (void)status;
  int rc = check_layout(L);
  if (rc) return rc;
  if (!x || !A || !A_scale) return MOE_ERR_INVALID_ARG;
  if (H < kQBlock || H % kQBlock != 0 || H > 32768) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(A) || !aligned16(A_scale)) return MOE_ERR_INVALID_ARG;
  return launch_dispatch(x, H, L->T, L->pair_row, L->k, (long long)L->T * L->k, A, A_scale, (cudaStream_t)stream);
}

extern "C" int moe_quant_weights(const uint16_t* W, int E, int N, int H, uint8_t* Wq, float* W_scale,
                                 moe_stream_t stream) {
  if (!W || !Wq || !W_scale) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 65535 || N < 128 || N % 128 || H < 128 || H % 128 || N > 32768 || H > 32768)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(Wq)) return MOE_ERR_INVALID_ARG;
  quant_weights_kernel<<<dim3(H / 128, N / 128, E), 256, 0, (cudaStream_t)stream>>>(W, N, H, Wq, W_scale);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_dequant_rows(const uint8_t* A, const float* A_scale, int H, const moe_layout_t* L,
                                uint16_t* Y, moe_stream_t stream) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!A || !A_scale || !Y) return MOE_ERR_INVALID_ARG;
  if (H < kQBlock || H % kQBlock != 0 || H > 32768) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const long long R = (long long)L->T * L->k;
  const int blocks = (int)std::max(1LL, std::min((R + 7) / 8, (long long)nsm * 8));
  dequant_rows_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(A, A_scale, H, to_dev(L), Y);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
