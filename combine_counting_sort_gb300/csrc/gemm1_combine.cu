// gemm1_combine.cu: moe_grouped_gemm1_combine, GEMM1 with the combine
// overlapped on the same SMs, gated per token.
//
// The TilePipe page ("Overlap"): a producer and a consumer on the same GPU
// synchronised by per-tile semaphores, so the consumer starts on a tile as
// soon as its producer is done with it; its "GEMM -> combine" driver runs the
// expert GEMM as the producer of the combine.  Here the consumer's unit is a
// token: its k expert outputs (all N columns of each of its k rows) must be
// stored before its weighted sum can be formed.
//
// One cooperative launch of the GEMM1 pipeline (gemm1.cuh), one CTA per SM, and:
//   epilogue warps  after storing a unit's Y rows, arrive on the unit's
//                   `stored` barrier;
//   warp 2          (counting) waits for that barrier, makes the stores
//                   visible at gpu scope with one fence, and bumps the
//                   completion counter of the token of every valid row of the
//                   unit (atom.release); the bump that brings a token to
//                   (N/256) x (its valid pairs) pushes the token onto a ready
//                   queue (atomic tail, slot published with st.release);
//   epilogue warps  once their CTA's GEMM work is done, pop tokens from the
//                   queue head (atomic ticket, bounded wait on the slot) and
//                   write out[t] = bf16( sum_j w[t,j] * Y[pair_row[t*k+j]] )
//                   with the same fp32 FMAs in the same slot order as
//                   moe_combine, so the output is bit-for-bit moe_combine's;
//                   8 rows x 64 bytes per lane in flight.
// Tokens with no valid pair are queued at the start (warp 3).  Every wait is
// bounded (timeout: MOE_ERR_TIMEOUT in *status).
//
// Under an expert-major tile order a token is complete only when its last
// expert is done, so most tokens become ready in the last few percent of the
// GEMM: the combine overlaps the GEMM's tail (CTAs finish their last units at
// different times) and needs no launch of its own.  Warpgroup 0 keeps 40
// registers (the promotion warps need the rest), too few to combine at a
// useful rate, so it does not combine.
#include "gemm1.cuh"
#include "host_util.h"

namespace moe {

constexpr int kCombHeader = 256;   // workspace bytes: queue head, queue tail
// Register split of this kernel: GEMM1's (40 for warpgroup 0: TMA, MMA and
// counting warps; 232 for the promotion warpgroups, which combine once their
// GEMM work is done), no spill.
constexpr uint32_t kRegsControlC = kRegsControl;
constexpr uint32_t kRegsEpilogueC = kRegsEpilogue;
static_assert(128 * kRegsControlC + 256 * kRegsEpilogueC <= 168u * kGemmThreads, "register split exceeds launch");

struct CombineParams {
  int32_t* qhead;     // pop ticket
  int32_t* qtail;     // push ticket
  unsigned long long* tr;   // trace slots (MOE_GC_TRACE_*), ns from %globaltimer
  int32_t* tok_cnt;   // [T] (row, N-block) stores completed per token
  int32_t* queue;     // [T] token + 1 per queue position, 0 until published
  uint16_t* out;      // [T][N]
  int T;
};

MOE_DEV int ld_relaxed_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MOE_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

MOE_DEV int valid_pairs(const LayoutDev& L, int t) {
  int v = 0;
  for (int j = 0; j < L.k; ++j) v += L.pair_row[(size_t)t * L.k + j] >= 0;
  return v;
}

MOE_DEV void push_token(const CombineParams& c, int t) {
  const int pos = atomicAdd(c.qtail, 1);
  st_release_gpu(c.queue + pos, t + 1);
  if (pos == c.T - 1) atomicMax(c.tr + MOE_GC_TRACE_LAST_PUSH, (unsigned long long)globaltimer_ns());
}

// Tokens with no valid pair (all ids invalid): nothing to wait for.  One warp
// of every CTA checks a strided share of the tokens.
MOE_DEV void queue_empty_tokens(const CombineParams& c, const LayoutDev& L) {
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 32 + lane; t < L.T; t += gridDim.x * 32)
    if (valid_pairs(L, t) == 0) push_token(c, t);
}

// Counting warp: per unit, after the epilogue's stores, bump the tokens of its rows.
MOE_DEV void count_loop(const GemmSmem& S, const GemmParams& g, const CombineParams& c) {
  GemmShared* sh = S.sh;
  const int lane = threadIdx.x & 31;
  const int nbn = g.N / kGemmBN;
  for (int j = 0;; ++j) {
    const int slot = j % kUnitRing;
    const uint32_t ph = (uint32_t)(j / kUnitRing) & 1u;
    if (!mbar_wait(smem_u32(&sh->ufull[slot]), ph, &sh->abort_flag, g.status, g.timeout_ns)) return;
    const int4 un = sh->unit[slot];
    const int rows = sh->unit_rows[slot];
    __syncwarp();
    if (un.x < 0) {
      if (lane == 0) mbar_arrive(smem_u32(&sh->uempty[slot]));
      return;
    }
    // the ring slot is handed back only after its stores are seen, so the
    // epilogue cannot arrive on this slot's `stored` barrier for a later unit first
    if (!mbar_wait(smem_u32(&sh->stored[slot]), ph, &sh->abort_flag, g.status, g.timeout_ns)) return;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh->uempty[slot]));
    // one fence makes the unit's Y stores (ordered before us by the barrier)
    // visible at gpu scope before every bump below: fence + relaxed atomic is
    // a release, without a fence per atomic
    fence_acq_rel_gpu();
    for (int i = lane; i < rows; i += 32) {
      const int r = un.w + i;
      const int t = g.L.row_pair[r] / g.L.k;
      const int now = atomicAdd(c.tok_cnt + t, 1) + 1;
      if (now % nbn == 0 && now == nbn * valid_pairs(g.L, t)) {
        fence_acq_rel_gpu();   // acquire every other bump of t (and the stores they released)
        push_token(c, t);
      }
    }
  }
}

// One token's weighted sum over its k rows, 256 * VEC columns per round: lane
// l owns columns [hh*256 + 8l, hh*256 + 8l + 8) of the round for hh < VEC, so
// every 16-byte load instruction of the warp covers 512 contiguous bytes;
// ROWS rows of VEC x 16 bytes per lane in flight; fp32 FMAs with the slots in
// ascending order (moe_combine's arithmetic, element by element).  Whole
// warp, converged.
template <int ROWS, int VEC>
MOE_DEV void combine_token(const LayoutDev& L, const uint16_t* __restrict__ Y, int D, int t, uint16_t* out) {
  const int lane = threadIdx.x & 31;
  const int k = L.k;
  int myrow = -1;
  float myw = 0.0f;
  if (lane < k) {
    myrow = L.pair_row[(size_t)t * k + lane];
    if (myrow >= 0) myw = L.row_weight[myrow];
  }
  for (int c0 = 0; c0 < D; c0 += 256 * VEC) {
    const int col = c0 + lane * 8;   // + hh * 256
    float acc[8 * VEC];
#pragma unroll
    for (int i = 0; i < 8 * VEC; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += ROWS) {
      uint4 v[ROWS][VEC];
      float wj[ROWS];
#pragma unroll
      for (int jj = 0; jj < ROWS; ++jj) {
        const int j = j0 + jj;
        const int r = __shfl_sync(0xffffffffu, myrow, j & 31);
        wj[jj] = __shfl_sync(0xffffffffu, myw, j & 31);
#pragma unroll
        for (int hh = 0; hh < VEC; ++hh) v[jj][hh] = make_uint4(0, 0, 0, 0);
        if (j < k && r >= 0) {
          const uint16_t* src = Y + (size_t)r * D + col;
#pragma unroll
          for (int hh = 0; hh < VEC; ++hh)
            if (col + hh * 256 < D) v[jj][hh] = __ldcg(reinterpret_cast<const uint4*>(src + hh * 256));
        } else {
          wj[jj] = 0.0f;
        }
      }
#pragma unroll
      for (int jj = 0; jj < ROWS; ++jj) {
        if (j0 + jj >= k) break;
#pragma unroll
        for (int hh = 0; hh < VEC; ++hh) {
          const uint32_t w4[4] = {v[jj][hh].x, v[jj][hh].y, v[jj][hh].z, v[jj][hh].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[hh * 8 + 2 * i] = fmaf(wj[jj], bf16_lo(w4[i]), acc[hh * 8 + 2 * i]);
            acc[hh * 8 + 2 * i + 1] = fmaf(wj[jj], bf16_hi(w4[i]), acc[hh * 8 + 2 * i + 1]);
          }
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < VEC; ++hh) {
      if (col + hh * 256 < D)
        *reinterpret_cast<uint4*>(out + (size_t)t * D + col + hh * 256) =
            make_uint4(pack_bf16x2(acc[hh * 8], acc[hh * 8 + 1]), pack_bf16x2(acc[hh * 8 + 2], acc[hh * 8 + 3]),
                       pack_bf16x2(acc[hh * 8 + 4], acc[hh * 8 + 5]), pack_bf16x2(acc[hh * 8 + 6], acc[hh * 8 + 7]));
    }
  }
}

// Pop tokens until the queue's T positions are all taken.  A position whose
// token is not published within the timeout ends the loop with MOE_ERR_TIMEOUT.
template <int ROWS, int VEC>
MOE_DEV void combine_loop(const GemmParams& g, const CombineParams& c) {
  const int lane = threadIdx.x & 31;
  for (;;) {
    int v = 0;
    if (lane == 0) v = atomicAdd(c.qhead, 1);
    v = __shfl_sync(0xffffffffu, v, 0);
    if (v >= g.L.T) return;
    int t = -1;
    const uint64_t w0 = globaltimer_ns();
    if (lane == 0) {
      // relaxed polling, one acquire fence once the slot is published
      int x = ld_relaxed_gpu(c.queue + v);
      if (x == 0) {
        const uint64_t t0 = globaltimer_ns();
        while ((x = ld_relaxed_gpu(c.queue + v)) == 0) {
          if (globaltimer_ns() - t0 > g.timeout_ns) {
            set_status(g.status, MOE_ERR_TIMEOUT);
            break;
          }
          __nanosleep(200);
        }
      }
      fence_acq_rel_gpu();
      t = x - 1;
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t < 0) return;
    const uint64_t w1 = globaltimer_ns();
    combine_token<ROWS, VEC>(g.L, g.Y, g.N, t, c.out);
    if (lane == 0) {
      atomicAdd(c.tr + MOE_GC_TRACE_WAIT_NS, (unsigned long long)(w1 - w0));
      atomicAdd(c.tr + MOE_GC_TRACE_WORK_NS, (unsigned long long)(globaltimer_ns() - w1));
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm1_combine_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                                 const __grid_constant__ GemmParams g, const __grid_constant__ CombineParams c) {
  extern __shared__ uint8_t smem_raw[];
  const GemmSmem S = gemm_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
  }
  if (threadIdx.x == 0) atomicCAS(c.tr + MOE_GC_TRACE_START, 0ull, (unsigned long long)globaltimer_ns());
  gemm_setup(S, /*extra_unit_consumers=*/1);   // the counting warp reads every unit too
  const int nbn = g.N / kGemmBN;
  const int KB = g.H / kGemmBK;
  const int units = g.L.num_tiles[0] * nbn;

  if (warp < kEpiWarp0) {
    regs_dealloc<kRegsControlC>();
    if (warp == 0) {
      uint32_t it = 0;
      int j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
        const Unit x = unit_of(g.L, u, nbn);
        ok = publish_unit(S.sh, j, x, g.status, g.timeout_ns) &&
             produce_unit(S, &tmA, &tmW, x, KB, it, g.status, g.timeout_ns);
      }
      if (ok) {
        Unit end = {-1, 0, 0, 0, 0};
        publish_unit(S.sh, j, end, g.status, g.timeout_ns);
      }
      drain_fills(S, it, g.timeout_ns);
    } else if (warp == 1) {
      mma_loop<false, true>(S, KB, g.status, g.timeout_ns);
    } else if (warp == 2) {
      count_loop(S, g, c);
    } else {
      queue_empty_tokens(c, g.L);
    }
  } else {
    regs_alloc<kRegsEpilogueC>();
    epilogue_loop<true, true, false, false, true, true>(S, g);
    if (warp == kEpiWarp0 && lane == 0) {   // this CTA's GEMM work is done
      const unsigned long long now = globaltimer_ns();
      atomicMin(c.tr + MOE_GC_TRACE_GEMM_FIRST_DONE, now);
      atomicMax(c.tr + MOE_GC_TRACE_GEMM_LAST_DONE, now);
    }
    combine_loop<8, 4>(g, c);
  }
  gemm_teardown(S);
  if (threadIdx.x == 0) atomicMax(c.tr + MOE_GC_TRACE_END, (unsigned long long)globaltimer_ns());
}

}  // namespace moe

using namespace moe;

size_t moe_gemm_combine_ws_bytes(int T) { return kCombHeader + 2 * sizeof(int32_t) * (size_t)T; }

int gemm1_check_args(const uint8_t* A, const float* A_scale, const uint8_t* W, const float* W_scale, int N,
                     int H, const moe_layout_t* L, const uint16_t* Y);

extern "C" int moe_grouped_gemm1_combine(const uint8_t* A, const float* A_scale, const uint8_t* W,
                                         const float* W_scale, int N, int H, const moe_layout_t* L, uint16_t* Y,
                                         uint16_t* out, void* ws, size_t ws_bytes, int32_t* status,
                                         moe_stream_t stream) {
  int rc = gemm1_check_args(A, A_scale, W, W_scale, N, H, L, Y);
  if (rc) return rc;
  if (!out || !ws || !aligned16(out) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_gemm_combine_ws_bytes(L->T)) return MOE_ERR_INVALID_ARG;
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
  char* base = reinterpret_cast<char*>(ws);
  CombineParams c;
  c.qhead = reinterpret_cast<int32_t*>(base);
  c.qtail = c.qhead + 1;
  c.tr = reinterpret_cast<unsigned long long*>(base + MOE_GC_TRACE_OFFSET);
  c.tok_cnt = reinterpret_cast<int32_t*>(base + kCombHeader);
  c.queue = c.tok_cnt + L->T;
  c.out = out;
  c.T = L->T;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, moe_gemm_combine_ws_bytes(L->T), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(base + MOE_GC_TRACE_OFFSET + 8 * MOE_GC_TRACE_GEMM_FIRST_DONE, 0xFF, 8, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, grouped_gemm1_combine_kernel) != cudaSuccess) return MOE_ERR_CUDA;
    if (128u * kRegsControlC + 256u * kRegsEpilogueC > (uint32_t)a.numRegs * (uint32_t)kGemmThreads)
      return MOE_ERR_UNSUPPORTED;
  }
  if (cudaFuncSetAttribute(grouped_gemm1_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsm);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, grouped_gemm1_combine_kernel, tmA, tmW, g, c) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
