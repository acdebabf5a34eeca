// stage1.cu: moe_stage1, the fused quant + dispatch + GEMM1 with
// producer/consumer overlap on a partitioned SM set.
//
// The TilePipe page ("Overlap"): the SMs are split between a producer that
// bumps a semaphore per finished tile and a consumer GEMM that waits on it;
// the producer's order is chosen to unblock the consumer's expert-major tile
// order as early as possible (earliest deadline first); the synchronisation
// granularity (per tile or per expert) trades flag traffic for earlier starts.
// The mori stage1 page ("How it works now"): GEMM1 gated per tile on ready
// signals in a static order, or --ready-first, where one scheduler publishes
// M-tiles in readiness order and workers take tickets with one atomic.
//
// One cooperative launch, one CTA per SM (co-residency is what makes the
// bounded waits below safe):
//   CTAs [0, S)   producers: every warp quantises tokens taken in token_order
//                 (tokens sorted by first expert, so rows of low experts land
//                 first) into one of two shared-memory row buffers, stores the
//                 block scales to the token's k rows and bulk-copies the code
//                 row to each of them; once a token's copies are complete (one
//                 token later) each of its rows is published with a release
//                 add on its tile's flag (or its expert's flag).  Rows too wide
//                 for two buffers per warp go out by 16-byte stores instead.
//                 With producers_join they then take GEMM work like the
//                 consumers.
//   CTAs [S, #SM) consumers: the GEMM1 pipeline of gemm1.cuh; the TMA warp
//                 acquires a unit's ready flag (bounded wait) before it hands
//                 the unit to the MMA and promotion warps and before the
//                 unit's first load; the unit ring's mbarrier carries that
//                 acquire on to the promotion warps' A_scale reads.
// Units come from a static expert-major stride, or from a global ticket
// counter (expert-major order, or positions of the ready queue filled by a
// scheduler warp in readiness order).
#include "gemm1.cuh"
#include "quant.cuh"
#include "host_util.h"

namespace moe {

constexpr int kWsHeader = 256;   // bytes: ticket counter, queue length

struct Stage1Params {
  GemmParams g;
  const uint16_t* x;
  uint8_t* A;
  float* A_scale;
  int S;              // producer CTAs
  int per_expert;     // flag granularity
  int ready_first;    // schedule
  int join;           // producers take GEMM work when done
  int use_tickets;
  int withhold_tile;  // test hook: rows of this tile are never published (-1: off)
  int trace;          // record stamps / counters in the workspace header
  unsigned long long* tr;  // trace slots
  int32_t* ticket;
  int32_t* qlen;
  int32_t* tile_flag;     // [max_tiles] rows landed
  int32_t* expert_flag;   // [E] rows landed
  int32_t* queue;         // [max_tiles] M-tiles in publish order
};

// Bounded wait until the unit's rows have all landed; then order the later
// async-proxy (TMA) reads after the acquired generic-proxy writes.
MOE_DEV bool wait_ready(const Stage1Params& p, int m, int e, int rows, volatile int* abort_flag,
                        bool count = false) {
  const int32_t* flag = p.per_expert ? p.expert_flag + e : p.tile_flag + m;
  const int target = p.per_expert ? p.g.L.count[e] : rows;
  if (ld_acquire_gpu(flag) < target) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
      if (ld_acquire_gpu(flag) >= target) {
        if (count && p.trace) {
          atomicAdd(p.tr + MOE_TRACE_WAIT_NS, (unsigned long long)(globaltimer_ns() - t0));
          atomicAdd(p.tr + MOE_TRACE_WAITED_UNITS, 1ull);
        }
        break;
      }
      if ((i & 7u) == 7u) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > p.g.timeout_ns) {
          *abort_flag = 1;
          set_status(p.g.status, MOE_ERR_TIMEOUT);
          return false;
        }
      }
      __nanosleep(64);
    }
  }
  fence_proxy_async_global();
  return true;
}

// Lane j < k publishes its row of the token (per-tile or per-expert flag),
// after a fence that orders the row's writes before the release.
MOE_DEV void publish_row(const Stage1Params& p, int row, const int* s_eoff, const int* s_toff) {
  if (row < 0) return;
  int lo = 0, hi = p.g.L.E;                     // expert of the row: largest e with eoff[e] <= row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_eoff[mid] <= row) lo = mid; else hi = mid;
  }
  const int m = s_toff[lo] + (row - s_eoff[lo]) / kGemmBM;
  if (m != p.withhold_tile) {
    __threadfence();
    red_release_gpu_add(p.per_expert ? p.expert_flag + lo : p.tile_flag + m, 1);
  }
}

// Producer warp: tokens token_order[i] for i = gw, gw + PW, ..., each
// quantised once in 2048-column chunks (4 KB of the row in flight) and stored
// to its k rows with 16-byte stores, then published.
MOE_DEV void produce_tokens(const Stage1Params& p, int gw, int PW, const int* s_eoff, const int* s_toff) {
  const int lane = threadIdx.x & 31;
  const LayoutDev& L = p.g.L;
  const int T = L.T, k = L.k;
  for (int i = gw; i < T; i += PW) {
    const int t = L.token_order[i];
    const int myrow = lane < k ? L.pair_row[(size_t)t * k + lane] : -1;
    for (int c0 = 0; c0 < p.g.H; c0 += 2048)
      quant_scatter_slice<4>(p.x, p.g.H, t, c0, k, p.g.R, myrow, p.A, p.A_scale);
    fence_proxy_async_global();
    __syncwarp();
    publish_row(p, myrow, s_eoff, s_toff);
  }
}

// The same with the code rows written by bulk copies (the TMA engine, not the
// warp's 16-byte stores, which set a producer SM's pace): the token's codes
// are staged in one of two row buffers of `stg` (2 x H bytes), and lane j < k
// copies the row to A row j.  A token is published one token later, once its
// copies are complete (wait_group 1), so the copies of token i overlap the
// quantisation of token i+1; that wait also frees the buffer token i+2 reuses.
MOE_DEV void produce_tokens_bulk(const Stage1Params& p, int gw, int PW, const int* s_eoff, const int* s_toff,
                                 uint32_t stg) {
  const int lane = threadIdx.x & 31;
  const LayoutDev& L = p.g.L;
  const int T = L.T, k = L.k, H = p.g.H;
  int prev_row = -1;
  bool have_prev = false;
  uint32_t buf = 0;
  for (int i = gw; i < T; i += PW) {
    const int t = L.token_order[i];
    const int myrow = lane < k ? L.pair_row[(size_t)t * k + lane] : -1;
    const uint32_t row_s = stg + buf * (uint32_t)H;
    for (int c0 = 0; c0 < H; c0 += 2048)
      quant_stage_slice<4>(p.x, H, t, c0, k, p.g.R, myrow, p.A_scale, row_s);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane < k) {
      if (myrow >= 0) bulk_copy_to_global(p.A + (size_t)myrow * H, row_s, (uint32_t)H);
      bulk_commit();
    }
    if (have_prev) {
      if (lane < k) bulk_wait<1>();            // the previous token's copies are complete
      fence_proxy_async_global();
      __syncwarp();
      publish_row(p, prev_row, s_eoff, s_toff);
    }
    prev_row = myrow;
    have_prev = true;
    buf ^= 1u;
  }
  if (have_prev) {
    if (lane < k) bulk_wait<0>();
    fence_proxy_async_global();
    __syncwarp();
    publish_row(p, prev_row, s_eoff, s_toff);
  }
}

// Scheduler warp (--ready-first): publish M-tiles into the queue as they complete.
MOE_DEV void schedule_ready(const Stage1Params& p, uint32_t* s_done) {
  const int lane = threadIdx.x & 31;
  const LayoutDev& L = p.g.L;
  const int nt = L.num_tiles[0];
  const int words = (nt + 31) / 32;
  for (int w = lane; w < words; w += 32) s_done[w] = 0u;
  __syncwarp();
  int published = 0;
  uint64_t t0 = globaltimer_ns();   // time of the last progress
  while (published < nt) {
    int progress = 0;
    for (int base = 0; base < nt; base += 32) {
      const int m = base + lane;
      bool ready = false;
      if (m < nt && !(s_done[m >> 5] & (1u << (m & 31)))) {
        if (p.per_expert) {
          const int e = L.tile_expert[m];
          ready = ld_acquire_gpu(p.expert_flag + e) >= L.count[e];
        } else {
          ready = ld_acquire_gpu(p.tile_flag + m) >= L.tile_rows[m];
        }
      }
      const unsigned b = __ballot_sync(0xffffffffu, ready);
      if (b) {
        if (ready) p.queue[published + __popc(b & lanemask_lt())] = m;
        __syncwarp();
        if (lane == 0) s_done[base >> 5] |= b;   // one writer per bitmap word
        __syncwarp();
        published += __popc(b);
        progress += __popc(b);
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.qlen, published);
      }
    }
    if (progress) {
      t0 = globaltimer_ns();
    } else {
      if (globaltimer_ns() - t0 > p.g.timeout_ns) {
        if (lane == 0) set_status(p.g.status, MOE_ERR_TIMEOUT);
        return;
      }
      __nanosleep(256);
    }
  }
}

// Consumer TMA thread: next unit index, or -1 when the work is done.
MOE_DEV int next_unit(const Stage1Params& p, int units, int nbn, int& cursor, int stride,
                      volatile int* abort_flag) {
  if (!p.use_tickets) {
    const int u = cursor;
    cursor += stride;
    return u < units ? u : -1;
  }
  const int v = atomicAdd(p.ticket, 1);
  if (v >= units) return -1;
  if (!p.ready_first) return v;
  const int pos = v / nbn;
  if (ld_acquire_gpu(p.qlen) <= pos) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
      if (ld_acquire_gpu(p.qlen) > pos) break;
      if ((i & 7u) == 7u) {
        if (*abort_flag) return -2;
        if (globaltimer_ns() - t0 > p.g.timeout_ns) {
          *abort_flag = 1;
          set_status(p.g.status, MOE_ERR_TIMEOUT);
          return -2;
        }
      }
      __nanosleep(64);
    }
  }
  const int m = __ldcg(p.queue + pos);
  return m * nbn + v % nbn;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    stage1_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ Stage1Params p) {
  extern __shared__ uint8_t smem_raw[];
  const GemmSmem S = gemm_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const LayoutDev& L = p.g.L;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
  }
  gemm_setup(S);
  const int nbn = p.g.N / kGemmBN;
  const int KB = p.g.H / kGemmBK;
  const bool producer = (int)blockIdx.x < p.S;
  if (p.trace && threadIdx.x == 0) atomicCAS(p.tr + MOE_TRACE_START, 0ull, (unsigned long long)globaltimer_ns());

  if (producer) {
    // the stage buffers are idle while producing: stage the expert offset tables there
    int* s_eoff = reinterpret_cast<int*>(S.stages);
    int* s_toff = s_eoff + (L.E + 1);
    uint32_t* s_done = reinterpret_cast<uint32_t*>(s_toff + (L.E + 1));
    for (int e = threadIdx.x; e <= L.E; e += blockDim.x) {
      s_eoff[e] = L.expert_offset[e];
      s_toff[e] = L.expert_tile_offset[e];
    }
    __syncthreads();
    const int nw = kGemmThreads / 32;
    const bool sched = p.ready_first && blockIdx.x == 0 && warp == nw - 1;
    if (sched) {
      schedule_ready(p, s_done);
    } else {
      int gw = blockIdx.x * nw + warp;
      int PW = p.S * nw;
      if (p.ready_first) { PW -= 1; if (gw > nw - 1) gw -= 1; }
      // two staging rows per warp after the offset tables and the scheduler's
      // bitmap, when they fit in the idle stage buffers
      const size_t bitmap_bytes = ((size_t)L.max_tiles + 31) / 32 * 4;
      const size_t table_end =
          ((size_t)(reinterpret_cast<uint8_t*>(s_done) - S.stages) + bitmap_bytes + 1023) & ~size_t(1023);
      if (table_end + (size_t)nw * 2 * p.g.H <= (size_t)kGemmStages * kStageBytes)
        produce_tokens_bulk(p, gw, PW, s_eoff, s_toff,
                            smem_u32(S.stages + table_end + (size_t)warp * 2 * p.g.H));
      else
        produce_tokens(p, gw, PW, s_eoff, s_toff);
    }
    // the stage buffers go back to the TMA (async proxy) after generic-proxy use
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (p.trace && threadIdx.x == 0) atomicMax(p.tr + MOE_TRACE_PRODUCED, (unsigned long long)globaltimer_ns());
    if (!p.join) {
      gemm_teardown(S);
      return;
    }
  }

  const int units = L.num_tiles[0] * nbn;
  if (warp < kEpiWarp0) {
    regs_dealloc<kRegsControl>();
    if (warp == 0) {
      // the whole warp runs the loop (converged, warp-uniform values); lane 0
      // claims units (ticket atomics, queue reads) and broadcasts them
      uint32_t it = 0;
      int j = 0;
      bool ok = true;
      int cursor = (int)blockIdx.x - p.S;
      const int stride = (int)gridDim.x - p.S;
      while (ok) {
        int u = 0;
        if (lane == 0) u = next_unit(p, units, nbn, cursor, stride, &S.sh->abort_flag);
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u == -2) { ok = false; break; }
        if (u < 0) break;
        const Unit x = unit_of(L, u, nbn);
        // the acquire of the unit's ready flag comes before the unit is handed
        // on: the ring's mbarrier (release here, acquire in the promotion warps)
        // orders the producers' A_scale writes before the promotion warps' reads
        ok = wait_ready(p, x.m, x.e, x.rows, &S.sh->abort_flag, lane == 0) &&
             publish_unit(S.sh, j, x, p.g.status, p.g.timeout_ns) &&
             produce_unit(S, &tmA, &tmW, x, KB, it, p.g.status, p.g.timeout_ns);
        ++j;
      }
      if (p.trace && lane == 0) {
        atomicAdd(p.tr + MOE_TRACE_UNITS, (unsigned long long)j);
        if (producer) atomicAdd(p.tr + MOE_TRACE_JOINED_UNITS, (unsigned long long)j);
      }
      if (ok) {
        Unit end = {-1, 0, 0, 0, 0};
        publish_unit(S.sh, j, end, p.g.status, p.g.timeout_ns);
      }
      drain_fills(S, it, p.g.timeout_ns);
    } else if (warp == 1) {
      mma_loop<false, true>(S, KB, p.g.status, p.g.timeout_ns);
    }
  } else {
    regs_alloc<kRegsEpilogue>();
    epilogue_loop<false, false, false, false, true, true>(S, p.g);
  }
  gemm_teardown(S);
  if (p.trace && threadIdx.x == 0) atomicMax(p.tr + MOE_TRACE_END, (unsigned long long)globaltimer_ns());
}

}  // namespace moe

using namespace moe;

size_t moe_stage1_ws_bytes(int T, int k, int E, int block_m) {
  const size_t tiles = (size_t)max_tiles_of(T, k, E, block_m);
  // header (ticket, queue length) + per-tile flags + per-expert flags + ready queue
  return kWsHeader + sizeof(int32_t) * (tiles + (size_t)E + tiles);
}

int gemm1_check_args(const uint8_t* A, const float* A_scale, const uint8_t* W, const float* W_scale, int N,
                     int H, const moe_layout_t* L, const uint16_t* Y);

extern "C" int moe_stage1(const uint16_t* x, int H, const moe_layout_t* L, const uint8_t* W,
                          const float* W_scale, int N, const moe_stage1_opts_t* opts, uint8_t* A,
                          float* A_scale, uint16_t* Y, void* ws, size_t ws_bytes, int32_t* status,
                          moe_stream_t stream) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!x || !W || !W_scale || !A || !A_scale || !Y || !ws || !opts) return MOE_ERR_INVALID_ARG;
  rc = gemm1_check_args(A, A_scale, W, W_scale, N, H, L, Y);
  if (rc) return rc;
  if (!aligned16(x) || !aligned16(A_scale) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_stage1_ws_bytes(L->T, L->k, L->E, L->block_m)) return MOE_ERR_INVALID_ARG;
  const int nsm = device_sm_count();
  if (nsm < 2) return MOE_ERR_CUDA;
  const int S = opts->comm_sms > 0 ? opts->comm_sms : std::min(16, nsm / 2);
  if (S >= nsm) return MOE_ERR_INVALID_ARG;
  if (opts->flags != MOE_FLAGS_PER_TILE && opts->flags != MOE_FLAGS_PER_EXPERT) return MOE_ERR_INVALID_ARG;
  if (opts->schedule != MOE_SCHED_EXPERT_MAJOR && opts->schedule != MOE_SCHED_READY_FIRST)
    return MOE_ERR_INVALID_ARG;
  // the producer CTAs stage the offset tables (and the scheduler its bitmap) in the idle stage buffers
  const long long table_bytes = 8LL * (L->E + 1);
  if (opts->schedule == MOE_SCHED_READY_FIRST &&
      (long long)L->max_tiles > ((long long)kGemmStages * kStageBytes - table_bytes) * 8)
    return MOE_ERR_UNSUPPORTED;

  const long long R = (long long)L->T * L->k;
  const int tiles = L->max_tiles;
  Stage1Params p;
  p.g.A_scale = A_scale;
  p.g.W_scale = W_scale;
  p.g.L = to_dev(L);
  p.g.N = N;
  p.g.H = H;
  p.g.R = R;
  p.g.Y = Y;
  p.g.status = status;
  p.g.timeout_ns = opts->timeout_ns > 0 ? (uint64_t)opts->timeout_ns : 1000000000ull;
  p.g.gather_row = nullptr;
  p.x = x;
  p.A = A;
  p.A_scale = A_scale;
  p.S = S;
  p.per_expert = opts->flags == MOE_FLAGS_PER_EXPERT;
  p.ready_first = opts->schedule == MOE_SCHED_READY_FIRST;
  p.join = opts->producers_join != 0;
  p.use_tickets = p.join || p.ready_first;
  p.withhold_tile = opts->withhold_tile;
  p.trace = opts->trace != 0;
  p.tr = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + MOE_TRACE_OFFSET);
  char* base = reinterpret_cast<char*>(ws);
  p.ticket = reinterpret_cast<int32_t*>(base);
  p.qlen = p.ticket + 1;
  p.tile_flag = reinterpret_cast<int32_t*>(base + kWsHeader);
  p.expert_flag = p.tile_flag + tiles;
  p.queue = p.expert_flag + L->E;

  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, kWsHeader + sizeof(int32_t) * ((size_t)tiles + L->E), s) != cudaSuccess)
    return MOE_ERR_CUDA;

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
  static const bool split_ok = register_split_fits(stage1_kernel);
  if (!split_ok) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(stage1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmemBytes) !=
      cudaSuccess)
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
  if (cudaLaunchKernelEx(&cfg, stage1_kernel, tmA, tmW, p) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
