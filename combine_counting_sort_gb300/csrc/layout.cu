// layout.cu: routing layout (stable counting sort of the T*k (token, slot)
// pairs by (group, expert)) and the top-k router helper.
//
// The counting sort of the mori stage1 page ("How it works now": a counting
// sort by (destination, first expert) so that a landed prefix of a run is a
// prefix of experts; recv_layout commit: per-expert counts, padding of every
// expert to the sort block, expert-major tables) as ONE launch: a cooperative
// grid of at most one block per SM (T <= 32: a single block in a plain launch,
// which needs neither barrier):
//
//   phase A  each block histograms its contiguous token range: experts of its
//            pairs and first (smallest) experts of its tokens, with
//            warp-aggregated shared-memory adds (__match_any_sync leaders);
//            the block's ids and weights stay staged in shared memory.
//   barrier  grid-wide barrier (bounded spin: MOE_ERR_TIMEOUT after 1 s).
//   phase B  the per-block histograms are scanned down the blocks, one warp
//            per expert column (in place: each entry becomes that block's
//            exclusive prefix; the column total goes to a totals array);
//            after a second grid barrier every block reads its own row of
//            prefixes and the totals, scans across experts (expert offsets,
//            tile offsets, first-expert offsets) in shared memory; block 0
//            writes the E-sized tables; the tile tables and the rowmap are
//            written one tile per warp over the whole grid.
//   phase C  stable ranks: the block's pairs, in (token, slot) order, are cut
//            into one contiguous slice per warp; per-warp histograms scanned
//            across the warps give each warp its first row per expert, and each
//            warp walks its slice 32 at a time (lanes with equal experts find
//            each other with __match_any_sync and take consecutive rows); the
//            token order by first expert is ranked the same way.
//
// Logical group g holds experts [g*E/G, (g+1)*E/G) (the Mojo EPDispatchKernel
// page's n_local_experts = n_experts / n_ranks), so the key (group, expert)
// orders like the expert id.
#include "common.cuh"
#include "host_util.h"

namespace moe {

constexpr int kLayoutThreads = 512;
constexpr int kLayoutMaxBlocks = 256;     // bound of the workspace's per-block histograms
constexpr int kChunkPairs = 4096;         // pairs staged in shared memory per pass
constexpr int kLayoutWarps = kLayoutThreads / 32;

struct LayoutArgs {
  const int32_t* ids;
  const float* w;
  LayoutDev L;
  int32_t* ws_hist;     // [E][kLayoutMaxBlocks]: expert e's count in block b at e * kLayoutMaxBlocks + b
  int32_t* ws_fhist;    // [E][kLayoutMaxBlocks]
  int32_t* ws_tot;      // [2][E] column totals of ws_hist / ws_fhist
  uint32_t* ws_barrier; // [2] zeroed in-stream before the launch
  int32_t* status;
  int tpb;              // tokens per block
  uint64_t timeout_ns;
  int quiet;            // 1: a negative id means "no route" and is skipped without an error status
};

__device__ __forceinline__ int first_expert(const int32_t* s_ids, int k, int E) {
  int fe = E;
  for (int j = 0; j < k; ++j) {
    int e = s_ids[j];
    if (e >= 0 && e < E && e < fe) fe = e;
  }
  return fe;
}

// Grid-wide barrier on counter `ctr` (all blocks co-resident: cooperative
// launch), bounded by timeout_ns; false (and MOE_ERR_TIMEOUT) if it gave up.
// `flag` is a shared int used to broadcast the outcome.
__device__ bool grid_barrier(uint32_t* ctr, int nblk, int32_t* status, uint64_t timeout_ns, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int timed_out = 0;
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint64_t tstart = globaltimer_ns();
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= (unsigned)nblk) break;
      if (globaltimer_ns() - tstart > timeout_ns) {
        set_status(status, MOE_ERR_TIMEOUT);
        timed_out = 1;
        break;
      }
      __nanosleep(64);
    }
    *flag = timed_out;
  }
  __syncthreads();
  return *flag == 0;
}

// One warp scans column `col` (nblk <= 256 contiguous entries) in place into
// exclusive prefixes and returns the column total (all lanes).  Rows of 32
// entries, one coalesced load per row: each row's warp scan on top of the
// rows before it.
__device__ int warp_column_scan(int32_t* col, int nblk) {
  const int lane = threadIdx.x & 31;
  const int rows = (nblk + 31) / 32;     // <= 8
  int v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int bb = i * 32 + lane;
    v[i] = (i < rows && bb < nblk) ? __ldcg(col + bb) : 0;
  }
  int base = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < rows) {
      int incl = v[i];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const int bb = i * 32 + lane;
      if (bb < nblk) col[bb] = base + incl - v[i];
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  return base;
}

// Exclusive scan over n <= 2*blockDim values held in shared memory (in place),
// returning the total.  `scratch` holds >= 32 ints.
__device__ int block_exclusive_scan(int* data, int n, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = blockDim.x >> 5;
  int a = (2 * tid < n) ? data[2 * tid] : 0;
  int b = (2 * tid + 1 < n) ? data[2 * tid + 1] : 0;
  int v = a + b;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? scratch[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    if (lane < nw) scratch[lane] = si - s;   // exclusive warp offsets
    if (lane == 31) scratch[32] = si;        // total
  }
  __syncthreads();
  int excl = scratch[warp] + incl - v;
  if (2 * tid < n) data[2 * tid] = excl;
  if (2 * tid + 1 < n) data[2 * tid + 1] = excl + a;
  int total = scratch[32];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kLayoutThreads) route_layout_kernel(LayoutArgs a) {
  extern __shared__ int smem_i[];
  const int E = a.L.E, k = a.L.k, T = a.L.T, BM = a.L.block_m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x, nblk = gridDim.x;

  int* hist = smem_i;             // [E]   block histogram, later the running row cursor
  int* fhist = hist + E;          // [E]   block first-expert histogram, later the token cursor
  int* eoff = fhist + E;          // [E+1] expert offsets
  int* toff = eoff + E + 1;       // [E+1] expert tile offsets
  int* foff = toff + E + 1;       // [E+1] first-expert offsets
  int* scratch = foff + E + 1;    // [64]
  int* s_ids = scratch + 64;      // [kChunkPairs]
  float* s_w = reinterpret_cast<float*>(s_ids + kChunkPairs);  // [kChunkPairs]

  const int t0 = min(T, b * a.tpb), t1 = min(T, t0 + a.tpb);
  const int chunk_tokens = max(1, kChunkPairs / k);
  const bool one_chunk = (t1 - t0) <= chunk_tokens;

  for (int e = tid; e < E; e += blockDim.x) { hist[e] = 0; fhist[e] = 0; }
  __syncthreads();

  // ---------------- phase A: block histograms
  for (int c0 = t0; c0 < t1; c0 += chunk_tokens) {
    const int c1 = min(t1, c0 + chunk_tokens);
    const int q0 = c0 * k, q1 = c1 * k;
    for (int p = q0 + tid; p < q1; p += blockDim.x) {
      s_ids[p - q0] = a.ids[p];
      s_w[p - q0] = a.w[p];
    }
    __syncthreads();
    for (int base = q0; base < q1; base += blockDim.x) {
      const int p = base + tid;
      int e = -1;
      if (p < q1) {
        e = s_ids[p - q0];
        if (e < 0 || e >= E) {
          if (!(a.quiet && e < 0)) set_status(a.status, MOE_ERR_EXPERT_ID);
          e = -1;
        }
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
    }
    for (int base = c0; base < c1; base += blockDim.x) {
      const int t = base + tid;
      int fe = -1;
      if (t < c1) {
        fe = first_expert(s_ids + (t - c0) * k, k, E);
        if (fe >= E) fe = -1;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, fe);
      if (fe >= 0 && lane == __ffs(peers) - 1) atomicAdd(&fhist[fe], __popc(peers));
    }
    __syncthreads();
  }
  if (nblk == 1) {
    // one block (small batches, a plain launch): its histograms are the totals
    // and its prefixes are zero; no workspace, no grid barrier
    for (int e = tid; e < E; e += blockDim.x) {
      const int tot = hist[e], ftot = fhist[e];
      hist[e] = 0;
      fhist[e] = 0;
      eoff[e] = tot;
      toff[e] = (tot + BM - 1) / BM;
      foff[e] = ftot;
    }
  } else {
    for (int e = tid; e < E; e += blockDim.x) {
      a.ws_hist[(size_t)e * kLayoutMaxBlocks + b] = hist[e];
      a.ws_fhist[(size_t)e * kLayoutMaxBlocks + b] = fhist[e];
    }

    // ---------------- phase B1: scan every expert column down the blocks (one warp per column)
    if (!grid_barrier(a.ws_barrier, nblk, a.status, a.timeout_ns, &scratch[63])) return;
    {
      const int nwarps = blockDim.x >> 5;
      for (int item = b * nwarps + warp; item < 2 * E; item += nblk * nwarps) {
        int32_t* col = (item < E ? a.ws_hist : a.ws_fhist) + (size_t)(item % E) * kLayoutMaxBlocks;
        const int total = warp_column_scan(col, nblk);
        if (lane == 0) a.ws_tot[item] = total;
      }
    }
    if (!grid_barrier(a.ws_barrier + 1, nblk, a.status, a.timeout_ns, &scratch[63])) return;

    // ---------------- phase B2: this block's prefixes, expert scans
    for (int e = tid; e < E; e += blockDim.x) {
      const int tot = __ldcg(a.ws_tot + e), ftot = __ldcg(a.ws_tot + E + e);
      hist[e] = __ldcg(a.ws_hist + (size_t)e * kLayoutMaxBlocks + b);     // this block's first row within expert e (relative)
      fhist[e] = __ldcg(a.ws_fhist + (size_t)e * kLayoutMaxBlocks + b);   // this block's first position within first-expert e
      eoff[e] = tot;
      toff[e] = (tot + BM - 1) / BM;
      foff[e] = ftot;
    }
  }
  __syncthreads();
  const int total_rows = block_exclusive_scan(eoff, E, scratch);
  const int total_tiles = block_exclusive_scan(toff, E, scratch);
  const int total_first = block_exclusive_scan(foff, E, scratch);
  if (tid == 0) { eoff[E] = total_rows; toff[E] = total_tiles; foff[E] = total_first; }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    hist[e] += eoff[e];
    fhist[e] += foff[e];
  }
  if (b == 0) {
    for (int e = tid; e <= E; e += blockDim.x) {
      if (e < E) {
        a.L.count[e] = eoff[e + 1] - eoff[e];
        a.L.ready_tokens[e] = foff[e + 1];
      }
      a.L.expert_offset[e] = eoff[e];
      a.L.expert_tile_offset[e] = toff[e];
    }
    const int epg = E / a.L.G;
    for (int g = tid; g <= a.L.G; g += blockDim.x) a.L.group_offset[g] = eoff[g * epg];
    if (tid == 0) a.L.num_tiles[0] = total_tiles;
  }
  // tile tables and rowmap: one warp per tile, grid-stride over all blocks'
  // warps; one search for the tile's expert, then the tile's BM rowmap slots
  // in coalesced runs of 32 (per-slot searches cost ~1 us more per call)
  {
    const int nwarps = blockDim.x >> 5;
    const int gw = b * nwarps + warp, gwstride = nblk * nwarps;
    const int cap = a.L.max_tiles;
    for (int m = gw; m < cap; m += gwstride) {
      int e = -1, begin = T * k, rows = 0;
      if (m < total_tiles) {
        int lo = 0, hi = E;                 // largest e with toff[e] <= m
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (toff[mid] <= m) lo = mid; else hi = mid;
        }
        e = lo;
        begin = eoff[e] + (m - toff[e]) * BM;
        rows = min(BM, eoff[e + 1] - begin);
      }
      if (lane == 0) {
        a.L.tile_expert[m] = e;
        a.L.tile_row_begin[m] = begin;
        a.L.tile_rows[m] = rows;
      }
      int32_t* slot = a.L.rowmap + (size_t)m * BM;
      for (int j = lane; j < BM; j += 32) slot[j] = j < rows ? begin + j : -1;
    }
  }
  __syncthreads();

  // ---------------- phase C: stable ranks within the block, all warps
  // Each chunk's pairs (then its tokens) are cut into one contiguous slice per
  // warp.  A per-warp histogram of the slice, scanned across the warps on top
  // of the block's running cursors, gives every warp its first row per
  // expert; each warp then ranks its slice 32 at a time (lanes with equal
  // keys find each other with __match_any_sync and take consecutive rows in
  // lane order), which keeps the (token, slot) order stable.
  int* whist = reinterpret_cast<int*>(s_w + kChunkPairs);   // [kLayoutWarps][E]
  int* wh = whist + warp * E;
  for (int c0 = t0; c0 < t1; c0 += chunk_tokens) {
    const int c1 = min(t1, c0 + chunk_tokens);
    const int q0 = c0 * k, q1 = c1 * k;
    if (!one_chunk) {
      __syncthreads();
      for (int p = q0 + tid; p < q1; p += blockDim.x) {
        s_ids[p - q0] = a.ids[p];
        s_w[p - q0] = a.w[p];
      }
      __syncthreads();
    }
    for (int pass = 0; pass < 2; ++pass) {
      // pass 0: pairs [q0, q1) keyed by expert; pass 1: tokens [c0, c1) keyed by first expert
      const int n = pass == 0 ? q1 - q0 : c1 - c0;
      int* cursor = pass == 0 ? hist : fhist;
      const int per = (((n + kLayoutWarps - 1) / kLayoutWarps) + 31) & ~31;
      const int s0 = min(n, warp * per), s1 = min(n, s0 + per);
      auto key_of = [&](int i) -> int {   // i < n; -1 for an invalid expert id
        if (pass == 0) {
          const int e = s_ids[i];
          return (e < 0 || e >= E) ? -1 : e;
        }
        const int fe = first_expert(s_ids + i * k, k, E);
        return fe >= E ? -1 : fe;
      };
      for (int i = tid; i < kLayoutWarps * E; i += blockDim.x) whist[i] = 0;
      __syncthreads();
      for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const int e = i < s1 ? key_of(i) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      for (int e = tid; e < E; e += blockDim.x) {
        int run = cursor[e];
        for (int w2 = 0; w2 < kLayoutWarps; ++w2) {
          const int c = whist[w2 * E + e];
          whist[w2 * E + e] = run;
          run += c;
        }
        cursor[e] = run;
      }
      __syncthreads();
      for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const int e = i < s1 ? key_of(i) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int pos = e >= 0 ? wh[e] + __popc(peers & lanemask_lt()) : -1;
        if (pass == 0) {
          if (i < s1) {
            const int p = q0 + i;
            a.L.pair_row[p] = pos;
            if (e >= 0) {
              a.L.row_pair[pos] = p;
              a.L.row_weight[pos] = s_w[i];
            }
          }
        } else if (e >= 0) {
          a.L.token_order[pos] = c0 + i;
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();   // whist is cleared for the next pass
    }
  }
}

// ---------------------------------------------------------------- router helper

// One warp per token: k rounds of a warp-wide arg-max (largest logit, ties to
// the lower expert id), then softmax weights over the selected logits.
template <int VPL>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                          int E, int k, int32_t* __restrict__ ids,
                                                          float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = i * 32 + lane;
      v[i] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
    }
    bool used[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) used[i] = (i * 32 + lane) >= E;
    float sel_l0 = 0.f, my_l = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      float best = -INFINITY;
      int bid = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = i * 32 + lane;
        if (!used[i] && (v[i] > best || (v[i] == best && e < bid))) { best = v[i]; bid = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
        if (ob > best || (ob == best && oi < bid)) { best = ob; bid = oi; }
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (i * 32 + lane == bid) used[i] = true;
      if (j == 0) sel_l0 = best;
      if (lane == j) { my_l = best; my_id = bid; }
    }
    const float ex = lane < k ? expf(my_l - sel_l0) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);   // slots in order
    if (lane < k) {
      ids[(size_t)t * k + lane] = my_id;
      w[(size_t)t * k + lane] = ex / sum;
    }
  }
}

}  // namespace moe

using namespace moe;

static size_t layout_smem_bytes(int E) {
  return sizeof(int) * (size_t)(2 * E + 3 * (E + 1) + 64 + kChunkPairs) + sizeof(float) * kChunkPairs +
         sizeof(int) * (size_t)kLayoutWarps * E;
}

size_t moe_layout_ws_bytes(int E) {
  return 256 + 2 * sizeof(int32_t) * (size_t)kLayoutMaxBlocks * E + 2 * sizeof(int32_t) * (size_t)E;
}

// Grid, workspace pointers and launch shared by both entry points.  `ws` is
// the caller's workspace or the library's fixed scratch.
int launch_layout(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L, void* ws,
                  int32_t* status, cudaStream_t s, int quiet) {
  int dev, nsm;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;

  const size_t smem = layout_smem_bytes(L->E);
  static_assert(kLayoutThreads * 2 >= 1024, "scan covers E <= 1024");
  if (cudaFuncSetAttribute(route_layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_layout_kernel, kLayoutThreads, smem) != cudaSuccess || per_sm < 1)
    return MOE_ERR_CUDA;
  // One block per SM at most, ~32 tokens per block.  The tile tables and the
  // rowmap (max_tiles x 128 slots, most of them -1 on small batches) are
  // written one tile per warp over the whole grid, and one SM writes them
  // slowly, so a grid of more than one block has at least one warp per tile
  // (blocks past the last token have empty ranges).  A single block (T <= 32)
  // runs as a plain launch with no workspace memset and no grid barrier.
  int nblk = (L->T + 31) / 32;
  if (nblk > 1) nblk = std::max(nblk, (L->max_tiles + kLayoutWarps - 1) / kLayoutWarps);
  nblk = std::min(nblk, std::min(nsm * per_sm, std::min(nsm, kLayoutMaxBlocks)));
  nblk = std::max(nblk, 1);
  const int tpb = (L->T + nblk - 1) / nblk;

  LayoutArgs a;
  a.ids = topk_ids;
  a.w = topk_w;
  a.L = to_dev(L);
  a.ws_barrier = reinterpret_cast<uint32_t*>(ws);
  a.ws_hist = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + 256);
  a.ws_fhist = a.ws_hist + (size_t)kLayoutMaxBlocks * L->E;
  a.ws_tot = a.ws_fhist + (size_t)kLayoutMaxBlocks * L->E;
  a.status = status;
  a.tpb = tpb;
  a.timeout_ns = 1000000000ull;
  a.quiet = quiet;

  if (nblk == 1) {
    route_layout_kernel<<<1, kLayoutThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  // the grid barriers' counters start at zero (the workspace, or the fixed
  // scratch, keeps whatever the previous call left; the histograms and totals
  // are fully written before they are read)
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kLayoutThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, route_layout_kernel, a) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" int moe_route_layout(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L,
                                void* ws, size_t ws_bytes, int32_t* status, moe_stream_t stream) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!topk_ids || !topk_w || !ws) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_layout_ws_bytes(L->E)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)ws & 15) != 0) return MOE_ERR_INVALID_ARG;
  return launch_layout(topk_ids, topk_w, L, ws, status, (cudaStream_t)stream, 0);
}

extern "C" int moe_router_topk(const float* logits, int T, int E, int k, int32_t* topk_ids,
                               float* topk_w, moe_stream_t stream) {
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int warps = 8;
  const int grid = std::min((T + warps - 1) / warps, 4096);
  if (E <= 256)
    router_topk_kernel<8><<<grid, warps * 32, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  else
    router_topk_kernel<32><<<grid, warps * 32, 0, s>>>(logits, T, E, k, topk_ids, topk_w);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- allocation-free variant
//
// moe_route_layout_noalloc: the same layout kernel, with its scratch in a
// fixed device array of this library instead of a caller workspace, for
// callers that cannot allocate device memory: a plugin inside a framework
// whose memory pool owns the whole device, a latency-critical path that must
// not pay the device-wide synchronisation a cudaMalloc can cause, or a
// deployment that sizes all memory once at load time.  The array (514 KiB +
// 256 B, for up to 256 experts) is reserved on every GPU that loads the
// library and stays there until the process exits.  The first call on a
// device looks its address up (make that call outside any stream capture);
// every call shares the array, so calls that can overlap on the GPU race.

namespace moe {
constexpr int kNoAllocMaxExperts = MOE_NOALLOC_MAX_EXPERTS;
// header (grid-barrier counters) + two per-block histograms of up to kLayoutMaxBlocks x 256
// experts + their column totals
constexpr size_t kNoAllocScratchBytes = 256 + 2 * sizeof(int32_t) * (size_t)kLayoutMaxBlocks * kNoAllocMaxExperts +
                                        2 * sizeof(int32_t) * (size_t)kNoAllocMaxExperts;
}  // namespace moe

static __device__ __align__(256) unsigned char g_layout_scratch[moe::kNoAllocScratchBytes];

#include <mutex>

// Device address of g_layout_scratch on each device (the symbol's name is only
// a host-side handle; kernels need this address).  Looked up again on every
// call made outside a stream capture, so a context torn down and created again
// (cudaDeviceReset) gets the new address; a call inside a capture uses the
// address of the last uncaptured call on that device, and the very first call
// on a device must not be inside a capture.
static void* g_scratch_addr[128];
static std::mutex g_scratch_mu;

static int layout_scratch_address(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return MOE_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
    if (cap != cudaStreamCaptureStatusNone) return MOE_ERR_CUDA;   // first call inside a capture
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

extern "C" int moe_route_layout_noalloc(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L,
                                        int32_t* status, moe_stream_t stream) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (L->E > kNoAllocMaxExperts) return MOE_ERR_UNSUPPORTED;   // beyond the fixed scratch
  void* ws = nullptr;
  rc = layout_scratch_address((cudaStream_t)stream, &ws);
  if (rc) return rc;
  return launch_layout(topk_ids, topk_w, L, ws, status, (cudaStream_t)stream, 0);
}

// ---------------------------------------------------------------- no-plan layout (small batches)
//
// The mori stage1 page's --no-plan ("How it works now"): no counting sort --
// one reservation atomic per worker and run, no histogram pass, no prefix sum
// over the batch, no grid rendezvous -- worth it while a batch is small
// ("What each mechanism is worth": -12 us at 256 tokens, -5 at 512, +23 at
// 1024).  Here: ONE block of 1024 threads.  Each warp reserves, per expert
// its 32 pairs route to, one run of consecutive slots with a single
// shared-memory atomic (lanes with equal experts find each other with
// __match_any_sync and take consecutive slots of the run), and the same for
// each token's first expert; one block scan over the E counts then gives the
// expert offsets and the tile tables, and every pair lands at its expert's
// offset plus its slot.  The tables are the counting sort's except for the
// order of the rows within an expert (and of the tokens within a
// first-expert group), which follows the atomics: as a multiset per expert
// they are the same.  No workspace, nothing to zero between calls.

namespace moe {
constexpr int kNoPlanThreads = 1024;
constexpr int kNoPlanPer = MOE_NOPLAN_MAX_PAIRS / kNoPlanThreads;   // pairs (and tokens) per thread

// Warp-aggregated reservation: every lane whose key is >= 0 gets a distinct
// slot of counter[key]; lanes with equal keys take consecutive slots, one
// atomic per key per warp.  Whole warp, converged.
__device__ __forceinline__ int reserve_slot(int* counter, int key) {
  const int lane = threadIdx.x & 31;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int leader = __ffs(peers) - 1;
  int base = 0;
  if (key >= 0 && lane == leader) base = atomicAdd(&counter[key], __popc(peers));
  base = __shfl_sync(0xffffffffu, base, leader);
  return key >= 0 ? base + __popc(peers & lanemask_lt()) : -1;
}

__global__ void __launch_bounds__(kNoPlanThreads, 1)
    route_layout_noplan_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, LayoutDev L,
                               int32_t* status) {
  extern __shared__ int smem_np[];
  const int E = L.E, k = L.k, T = L.T, BM = L.block_m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = T * k;
  int* cnt = smem_np;          // [E]   pairs per expert (the reservation counters)
  int* fcnt = cnt + E;         // [E]   tokens per first expert
  int* eoff = fcnt + E;        // [E+1] expert offsets
  int* toff = eoff + E + 1;    // [E+1] expert tile offsets
  int* foff = toff + E + 1;    // [E+1] first-expert offsets
  int* scratch = foff + E + 1; // [64]
  int* s_ids = scratch + 64;   // [P]   the batch's expert ids, staged once
  float* s_w = reinterpret_cast<float*>(s_ids + P);   // [P]
  for (int e = tid; e < E; e += blockDim.x) { cnt[e] = 0; fcnt[e] = 0; }
  // one coalesced pass over the inputs: every later read comes from shared memory
  for (int p = tid; p < P; p += blockDim.x) {
    s_ids[p] = __ldcs(ids + p);
    s_w[p] = __ldcs(w + p);
  }
  __syncthreads();

  const int rounds = (max(P, T) + kNoPlanThreads - 1) / kNoPlanThreads;   // block-uniform
  // (key << 16) | slot per pair and per token (-1: none); keys < 1024, slots < 2^15
  int pk[kNoPlanPer], tk[kNoPlanPer];
#pragma unroll
  for (int i = 0; i < kNoPlanPer; ++i) {
    pk[i] = -1;
    tk[i] = -1;
    if (i < rounds) {
      const int p = tid + i * kNoPlanThreads;
      int e = -1;
      if (p < P) {
        e = s_ids[p];
        if (e < 0 || e >= E) { set_status(status, MOE_ERR_EXPERT_ID); e = -1; }
      }
      const int ps = reserve_slot(cnt, e);
      if (e >= 0) pk[i] = (e << 16) | ps;
      const int t = tid + i * kNoPlanThreads;
      int fe = -1;
      if (t < T) {
        fe = first_expert(s_ids + (size_t)t * k, k, E);
        if (fe >= E) fe = -1;
      }
      const int ts = reserve_slot(fcnt, fe);
      if (fe >= 0) tk[i] = (fe << 16) | ts;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    eoff[e] = cnt[e];
    toff[e] = (cnt[e] + BM - 1) / BM;
    foff[e] = fcnt[e];
  }
  __syncthreads();
  const int total_rows = block_exclusive_scan(eoff, E, scratch);
  const int total_tiles = block_exclusive_scan(toff, E, scratch);
  const int total_first = block_exclusive_scan(foff, E, scratch);
  if (tid == 0) { eoff[E] = total_rows; toff[E] = total_tiles; foff[E] = total_first; }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {
    if (e < E) {
      L.count[e] = cnt[e];
      L.ready_tokens[e] = foff[e + 1];
    }
    L.expert_offset[e] = eoff[e];
    L.expert_tile_offset[e] = toff[e];
  }
  const int epg = E / L.G;
  for (int g = tid; g <= L.G; g += blockDim.x) L.group_offset[g] = eoff[g * epg];
  if (tid == 0) L.num_tiles[0] = total_tiles;
  // every pair to its expert's offset plus its slot; every token after its first expert's offset
#pragma unroll
  for (int i = 0; i < kNoPlanPer; ++i) {
    if (i < rounds) {
      const int p = tid + i * kNoPlanThreads;
      if (p < P) {
        if (pk[i] >= 0) {
          const int row = eoff[pk[i] >> 16] + (pk[i] & 0xFFFF);
          L.pair_row[p] = row;
          L.row_pair[row] = p;
          L.row_weight[row] = s_w[p];
        } else {
          L.pair_row[p] = -1;
        }
      }
      const int t = tid + i * kNoPlanThreads;
      if (tk[i] >= 0) L.token_order[foff[tk[i] >> 16] + (tk[i] & 0xFFFF)] = t;
    }
  }
  // tile tables and rowmap, one warp per tile (as the counting-sort layout)
  for (int m = warp; m < L.max_tiles; m += kNoPlanThreads / 32) {
    int e = -1, begin = T * k, rows = 0;
    if (m < total_tiles) {
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (toff[mid] <= m) lo = mid; else hi = mid;
      }
      e = lo;
      begin = eoff[e] + (m - toff[e]) * BM;
      rows = min(BM, eoff[e + 1] - begin);
    }
    if (lane == 0) {
      L.tile_expert[m] = e;
      L.tile_row_begin[m] = begin;
      L.tile_rows[m] = rows;
    }
    int32_t* slot = L.rowmap + (size_t)m * BM;
    for (int j = lane; j < BM; j += 32) slot[j] = j < rows ? begin + j : -1;
  }
}
}  // namespace moe

extern "C" int moe_route_layout_noplan(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L,
                                       int32_t* status, moe_stream_t stream) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((long long)L->T * L->k > MOE_NOPLAN_MAX_PAIRS) return MOE_ERR_UNSUPPORTED;
  const size_t smem = sizeof(int) * (size_t)(2 * L->E + 3 * (L->E + 1) + 64 + 2 * (size_t)L->T * L->k);
  if (cudaFuncSetAttribute(route_layout_noplan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  route_layout_noplan_kernel<<<1, kNoPlanThreads, smem, (cudaStream_t)stream>>>(topk_ids, topk_w, to_dev(L), status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
