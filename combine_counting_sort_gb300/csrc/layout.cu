// layout.cu: routing layout (stable counting sort of the T*k (token, slot)
// pairs by (group, expert)) and the top-k router helper.
//
// The counting sort of the mori stage1 page ("How it works now": a counting
// sort by (destination, first expert) so that a landed prefix of a run is a
// prefix of experts; recv_layout commit: per-expert counts, padding of every
// expert to the sort block, expert-major tables) as ONE launch: a cooperative
// grid of at most 64 blocks, about 1024 pairs each (T <= 32: a single block
// in a plain launch, which needs no barrier):
//
//   phase A  each block counts its contiguous token range by both keys (the
//            expert of each pair, the first (smallest) expert of each token):
//            every warp histograms its own slice with warp-aggregated
//            shared-memory adds (__match_any_sync leaders), and the slice
//            histograms, scanned across the warps, become each warp's first
//            position within the block; the block totals go to its row of a
//            table in the workspace.  The block's ids and weights stay
//            staged in shared memory.
//   barrier  one grid-wide barrier (bounded spin: MOE_ERR_TIMEOUT after 1 s).
//   phase B  every block reads the whole table (rows of 2E contiguous counts)
//            and sums each column over the blocks before it (its first row
//            per expert within the expert) and over all blocks (the totals);
//            one scan across experts gives expert offsets, tile offsets and
//            first-expert offsets; block 0 writes the E-sized tables; the
//            tile tables and the rowmap are written one tile per warp over
//            the whole grid.
//   phase C  stable ranks: each warp walks its slice 32 keys at a time
//            (lanes with equal keys find each other with __match_any_sync
//            and take consecutive rows in lane order), the token order by
//            first expert the same way.  A block whose range exceeds one
//            staged chunk stages, histograms and ranks chunk by chunk.
//
// Logical group g holds experts [g*E/G, (g+1)*E/G) (the Mojo EPDispatchKernel
// page's n_local_experts = n_experts / n_ranks), so the key (group, expert)
// orders like the expert id.
#include "common.cuh"
#include "host_util.h"

namespace moe {

constexpr int kLayoutThreads = 512;
constexpr int kLayoutGridCap = 64;        // blocks of one grid at most (each reads every block's row)
constexpr int kLayoutPairsPerBlock = 1024;
constexpr int kChunkPairs = 4096;         // pairs staged in shared memory per pass
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kStageRounds = kChunkPairs / kLayoutThreads;   // staged pairs per thread
// phase B's partial column sums: 2 x (row groups x row stride) <= 2 x 4 x kLayoutThreads ints
constexpr int kPartInts = 8 * kLayoutThreads;
static_assert(kPartInts % 4 == 0, "the arrays after it stay 16-byte aligned at their start");
static_assert(kChunkPairs % kLayoutThreads == 0, "whole staging rounds");

// Row stride (ints) of the workspace table of per-block counts: 2E rounded up
// to whole 16-byte vectors.
__host__ __device__ __forceinline__ int layout_row_stride(int E) { return (2 * E + 3) & ~3; }

struct LayoutArgs {
  const int32_t* ids;
  const float* w;
  LayoutDev L;
  int32_t* ws_tab;      // [nblk][2E]: block b's expert counts, then its first-expert counts
  uint32_t* ws_barrier; // [1] zeroed in-stream before the launch
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

// Exclusive scans, in place, of three arrays of n <= 2*blockDim values held in
// shared memory, in one pass; tot[i] receives array i's total.  `scratch`
// holds >= 3 * 32 + 3 ints.
__device__ void block_exclusive_scan3(int* d0, int* d1, int* d2, int n, int* scratch, int* tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = blockDim.x >> 5;
  int* d[3] = {d0, d1, d2};
  int a[3], v[3], incl[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    a[i] = (2 * tid < n) ? d[i][2 * tid] : 0;
    v[i] = a[i] + ((2 * tid + 1 < n) ? d[i][2 * tid + 1] : 0);
    incl[i] = v[i];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int u = __shfl_up_sync(0xffffffffu, incl[i], o);
      if (lane >= o) incl[i] += u;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int i = 0; i < 3; ++i) scratch[i * 32 + warp] = incl[i];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int w = lane < nw ? scratch[i * 32 + lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += u;
      }
      if (lane < nw) scratch[i * 32 + lane] = wi - w;   // exclusive warp offsets
      if (lane == 31) scratch[96 + i] = wi;            // total
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int excl = scratch[i * 32 + warp] + incl[i] - v[i];
    if (2 * tid < n) d[i][2 * tid] = excl;
    if (2 * tid + 1 < n) d[i][2 * tid + 1] = excl + a[i];
    tot[i] = scratch[96 + i];
  }
  __syncthreads();
}

// Slice of the block's keys ranked by warp `warp`: a contiguous run of whole
// 32-key rounds, one run per warp, in key order.
__device__ __forceinline__ void warp_slice(int n, int warp, int& s0, int& s1) {
  const int per = (((n + kLayoutWarps - 1) / kLayoutWarps) + 31) & ~31;
  s0 = min(n, warp * per);
  s1 = min(n, s0 + per);
}

__global__ void __launch_bounds__(kLayoutThreads) route_layout_kernel(LayoutArgs a) {
  extern __shared__ __align__(16) int smem_i[];
  const int E = a.L.E, k = a.L.k, T = a.L.T, BM = a.L.block_m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x, nblk = gridDim.x;

  int* part = smem_i;             // [kPartInts] phase B column sums (first: 16-byte aligned, int4 stores)
  int* hist = part + kPartInts;   // [E]   block histogram, later the block's first row per expert
  int* fhist = hist + E;          // [E]   block first-expert histogram, later the block's first position
  int* eoff = fhist + E;          // [E+1] expert offsets
  int* toff = eoff + E + 1;       // [E+1] expert tile offsets
  int* foff = toff + E + 1;       // [E+1] first-expert offsets
  int* scratch = foff + E + 1;    // [128]
  int* s_ids = scratch + 128;     // [kChunkPairs]
  float* s_w = reinterpret_cast<float*>(s_ids + kChunkPairs);   // [kChunkPairs]
  int* whist = reinterpret_cast<int*>(s_w + kChunkPairs);       // [2][kLayoutWarps][E]

  const int t0 = min(T, b * a.tpb), t1 = min(T, t0 + a.tpb);
  const int chunk_tokens = max(1, kChunkPairs / k);
  const bool one_chunk = (t1 - t0) <= chunk_tokens;

  // key of item i of a staged chunk: pass 0 the expert of pair i, pass 1 the
  // first (smallest) expert of token i; -1 for an invalid id
  auto key_of = [&](int pass, int i) -> int {
    if (pass == 0) {
      const int e = s_ids[i];
      return (e < 0 || e >= E) ? -1 : e;
    }
    const int fe = first_expert(s_ids + i * k, k, E);
    return fe >= E ? -1 : fe;
  };
  // stage pairs [q0, q1) (at most kChunkPairs): every load issued before the
  // first store, so the chunk costs one memory round trip
  auto stage = [&](int q0, int q1) {
    int vi[kStageRounds];
    float vw[kStageRounds];
#pragma unroll
    for (int j = 0; j < kStageRounds; ++j) {
      const int p = q0 + tid + j * kLayoutThreads;
      if (p < q1) {
        vi[j] = __ldg(a.ids + p);
        vw[j] = __ldg(a.w + p);
      }
    }
#pragma unroll
    for (int j = 0; j < kStageRounds; ++j) {
      const int p = q0 + tid + j * kLayoutThreads;
      if (p < q1) {
        s_ids[p - q0] = vi[j];
        s_w[p - q0] = vw[j];
      }
    }
  };

  // one chunk: its loads are in flight while the histograms are cleared
  int vi[kStageRounds];
  float vw[kStageRounds];
  if (one_chunk) {
#pragma unroll
    for (int j = 0; j < kStageRounds; ++j) {
      const int p = t0 * k + tid + j * kLayoutThreads;
      if (p < t1 * k) {
        vi[j] = __ldg(a.ids + p);
        vw[j] = __ldg(a.w + p);
      }
    }
  }
  for (int e = tid; e < E; e += blockDim.x) { hist[e] = 0; fhist[e] = 0; }
  if (one_chunk)
    for (int i = tid; i < 2 * kLayoutWarps * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();

  // ---------------- phase A: block histograms
  if (one_chunk) {
    // One chunk (every grid this library launches up to T*k = 64 * 4096
    // pairs): per-warp slice histograms of both keys, kept for phase C, then
    // scanned across the warps in place (each entry becomes the warp's first
    // position within the block) with the block totals left in hist / fhist.
    const int q0 = t0 * k, q1 = t1 * k;
#pragma unroll
    for (int j = 0; j < kStageRounds; ++j) {
      const int p = q0 + tid + j * kLayoutThreads;
      if (p < q1) {
        s_ids[p - q0] = vi[j];
        s_w[p - q0] = vw[j];
      }
    }
    __syncthreads();
    for (int i = q0 + tid; i < q1; i += blockDim.x) {
      const int e = s_ids[i - q0];
      if (e >= E || (e < 0 && !a.quiet)) set_status(a.status, MOE_ERR_EXPERT_ID);
    }
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      int s0, s1;
      warp_slice(pass == 0 ? q1 - q0 : t1 - t0, warp, s0, s1);
      int* wh = whist + (pass * kLayoutWarps + warp) * E;
      for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const int e = i < s1 ? key_of(pass, i) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
    for (int c = tid; c < 2 * E; c += blockDim.x) {
      int* col = whist + (c < E ? 0 : kLayoutWarps * E) + (c % E);
      int v[kLayoutWarps];
#pragma unroll
      for (int w2 = 0; w2 < kLayoutWarps; ++w2) v[w2] = col[w2 * E];
      int run = 0;
#pragma unroll
      for (int w2 = 0; w2 < kLayoutWarps; ++w2) {
        col[w2 * E] = run;
        run += v[w2];
      }
      (c < E ? hist : fhist)[c % E] = run;
    }
  } else {
    for (int c0 = t0; c0 < t1; c0 += chunk_tokens) {
      const int c1 = min(t1, c0 + chunk_tokens);
      const int q0 = c0 * k, q1 = c1 * k;
      stage(q0, q1);
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
        const int fe = t < c1 ? key_of(1, t - c0) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, fe);
        if (fe >= 0 && lane == __ffs(peers) - 1) atomicAdd(&fhist[fe], __popc(peers));
      }
      __syncthreads();
    }
  }
  __syncthreads();

  // ---------------- phase B: every block's prefixes and the totals
  if (nblk == 1) {
    // one block (small batches, a plain launch): its histograms are the totals
    // and its prefixes are zero; no workspace, no grid barrier
    for (int e = tid; e < E; e += blockDim.x) {
      eoff[e] = hist[e];
      toff[e] = (hist[e] + BM - 1) / BM;
      foff[e] = fhist[e];
      hist[e] = 0;
      fhist[e] = 0;
    }
  } else {
    // this block's row of the table [nblk][RS] (expert counts, then
    // first-expert counts, padded to 16-byte vectors)
    const int RS = layout_row_stride(E);
    int32_t* row = a.ws_tab + (size_t)b * RS;
    for (int c = tid; c < RS; c += blockDim.x) row[c] = c < 2 * E ? (c < E ? hist : fhist)[c % E] : 0;
    if (!grid_barrier(a.ws_barrier, nblk, a.status, a.timeout_ns, &scratch[127])) return;
    // every block reads the whole table: each thread one 16-byte vector of
    // columns in a group of rows, 16 rows in flight at a time; the column sums
    // over the blocks before this one and over all blocks meet in shared
    // memory (part: [2][ngroups][RS], prefixes then totals)
    const int nvec = RS / 4;
    const int ngroups = max(1, kLayoutThreads / nvec);
    for (int i = tid; i < 2 * ngroups * RS; i += blockDim.x) part[i] = 0;
    __syncthreads();
    for (int vt = tid; vt < nvec * ngroups; vt += blockDim.x) {
      const int vc = vt % nvec, g = vt / nvec;
      int4 pre = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
      for (int r0 = g; r0 < nblk; r0 += 16 * ngroups) {
        int4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = r0 + i * ngroups;
          v[i] = r < nblk ? __ldcg(reinterpret_cast<const int4*>(a.ws_tab + (size_t)r * RS) + vc)
                          : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = r0 + i * ngroups;
          tot.x += v[i].x; tot.y += v[i].y; tot.z += v[i].z; tot.w += v[i].w;
          if (r < b) { pre.x += v[i].x; pre.y += v[i].y; pre.z += v[i].z; pre.w += v[i].w; }
        }
      }
      reinterpret_cast<int4*>(part + g * RS)[vc] = pre;
      reinterpret_cast<int4*>(part + (ngroups + g) * RS)[vc] = tot;
    }
    __syncthreads();
    for (int c = tid; c < 2 * E; c += blockDim.x) {
      int pre = 0, tot = 0;
      for (int g = 0; g < ngroups; ++g) {
        pre += part[g * RS + c];
        tot += part[(ngroups + g) * RS + c];
      }
      if (c < E) { hist[c] = pre; eoff[c] = tot; toff[c] = (tot + BM - 1) / BM; }
      else { fhist[c - E] = pre; foff[c - E] = tot; }
    }
  }
  __syncthreads();
  int tot3[3];
  block_exclusive_scan3(eoff, toff, foff, E, scratch, tot3);
  const int total_tiles = tot3[1];
  if (tid == 0) { eoff[E] = tot3[0]; toff[E] = tot3[1]; foff[E] = tot3[2]; }
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
  // in coalesced runs of 32
  {
    const int gw = b * kLayoutWarps + warp, gwstride = nblk * kLayoutWarps;
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
  // Each warp walks its slice 32 keys at a time: lanes with equal keys find
  // each other with __match_any_sync and take consecutive positions in lane
  // order after the warp's running first position for that key, which keeps
  // the (token, slot) order stable.  One chunk: the slice histograms of phase
  // A, scanned, are the warps' first positions within the block.  More
  // chunks: each chunk is staged again, histogrammed per warp and scanned on
  // top of the block's running cursors.
  auto rank = [&](int pass, int q0, int c0, int n, int* cursor_base, int* wh) {
    int s0, s1;
    warp_slice(n, warp, s0, s1);
    for (int base = s0; base < s1; base += 32) {
      const int i = base + lane;
      const int e = i < s1 ? key_of(pass, i) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int pos = e >= 0 ? cursor_base[e] + wh[e] + __popc(peers & lanemask_lt()) : -1;
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
  };
  if (one_chunk) {
    rank(0, t0 * k, t0, (t1 - t0) * k, hist, whist + warp * E);
    rank(1, t0 * k, t0, t1 - t0, fhist, whist + (kLayoutWarps + warp) * E);
    return;
  }
  for (int c0 = t0; c0 < t1; c0 += chunk_tokens) {
    const int c1 = min(t1, c0 + chunk_tokens);
    const int q0 = c0 * k, q1 = c1 * k;
    __syncthreads();
    stage(q0, q1);
    __syncthreads();
    for (int pass = 0; pass < 2; ++pass) {
      const int n = pass == 0 ? q1 - q0 : c1 - c0;
      int* cursor = pass == 0 ? hist : fhist;
      int* wh = whist + warp * E;
      for (int i = tid; i < kLayoutWarps * E; i += blockDim.x) whist[i] = 0;
      __syncthreads();
      int s0, s1;
      warp_slice(n, warp, s0, s1);
      for (int base = s0; base < s1; base += 32) {
        const int i = base + lane;
        const int e = i < s1 ? key_of(pass, i) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w2 = 0; w2 < kLayoutWarps; ++w2) {
          const int c = whist[w2 * E + e];
          whist[w2 * E + e] = run;
          run += c;
        }
        whist[kLayoutWarps * E + e] = run;   // this chunk's count of key e
      }
      __syncthreads();
      rank(pass, q0, c0, n, cursor, wh);
      __syncthreads();
      for (int e = tid; e < E; e += blockDim.x) cursor[e] += whist[kLayoutWarps * E + e];
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
  return sizeof(int) * (size_t)(2 * E + 3 * (E + 1) + 128 + kChunkPairs) + sizeof(float) * kChunkPairs +
         sizeof(int) * (size_t)2 * kLayoutWarps * E + sizeof(int) * (size_t)kPartInts;
}

size_t moe_layout_ws_bytes(int E) {
  return 256 + sizeof(int32_t) * (size_t)kLayoutGridCap * layout_row_stride(E);
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
  // About kLayoutPairsPerBlock pairs per block, at most kLayoutGridCap
  // blocks (every block reads every block's row of counts after the barrier,
  // so the grid stays small) and one per SM.  The tile tables and the rowmap
  // (max_tiles x 128 slots, most of them -1 on small batches) are written one
  // tile per warp over the whole grid, so a grid of more than one block has
  // at least one warp per two tiles (blocks past the last token have empty
  // ranges).  A single block (T <= 32) runs as a plain launch with no
  // workspace memset and no grid barrier.
  const long long pairs = (long long)L->T * L->k;
  int nblk = L->T <= 32 ? 1 : (int)std::min<long long>((pairs + kLayoutPairsPerBlock - 1) / kLayoutPairsPerBlock,
                                                        kLayoutGridCap);
  if (L->T > 32) nblk = std::max(nblk, std::min(kLayoutGridCap, (L->max_tiles + 2 * kLayoutWarps - 1) / (2 * kLayoutWarps)));
  nblk = std::min(nblk, std::min(nsm * per_sm, std::min(nsm, kLayoutGridCap)));
  nblk = std::max(nblk, 1);
  const int tpb = (L->T + nblk - 1) / nblk;

  LayoutArgs a;
  a.ids = topk_ids;
  a.w = topk_w;
  a.L = to_dev(L);
  a.ws_barrier = reinterpret_cast<uint32_t*>(ws);
  a.ws_tab = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + 256);
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
// deployment that sizes all memory once at load time.  The array (128 KiB +
// 256 B, for up to 256 experts) is reserved on every GPU that loads the
// library and stays there until the process exits.  The first call on a
// device looks its address up (make that call outside any stream capture);
// every call shares the array, so calls that can overlap on the GPU race.

namespace moe {
constexpr int kNoAllocMaxExperts = MOE_NOALLOC_MAX_EXPERTS;
// header (grid-barrier counter) + one row of 2 x 256 counts per block of the grid
constexpr size_t kNoAllocScratchBytes = 256 + sizeof(int32_t) * (size_t)kLayoutGridCap * 2 * kNoAllocMaxExperts;
static_assert(2 * kNoAllocMaxExperts % 4 == 0, "whole 16-byte rows");
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
