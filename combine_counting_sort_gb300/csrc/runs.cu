// runs.cu: per-(token, logical group) send runs -- one FP8 row per token and
// group it routes into -- and their dispatch.
//
// The mori stage1 page ("What": the sender quantises each token once into a
// send buffer grouped by destination; "How it works now": a counting sort by
// (destination, first expert) places every token's row so that a landed prefix
// of a run is a prefix of experts; the quant writes each row once to every run
// it is in).  On one GPU the destinations are the logical groups: run g holds
// one row for every token with a route into group g, ordered by (the token's
// smallest expert in g, token).  GEMM1 then gathers its A rows from the runs
// (moe_grouped_gemm1_gather) instead of reading a dense T*k-row buffer, so the
// dispatch writes one row per (token, group) instead of one per (token, slot).
//
// The runs are computed with the routing layout's own counting sort: item
// (t, g) gets the key "smallest expert of t in g" (-1 when t has no route into
// g, skipped quietly), and the stable sort of the T*G items by that key is
// exactly the run order (the key's expert id also orders the groups).  So
// send_row[t*G + g] is the sort's pair_row, run_offset its group offsets, and
// run_ready[e] the end of key e's rows.
#include "common.cuh"
#include "host_util.h"

int launch_layout(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L, void* ws,
                  int32_t* status, cudaStream_t s, int quiet);
int launch_dispatch(const uint16_t* x, int H, int T, const int32_t* rows, int per_token, long long R, uint8_t* A,
                    float* A_scale, cudaStream_t stream);

namespace moe {

// keys[t*G + g] = smallest expert of token t within group g, or -1.  Ids
// outside [0, E) are ignored here (moe_route_layout reports them).
__global__ void __launch_bounds__(256) send_keys_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int G,
                                                        int32_t* __restrict__ keys) {
  const int epg = E / G;
  const long long n = (long long)T * G;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / G), g = (int)(i % G);
    int best = E;
    for (int j = 0; j < k; ++j) {
      const int e = ids[(size_t)t * k + j];
      if (e >= g * epg && e < (g + 1) * epg && e < best) best = e;
    }
    keys[i] = best < E ? best : -1;
  }
}

struct SendDev {
  int32_t* run_offset;
  int32_t* send_token;
  int32_t* send_row;
  int32_t* run_ready;
  int32_t* gather_row;
};

// From the sorted items: the token of every send row, run_ready, and the send
// row every dense row of the routing layout reads.
__global__ void __launch_bounds__(256) send_finalize_kernel(const int32_t* __restrict__ ids, LayoutDev L, SendDev S,
                                                            const int32_t* __restrict__ item_of_row,
                                                            const int32_t* __restrict__ key_offset, long long smax) {
  const int G = L.G, E = L.E, k = L.k, epg = E / G;
  const long long R = (long long)L.T * k;
  const int sends = key_offset[E];
  const int dense = L.expert_offset[E];
  const long long n = max(max(R, smax), (long long)E);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    if (i < smax) S.send_token[i] = i < sends ? item_of_row[i] / G : -1;
    if (i < E) S.run_ready[i] = key_offset[i + 1];
    if (i < R) {
      int gr = -1;
      if (i < dense) {
        const int p = L.row_pair[i];
        gr = S.send_row[(size_t)(p / k) * G + ids[p] / epg];
      }
      S.gather_row[i] = gr;
    }
  }
}

// Workspace carve-up of moe_send_layout (every piece 256-byte aligned).
struct SendWs {
  size_t layout_ws, keys, item_of_row, weights, count, key_offset, tile_offset, ready, rowmap, tile_expert,
      tile_begin, tile_rows, num_tiles, token_order, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline SendWs send_ws(int T, int E, int G) {
  const size_t items = (size_t)T * G;
  const size_t tiles = (size_t)max_tiles_of(T, G, E, MOE_BLOCK_M);
  SendWs w;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
  w.layout_ws = take(moe_layout_ws_bytes(E));
  w.keys = take(4 * items);
  w.item_of_row = take(4 * items);
  w.weights = take(4 * items);
  w.count = take(4 * (size_t)E);
  w.key_offset = take(4 * ((size_t)E + 1));
  w.tile_offset = take(4 * ((size_t)E + 1));
  w.ready = take(4 * (size_t)E);
  w.rowmap = take(4 * tiles * MOE_BLOCK_M);
  w.tile_expert = take(4 * tiles);
  w.tile_begin = take(4 * tiles);
  w.tile_rows = take(4 * tiles);
  w.num_tiles = take(4);
  w.token_order = take(4 * (size_t)T);
  w.total = o;
  return w;
}

}  // namespace moe

using namespace moe;

size_t moe_send_ws_bytes(int T, int k, int E, int G) {
  (void)k;
  return send_ws(T, E, G).total;
}

long long moe_max_send_rows(int T, int k, int G) { return (long long)T * std::min(G, k); }

static int check_runs(const moe_layout_t* L, const moe_send_runs_t* S) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (!S || !S->run_offset || !S->send_token || !S->send_row || !S->run_ready || !S->gather_row)
    return MOE_ERR_INVALID_ARG;
  if (L->G > 32) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

extern "C" int moe_send_layout(const int32_t* topk_ids, const moe_layout_t* L, const moe_send_runs_t* S, void* ws,
                               size_t ws_bytes, int32_t* status, moe_stream_t stream) {
  int rc = check_runs(L, S);
  if (rc) return rc;
  if (!topk_ids || !ws || ((uintptr_t)ws & 255) != 0) return MOE_ERR_INVALID_ARG;
  const int T = L->T, E = L->E, G = L->G;
  if ((long long)T * G >= ((long long)1 << 31)) return MOE_ERR_INVALID_ARG;
  const SendWs w = send_ws(T, E, G);
  if (ws_bytes < w.total) return MOE_ERR_INVALID_ARG;
  char* base = reinterpret_cast<char*>(ws);
  auto at = [&](size_t off) { return reinterpret_cast<int32_t*>(base + off); };
  cudaStream_t s = (cudaStream_t)stream;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const long long items = (long long)T * G;
  send_keys_kernel<<<(int)std::max(1LL, std::min((items + 255) / 256, (long long)nsm * 8)), 256, 0, s>>>(
      topk_ids, T, L->k, E, G, at(w.keys));
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // the counting sort of the (token, group) items by key
  moe_layout_t Li;
  Li.T = T; Li.k = G; Li.E = E; Li.G = G; Li.block_m = MOE_BLOCK_M;
  Li.max_tiles = (int32_t)max_tiles_of(T, G, E, MOE_BLOCK_M);
  Li.count = at(w.count);
  Li.expert_offset = at(w.key_offset);
  Li.expert_tile_offset = at(w.tile_offset);
  Li.group_offset = S->run_offset;
  Li.ready_tokens = at(w.ready);
  Li.pair_row = S->send_row;
  Li.row_pair = at(w.item_of_row);
  Li.row_weight = reinterpret_cast<float*>(at(w.weights));
  Li.rowmap = at(w.rowmap);
  Li.tile_expert = at(w.tile_expert);
  Li.tile_row_begin = at(w.tile_begin);
  Li.tile_rows = at(w.tile_rows);
  Li.num_tiles = at(w.num_tiles);
  Li.token_order = at(w.token_order);
  // the sort copies a weight per item; the keys serve as that (ignored) input
  rc = launch_layout(at(w.keys), reinterpret_cast<const float*>(at(w.keys)), &Li, base + w.layout_ws, status, s,
                     /*quiet=*/1);
  if (rc) return rc;
  SendDev d;
  d.run_offset = S->run_offset;
  d.send_token = S->send_token;
  d.send_row = S->send_row;
  d.run_ready = S->run_ready;
  d.gather_row = S->gather_row;
  const long long smax = moe_max_send_rows(T, L->k, G);
  const long long n = std::max(std::max((long long)T * L->k, smax), (long long)E);
  send_finalize_kernel<<<(int)std::max(1LL, std::min((n + 255) / 256, (long long)nsm * 8)), 256, 0, s>>>(
      topk_ids, to_dev(L), d, at(w.item_of_row), at(w.key_offset), smax);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_dispatch_quant_runs(const uint16_t* x, int H, const moe_layout_t* L, const moe_send_runs_t* S,
                                       uint8_t* A_send, float* A_send_scale, int32_t* status, moe_stream_t stream) {
  (void)status;
  int rc = check_runs(L, S);
  if (rc) return rc;
  if (!x || !A_send || !A_send_scale) return MOE_ERR_INVALID_ARG;
  if (H < MOE_QBLOCK || H % MOE_QBLOCK != 0 || H > 32768) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(A_send) || !aligned16(A_send_scale)) return MOE_ERR_INVALID_ARG;
  return launch_dispatch(x, H, L->T, S->send_row, L->G, moe_max_send_rows(L->T, L->k, L->G), A_send, A_send_scale,
                         (cudaStream_t)stream);
}
