/*
 * moe.h: C ABI of the single-GPU MoE stage1 + combine library (libmoe.so, sm_103a).
 *
 * The path: a stable counting-sort routing layout of each token's top-k
 * (expert, weight) pairs; a dispatch that quantises each token once to FP8
 * e4m3 with fp32 per-128 block scales and scatters it into its expert-major
 * rows; GEMM1 as a grouped FP8 GEMM that reads those rows in place; a fused
 * stage1 that overlaps the dispatch (producer SMs) with GEMM1 (consumer SMs)
 * through per-tile ready flags; and a combine that gathers each token's k
 * expert outputs back into token order, weighted by the router weights.
 *
 * Sources, by page title and section:
 *  [mori]     "poc(cco): MegaMoE stage1 dispatch over SDMA" (mori PR #1).
 *  [mojo]     "EPDispatchKernel" (Mojo ep_comm API page).
 *  [tilepipe] "TilePipe: MoE Communication and Overlap Kernels with CuteDSL".
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers are device memory owned by the caller;
 *    the library never allocates, frees or keeps them, and keeps no global
 *    mutable state (the one exception is the fixed scratch array behind
 *    moe_route_layout_noalloc).  Host pointers (struct arguments) are read
 *    during the call only.
 *  - bf16 tensors are passed as uint16_t bit patterns; fp8 tensors as uint8_t
 *    e4m3 codes ("fn" variant: no infinities, max 448).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *    stream) and never synchronises the host.  Calls capture into CUDA graphs.
 *  - The return code reports argument and launch errors found on the host.
 *    Errors found on the device are written to `*status` (a device int32 that
 *    the caller zeroes; the first error wins) and are read after a sync.
 *  - One call at a time per workspace: two calls that share a workspace or
 *    output buffers must be ordered on one stream.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t;   /* same handle as cudaStream_t */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, workspace too small */
  MOE_ERR_UNSUPPORTED = 2,   /* device is not sm_100-class / shape beyond a kernel limit /
                                the GEMM kernel's compiled register count cannot hold its
                                warp-role register split (nothing is launched) */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  MOE_ERR_EXPERT_ID = 4,     /* device: an expert id outside [0, E); the pair was skipped */
  MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up (stage1 flag never set) */
} moe_status;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* Sort block: rows per GEMM1 M-tile and padding unit of every expert
 * ([mori] recv_layout commit: each expert padded to the sort block of 128). */
#define MOE_BLOCK_M 128
/* Quantisation block along the hidden dimension (fp32 scale per 128 values). */
#define MOE_QBLOCK 128

/* ---------------------------------------------------------------------------
 * Sizes.  One function sizes every table and workspace; the kernels index them
 * with the same numbers.
 *   T tokens, k routes per token, E experts in G logical groups (group g holds
 *   experts [g*E/G, (g+1)*E/G): [mojo] n_local_experts = n_experts / n_ranks).
 * Limits: 1 <= T <= 2^20, 1 <= k <= 32, k <= E <= 1024, E % G == 0,
 * T*k < 2^31, block_m == 128.
 * ------------------------------------------------------------------------- */
typedef struct moe_layout_sizes {
  int64_t pairs;             /* T*k: rows of the dense dispatch buffer */
  int64_t max_tiles;         /* min(T*k, (T*k + E*(block_m-1)) / block_m) */
  int64_t rowmap_len;        /* max_tiles * block_m */
  size_t layout_ws_bytes;    /* workspace for moe_route_layout */
  size_t stage1_ws_bytes;    /* workspace for moe_stage1 */
  size_t gemm_combine_ws_bytes; /* workspace for moe_grouped_gemm1_combine */
  int64_t max_send_rows;     /* T * min(G, k): capacity of the per-(token, group) send runs */
  size_t send_ws_bytes;      /* workspace for moe_send_layout */
} moe_layout_sizes_t;

int moe_layout_sizes(int T, int k, int E, int G, int block_m, moe_layout_sizes_t* out);

/* ---------------------------------------------------------------------------
 * Layout tables ([mori] recv_layout commit: counts per expert, padding to the
 * sort block, rowmap / srcmap / weights / tile tables; [mojo] ep_final_layout:
 * each routed row written to its final contiguous per-expert row).
 * The caller fills the shape fields and the device pointers (sizes from
 * moe_layout_sizes); moe_route_layout writes the tables, the other calls read
 * them.  Pair p = t*k + j is token t's j-th route.
 * ------------------------------------------------------------------------- */
typedef struct moe_layout {
  int32_t T, k, E, G, block_m, max_tiles;          /* host values */
  int32_t* count;              /* [E]   pairs routed to expert e */
  int32_t* expert_offset;      /* [E+1] exclusive prefix of count: first dense row of e */
  int32_t* expert_tile_offset; /* [E+1] exclusive prefix of ceil(count/block_m) */
  int32_t* group_offset;       /* [G+1] expert_offset[g*E/G]: a group's run of rows */
  int32_t* ready_tokens;       /* [E]   inclusive prefix of first-expert counts */
  int32_t* pair_row;           /* [T*k] dense row of pair p (-1 if its id was invalid) */
  int32_t* row_pair;           /* [T*k] pair held by dense row r */
  float* row_weight;           /* [T*k] router weight of the pair held by row r */
  int32_t* rowmap;             /* [max_tiles*block_m] dense row of tile slot, or -1 */
  int32_t* tile_expert;        /* [max_tiles] expert of tile m, -1 past num_tiles */
  int32_t* tile_row_begin;     /* [max_tiles] first dense row of tile m, T*k past num_tiles */
  int32_t* tile_rows;          /* [max_tiles] valid rows of tile m (1..block_m), 0 past num_tiles */
  int32_t* num_tiles;          /* [1]   tiles in use */
  int32_t* token_order;        /* [T]   tokens stably sorted by first (smallest) expert */
} moe_layout_t;

/* moe_route_layout: histogram, prefix sums and stable ranks of the T*k pairs
 * sorted by (group, expert), rows within an expert in ascending pair order
 * ([mori] "How it works now": counting sort so that a landed prefix of a run
 * is a prefix of experts).  Also the token order by first expert that the
 * stage1 producer walks, so that every token of expert e sits before
 * ready_tokens[e].
 *   topk_ids  device int32 [T, k] row-major; ids outside [0,E) are skipped and
 *             raise MOE_ERR_EXPERT_ID in *status (the tables then cover only
 *             the valid pairs).
 *   topk_w    device f32 [T, k] router weights (copied to row_weight).
 *   ws        device workspace of at least layout_ws_bytes (contents ignored;
 *             the call initialises what it uses, in-stream).
 * One launch: a cooperative grid of at most 64 blocks (one per SM) with one
 * grid-wide barrier (bounded: a barrier not reached within 1 s writes
 * MOE_ERR_TIMEOUT to *status and the kernel returns), or, for T <= 32, a
 * single block in a plain launch without it. */
int moe_route_layout(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L,
                     void* ws, size_t ws_bytes, int32_t* status, moe_stream_t stream);

/* moe_route_layout_noalloc: moe_route_layout for callers that cannot
 * allocate device memory: a plugin inside a framework whose memory pool owns
 * the whole device (a raw cudaMalloc would fail or fragment the pool), a
 * latency-critical path that must not pay the device-wide synchronisation a
 * cudaMalloc can cause, or a deployment that sizes all memory once at load
 * time.  The scratch lives in a fixed array inside this library, so the
 * caller passes only inputs and outputs.  The source pages have no
 * counterpart of this entry point.
 *   Limit: E <= MOE_NOALLOC_MAX_EXPERTS (larger E returns MOE_ERR_UNSUPPORTED);
 *   other limits and outputs as moe_route_layout.
 *   The array (about 128 KiB) is reserved on every GPU that loads the library
 *   until the process exits.  Every call made outside a stream capture looks
 *   up the array's device address (so a context reset is followed); a call
 *   inside a capture reuses the address of the last uncaptured call on that
 *   device, so make the first call on each device (and the first one after a
 *   cudaDeviceReset) outside any stream capture: a first call inside a
 *   capture returns MOE_ERR_CUDA.
 *   All calls share the one array: calls that can overlap on the GPU (other
 *   streams, other threads) race and must be ordered by the caller. */
#define MOE_NOALLOC_MAX_EXPERTS 256
int moe_route_layout_noalloc(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L,
                             int32_t* status, moe_stream_t stream);

/* moe_route_layout_noplan: the layout without the counting sort, for small
 * batches ([mori] "How it works now", --no-plan: one reservation atomic per
 * worker and run, no histogram, no prefix sum over the batch, no grid
 * rendezvous; "What each mechanism is worth": a gain at 256 and 512 tokens, a
 * loss at 1024).  One block: each warp reserves one run of consecutive slots
 * per expert its pairs route to with a single shared-memory atomic, then one
 * scan over the E counts places the runs.  Every table equals
 * moe_route_layout's EXCEPT the order of the rows within an expert
 * (pair_row, row_pair, row_weight) and of the tokens within a first-expert
 * group (token_order): those follow the atomics and change from call to call;
 * as a multiset per expert (per first expert) they are the same.  Counts,
 * offsets, tile tables, rowmap, group offsets and ready_tokens are identical.
 *   Limit: T * k <= MOE_NOPLAN_MAX_PAIRS (larger returns MOE_ERR_UNSUPPORTED).
 *   No workspace: everything lives in the block's shared memory.  Invalid
 *   ids as moe_route_layout. */
#define MOE_NOPLAN_MAX_PAIRS 16384
int moe_route_layout_noplan(const int32_t* topk_ids, const float* topk_w, const moe_layout_t* L,
                            int32_t* status, moe_stream_t stream);

/* moe_dispatch_quant: quantise each token once and store it to each of its k
 * rows ([mori] "How it works now" and the quant-once commit: read and quantise
 * a token once, store it to every run it is in).  Per token t and block b of
 * 128 values: amax = max|x|, scale = amax/448 (fp32), code = e4m3(x/scale)
 * (fp32 IEEE division, round to nearest even, saturating); amax == 0 gives
 * scale 0 and zero codes.
 *   x        device bf16 [T, H] row-major, H % 128 == 0, H <= 32768.
 *   A        device u8 [T*k, H] row-major: row pair_row[t*k+j] = codes of token t.
 *   A_scale  device f32 [H/128, T*k]: A_scale[b*T*k + r] = scale of row r, block b.
 * Rows of invalid pairs are not written. */
int moe_dispatch_quant(const uint16_t* x, int H, const moe_layout_t* L, uint8_t* A,
                       float* A_scale, int32_t* status, moe_stream_t stream);

/* moe_grouped_gemm1: Y[r, n] = bf16( sum_k (A[r,k]*sa[r,k/128]) * (W[e,n,k]*sb[e,n/128,k/128]) )
 * for every dense row r of expert e ([mori] "What": GEMM1 reads its A rows in
 * place through the rowmap).  One persistent tcgen05 kernel: M-tiles of 128
 * rows from the tile tables in expert-major order, FP8 operands by TMA,
 * fp32 accumulation with the block scales applied per 128 of K.
 *   A, A_scale  as written by moe_dispatch_quant (A must be 16-byte aligned).
 *   W           device u8 [E, N, H] e4m3 codes, row n of expert e is K-contiguous.
 *   W_scale     device f32 [E, N/128, H/128].
 *   Y           device bf16 [T*k, N] row-major; only valid rows are written.
 * N % 256 == 0, H % 128 == 0, N, H <= 32768. */
int moe_grouped_gemm1(const uint8_t* A, const float* A_scale, const uint8_t* W,
                      const float* W_scale, int N, int H, const moe_layout_t* L, uint16_t* Y,
                      int32_t* status, moe_stream_t stream);

/* moe_grouped_gemm1_pair: moe_grouped_gemm1 on CTA pairs.  Same arguments,
 * same Y (the same fp32 partials folded in the same order).  A 2-CTA cluster
 * runs tcgen05 MMAs of M = 256 (two consecutive M-tiles of one expert; the
 * second empty when the expert has an odd tile count) against 256 columns,
 * each SM holding its 128 rows of A and 128 of the 256 W rows.
 * MOE_ERR_UNSUPPORTED on a device with fewer than two SMs. */
int moe_grouped_gemm1_pair(const uint8_t* A, const float* A_scale, const uint8_t* W,
                           const float* W_scale, int N, int H, const moe_layout_t* L, uint16_t* Y,
                           int32_t* status, moe_stream_t stream);

/* moe_combine: out[t, :] = bf16( sum_{j<k} w[t,j] * Y[pair_row[t*k+j], :] ),
 * accumulated in fp32 with the slots in ascending order; w is read as
 * row_weight[pair_row[t*k+j]] ([tilepipe] "Communication Kernels": the
 * combine that returns expert outputs to token order).
 *   Y    device bf16 [T*k, D] (D % 8 == 0), out device bf16 [T, D].
 * A pair whose pair_row is -1 contributes nothing. */
int moe_combine(const uint16_t* Y, int D, const moe_layout_t* L, uint16_t* out, int32_t* status,
                moe_stream_t stream);

/* moe_grouped_gemm1_combine: moe_grouped_gemm1 and moe_combine (D = N) in one
 * cooperative launch, the combine of a token overlapping the rest of the GEMM
 * ([tilepipe] "Overlap": producer and consumer on one GPU synchronised by
 * per-tile semaphores; its "GEMM -> combine" driver).  After the epilogue
 * stores a unit's rows, a counting warp bumps a completion counter per token
 * (release); the bump that completes a token (N/256 per valid pair) puts it on
 * a ready queue; combining warps (one per CTA during the GEMM, all of a CTA's
 * warps once its GEMM work is done) pop tokens and write out[t] with the
 * arithmetic of moe_combine.  Y and out are bit-for-bit what
 * moe_grouped_gemm1 followed by moe_combine write.
 *   Arguments as moe_grouped_gemm1, plus out device bf16 [T, N] and ws, a
 *   device workspace of at least gemm_combine_ws_bytes (16-byte aligned;
 *   zeroed in-stream by the call).  A token not complete within the bounded
 *   wait (2 s) writes MOE_ERR_TIMEOUT to *status. */
/* Trace slots (uint64, ns from %globaltimer) in the gemm1_combine workspace
 * header, written by every call: kernel start, the first and the last CTA to
 * finish its GEMM work, kernel end, the last push onto the ready queue, and
 * the combining warps' total waiting and working time. */
#define MOE_GC_TRACE_OFFSET 64
#define MOE_GC_TRACE_START 0
#define MOE_GC_TRACE_GEMM_FIRST_DONE 1
#define MOE_GC_TRACE_GEMM_LAST_DONE 2
#define MOE_GC_TRACE_END 3
#define MOE_GC_TRACE_LAST_PUSH 4     /* the last token put on the ready queue */
#define MOE_GC_TRACE_WAIT_NS 5       /* total ns combining warps waited for queued tokens */
#define MOE_GC_TRACE_WORK_NS 6       /* total ns combining warps spent combining */
int moe_grouped_gemm1_combine(const uint8_t* A, const float* A_scale, const uint8_t* W,
                              const float* W_scale, int N, int H, const moe_layout_t* L, uint16_t* Y,
                              uint16_t* out, void* ws, size_t ws_bytes, int32_t* status,
                              moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Per-(token, group) send runs: one FP8 row per token and logical group it
 * routes into ([mori] "What": the sender quantises each token once into a send
 * buffer grouped by destination; "How it works now": a counting sort by
 * (destination, first expert) places every token's row so that a landed prefix
 * of a run is a prefix of experts).  Run g holds one row for every token with
 * a route into group g, ordered by (the token's smallest expert in g, token);
 * GEMM1 gathers its A rows from the runs, so the dispatch writes one row per
 * (token, group) instead of one per (token, slot).  G <= 32.
 * ------------------------------------------------------------------------- */
typedef struct moe_send_runs {
  int32_t* run_offset;   /* [G+1] first send row of run g */
  int32_t* send_token;   /* [max_send_rows] token held by send row s, -1 past the last */
  int32_t* send_row;     /* [T*G] send row of (token t, group g), -1 if t has no route into g */
  int32_t* run_ready;    /* [E] for expert e of group g: end of the prefix of run g that holds
                            every token routed to e */
  int32_t* gather_row;   /* [T*k] send row that dense row r of the layout reads, -1 past the
                            valid rows */
} moe_send_runs_t;

/* moe_send_layout: the send runs of a routing layout (computed by
 * moe_route_layout from the same topk_ids).  ws: device workspace of at least
 * send_ws_bytes, 256-byte aligned (contents ignored).  Ids outside [0, E) are
 * left out (moe_route_layout reports them). */
int moe_send_layout(const int32_t* topk_ids, const moe_layout_t* L, const moe_send_runs_t* S, void* ws,
                    size_t ws_bytes, int32_t* status, moe_stream_t stream);

/* moe_dispatch_quant_runs: quantise each token once (the rule of
 * moe_dispatch_quant) and store it to its send rows.
 *   A_send        device u8 [max_send_rows, H]: row send_row[t*G + g] = codes of t.
 *   A_send_scale  device f32 [H/128, max_send_rows] (block-major, as A_scale). */
int moe_dispatch_quant_runs(const uint16_t* x, int H, const moe_layout_t* L, const moe_send_runs_t* S,
                            uint8_t* A_send, float* A_send_scale, int32_t* status, moe_stream_t stream);

/* moe_grouped_gemm1_gather: moe_grouped_gemm1 with A gathered: dense row r of
 * the layout reads row gather_row[r] of A_send (half of each tile's rows by
 * TMA tile::gather4, half by 16-byte cp.async copies, into the swizzled
 * shared-memory stage) and its scales from A_send_scale at that row.  Y is
 * the dense [T*k, N] output, as moe_grouped_gemm1's.  send_rows: rows of
 * A_send (max_send_rows). */
int moe_grouped_gemm1_gather(const uint8_t* A_send, const float* A_send_scale, const uint8_t* W,
                             const float* W_scale, int N, int H, const moe_layout_t* L,
                             const int32_t* gather_row, long long send_rows, uint16_t* Y, int32_t* status,
                             moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * MXFP8 variant: e8m0 (power-of-two) scales per 32 values, applied by the
 * tensor core's block-scaled MMA instead of in software ([mori] first commit:
 * "GEMM1 reads its A rows and e8m0 scales through a rowmap"; quant-LDS commit:
 * the e8m0 scales packed four per 32-bit word).  The pages give neither the
 * block size nor the rule; this library takes 32 values per block (for the
 * activations along H, for each weight row along K) and
 *   X = the smallest integer with 448 * 2^X >= amax (amax / 448 rounded up to
 *       a power of two), clamped to [-127, 127]; amax == 0 gives X = -127;
 *   e8m0 code = X + 127; value code = e4m3(x * 2^-X) (round to nearest even,
 *   saturating).
 * Scale-factor layouts (MMA-ready; byte (i % 32) * 16 + (i / 32) * 4 + j of a
 * 512-byte atom holds row i's code of 32-value chunk j of a 128-value K block):
 *   A_sf  u8 [max_tiles][H/128][512]: atom of (M-tile m, K block kb); row i is
 *         slot i of tile m (dense row tile_row_begin[m] + i).  Slots past the
 *         tile's rows are never written (their content is ignored).
 *   W_sf  u8 [E][H/128][N/128][512]: atom of (expert e, K block kb, weight
 *         rows [128 nb, 128 nb + 128)).
 * Buffers must be 16-byte aligned.  E <= 1024, H % 128 == 0, H <= 32768.
 * ------------------------------------------------------------------------- */

/* moe_dispatch_quant_mx: quantise each token once (MX rule above) and store
 * it to each of its k rows: A as moe_dispatch_quant, scales into A_sf at the
 * row's tile slot.  Rows of invalid pairs are not written. */
int moe_dispatch_quant_mx(const uint16_t* x, int H, const moe_layout_t* L, uint8_t* A, uint8_t* A_sf,
                          int32_t* status, moe_stream_t stream);

/* moe_quant_weights_mx: expert weights bf16 [E, N, H] -> e4m3 codes [E, N, H]
 * and W_sf (layout above), one scale per weight row and 32 values of K.
 * N % 128 == 0, H % 128 == 0. */
int moe_quant_weights_mx(const uint16_t* W, int E, int N, int H, uint8_t* Wq, uint8_t* W_sf,
                         moe_stream_t stream);

/* moe_grouped_gemm1_mx: Y[r, n] = bf16( sum_k (A[r,k] 2^XA[r,k/32]) (W[e,n,k] 2^XW[e,n,k/32]) )
 * for every dense row r of expert e: one persistent tcgen05 kernel with
 * kind::mxf8f6f4 block-scaled MMAs (M128 N256 K32), scales copied from A_sf /
 * W_sf into tensor memory per K block, fp32 accumulation in tensor memory over
 * the whole K, bf16 (round to nearest even) for the valid rows only.
 * N % 256 == 0, H % 128 == 0, N, H <= 32768. */
int moe_grouped_gemm1_mx(const uint8_t* A, const uint8_t* A_sf, const uint8_t* W, const uint8_t* W_sf, int N,
                         int H, const moe_layout_t* L, uint16_t* Y, int32_t* status, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Fused stage1 ([tilepipe] "Overlap": SMs partitioned between a producer that
 * bumps a semaphore per finished tile and a consumer GEMM waiting on it,
 * producer order chosen to unblock the expert-major GEMM order as early as
 * possible, sync granularity per tile or per expert; [mori] "How it works
 * now": GEMM1 gated per tile on ready signals, or --ready-first, a scheduler
 * publishing m-tiles in readiness order with workers taking tickets).
 * Computes exactly what moe_dispatch_quant followed by moe_grouped_gemm1 does
 * (same A, A_scale and Y bits), in one cooperative launch of one CTA per SM.
 * ------------------------------------------------------------------------- */
typedef enum moe_flag_granularity { MOE_FLAGS_PER_TILE = 0, MOE_FLAGS_PER_EXPERT = 1 } moe_flag_granularity;
typedef enum moe_schedule { MOE_SCHED_EXPERT_MAJOR = 0, MOE_SCHED_READY_FIRST = 1 } moe_schedule;

typedef struct moe_stage1_opts {
  int32_t comm_sms;          /* producer CTAs (1..#SMs-1); 0 = default (16) */
  int32_t flags;             /* moe_flag_granularity */
  int32_t schedule;          /* moe_schedule */
  int32_t producers_join;    /* 1: producer CTAs take GEMM work once their tokens are done */
  int64_t timeout_ns;        /* bound of every wait on a flag; 0 = default (1 s) */
  int32_t withhold_tile;     /* test hook: >= 0 never publishes this M-tile's rows (the
                                consumer must time out); -1 = off */
  int32_t trace;             /* 1: record timestamps / wait counters in the workspace
                                header (int64 slots MOE_TRACE_*, ns from %globaltimer) */
} moe_stage1_opts_t;

/* Trace slots (int64) of the stage1 workspace header when opts.trace = 1. */
#define MOE_TRACE_OFFSET 64          /* byte offset of slot 0 in the workspace */
#define MOE_TRACE_START 0            /* kernel start (first CTA to stamp) */
#define MOE_TRACE_PRODUCED 1         /* last producer CTA done with its tokens */
#define MOE_TRACE_WAIT_NS 2          /* total ns consumers spent waiting for ready flags */
#define MOE_TRACE_WAITED_UNITS 3     /* units whose first load had to wait */
#define MOE_TRACE_END 4              /* last CTA done */
#define MOE_TRACE_JOINED_UNITS 5     /* units taken by producer CTAs after joining */
#define MOE_TRACE_UNITS 6            /* units processed in total */

/*   x, H, L        as moe_dispatch_quant; W, W_scale, N as moe_grouped_gemm1.
 *   A, A_scale, Y  outputs as the unfused calls.
 *   ws             device workspace of at least stage1_ws_bytes (initialised
 *                  in-stream by the call). */
int moe_stage1(const uint16_t* x, int H, const moe_layout_t* L, const uint8_t* W,
               const float* W_scale, int N, const moe_stage1_opts_t* opts, uint8_t* A,
               float* A_scale, uint16_t* Y, void* ws, size_t ws_bytes, int32_t* status,
               moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Helpers (input preparation and the identity expert of the bandwidth sweep).
 * ------------------------------------------------------------------------- */

/* moe_router_topk: per token, the k largest of E logits (ties to the lower
 * expert id; slots in descending order) and weights softmax-renormalised over
 * the k selected: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) in fp32.
 *   logits device f32 [T, E] (E <= 1024); topk_ids device int32 [T, k];
 *   topk_w device f32 [T, k]. */
int moe_router_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                    moe_stream_t stream);

/* moe_quant_weights: expert weights bf16 [E, N, H] -> e4m3 codes [E, N, H]
 * and fp32 scales [E, N/128, H/128], one scale per 128x128 block with the
 * activations' amax/448 rule.  N % 128 == 0, H % 128 == 0. */
int moe_quant_weights(const uint16_t* W, int E, int N, int H, uint8_t* Wq, float* W_scale,
                      moe_stream_t stream);

/* moe_dequant_rows: the identity expert, Y[r, :] = bf16(code * scale) for every
 * valid dense row r (Y device bf16 [T*k, H]). */
int moe_dequant_rows(const uint8_t* A, const float* A_scale, int H, const moe_layout_t* L,
                     uint16_t* Y, moe_stream_t stream);

/* Number of SMs of the current device (0 on error): the persistent grids'
 * size. */
int moe_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
