// common.cuh: shared device helpers of the MoE stage1 + combine kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA tensor loads and the tcgen05 tensor
// core (TMEM allocation, MMA, commit, TMEM loads), plus status reporting and
// the bounded waits every spin loop goes through.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda.h>
#include <stdint.h>

#include "../../include/moe.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

constexpr int kBlockM = MOE_BLOCK_M;   // rows per M-tile / sort block
constexpr int kQBlock = MOE_QBLOCK;    // quantisation block along H

// Device view of the layout tables (the host struct by value).
struct LayoutDev {
  int32_t T, k, E, G, block_m, max_tiles;
  int32_t* count;
  int32_t* expert_offset;
  int32_t* expert_tile_offset;
  int32_t* group_offset;
  int32_t* ready_tokens;
  int32_t* pair_row;
  int32_t* row_pair;
  float* row_weight;
  int32_t* rowmap;
  int32_t* tile_expert;
  int32_t* tile_row_begin;
  int32_t* tile_rows;
  int32_t* num_tiles;
  int32_t* token_order;
};

inline LayoutDev to_dev(const moe_layout_t* L) {
  LayoutDev d;
  d.T = L->T; d.k = L->k; d.E = L->E; d.G = L->G; d.block_m = L->block_m; d.max_tiles = L->max_tiles;
  d.count = L->count; d.expert_offset = L->expert_offset; d.expert_tile_offset = L->expert_tile_offset;
  d.group_offset = L->group_offset; d.ready_tokens = L->ready_tokens; d.pair_row = L->pair_row;
  d.row_pair = L->row_pair; d.row_weight = L->row_weight; d.rowmap = L->rowmap;
  d.tile_expert = L->tile_expert; d.tile_row_begin = L->tile_row_begin; d.tile_rows = L->tile_rows;
  d.num_tiles = L->num_tiles; d.token_order = L->token_order;
  return d;
}

// ---------------------------------------------------------------- status / time

MOE_DEV void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

MOE_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

MOE_DEV uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %lanemask_lt;" : "=r"(m));
  return m;
}

MOE_DEV int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MOE_DEV void red_release_gpu_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

MOE_DEV void st_release_gpu(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Generic-proxy writes made visible to later async-proxy (TMA) reads.
MOE_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- bf16 / fp8

MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 values as one packed pair (lo in the low half), the operand form of the .f32x2 instructions.
MOE_DEV unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// A packed pair of fp32 values (low half first) -> two bf16 values.
MOE_DEV uint32_t pack_bf16x2_from_pair(unsigned long long v) {
  return pack_bf16x2(__uint_as_float((uint32_t)v), __uint_as_float((uint32_t)(v >> 32)));
}

// Two fp32 -> two e4m3 codes (round to nearest even, saturate to +-448); lo in the low byte.
MOE_DEV uint16_t e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Two e4m3 codes (low byte first) -> two floats (exact: e4m3 is a subset of fp16).
MOE_DEV float2 e4m3x2_to_float2(uint16_t codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)codes, __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// bf16 of the exact product a*b (one rounding to nearest even), from the
// fp32 product and its exact error: the fp32 rounding can land exactly on a
// bf16 midpoint, where the sign of the error decides the direction.
MOE_DEV uint16_t bf16_of_product(float a, float b) {
  float hi = a * b;
  float lo = fmaf(a, b, -hi);
  uint32_t u = __float_as_uint(hi);
  if ((u & 0xFFFFu) == 0x8000u && lo != 0.0f && (u & 0x7F800000u) != 0x7F800000u) {
    bool same_sign = (lo > 0.0f) == (hi > 0.0f);
    return same_sign ? (uint16_t)((u + 0x8000u) >> 16) : (uint16_t)(u >> 16);
  }
  __nv_bfloat16 r = __float2bfloat16_rn(hi);
  return *reinterpret_cast<uint16_t*>(&r);
}

// ---------------------------------------------------------------- shared memory / mbarrier

// One lane of a converged warp (elect.sync): tcgen05 / TMA issue from a
// warp whose other lanes run the same (warp-uniform) loop.
MOE_DEV bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

MOE_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
MOE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
MOE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's abort
// flag plus MOE_ERR_TIMEOUT in *status) once `timeout_ns` has passed, or
// false at once when another role of the CTA has aborted.
MOE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                       uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        set_status(status, MOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- cp.async (4-byte)

// Asynchronous 4-byte copy global -> shared (zero-filled when src_bytes == 0,
// in which case nothing is read).  Completion is tracked per thread by commit
// groups.
MOE_DEV void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}
MOE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MOE_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- TMA

MOE_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

MOE_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

MOE_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / bulk copy) reads of them.
MOE_DEV void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Bulk copy shared -> global (this thread's bulk async-group); the source must
// be visible to the async proxy first (fence.proxy.async.shared::cta).
MOE_DEV void bulk_copy_to_global(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes) : "memory");
}
MOE_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all but this thread's newest N bulk groups are complete (their writes performed)
template <int N>
MOE_DEV void bulk_wait() { asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- tcgen05 / TMEM

MOE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
MOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols)
               : "memory");
}
// Warpgroup register re-split (whole warpgroup, converged).
template <uint32_t N>
MOE_DEV void regs_dealloc() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(N)); }
template <uint32_t N>
MOE_DEV void regs_alloc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(N)); }

MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, FP8 e4m3 operands, fp32 accumulator.
MOE_DEV void umma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
MOE_DEV void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

// Shared-memory matrix descriptor: K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart),
// exactly the layout a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes.
// Fields: start address >> 4 (bits 0-13), leading-dimension byte offset >> 4
// (bits 16-29, unused for this layout), stride-dimension byte offset >> 4
// (bits 32-45), descriptor version 1 (bits 46-47), swizzle mode 2 = 128B (bits 61-63).
MOE_DEV uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// ---------------------------------------------------------------- CTA pairs (2-CTA clusters)
//
// A pair of CTAs on two SMs of a cluster runs one tcgen05 MMA of M = 256:
// each CTA holds 128 rows of A and half of B's N rows in its own shared
// memory, and receives its 128 rows of D in its own tensor memory.  The
// allocation, the MMAs and their commits all name cta_group::2.

MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of offset `addr` in CTA `rank` of this cluster.
MOE_DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive (relaxed, cluster scope) on an mbarrier given by its shared::cluster
// address.  Relaxed is enough where what the arrival reports is already
// complete when it is issued (tensor-memory loads waited for with wait::ld).
MOE_DEV void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}

// Every thread of both CTAs (release / acquire at cluster scope).
MOE_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Pair allocation: one warp of each CTA of the pair runs these together.
MOE_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
MOE_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols)
               : "memory");
}

// Pair MMA (issued by the even CTA only): D[tmem] (+)= A * B^T with M = 256,
// the descriptors' shared-memory offsets read in both CTAs.
MOE_DEV void umma_f8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on the mbarrier at offset `bar` of every CTA in `mask` when the
// pair MMAs issued so far by this thread complete.
MOE_DEV void umma_commit_pair_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      :: "r"(bar), "h"(mask) : "memory");
}

// TMA loads into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (`bar` a shared::cluster address).
MOE_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}
MOE_DEV void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4: fp32 D (bits 4-5 = 1), A and B e4m3
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
constexpr uint32_t idesc_f8_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace moe
