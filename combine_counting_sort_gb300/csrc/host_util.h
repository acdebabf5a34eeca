// host_util.h: host-side validation and TMA descriptor encoding shared by the
// entry points of libmoe.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/moe.h"

// Bytes of the moe_route_layout workspace (defined next to the kernel).
size_t moe_layout_ws_bytes(int E);
// Bytes of the moe_stage1 workspace (defined next to the kernel).
size_t moe_stage1_ws_bytes(int T, int k, int E, int block_m);
// Bytes of the moe_grouped_gemm1_combine workspace (defined next to the kernel).
size_t moe_gemm_combine_ws_bytes(int T);
// Bytes of the moe_send_layout workspace and capacity of the send runs (defined next to the kernels).
size_t moe_send_ws_bytes(int T, int k, int E, int G);
long long moe_max_send_rows(int T, int k, int G);

namespace moe {

inline int64_t max_tiles_of(int64_t T, int64_t k, int64_t E, int64_t bm) {
  return std::min(T * k, (T * k + E * (bm - 1)) / bm);
}

inline int check_shape(int T, int k, int E, int G, int block_m) {
  if (T < 1 || T > (1 << 20)) return MOE_ERR_INVALID_ARG;
  if (k < 1 || k > 32 || E < k || E > 1024) return MOE_ERR_INVALID_ARG;
  if (G < 1 || E % G != 0) return MOE_ERR_INVALID_ARG;
  if (block_m != MOE_BLOCK_M) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * k >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

inline int check_layout(const moe_layout_t* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  int rc = check_shape(L->T, L->k, L->E, L->G, L->block_m);
  if (rc) return rc;
  if (L->max_tiles != max_tiles_of(L->T, L->k, L->E, L->block_m)) return MOE_ERR_INVALID_ARG;
  if (!L->count || !L->expert_offset || !L->expert_tile_offset || !L->group_offset ||
      !L->ready_tokens || !L->pair_row || !L->row_pair || !L->row_weight || !L->rowmap ||
      !L->tile_expert || !L->tile_row_begin || !L->tile_rows || !L->num_tiles || !L->token_order)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

inline int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// sm_100-class (tcgen05) device?
inline bool device_has_tcgen05() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  return major == 10;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda, so the library loads on machines without a driver).  Looked
// up once, by the first call that needs it (a thread-safe static initialiser);
// null where there is no driver, and the entry points then return MOE_ERR_CUDA.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
  }();
  return fn;
}

// 2-D / 3-D uint8 tensor map with the 128-byte swizzle; dims innermost first,
// strides in bytes for dims 1.., box in elements.
inline bool encode_u8_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d, s,
                   b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace moe
