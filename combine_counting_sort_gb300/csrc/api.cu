// api.cu: sizes, status strings and device queries of the C ABI.
#include "host_util.h"

using namespace moe;

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_EXPERT_ID: return "MOE_ERR_EXPERT_ID";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

extern "C" int moe_layout_sizes(int T, int k, int E, int G, int block_m, moe_layout_sizes_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  int rc = check_shape(T, k, E, G, block_m);
  if (rc) return rc;
  out->pairs = (int64_t)T * k;
  out->max_tiles = max_tiles_of(T, k, E, block_m);
  out->rowmap_len = out->max_tiles * block_m;
  out->layout_ws_bytes = moe_layout_ws_bytes(E);
  out->stage1_ws_bytes = moe_stage1_ws_bytes(T, k, E, block_m);
  out->gemm_combine_ws_bytes = moe_gemm_combine_ws_bytes(T);
  out->max_send_rows = moe_max_send_rows(T, k, G);
  out->send_ws_bytes = moe_send_ws_bytes(T, k, E, G);
  return MOE_OK;
}

extern "C" int moe_device_sm_count(void) { return device_sm_count(); }
