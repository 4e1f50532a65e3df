// Internal declarations of libhisparse (sm_103a). Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "hisparse.h"

#define HS_ROW_BYTES (HS_LATENT_DIM * 2)   // 1152 bytes per latent row
#define HS_ROW_VEC16 (HS_ROW_BYTES / 16)   // 72 16-byte chunks per row
#define HS_MAX_SLOTS 8192                  // S limit (the LRU sort runs in SMEM)
#define HS_MAX_STEP 16

// Host-side state of a hot buffer. Device arrays are owned by the library.
struct hs_buffer {
  int device;
  int32_t max_reqs, S, n_step, S_tot, max_ctx, block_size, hbt_stride;
  __nv_bfloat16 *hot_kv;                 // caller's, [max_reqs*S_tot][576]
  const __nv_bfloat16 *host_pool;        // device-addressable view of the pool
  int64_t host_pool_rows;
  const int32_t *hbt;                    // caller's, [max_reqs][hbt_stride]

  // persistent maps
  int32_t *token_slot;   // [max_reqs][max_ctx], -1 = not resident
  int32_t *slot_token;   // [max_reqs][S], -1 = empty
  int64_t *slot_ts;      // [max_reqs][S], -1 = empty

  // per-call scratch (epoch-stamped, so nothing needs clearing per call)
  uint32_t *pos_mark;    // [max_reqs][max_ctx]: epoch at which a position was claimed
  uint32_t *slot_mark;   // [max_reqs][S]: epoch at which a slot was found needed
  uint32_t *req_mark;    // [max_reqs]: epoch at which a request appeared
  uint32_t *fail_mark;   // [max_reqs]: epoch at which a request overflowed
  int32_t *counters;     // [2*max_reqs + 1]: need, miss per request; copy count
  int32_t *miss_list;    // [max_reqs][S]
  int64_t *copy_src;     // [max_reqs*S] host pool rows
  int32_t *copy_dst;     // [max_reqs*S] hot rows
  int32_t *pred;         // [max_reqs*n_step] argmax per verify row
  uint32_t *status;      // device status word

  int64_t clock;         // LRU clock: swap-in and commit calls made so far
};

// error reporting (hs_api.cu)
int hs_set_error(int code, const char *fmt, ...);

#define HS_CUDA_TRY(expr)                                                      \
  do {                                                                         \
    cudaError_t e_ = (expr);                                                   \
    if (e_ != cudaSuccess)                                                     \
      return hs_set_error(HS_ERR_CUDA, "%s failed: %s", #expr,                 \
                          cudaGetErrorString(e_));                             \
  } while (0)

#define HS_LAUNCH_CHECK(what)                                                  \
  do {                                                                         \
    cudaError_t e_ = cudaGetLastError();                                       \
    if (e_ != cudaSuccess)                                                     \
      return hs_set_error(HS_ERR_CUDA, "launch of %s failed: %s", what,        \
                          cudaGetErrorString(e_));                             \
  } while (0)

int hs_check_device_ptr(const void *p, const char *name, bool allow_null);
int hs_check_buffer(const hs_buffer *buf);
