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
#define HS_MAX_REQS 16384                  // requests per buffer (swap-in gather prefix in SMEM)
#define HS_MAX_LAYERS 64                   // caches per hs_swap_apply_plan / hs_backup_pages call

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
  int32_t *lru_order;    // [max_reqs][S]: slots in ascending (ts, slot) order

  // per-call scratch (epoch-stamped, so nothing needs clearing per call)
  uint32_t *pos_mark;    // [max_reqs][max_ctx]: epoch at which a position was claimed
  uint64_t *copy_desc;   // [max_reqs][S]: (host pool row << 16) | hot slot, per miss
  int32_t *copy_cnt;     // [max_reqs]: misses to copy in the current call
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
// The device-accessible alias of p (device memory, or page-locked host memory
// mapped into the device's address space); `align`-byte alignment required.
int hs_device_alias(const void *p, const void **out, const char *name, int align = 16);

// ---- block helpers shared by the swap-in and commit kernels -----------------

// Exclusive prefix sum of one int per thread over the block; *total gets the
// sum. `tmp` is 33 ints of shared memory. Every thread of the block calls it.
__device__ __forceinline__ int hs_block_exscan(int v, int *tmp, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int incl = v;
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) tmp[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = lane < nw ? tmp[lane] : 0;
    int xi = x;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += y;
    }
    tmp[lane] = xi - x;
    if (lane == 31) tmp[32] = xi;
  }
  __syncthreads();
  const int res = tmp[w] + incl - v;
  *total = tmp[32];
  __syncthreads();
  return res;
}

// The LRU order after a call that gave every slot in `touched` the newest
// timestamp: the untouched slots keep their order, the touched ones follow in
// slot order -- which is again the order by ascending (ts, slot). `order` is
// the current order (shared memory), `touched` a bitmap of S bits (shared
// memory); the new order is written to `out` (global). Every thread calls it.
__device__ __forceinline__ void hs_lru_reorder(const int32_t *order, const uint32_t *touched,
                                               int S, int32_t *out, int *tmp) {
  const int E = (S + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * E, hi = min(S, lo + E);
  int cu = 0, ct = 0;
  for (int i = lo; i < hi; ++i) {
    const int s = order[i];
    cu += !((touched[s >> 5] >> (s & 31)) & 1u);
    ct += (touched[i >> 5] >> (i & 31)) & 1u;
  }
  int tot_u, tot_t;
  int ku = hs_block_exscan(cu, tmp, &tot_u);
  int kt = hs_block_exscan(ct, tmp, &tot_t) + tot_u;
  for (int i = lo; i < hi; ++i) {
    const int s = order[i];
    if (!((touched[s >> 5] >> (s & 31)) & 1u)) out[ku++] = s;
    if ((touched[i >> 5] >> (i & 31)) & 1u) out[kt++] = i;
  }
}
int hs_check_buffer(const hs_buffer *buf);
