// Internal declarations of libhisparse (sm_103a). Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "hisparse.h"

#define HS_ROW_BYTES (HS_LATENT_DIM * 2)   // 1152 bytes per latent row
#define HS_ROW_VEC16 (HS_ROW_BYTES / 16)   // 72 16-byte chunks per row
#define HS_MAX_SLOTS 8192                  // S limit (the LRU sort runs in SMEM)
#define HS_MAX_STEP 16
#define HS_MAX_REQS 16384                  // requests per buffer (swap-in gather prefix in SMEM)
#define HS_MAX_LAYERS 64                   // caches per hs_swap_apply_plan / hs_backup_pages call
#define HS_MAX_GROUPS 8                    // request groups of one hs_swap_in_attn_decode call
#define HS_SIDE_STREAMS 3                  // one for the gathers, two for the attention launches

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
  int32_t *lru_order;    // [max_reqs][S]: slots in ascending (ts, slot) order, a ring
  int32_t *lru_head;     // [max_reqs]: ring position of each request's order's first slot

  // per-call scratch (epoch-stamped, so nothing needs clearing per call)
  uint32_t *pos_mark;    // [max_reqs][max_ctx]: epoch at which a position was claimed
  uint64_t *copy_desc;   // [max_reqs][S]: (host pool row << 16) | hot slot, per miss
  int32_t *copy_cnt;     // [max_reqs]: misses to copy in the current call
  int32_t *pred;         // [max_reqs*n_step] argmax per verify row
  int32_t *row_count;    // [max_reqs] verify rows done per request in a call (0 between calls)
  uint32_t *verify_claim; // [max_reqs]: low 32 bits of the clock of the last commit of a request
  int32_t *req_group;    // [max_reqs]: group of the request's first row in the latest swap-in
  uint32_t *status;      // device status word

  // streams and events of hs_swap_in_attn_decode (created with the buffer)
  cudaStream_t side[HS_SIDE_STREAMS];
  cudaEvent_t ev_fork, ev_gather[HS_MAX_GROUPS], ev_join[HS_SIDE_STREAMS];

  int64_t clock;         // LRU clock: swap-in and commit calls made so far
  int32_t copy_sms;      // SMs the copy kernels may spread over (0 = all)
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

int hs_check_buffer(const hs_buffer *buf);

// ---- launchers shared by hs_swap_in and hs_swap_in_attn_decode (hs_swap.cu)

// The metadata kernel over rows [0, R) of a call. Rows [group_end[g-1],
// group_end[g]) form group g (n_groups >= 1, group_end ascending, the last
// = R); each request's first-row group goes to buf->req_group. The caller
// advances buf->clock first.
int hs_swap_plan_launch(hs_buffer *buf, const int32_t *req_id_per_row,
                        const int32_t *row_causal_len, const int32_t *kv_len, const int32_t *topk,
                        int32_t R, int32_t K, int32_t n_groups, const int32_t *group_end,
                        int32_t *out_slot_idx, int32_t *out_valid, int64_t *stats,
                        cudaStream_t stream);
// The copies of the misses of group g's requests (those whose first row lies
// in group g) and the slot table of rows [row_lo, row_hi). ctas_per_sm
// blocks of `threads` (a multiple of 32, at most 512) per SM of the buffer's
// copy SMs; pdl: a programmatic dependent launch of the kernel before it in
// the stream.
int hs_swap_gather_launch(hs_buffer *buf, const int32_t *req_id_per_row,
                          const int32_t *row_causal_len, const int32_t *kv_len,
                          const int32_t *topk, int32_t R, int32_t K, int32_t g, int32_t row_lo,
                          int32_t row_hi, int32_t *out_slot_idx, int32_t *out_valid,
                          int ctas_per_sm, int threads, bool pdl, cudaStream_t stream);

// ---- attention launcher (hs_attn.cu) ----------------------------------------

// hs_sparse_attn_decode_mixed with the launch made a programmatic dependent
// one (pdl) or a plain one.
int hs_attn_launch(const void *q, const void *kv_resident, int64_t n_resident, const void *kv_hot,
                   int64_t n_hot, const int32_t *row_req, const int32_t *fully_resident,
                   int32_t n_reqs, const int32_t *idx, int32_t R, int32_t H, int32_t K,
                   float scale, void *out, float *lse, uint32_t *status, bool pdl,
                   cudaStream_t stream);
// Rows of H heads that one wave of the attention kernel holds on the current
// device (two-SM clusters resident at once, per row's head groups); >= 1.
int hs_attn_wave_rows(int32_t H, int32_t *rows);
// The attention kernel's attributes (registers, static shared memory) and the
// threads and dynamic shared memory of one CTA.
int hs_attn_block_attrs(cudaFuncAttributes *attr, int *threads, size_t *dyn_smem);
// The same for the swap-in gather kernel (its dynamic shared memory depends
// on the launch: 4 * (max_reqs + 1) bytes).
int hs_gather_func_attrs(cudaFuncAttributes *attr);

// ---- argmax of one logits row (greedy verify) -------------------------------

#define HS_ARGMAX_THREADS 256   // a block per row: 8 per SM, every row of a call in one wave

// The index of the largest of logits[0 .. V-1] (fp32 or bf16 as dtype says),
// the lowest index among equals, for the block's thread 0 (others: unspecified).
// 16-byte streaming loads over the aligned body, eight in flight per thread;
// scalar loads for the unaligned head and the tail. Every thread of the block
// (HS_ARGMAX_THREADS of them) calls it.
template <int DTYPE>
__device__ __forceinline__ int32_t hs_row_argmax(const char *base, int32_t V) {
  struct Best {
    float v;
    int32_t i;
  };
  auto take = [](Best &b, float v, int32_t i) {
    if (v > b.v || (v == b.v && i < b.i)) { b.v = v; b.i = i; }
  };
  constexpr int NT = HS_ARGMAX_THREADS;
  const int64_t elem = (DTYPE == HS_LOGITS_F32) ? 4 : 2;
  const int per16 = 16 / (int)elem;
  auto load = [&](int32_t i) -> float {
    if (DTYPE == HS_LOGITS_F32) return reinterpret_cast<const float *>(base)[i];
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
  };
  auto take16 = [&](Best &b, const uint4 w, int32_t i0) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (DTYPE == HS_LOGITS_F32) {
        take(b, __uint_as_float(ws[q]), i0 + q);
      } else {
        take(b, __uint_as_float(ws[q] << 16), i0 + 2 * q);
        take(b, __uint_as_float(ws[q] & 0xFFFF0000u), i0 + 2 * q + 1);
      }
    }
  };
  Best best{-INFINITY, INT32_MAX};
  const uintptr_t addr = reinterpret_cast<uintptr_t>(base);
  int head = (int)(((16 - (addr & 15)) & 15) / elem);
  if ((addr & (elem - 1)) != 0) head = V;     // misaligned elements: all scalar
  if (head > V) head = V;
  const int nvec = (V - head) / per16;
  for (int i = threadIdx.x; i < head; i += NT) take(best, load(i), i);
  const uint4 *body = reinterpret_cast<const uint4 *>(base + (int64_t)head * elem);
  int k = threadIdx.x;
  for (; k + 7 * NT < nvec; k += 8 * NT) {
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = __ldcs(body + k + u * NT);
#pragma unroll
    for (int u = 0; u < 8; ++u) take16(best, w[u], head + (k + u * NT) * per16);
  }
  for (; k < nvec; k += NT) take16(best, __ldcs(body + k), head + k * per16);
  for (int i = head + nvec * per16 + threadIdx.x; i < V; i += NT) take(best, load(i), i);
  for (int off = 16; off; off >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, best.v, off);
    const int32_t i = __shfl_xor_sync(0xffffffffu, best.i, off);
    take(best, v, i);
  }
  __shared__ float wv[NT / 32];
  __shared__ int32_t wi[NT / 32];
  if ((threadIdx.x & 31) == 0) {
    wv[threadIdx.x >> 5] = best.v;
    wi[threadIdx.x >> 5] = best.i;
  }
  __syncthreads();
  Best b{-INFINITY, INT32_MAX};
  if (threadIdx.x == 0)
    for (int w = 0; w < NT / 32; ++w) take(b, wv[w], wi[w]);
  return b.i;
}
