// Hot-buffer lifetime, status, error text, the fully-resident index
// conversion (a1) and the host-read probe.
//
// a1 follows "vllm 分析(十二) HiSparse 下篇", HiSparseCacheHandle.resolve_topk:
// with fully_resident set, each row's top-k logical positions become physical
// cache rows through the request's block table (block size and physical block
// stride as parameters).

#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "hs_internal.cuh"

static thread_local char g_err[512] = "no error";

int hs_set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

extern "C" const char *hs_last_error_string(void) { return g_err; }

int hs_check_device_ptr(const void *p, const char *name, bool allow_null) {
  if (!p && !allow_null)
    return hs_set_error(HS_ERR_INVALID_ARG, "%s is NULL", name);
  return HS_OK;
}

int hs_device_alias(const void *p, const void **out, const char *name, int align) {
  if (!p) return hs_set_error(HS_ERR_INVALID_ARG, "%s is NULL", name);
  if ((uintptr_t)p % (uintptr_t)align)
    return hs_set_error(HS_ERR_INVALID_ARG, "%s must be %d-byte aligned", name, align);
  cudaPointerAttributes attr;
  HS_CUDA_TRY(cudaPointerGetAttributes(&attr, p));
  *out = nullptr;
  if (attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeDevice ||
      attr.type == cudaMemoryTypeManaged)
    *out = attr.devicePointer;
  if (!*out)
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "%s is not page-locked mapped host memory or device memory", name);
  return HS_OK;
}

int hs_check_buffer(const hs_buffer *buf) {
  if (!buf) return hs_set_error(HS_ERR_INVALID_ARG, "buffer is NULL");
  int dev = -1;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != buf->device)
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "current device %d is not the buffer's device %d", dev,
                        buf->device);
  return HS_OK;
}

// ---------------------------------------------------------------- buffer --

static void free_buffer(hs_buffer *b) {
  if (!b) return;
  void *ptrs[] = {b->token_slot, b->slot_token, b->slot_ts, b->lru_order, b->lru_head, b->pos_mark,
                  b->copy_desc,  b->copy_cnt,   b->pred,    b->row_count, b->verify_claim,
                  b->req_group,  b->status};
  for (void *p : ptrs)
    if (p) cudaFree(p);
  for (cudaStream_t &st : b->side)
    if (st) cudaStreamDestroy(st);
  if (b->ev_fork) cudaEventDestroy(b->ev_fork);
  for (cudaEvent_t &e : b->ev_gather)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t &e : b->ev_join)
    if (e) cudaEventDestroy(e);
  free(b);
}

// Every request starts with all slots empty (ts = -1): LRU order = slot order.
__global__ void k_order_init(int32_t *order, int32_t S, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    order[i] = (int32_t)(i % S);
}

extern "C" int hs_buffer_create(const hs_buffer_desc *d, hs_buffer **out) {
  if (!d || !out) return hs_set_error(HS_ERR_INVALID_ARG, "desc/out is NULL");
  *out = nullptr;
  if (d->max_reqs < 1 || d->max_reqs > HS_MAX_REQS || d->slots_per_req < 1 ||
      d->slots_per_req > HS_MAX_SLOTS ||
      d->step_slots < 1 || d->step_slots > HS_MAX_STEP || d->max_ctx < 1 ||
      d->block_size < 1 || d->host_pool_rows < 1)
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "bad sizes: max_reqs=%d (1..16384) S=%d (1..%d) step_slots=%d (1..%d) "
                        "max_ctx=%d block_size=%d host_pool_rows=%lld",
                        d->max_reqs, d->slots_per_req, HS_MAX_SLOTS, d->step_slots,
                        HS_MAX_STEP, d->max_ctx, d->block_size,
                        (long long)d->host_pool_rows);
  int64_t need_blocks = ((int64_t)d->max_ctx + d->block_size - 1) / d->block_size;
  if (d->hbt_stride < need_blocks)
    return hs_set_error(HS_ERR_INVALID_ARG, "hbt_stride %d < ceil(max_ctx/block_size) %lld",
                        d->hbt_stride, (long long)need_blocks);
  if (!d->hot_kv || !d->host_pool || !d->host_block_table)
    return hs_set_error(HS_ERR_INVALID_ARG, "hot_kv/host_pool/host_block_table is NULL");
  if (((uintptr_t)d->hot_kv & 15) || ((uintptr_t)d->host_pool & 15))
    return hs_set_error(HS_ERR_INVALID_ARG, "hot_kv and host_pool must be 16-byte aligned");
  int64_t S_tot = (int64_t)d->slots_per_req + d->step_slots;
  if ((int64_t)d->max_reqs * S_tot > INT32_MAX ||
      (int64_t)d->max_reqs * d->max_ctx > ((int64_t)1 << 40))
    return hs_set_error(HS_ERR_INVALID_ARG, "buffer too large for int32 hot-row indices");

  // The host pool must be addressable by the device: page-locked mapped host
  // memory (its device alias is used) or device memory.
  cudaPointerAttributes attr;
  HS_CUDA_TRY(cudaPointerGetAttributes(&attr, d->host_pool));
  const void *pool_dev = nullptr;
  if (attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeDevice ||
      attr.type == cudaMemoryTypeManaged)
    pool_dev = attr.devicePointer;
  if (!pool_dev)
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "host_pool is not page-locked mapped host memory or device memory");

  hs_buffer *b = (hs_buffer *)calloc(1, sizeof(hs_buffer));
  if (!b) return hs_set_error(HS_ERR_INVALID_ARG, "out of host memory");
  HS_CUDA_TRY(cudaGetDevice(&b->device));
  b->max_reqs = d->max_reqs;
  b->S = d->slots_per_req;
  b->n_step = d->step_slots;
  b->S_tot = (int32_t)S_tot;
  b->max_ctx = d->max_ctx;
  b->block_size = d->block_size;
  b->hbt_stride = d->hbt_stride;
  b->hot_kv = (__nv_bfloat16 *)d->hot_kv;
  b->host_pool = (const __nv_bfloat16 *)pool_dev;
  b->host_pool_rows = d->host_pool_rows;
  b->hbt = d->host_block_table;

  const size_t R = (size_t)d->max_reqs, S = (size_t)d->slots_per_req,
               C = (size_t)d->max_ctx;
  struct { void **p; size_t bytes; int fill; } plan[] = {
      {(void **)&b->token_slot, R * C * 4, 0xFF},
      {(void **)&b->slot_token, R * S * 4, 0xFF},
      {(void **)&b->slot_ts, R * S * 8, 0xFF},
      {(void **)&b->lru_order, R * S * 4, 0},
      {(void **)&b->lru_head, R * 4, 0},
      {(void **)&b->pos_mark, R * C * 4, 0},
      {(void **)&b->copy_desc, R * S * 8, 0},
      {(void **)&b->copy_cnt, R * 4, 0},
      {(void **)&b->pred, R * (size_t)d->step_slots * 4, 0},
      {(void **)&b->row_count, R * 4, 0},
      {(void **)&b->verify_claim, R * 4, 0},
      {(void **)&b->req_group, R * 4, 0xFF},
      {(void **)&b->status, 4, 0},
  };
  for (auto &e : plan) {
    cudaError_t err = cudaMalloc(e.p, e.bytes);
    if (err == cudaSuccess) err = cudaMemset(*e.p, e.fill, e.bytes);
    if (err != cudaSuccess) {
      free_buffer(b);
      return hs_set_error(HS_ERR_CUDA, "allocating %zu bytes of buffer metadata: %s",
                          e.bytes, cudaGetErrorString(err));
    }
  }
  // the side streams and events of hs_swap_in_attn_decode
  {
    cudaError_t err = cudaSuccess;
    for (cudaStream_t &st : b->side)
      if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&b->ev_fork, cudaEventDisableTiming);
    for (cudaEvent_t &e : b->ev_gather)
      if (err == cudaSuccess) err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    for (cudaEvent_t &e : b->ev_join)
      if (err == cudaSuccess) err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (err != cudaSuccess) {
      free_buffer(b);
      return hs_set_error(HS_ERR_CUDA, "creating the buffer's streams and events: %s",
                          cudaGetErrorString(err));
    }
  }
  k_order_init<<<(int)std::min<size_t>(R * S / 256 + 1, 65535), 256>>>(b->lru_order, b->S,
                                                                        (int64_t)R * S);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  if (err != cudaSuccess) {
    free_buffer(b);
    return hs_set_error(HS_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(err));
  }
  *out = b;
  return HS_OK;
}

extern "C" int hs_buffer_destroy(hs_buffer *buf) {
  free_buffer(buf);
  return HS_OK;
}

extern "C" int64_t hs_buffer_clock(const hs_buffer *buf) { return buf ? buf->clock : -1; }

extern "C" int hs_buffer_set_copy_sms(hs_buffer *buf, int32_t n_sms) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (n_sms < 0) return hs_set_error(HS_ERR_INVALID_ARG, "n_sms %d < 0", n_sms);
  buf->copy_sms = n_sms;
  return HS_OK;
}

__global__ void k_request_reset(int32_t *token_slot, int32_t *slot_token, int64_t *slot_ts,
                                int32_t *order, int32_t *head, int32_t S, int32_t max_ctx,
                                int32_t req) {
  if (threadIdx.x == 0) head[req] = 0;
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    int64_t k = (int64_t)req * S + s;
    int32_t t = slot_token[k];
    if (t >= 0 && t < max_ctx) token_slot[(int64_t)req * max_ctx + t] = -1;
    slot_token[k] = -1;
    slot_ts[k] = -1;
    order[k] = s;      // all empty: slot order
  }
}

extern "C" int hs_request_reset(hs_buffer *buf, int32_t req, hs_stream_t stream) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (req < 0 || req >= buf->max_reqs)
    return hs_set_error(HS_ERR_INVALID_ARG, "req %d outside [0, %d)", req, buf->max_reqs);
  k_request_reset<<<1, 1024, 0, stream>>>(buf->token_slot, buf->slot_token, buf->slot_ts,
                                          buf->lru_order, buf->lru_head, buf->S, buf->max_ctx,
                                          req);
  HS_LAUNCH_CHECK("k_request_reset");
  return HS_OK;
}

extern "C" int hs_get_status(hs_buffer *buf, hs_stream_t stream, uint32_t *out_bits) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (!out_bits) return hs_set_error(HS_ERR_INVALID_ARG, "out_bits is NULL");
  uint32_t v = 0;
  HS_CUDA_TRY(cudaMemcpyAsync(&v, buf->status, 4, cudaMemcpyDeviceToHost, stream));
  HS_CUDA_TRY(cudaMemsetAsync(buf->status, 0, 4, stream));
  HS_CUDA_TRY(cudaStreamSynchronize(stream));
  *out_bits = v;
  return HS_OK;
}

extern "C" int hs_buffer_dump(hs_buffer *buf, hs_stream_t stream, int32_t *token_slot,
                              int32_t *slot_token, int64_t *slot_ts) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  HS_CUDA_TRY(cudaStreamSynchronize(stream));
  size_t R = buf->max_reqs, S = buf->S, C = buf->max_ctx;
  if (token_slot)
    HS_CUDA_TRY(cudaMemcpy(token_slot, buf->token_slot, R * C * 4, cudaMemcpyDeviceToHost));
  if (slot_token)
    HS_CUDA_TRY(cudaMemcpy(slot_token, buf->slot_token, R * S * 4, cudaMemcpyDeviceToHost));
  if (slot_ts)
    HS_CUDA_TRY(cudaMemcpy(slot_ts, buf->slot_ts, R * S * 8, cudaMemcpyDeviceToHost));
  return HS_OK;
}

// --------------------------------------------------------------- resolve --
// One thread per 4 entries of a row (16-byte loads and stores of topk and
// out_idx when K % 4 == 0), one block per row; the valid count is a block
// reduction, so out_valid needs no clearing.

template <bool VEC>
__global__ void __launch_bounds__(256) k_resolve_topk(
    const int32_t *__restrict__ req_id, const int32_t *__restrict__ clen,
    const int32_t *__restrict__ bt, int32_t bt_stride, const int32_t *__restrict__ topk,
    int32_t K, int32_t bs, int32_t stride, int32_t *__restrict__ out,
    int32_t *__restrict__ out_valid, uint32_t *status) {
  // the attention launched after this kernel may begin its prologue now; it
  // reads this kernel's output only after this kernel has finished
  asm volatile("griddepcontrol.launch_dependents;\n");
  const int r = blockIdx.x;
  // No branch on the request id before the top-k loads: the id, the causal
  // length and the row's entries are read together, and only the block-table
  // lookups wait for them. A row with no request (id < 0) gives -1
  // everywhere, no valid entry and the index status bit.
  const int32_t b = req_id[r];
  const int32_t n = clen[r];
  const bool none = b < 0;
  const int32_t *bt_row = bt + (int64_t)(none ? 0 : b) * bt_stride;
  const int32_t *tk = topk + (int64_t)r * K;
  int32_t *o = out + (int64_t)r * K;
  int cnt = 0;
  bool bad = none && K > 0;
  auto conv = [&](int32_t t) -> int32_t {
    if (t < 0 || none) return -1;
    if (t >= n) { bad = true; return -1; }
    int32_t blk = bt_row[t / bs];
    if (blk < 0) { bad = true; return -1; }
    ++cnt;
    return blk * stride + t % bs;
  };
  if (VEC) {
    const int4 *tk4 = reinterpret_cast<const int4 *>(tk);
    int4 *o4 = reinterpret_cast<int4 *>(o);
#pragma unroll 2
    for (int j = threadIdx.x; j < K / 4; j += blockDim.x) {
      int4 t = tk4[j];
      int4 v;
      v.x = conv(t.x); v.y = conv(t.y); v.z = conv(t.z); v.w = conv(t.w);
      o4[j] = v;
    }
  } else {
    for (int j = threadIdx.x; j < K; j += blockDim.x) o[j] = conv(tk[j]);
  }
  if (status && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, HS_STATUS_INDEX);
  if (out_valid) {
    __shared__ int warp_sum[8];
    for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += warp_sum[w];
      out_valid[r] = s;
    }
  }
}

extern "C" int hs_resolve_topk(const int32_t *req_id_per_row, const int32_t *row_causal_len,
                               const int32_t *block_table, int32_t bt_stride,
                               const int32_t *topk, int32_t R, int32_t K, int32_t block_size,
                               int32_t phys_block_stride, int32_t *out_idx, int32_t *out_valid,
                               uint32_t *status, hs_stream_t stream) {
  if (R < 0 || K < 0 || block_size < 1 || phys_block_stride < 1 || bt_stride < 1)
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "bad sizes: R=%d K=%d block_size=%d phys_block_stride=%d bt_stride=%d",
                        R, K, block_size, phys_block_stride, bt_stride);
  if (R == 0) return HS_OK;
  if (!req_id_per_row || !row_causal_len || !block_table || (K > 0 && (!topk || !out_idx)))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL input or output pointer");
  bool vec = (K % 4 == 0) && (((uintptr_t)topk | (uintptr_t)out_idx) & 15) == 0;
  if (vec)
    k_resolve_topk<true><<<R, 256, 0, stream>>>(req_id_per_row, row_causal_len, block_table,
                                                bt_stride, topk, K, block_size,
                                                phys_block_stride, out_idx, out_valid, status);
  else
    k_resolve_topk<false><<<R, 256, 0, stream>>>(req_id_per_row, row_causal_len, block_table,
                                                 bt_stride, topk, K, block_size,
                                                 phys_block_stride, out_idx, out_valid, status);
  HS_LAUNCH_CHECK("k_resolve_topk");
  return HS_OK;
}

// ------------------------------------------------------------ read probe --

__global__ void __launch_bounds__(256) k_read_probe(const uint4 *__restrict__ src, size_t n16,
                                                    uint64_t *sink) {
  uint64_t acc = 0;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t step = (size_t)gridDim.x * blockDim.x;
  for (; i + 3 * step < n16; i += 4 * step) {
    uint4 a = src[i], b = src[i + step], c = src[i + 2 * step], d = src[i + 3 * step];
    acc += (uint64_t)a.x ^ b.y ^ c.z ^ d.w;
  }
  for (; i < n16; i += step) acc += src[i].x;
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  __shared__ uint64_t ws[8];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t s = 0;
    for (int w = 0; w < 8; ++w) s += ws[w];
    sink[blockIdx.x] = s;
  }
}

extern "C" int hs_read_probe(const void *src, size_t bytes, uint64_t *sink, int32_t blocks,
                             hs_stream_t stream) {
  if (!src || !sink || blocks < 1 || (bytes & 15) || ((uintptr_t)src & 15))
    return hs_set_error(HS_ERR_INVALID_ARG, "bad read-probe arguments");
  k_read_probe<<<blocks, 256, 0, stream>>>((const uint4 *)src, bytes / 16, sink);
  HS_LAUNCH_CHECK("k_read_probe");
  return HS_OK;
}
