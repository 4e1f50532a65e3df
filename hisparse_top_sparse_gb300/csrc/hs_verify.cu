// a7-a8: greedy verify of [anchor, drafts] and commit of the accepted prefix.
//
// "投机解码的 KV 流转：prefill 阶段 DFlash 也要吃下整个 prompt", section ④: the
// target runs once over the anchor and the d drafts; the logits at input i
// check draft i+1, the first mismatch yields the correction token, and when
// every draft passes the last input's logits yield one more token. Only the
// KV of the agreeing prefix (anchor + accepted drafts) is kept; the token
// picked last has no KV until the next round, where it is the anchor at
// position L (section ⑥ and the closing table).
//
// Two launches:
//   k_verify_argmax  block per (request, input) row: streaming argmax over the
//                    vocabulary with 16-byte loads, ties to the lowest index
//   k_verify_commit  block per request: accepted length, next token, host-pool
//                    write of the kept rows through the mapped pool, LRU slot
//                    choice (the head of the request's (ts, slot) order, which
//                    is then rotated), hot-slot write and the kv_len update

#include <float.h>

#include "hs_internal.cuh"

namespace {

template <int DTYPE>
__global__ void __launch_bounds__(HS_ARGMAX_THREADS) k_verify_argmax(const void *__restrict__ logits,
                                                                    int32_t V, int32_t rows_per_req,
                                                                    int32_t n_step,
                                                                    int32_t *__restrict__ pred) {
  const int64_t row = blockIdx.x;
  const int64_t elem = (DTYPE == HS_LOGITS_F32) ? 4 : 2;
  const int32_t best = hs_row_argmax<DTYPE>(
      reinterpret_cast<const char *>(logits) + row * (int64_t)V * elem, V);
  if (threadIdx.x == 0) {
    const int64_t req = row / rows_per_req, i = row % rows_per_req;
    pred[req * n_step + i] = best;
  }
}

__global__ void __launch_bounds__(256) k_verify_commit(
    int32_t d, const int32_t *__restrict__ drafts, const int32_t *__restrict__ pred,
    const uint4 *__restrict__ step_kv, const int32_t *__restrict__ req_ids,
    int32_t *kv_len, int32_t *accept_len, int32_t *next_token, int32_t max_reqs, int32_t S,
    int32_t S_tot, int32_t n_step, int32_t max_ctx, int32_t block_size, int32_t hbt_stride,
    const int32_t *__restrict__ hbt, int64_t pool_rows, uint4 *pool, uint4 *hot,
    int32_t *token_slot, int32_t *slot_token, int64_t *slot_ts, int32_t *lru_order,
    uint32_t *status, int64_t now) {
  const int b = blockIdx.x;
  __shared__ int sm_m, sm_L, sm_ok;
  __shared__ int32_t chosen[HS_MAX_STEP];
  const int32_t req = req_ids ? req_ids[b] : b;
  if (threadIdx.x == 0) {
    const int32_t *p = pred + (int64_t)b * n_step;
    int m = 0;
    while (m < d && drafts[(int64_t)b * d + m] == p[m]) ++m;
    accept_len[b] = m;
    next_token[b] = p[m];
    int ok = 1;
    int L = 0;
    if (req < 0 || req >= max_reqs) {
      ok = 0;
      atomicOr(status, HS_STATUS_INDEX);
    } else {
      L = kv_len[req];
      if ((int64_t)L + m + 1 > max_ctx || m + 1 > S) {
        ok = 0;
        atomicOr(status, HS_STATUS_CAPACITY);
      }
    }
    sm_m = m; sm_L = L; sm_ok = ok;
  }
  __syncthreads();
  if (!sm_ok) return;
  const int n = sm_m + 1, L = sm_L;
  const int64_t sbase = (int64_t)req * S;

  // The victims are the first n slots of the LRU order (ascending (ts, slot),
  // nothing protected). They take the current time, so the new order is the
  // rest of the order followed by the victims in slot order.
  extern __shared__ int32_t ord[];                 // [S]
  int32_t *lru = lru_order + sbase;
  for (int i = threadIdx.x; i < S; i += blockDim.x) ord[i] = lru[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 0; k < n; ++k) chosen[k] = ord[k];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < S - n; i += blockDim.x) lru[i] = ord[n + i];
  if (threadIdx.x == 0) {
    int32_t sorted[HS_MAX_STEP];
    for (int k = 0; k < n; ++k) {               // insertion sort of at most 16 slots
      int32_t v = chosen[k];
      int j = k;
      while (j > 0 && sorted[j - 1] > v) { sorted[j] = sorted[j - 1]; --j; }
      sorted[j] = v;
    }
    for (int k = 0; k < n; ++k) lru[S - n + k] = sorted[k];
  }

  // map updates (one thread per kept position)
  const int64_t cbase = (int64_t)req * max_ctx;
  if (threadIdx.x < n) {
    const int k = threadIdx.x;
    const int32_t s = chosen[k], t = L + k;
    const int32_t old = slot_token[sbase + s];
    if (old >= 0 && old < max_ctx) token_slot[cbase + old] = -1;
    slot_token[sbase + s] = t;
    token_slot[cbase + t] = s;
    slot_ts[sbase + s] = now;
  }
  // row copies: kept step rows -> host pool rows and hot slots
  const int32_t *hbt_row = hbt + (int64_t)req * hbt_stride;
  for (int e = threadIdx.x; e < n * HS_ROW_VEC16; e += blockDim.x) {
    const int k = e / HS_ROW_VEC16, c = e % HS_ROW_VEC16;
    const int32_t t = L + k;
    const uint4 v = step_kv[((int64_t)b * (d + 1) + k) * HS_ROW_VEC16 + c];
    const int32_t hb = hbt_row[t / block_size];
    const int64_t hr = (int64_t)hb * block_size + t % block_size;
    if (hb >= 0 && hr < pool_rows) pool[hr * HS_ROW_VEC16 + c] = v;
    else if (c == 0) atomicOr(status, HS_STATUS_INDEX);
    hot[((int64_t)req * S_tot + chosen[k]) * HS_ROW_VEC16 + c] = v;
  }
  if (threadIdx.x == 0) kv_len[req] = L + n;
}

}  // namespace

extern "C" int hs_verify_finalize(hs_buffer *buf, const void *logits, int32_t logits_dtype,
                                  int32_t B, int32_t d, int32_t V, const int32_t *draft_tokens,
                                  const void *step_kv, const int32_t *req_ids, int32_t *kv_len,
                                  int32_t *accept_len, int32_t *next_token, hs_stream_t stream) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (B < 1 || B > buf->max_reqs || d < 0 || d + 1 > buf->n_step || V < 1)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes B=%d (1..%d) d=%d (d+1<=%d) V=%d", B,
                        buf->max_reqs, d, buf->n_step, V);
  if (logits_dtype != HS_LOGITS_F32 && logits_dtype != HS_LOGITS_BF16)
    return hs_set_error(HS_ERR_INVALID_ARG, "logits_dtype %d", logits_dtype);
  if (!logits || (d > 0 && !draft_tokens) || !step_kv || !kv_len || !accept_len || !next_token)
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL argument");
  if ((uintptr_t)step_kv & 15)
    return hs_set_error(HS_ERR_INVALID_ARG, "step_kv must be 16-byte aligned");
  buf->clock += 1;
  const int rows = B * (d + 1);
  if (logits_dtype == HS_LOGITS_F32)
    k_verify_argmax<HS_LOGITS_F32><<<rows, HS_ARGMAX_THREADS, 0, stream>>>(logits, V, d + 1, buf->n_step,
                                                             buf->pred);
  else
    k_verify_argmax<HS_LOGITS_BF16><<<rows, HS_ARGMAX_THREADS, 0, stream>>>(logits, V, d + 1, buf->n_step,
                                                              buf->pred);
  HS_LAUNCH_CHECK("k_verify_argmax");
  k_verify_commit<<<B, 256, (size_t)buf->S * sizeof(int32_t), stream>>>(
      d, draft_tokens, buf->pred, reinterpret_cast<const uint4 *>(step_kv), req_ids, kv_len,
      accept_len, next_token, buf->max_reqs, buf->S, buf->S_tot, buf->n_step, buf->max_ctx,
      buf->block_size, buf->hbt_stride, buf->hbt, buf->host_pool_rows,
      reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(buf->host_pool)),
      reinterpret_cast<uint4 *>(buf->hot_kv), buf->token_slot, buf->slot_token, buf->slot_ts,
      buf->lru_order, buf->status, buf->clock);
  HS_LAUNCH_CHECK("k_verify_commit");
  return HS_OK;
}
