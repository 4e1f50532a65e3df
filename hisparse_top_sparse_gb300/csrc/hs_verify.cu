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
// One launch, k_verify: a block per (request, input) row takes the streaming
// argmax over the vocabulary (16-byte loads, ties to the lowest index); the
// last of a request's rows to finish then, with the whole block, takes the
// accepted length and next token and commits: host-pool write of the kept
// rows through the mapped pool, LRU slot choice (the first slots of the
// request's (ts, slot) order, a ring whose head then moves past them, so the
// commit writes as many order entries as it keeps rows), hot-slot write,
// kv_len update.

#include <float.h>

#include "hs_internal.cuh"

namespace {

struct CommitArgs {
  int32_t d;
  const int32_t *drafts;
  int32_t *pred;
  const uint4 *step_kv;
  const int32_t *req_ids;
  int32_t *kv_len, *accept_len, *next_token;
  int32_t max_reqs, S, S_tot, n_step, max_ctx, block_size, hbt_stride;
  const int32_t *hbt;
  int64_t pool_rows;
  uint4 *pool, *hot;
  int32_t *token_slot, *slot_token;
  int64_t *slot_ts;
  int32_t *lru_order, *lru_head;
  uint32_t *verify_claim;
  uint32_t *status;
  int64_t now;
};

// Acceptance and commit of batch request b, by a whole block (HS_ARGMAX_THREADS
// threads): longest agreeing prefix m and next token; then the m + 1 kept step
// rows go to the host pool and to the first m + 1 slots of the LRU order
// (nothing protected), which take the current time and move to the order's
// end; the maps and kv_len follow.
__device__ __forceinline__ void commit_request(const int b, const CommitArgs &ca) {
  const int32_t d = ca.d;
  const int32_t *drafts = ca.drafts;
  const int32_t *pred = ca.pred;
  const uint4 *step_kv = ca.step_kv;
  const int32_t *req_ids = ca.req_ids;
  int32_t *kv_len = ca.kv_len, *accept_len = ca.accept_len, *next_token = ca.next_token;
  const int32_t max_reqs = ca.max_reqs, S = ca.S, S_tot = ca.S_tot, n_step = ca.n_step,
                max_ctx = ca.max_ctx, block_size = ca.block_size, hbt_stride = ca.hbt_stride;
  const int32_t *hbt = ca.hbt;
  const int64_t pool_rows = ca.pool_rows;
  uint4 *pool = ca.pool, *hot = ca.hot;
  int32_t *token_slot = ca.token_slot, *slot_token = ca.slot_token, *lru_order = ca.lru_order;
  int64_t *slot_ts = ca.slot_ts;
  uint32_t *status = ca.status;
  const int64_t now = ca.now;
  __shared__ int sm_m, sm_L, sm_ok;
  __shared__ int32_t chosen[HS_MAX_STEP];
  const int32_t req = req_ids ? req_ids[b] : b;
  if (threadIdx.x == 0) {
    const int32_t *p = pred + (int64_t)b * n_step;   // rows written by other blocks
    int m = 0;
    while (m < d && drafts[(int64_t)b * d + m] == __ldcg(p + m)) ++m;
    accept_len[b] = m;
    next_token[b] = __ldcg(p + m);
    int ok = 1;
    int L = 0;
    if (req < 0 || req >= max_reqs) {
      ok = 0;
      atomicOr(status, HS_STATUS_INDEX);
    } else if (atomicExch(ca.verify_claim + req, (uint32_t)now) == (uint32_t)now) {
      // the request appears twice in req_ids: only its first claimant commits
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
  // rest of the order followed by the victims in slot order. The order is a
  // ring from lru_head[req]: the victims' ring positions take them back in
  // slot order and the head moves past them (n entries written, not S).
  int32_t *lru = lru_order + sbase;
  const int head = ca.lru_head[req];
  if ((int)threadIdx.x < n) {
    int p = head + (int)threadIdx.x;
    if (p >= S) p -= S;
    chosen[threadIdx.x] = lru[p];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t sorted[HS_MAX_STEP];
    for (int k = 0; k < n; ++k) {               // insertion sort of at most 16 slots
      int32_t v = chosen[k];
      int j = k;
      while (j > 0 && sorted[j - 1] > v) { sorted[j] = sorted[j - 1]; --j; }
      sorted[j] = v;
    }
    for (int k = 0; k < n; ++k) {
      int p = head + k;
      if (p >= S) p -= S;
      lru[p] = sorted[k];
    }
    ca.lru_head[req] = head + n >= S ? head + n - S : head + n;
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


// Block per logits row: its argmax into pred; the request's last row to finish
// (a count per request, put back to 0) then commits the request with the
// whole block.
template <int DTYPE>
__global__ void __launch_bounds__(HS_ARGMAX_THREADS) k_verify(const void *__restrict__ logits,
                                                             int32_t V, int32_t *row_count,
                                                             const __grid_constant__ CommitArgs ca) {
  __shared__ int s_last;
  const int64_t row = blockIdx.x;
  const int rows_per_req = ca.d + 1;
  const int64_t elem = (DTYPE == HS_LOGITS_F32) ? 4 : 2;
  const int32_t best = hs_row_argmax<DTYPE>(
      reinterpret_cast<const char *>(logits) + row * (int64_t)V * elem, V);
  const int b = (int)(row / rows_per_req);
  if (threadIdx.x == 0) {
    ca.pred[(int64_t)b * ca.n_step + row % rows_per_req] = best;
    __threadfence();
    s_last = atomicAdd(&row_count[b], 1) == ca.d;
    if (s_last) {
      __threadfence();   // every row of request b has its pred
      row_count[b] = 0;
    }
  }
  __syncthreads();
  if (s_last) commit_request(b, ca);
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
  CommitArgs ca;
  ca.d = d; ca.drafts = draft_tokens; ca.pred = buf->pred;
  ca.step_kv = reinterpret_cast<const uint4 *>(step_kv); ca.req_ids = req_ids;
  ca.kv_len = kv_len; ca.accept_len = accept_len; ca.next_token = next_token;
  ca.max_reqs = buf->max_reqs; ca.S = buf->S; ca.S_tot = buf->S_tot; ca.n_step = buf->n_step;
  ca.max_ctx = buf->max_ctx; ca.block_size = buf->block_size; ca.hbt_stride = buf->hbt_stride;
  ca.hbt = buf->hbt; ca.pool_rows = buf->host_pool_rows;
  ca.pool = reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(buf->host_pool));
  ca.hot = reinterpret_cast<uint4 *>(buf->hot_kv);
  ca.token_slot = buf->token_slot; ca.slot_token = buf->slot_token; ca.slot_ts = buf->slot_ts;
  ca.lru_order = buf->lru_order; ca.lru_head = buf->lru_head;
  ca.verify_claim = buf->verify_claim; ca.status = buf->status;
  ca.now = buf->clock;
  if (logits_dtype == HS_LOGITS_F32)
    k_verify<HS_LOGITS_F32><<<rows, HS_ARGMAX_THREADS, 0, stream>>>(logits, V, buf->row_count, ca);
  else
    k_verify<HS_LOGITS_BF16><<<rows, HS_ARGMAX_THREADS, 0, stream>>>(logits, V, buf->row_count, ca);
  HS_LAUNCH_CHECK("k_verify");
  return HS_OK;
}
