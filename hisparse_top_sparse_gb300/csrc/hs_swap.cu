// a2-a5: swap-in of host-backed KV into the per-request hot buffer.
//
// "vllm 分析(十二) HiSparse 下篇", HiSparseCacheHandle.resolve_topk: when a
// request is not fully resident, runtime.swap_in takes (request of each row,
// block table, top-k) and returns the hot cache with indices into it.
// "hiSparse-MTP", section 1 and the core state maps: the coordinator keeps a
// device buffer of LRU slots per request, the slot -> position and position ->
// slot maps, and the host pool that holds every position's KV.
//
// One call = five launches on the caller's stream:
//   k_swap_begin   zero the per-request need/miss counters and the copy count
//   k_swap_probe   warp per 32 entries of a row: classify, claim each needed
//                  position once per call (epoch-stamped marks), mark hit slots,
//                  compact misses with __ballot_sync / __popc into a per-request
//                  list
//   k_swap_assign  block per request: capacity check, hit timestamps, sort the
//                  misses ascending and the unneeded slots by (ts, slot) in
//                  shared memory (bitonic), pair them in order, update the maps
//                  and emit (host row, hot row) copy descriptors
//   k_swap_gather  copy every missed 1152-byte row from the device-mapped
//                  page-locked host pool with 16-byte loads and stores
//   k_swap_table   block per row: the hot-row index table and valid counts

#include "hs_internal.cuh"

namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void k_swap_begin(int32_t *counters, int32_t n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    counters[i] = 0;
}

struct SwapArgs {
  const int32_t *req_id, *clen, *kv_len, *topk;
  int32_t R, K;
  int32_t max_reqs, S, S_tot, max_ctx, block_size, hbt_stride;
  const int32_t *hbt;
  int32_t *token_slot, *slot_token;
  int64_t *slot_ts;
  uint32_t *pos_mark, *slot_mark, *req_mark, *fail_mark;
  int32_t *need_cnt, *miss_cnt, *copy_cnt;
  int32_t *miss_list;
  int64_t *copy_src;
  int32_t *copy_dst;
  int64_t *stats;
  uint32_t *status;
  uint32_t epoch;
  int64_t now;
};

__global__ void __launch_bounds__(kWarpsPerBlock * 32) k_swap_probe(SwapArgs a) {
  const int lane = threadIdx.x & 31;
  const int chunks = (a.K + 31) / 32;
  const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (gw >= (int64_t)a.R * chunks) return;
  const int r = (int)(gw / chunks);
  const int j = (int)(gw % chunks) * 32 + lane;
  const int32_t b = a.req_id[r];
  if (b < 0 || b >= a.max_reqs) {
    if (lane == 0) atomicOr(a.status, HS_STATUS_INDEX);
    return;
  }
  const int32_t n = a.clen[r];
  const int32_t L = a.kv_len[b];
  const int32_t t = (j < a.K) ? a.topk[(int64_t)r * a.K + j] : -1;
  const bool in_range = t >= 0 && t < n;
  const bool bad = (t >= 0 && t >= n) || (t >= 0 && t < L && t >= a.max_ctx);
  if (__ballot_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, HS_STATUS_INDEX);
  if (lane == 0) a.req_mark[b] = a.epoch;
  const bool committed = in_range && t < L && t < a.max_ctx;

  // claim: the first thread to stamp a position in this call owns it
  bool first = false;
  int32_t s = -1;
  if (committed) {
    const uint32_t old = atomicExch(&a.pos_mark[(int64_t)b * a.max_ctx + t], a.epoch);
    first = (old != a.epoch);
    if (first) {
      s = a.token_slot[(int64_t)b * a.max_ctx + t];
      if (s >= 0) a.slot_mark[(int64_t)b * a.S + s] = a.epoch;   // hit: protect slot
    }
  }
  const unsigned first_mask = __ballot_sync(0xffffffffu, first);
  const bool miss = first && s < 0;
  const unsigned miss_mask = __ballot_sync(0xffffffffu, miss);
  int base = 0;
  if (lane == 0) {
    if (first_mask) atomicAdd(&a.need_cnt[b], __popc(first_mask));
    if (miss_mask) base = atomicAdd(&a.miss_cnt[b], __popc(miss_mask));
  }
  base = __shfl_sync(0xffffffffu, base, 0);
  if (miss) {
    const int pos = base + __popc(miss_mask & ((1u << lane) - 1u));
    if (pos < a.S) a.miss_list[(int64_t)b * a.S + pos] = t;   // beyond S: overflow, refused later
  }
}

// In-place ascending bitonic sort of n (a power of two) keys in shared memory.
template <typename T>
__device__ void block_bitonic_sort(T *keys, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const T x = keys[i], y = keys[ixj];
          const bool up = (i & k) == 0;
          if ((x > y) == up) { keys[i] = y; keys[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Victim key: (ts + 1) in the high bits, slot in the low 16; needed slots sort last.
__global__ void __launch_bounds__(1024) k_swap_assign(SwapArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int b = blockIdx.x;
  if (a.req_mark[b] != a.epoch) return;
  const int need = a.need_cnt[b];
  const int nm = a.miss_cnt[b];
  const int64_t sbase = (int64_t)b * a.S;
  if (need > a.S) {  // refused: nothing about this request changes
    if (threadIdx.x == 0) {
      atomicOr(a.status, HS_STATUS_CAPACITY);
      a.fail_mark[b] = a.epoch;
    }
    return;
  }
  if (threadIdx.x == 0 && a.stats) {
    atomicAdd((unsigned long long *)&a.stats[0], (unsigned long long)(need - nm));
    atomicAdd((unsigned long long *)&a.stats[1], (unsigned long long)nm);
  }
  // hits take the current time
  for (int s = threadIdx.x; s < a.S; s += blockDim.x)
    if (a.slot_mark[sbase + s] == a.epoch) a.slot_ts[sbase + s] = a.now;
  if (nm == 0) return;

  const int nS = pow2_ceil(a.S);
  const int nM = pow2_ceil(nm);
  uint64_t *vkey = reinterpret_cast<uint64_t *>(smem);
  int32_t *mkey = reinterpret_cast<int32_t *>(smem + (size_t)nS * sizeof(uint64_t));
  __shared__ int copy_base;
  for (int s = threadIdx.x; s < nS; s += blockDim.x) {
    uint64_t key = ~0ull;
    if (s < a.S && a.slot_mark[sbase + s] != a.epoch)
      key = ((uint64_t)(a.slot_ts[sbase + s] + 1) << 16) | (uint64_t)s;
    vkey[s] = key;
  }
  for (int i = threadIdx.x; i < nM; i += blockDim.x)
    mkey[i] = (i < nm) ? a.miss_list[sbase + i] : INT32_MAX;
  if (threadIdx.x == 0) copy_base = atomicAdd(a.copy_cnt, nm);
  __syncthreads();
  block_bitonic_sort(mkey, nM);
  block_bitonic_sort(vkey, nS);

  const int64_t cbase = (int64_t)b * a.max_ctx;
  const int32_t *hbt_row = a.hbt + (int64_t)b * a.hbt_stride;
  for (int i = threadIdx.x; i < nm; i += blockDim.x) {
    const int32_t t = mkey[i];
    if (vkey[i] == ~0ull) {   // fewer victims than misses: the maps are inconsistent
      atomicOr(a.status, HS_STATUS_CAPACITY);
      a.copy_src[copy_base + i] = -1;
      a.copy_dst[copy_base + i] = 0;
      continue;
    }
    const int32_t s = (int32_t)(vkey[i] & 0xFFFF);
    const int32_t old = a.slot_token[sbase + s];
    if (old >= 0 && old < a.max_ctx) a.token_slot[cbase + old] = -1;   // not needed now
    a.slot_token[sbase + s] = t;
    a.token_slot[cbase + t] = s;
    a.slot_ts[sbase + s] = a.now;
    const int32_t hb = hbt_row[t / a.block_size];
    int64_t src = -1;
    if (hb >= 0) src = (int64_t)hb * a.block_size + t % a.block_size;
    else atomicOr(a.status, HS_STATUS_INDEX);
    a.copy_src[copy_base + i] = src;
    a.copy_dst[copy_base + i] = b * a.S_tot + s;
  }
}

// Flattened (copy, 16-byte chunk) space; four independent 16-byte loads in
// flight per thread per iteration to cover the host-link latency.
__global__ void __launch_bounds__(256) k_swap_gather(const int32_t *__restrict__ copy_cnt,
                                                     const int64_t *__restrict__ copy_src,
                                                     const int32_t *__restrict__ copy_dst,
                                                     const uint4 *__restrict__ pool,
                                                     int64_t pool_rows, uint4 *__restrict__ hot,
                                                     uint32_t *status) {
  const int64_t total = (int64_t)(*copy_cnt) * HS_ROW_VEC16;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  constexpr int U = 4;
  for (; i < total; i += U * step) {
    uint4 v[U];
    int64_t dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * step;
      dst[u] = -1;
      if (k < total) {
        const int64_t e = k / HS_ROW_VEC16;
        const int c = (int)(k - e * HS_ROW_VEC16);
        const int64_t src = copy_src[e];
        if (src >= 0 && src < pool_rows) {
          v[u] = pool[src * HS_ROW_VEC16 + c];
          dst[u] = (int64_t)copy_dst[e] * HS_ROW_VEC16 + c;
        } else if (c == 0) {
          atomicOr(status, HS_STATUS_INDEX);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] >= 0) hot[dst[u]] = v[u];
  }
}

__global__ void __launch_bounds__(256) k_swap_table(SwapArgs a, int32_t *__restrict__ out,
                                                    int32_t *__restrict__ out_valid) {
  const int r = blockIdx.x;
  const int32_t b = a.req_id[r];
  int32_t *o = out + (int64_t)r * a.K;
  const int32_t *tk = a.topk + (int64_t)r * a.K;
  int cnt = 0;
  if (b < 0 || b >= a.max_reqs) {
    for (int j = threadIdx.x; j < a.K; j += blockDim.x) o[j] = -1;
  } else {
    const int32_t n = a.clen[r];
    const int32_t L = a.kv_len[b];
    const bool failed = a.fail_mark[b] == a.epoch;
    const int32_t row0 = b * a.S_tot;
    const int32_t *ts_row = a.token_slot + (int64_t)b * a.max_ctx;
    for (int j = threadIdx.x; j < a.K; j += blockDim.x) {
      const int32_t t = tk[j];
      int32_t v = -1;
      if (t >= 0 && t < n) {
        if (t >= L) {
          if (t - L < a.S_tot - a.S) v = row0 + a.S + (t - L);
        } else if (!failed && t < a.max_ctx) {
          const int32_t s = ts_row[t];
          if (s >= 0) v = row0 + s;
        }
      }
      cnt += (v >= 0);
      o[j] = v;
    }
  }
  if (out_valid) {
    __shared__ int ws[8];
    for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = 0;
      for (int w = 0; w < 8; ++w) s += ws[w];
      out_valid[r] = s;
    }
  }
}

}  // namespace

extern "C" int hs_swap_in(hs_buffer *buf, const int32_t *req_id_per_row,
                          const int32_t *row_causal_len, const int32_t *kv_len,
                          const int32_t *topk, int32_t R, int32_t K, int32_t *out_slot_idx,
                          int32_t *out_valid, int64_t *stats, hs_stream_t stream) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (R < 0 || K < 0) return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes R=%d K=%d", R, K);
  if (R > 0 && (!req_id_per_row || !row_causal_len || !kv_len))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL row descriptor");
  if (R > 0 && K > 0 && (!topk || !out_slot_idx))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL topk or out_slot_idx");

  buf->clock += 1;  // the LRU clock advances once per call, even an empty one
  if (R == 0) return HS_OK;

  SwapArgs a;
  a.req_id = req_id_per_row; a.clen = row_causal_len; a.kv_len = kv_len; a.topk = topk;
  a.R = R; a.K = K;
  a.max_reqs = buf->max_reqs; a.S = buf->S; a.S_tot = buf->S_tot; a.max_ctx = buf->max_ctx;
  a.block_size = buf->block_size; a.hbt_stride = buf->hbt_stride; a.hbt = buf->hbt;
  a.token_slot = buf->token_slot; a.slot_token = buf->slot_token; a.slot_ts = buf->slot_ts;
  a.pos_mark = buf->pos_mark; a.slot_mark = buf->slot_mark; a.req_mark = buf->req_mark;
  a.fail_mark = buf->fail_mark;
  a.need_cnt = buf->counters; a.miss_cnt = buf->counters + buf->max_reqs;
  a.copy_cnt = buf->counters + 2 * buf->max_reqs;
  a.miss_list = buf->miss_list; a.copy_src = buf->copy_src; a.copy_dst = buf->copy_dst;
  a.stats = stats; a.status = buf->status;
  a.epoch = (uint32_t)buf->clock;
  a.now = buf->clock;

  const int ncnt = 2 * buf->max_reqs + 1;
  k_swap_begin<<<(ncnt + 255) / 256, 256, 0, stream>>>(buf->counters, ncnt);
  HS_LAUNCH_CHECK("k_swap_begin");
  if (K > 0) {
    const int64_t warps = (int64_t)R * ((K + 31) / 32);
    const int64_t blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > INT32_MAX) return hs_set_error(HS_ERR_UNSUPPORTED, "R*K too large");
    k_swap_probe<<<(int)blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
    HS_LAUNCH_CHECK("k_swap_probe");
  }
  int nS = 1;
  while (nS < buf->S) nS <<= 1;
  const size_t smem = (size_t)nS * 8 + (size_t)nS * 4;
  static bool attr_set[64] = {false};
  if (buf->device >= 64 || !attr_set[buf->device]) {   // the kernel also has static SMEM
    HS_CUDA_TRY(cudaFuncSetAttribute(k_swap_assign, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(HS_MAX_SLOTS * 12)));
    if (buf->device < 64) attr_set[buf->device] = true;
  }
  k_swap_assign<<<buf->max_reqs, 1024, smem, stream>>>(a);
  HS_LAUNCH_CHECK("k_swap_assign");
  int dev_sms = 152;
  cudaDeviceGetAttribute(&dev_sms, cudaDevAttrMultiProcessorCount, buf->device);
  k_swap_gather<<<dev_sms * 8, 256, 0, stream>>>(
      a.copy_cnt, buf->copy_src, buf->copy_dst, reinterpret_cast<const uint4 *>(buf->host_pool),
      buf->host_pool_rows, reinterpret_cast<uint4 *>(buf->hot_kv), buf->status);
  HS_LAUNCH_CHECK("k_swap_gather");
  if (K > 0) {
    k_swap_table<<<R, 256, 0, stream>>>(a, out_slot_idx, out_valid);
    HS_LAUNCH_CHECK("k_swap_table");
  } else if (out_valid) {
    HS_CUDA_TRY(cudaMemsetAsync(out_valid, 0, (size_t)R * 4, stream));
  }
  return HS_OK;
}
