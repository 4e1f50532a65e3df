// a2-a5: swap-in of host-backed KV into the per-request hot buffer.
//
// "vllm 分析(十二) HiSparse 下篇", HiSparseCacheHandle.resolve_topk: when a
// request is not fully resident, runtime.swap_in takes (request of each row,
// block table, top-k) and returns the hot cache with indices into it.
// "hiSparse-MTP", section 1 and the core state maps: the coordinator keeps a
// device buffer of LRU slots per request, the slot -> position and position ->
// slot maps, and the host pool that holds every position's KV.
//
// Two launches. k_swap_request: one 1024-thread block per request that has
// rows in the call works through that request alone:
//   probe   every entry of the request's rows: classify it and look up its
//           position's slot; a hit sets the slot's flag in shared memory (a
//           plain byte store; distinct hits = flagged slots), a miss claims its
//           position once per call (a shared-memory bitmap of the request's
//           positions, or epoch-stamped marks when it does not fit) and the
//           first claims are compacted with __ballot_sync / __popc into a
//           shared-memory list (one shared atomic per warp and round)
//   assign  the victims are the first slots of the request's
//           LRU order (a persistent array kept in ascending (ts, slot) order,
//           a ring from the request's head: commits rotate it; this kernel
//           writes the new order from position 0)
//           that hold no needed position; the misses, in ascending position
//           order (their ranks in a bitmap of miss positions), take them in
//           order; hits and victims take the current time and move to the end
//           of the order in slot order. Victims and the new order come from
//           warp ballots over the order (held in registers from the start)
//           with one scan of the 32 warp counts -- no sort over all S slots;
//           the count of slots free for victims is also the capacity check
//   publish (host pool row, hot slot) of every miss
// k_swap_gather is a programmatic dependent launch of k_swap_request: its
// blocks take the SMs the metadata kernel leaves free and wait
// (griddepcontrol.wait) until its copy lists are complete.
// k_swap_gather: every SM copies a share of every request's missed 1152-byte
// rows from the device-mapped page-locked host pool with 16-byte loads (four
// in flight per thread): reads over the host link need requests in flight
// from all SMs to reach the link's bandwidth. While those loads are in
// flight, the same threads write the slot table: the hot-row index of every
// entry of every row and the valid count of every row.
// Rows are found by scanning the row descriptors, 1024 rows of the request at
// a time.

#include "hs_internal.cuh"

namespace {

constexpr int SW_THREADS = 1024;
constexpr int ROW_CHUNK = 1024;   // rows of one request handled per pass
constexpr int PB = 8;             // entries per thread per probe / table round

struct SwapArgs {
  const int32_t *req_id, *clen, *kv_len, *topk;
  int32_t R, K;
  int32_t max_reqs, S, S_tot, max_ctx, block_size, hbt_stride;
  const int32_t *hbt;
  int32_t *token_slot, *slot_token;
  int64_t *slot_ts;
  int32_t *lru_order, *lru_head;
  uint32_t *pos_mark;
  uint64_t *copy_desc;
  int32_t *copy_cnt;
  const uint4 *pool;
  int64_t pool_rows;
  uint4 *hot;
  int64_t *stats;
  uint32_t *status;
  uint32_t epoch;
  int64_t now;
  int32_t *req_group;                 // [max_reqs]: group of the request's first row
  int32_t n_groups;
  int32_t group_end[HS_MAX_GROUPS];   // rows [group_end[g-1], group_end[g]) form group g
};

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

__host__ __device__ inline int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Misses are put in ascending position order by rank in a bitmap of the
// request's committed positions (one bit per position, a prefix count per
// 32-bit word) when that fits in shared memory, else by a bitonic sort.
constexpr int RANK_MAX_WORDS = 8192;   // positions < 262144

__host__ __device__ inline int rank_words(int max_ctx) {
  const int w = (max_ctx + 31) / 32;
  return w <= RANK_MAX_WORDS ? w : 0;
}

// Shared-memory layout (bytes): mkey[nS] i32 (misses) | vict[S] i32 (victim
// slots) | hit / touched flags [S] u8, padded to 4 | rows[ROW_CHUNK] i32 |
// miss bitmap [W] u32 | its word prefix counts [W] i32 | needed-position
// bitmap [W] u32 (W = rank_words(max_ctx); with W = 0 the claims go through
// pos_mark and the misses are sorted)
__host__ __device__ inline size_t swap_smem_bytes(int S, int max_ctx) {
  const int nS = pow2_ceil(S);
  return (size_t)nS * 4 + (size_t)S * 4 + (size_t)((S + 3) / 4) * 4 + ROW_CHUNK * 4 +
         (size_t)rank_words(max_ctx) * 12;
}
constexpr int ORD_REGS = HS_MAX_SLOTS / SW_THREADS;   // LRU order entries a thread holds

// Exclusive scan over the block's 32 warps of one count per warp (every lane
// passes its warp's count): the warp's offset, and the total in *total.
// tmp holds 33 ints; every thread calls it.
__device__ __forceinline__ int warp_exscan(int cnt, int *tmp, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) tmp[w] = cnt;
  __syncthreads();
  if (w == 0) {
    const int x = tmp[lane];
    int xi = x;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += y;
    }
    tmp[lane] = xi - x;
    if (lane == 31) tmp[32] = xi;
  }
  __syncthreads();
  const int r = tmp[w];
  *total = tmp[32];
  __syncthreads();
  return r;
}

// Rows of request b among rows [from, R): fills rows[] with up to ROW_CHUNK of
// them (in row order) and returns the count and the next scan position.
__device__ int collect_rows(const SwapArgs &a, int b, int from, int *rows, int *next, int *s_cnt) {
  if (threadIdx.x == 0) *s_cnt = 0;
  __syncthreads();
  int r = from;
  for (; r < a.R; r += SW_THREADS) {
    const int rr = r + (int)threadIdx.x;
    const bool mine = rr < a.R && a.req_id[rr] == b;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    __shared__ int warp_base[SW_THREADS / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane == 0) warp_base[w] = __popc(m);
    __syncthreads();
    // exclusive prefix over warps, in row order (one warp's shuffle scan)
    __shared__ int total;
    if (w == 0) {
      const int x = warp_base[lane];
      int xi = x;
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xi, off);
        if (lane >= off) xi += y;
      }
      warp_base[lane] = *s_cnt + xi - x;
      if (lane == 31) total = *s_cnt + xi;
    }
    __syncthreads();
    if (mine) {
      const int pos = warp_base[w] + __popc(m & ((1u << lane) - 1u));
      if (pos < ROW_CHUNK) rows[pos] = rr;
    }
    __syncthreads();
    const int t = total;
    if (threadIdx.x == 0) *s_cnt = t < ROW_CHUNK ? t : ROW_CHUNK;
    __syncthreads();
    if (t >= ROW_CHUNK) {
      // the chunk is full: resume after the last row placed in it
      r = rows[ROW_CHUNK - 1] + 1;
      *next = r;
      return ROW_CHUNK;
    }
  }
  *next = a.R;
  return *s_cnt;
}

__global__ void __launch_bounds__(SW_THREADS, 1) k_swap_request(SwapArgs a,
                                                                 int32_t *__restrict__ out,
                                                                 int32_t *__restrict__ out_valid) {
  // the gather launched after this kernel may take its SMs now; it reads this
  // kernel's copy lists only after this kernel has finished
  asm volatile("griddepcontrol.launch_dependents;\n");
  extern __shared__ __align__(16) unsigned char smem[];
  const int b = blockIdx.x;
  const int nS = pow2_ceil(a.S);
  int32_t *mkey = reinterpret_cast<int32_t *>(smem);
  int32_t *vict = mkey + nS;
  // hit / touched flag per slot: plain byte stores (every writer stores 1)
  uint8_t *hit = reinterpret_cast<uint8_t *>(vict + a.S);
  int32_t *rows = reinterpret_cast<int32_t *>(hit + (a.S + 3) / 4 * 4);
  const int nW = rank_words(a.max_ctx);
  uint32_t *pbm = reinterpret_cast<uint32_t *>(rows + ROW_CHUNK);
  int32_t *pwp = reinterpret_cast<int32_t *>(pbm + nW);
  uint32_t *pneed = reinterpret_cast<uint32_t *>(pwp + nW);
  __shared__ int s_miss, s_cnt, s_any, s_bad, s_first;
  __shared__ int scan_tmp[33];

  if (threadIdx.x == 0) { s_miss = 0; s_any = 0; s_bad = 0; a.copy_cnt[b] = 0; }
  for (int i = threadIdx.x; i < (a.S + 3) / 4; i += SW_THREADS) reinterpret_cast<uint32_t *>(hit)[i] = 0u;
  __syncthreads();

  const int32_t L = a.kv_len[b];
  const int64_t cbase = (int64_t)b * a.max_ctx;
  const int64_t sbase = (int64_t)b * a.S;
  // the request's LRU order, loaded now (its latency hides behind the probe)
  // in the layout of the victim pass: order position w * CH + 32 j + lane
  // belongs to warp w, round j < NR
  const int lane = threadIdx.x & 31;
  const int CH = ((a.S + 31) / 32 + 31) / 32 * 32;   // order positions per warp
  const int NR = CH / 32;                             // rounds (at most ORD_REGS)
  // (the order is a ring from position lru_head[b]: commits rotate it)
  const int head = a.lru_head[b];
  int32_t ordv[ORD_REGS];
#pragma unroll
  for (int j = 0; j < ORD_REGS; ++j) {
    const int i = (int)(threadIdx.x >> 5) * CH + j * 32 + lane;
    int p = head + i;
    if (p >= a.S) p -= a.S;
    ordv[j] = j < NR && i < a.S ? a.lru_order[sbase + p] : -1;
  }
  // a position is claimed once per call: first setter of its bit in the
  // needed-position bitmap (or of its pos_mark epoch when that does not fit)
  const bool use_bm = nW > 0;
  if (use_bm)
    for (int w = threadIdx.x; w < (L + 31) / 32; w += SW_THREADS) pneed[w] = 0u;
  __syncthreads();

  // ---- probe ----------------------------------------------------------------
  for (int from = 0; from < a.R;) {
    int next;
    const int n = collect_rows(a, b, from, rows, &next, &s_cnt);
    from = next;
    if (n == 0) break;
    if (threadIdx.x == 0) {
      if (!s_any) s_first = rows[0];   // rows come in ascending order
      s_any = 1;
    }
    if (out_valid)   // counted by the gather's table pass
      for (int i = threadIdx.x; i < n; i += SW_THREADS) out_valid[rows[i]] = 0;
    const int items = n * a.K;
    // PB entries per thread per round. Every committed entry looks up its
    // position's slot; a hit marks the slot (distinct hits = marked slots),
    // and only a miss claims its position, so that a position missed by
    // several rows gets one slot. The loads of a round are in flight together.
    // Entry i = r * K + j of the chunk is row rows[r], column j; a thread
    // starts at entry threadIdx.x and steps by SW_THREADS, carrying (r, j)
    // instead of dividing every entry by K.
    int r = 0, j = 0, dq = 0, dr = 0;
    if (items > 0) {
      r = (int)threadIdx.x / a.K;
      j = (int)threadIdx.x % a.K;
      dq = SW_THREADS / a.K;
      dr = SW_THREADS % a.K;
    }
    for (int base = 0; base < items; base += SW_THREADS * PB) {
      int32_t t[PB], clen[PB], sl[PB];
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        t[u] = -1;
        clen[u] = 0;
        if (r < n) {
          const int row = rows[r];
          t[u] = a.topk[(int64_t)row * a.K + j];
          clen[u] = a.clen[row];
        }
        r += dq;
        j += dr;
        if (j >= a.K) {
          j -= a.K;
          ++r;
        }
      }
      bool bad = false;
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        const bool committed = t[u] >= 0 && t[u] < clen[u] && t[u] < L && t[u] < a.max_ctx;
        bad |= t[u] >= 0 && (t[u] >= clen[u] || (t[u] < L && t[u] >= a.max_ctx));
        sl[u] = committed ? a.token_slot[cbase + t[u]] : INT32_MIN;
      }
      unsigned mm[PB];
      int my_total = 0;
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        if (sl[u] >= 0 && sl[u] < a.S) hit[sl[u]] = 1;
        bool first = false;
        if (sl[u] < 0 && sl[u] != INT32_MIN) {      // a committed position not in the buffer
          if (use_bm) {
            const uint32_t bit = 1u << (t[u] & 31);
            first = !(atomicOr(&pneed[t[u] >> 5], bit) & bit);
          } else {
            first = atomicExch(&a.pos_mark[cbase + t[u]], a.epoch) != a.epoch;
          }
        }
        mm[u] = __ballot_sync(0xffffffffu, first);
        my_total += __popc(mm[u]);
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) s_bad = 1;
      if (my_total) {
        int mbase = 0;
        if (lane == 0) mbase = atomicAdd(&s_miss, my_total);
        mbase = __shfl_sync(0xffffffffu, mbase, 0);
#pragma unroll
        for (int u = 0; u < PB; ++u) {
          if ((mm[u] >> lane) & 1u) {
            const int pos = mbase + __popc(mm[u] & ((1u << lane) - 1u));
            if (pos < a.S) mkey[pos] = t[u];   // beyond S the request is refused below
          }
          mbase += __popc(mm[u]);
        }
      }
    }
    __syncthreads();
  }
  __syncthreads();
  if (!s_any) return;                    // no rows of this request in the call
  if (threadIdx.x == 0) {
    if (s_bad) atomicOr(a.status, HS_STATUS_INDEX);
    int g = 0;
    while (g < a.n_groups - 1 && s_first >= a.group_end[g]) ++g;
    a.req_group[b] = g;                  // its misses are copied with group g
  }

  // ---- assign ---------------------------------------------------------------
  // victims: the first nm slots of the LRU order (ascending (ts, slot)) that
  // hold no position needed in this call. Order position i = w * CH + 32 j +
  // lane belongs to warp w, round j (held in ordv since the start); ranks come
  // from warp ballots and one scan of the warp counts, so the writes of a warp
  // are contiguous. The count of such free slots also settles the capacity:
  // the distinct hits are the other S - n_free slots.
  const int nm = s_miss;
  const int w = threadIdx.x >> 5;
  unsigned fm[ORD_REGS];                              // free (not hit) slots, by round
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < ORD_REGS; ++j) {
    const int i = w * CH + j * 32 + lane;
    fm[j] = __ballot_sync(0xffffffffu, j < NR && i < a.S && !hit[ordv[j]]);
    cnt += __popc(fm[j]);
  }
  int n_free;
  int k = warp_exscan(cnt, scan_tmp, &n_free);
  const bool failed = nm > n_free;                    // hits + misses > S
  if (failed) {
    if (threadIdx.x == 0) {
      atomicOr(a.status, HS_STATUS_CAPACITY);
      a.copy_cnt[b] = -1;   // the table gives the request's committed entries -1
    }
  } else {
    if (threadIdx.x == 0 && a.stats) {
      atomicAdd((unsigned long long *)&a.stats[0], (unsigned long long)(a.S - n_free));
      atomicAdd((unsigned long long *)&a.stats[1], (unsigned long long)nm);
    }
    int32_t *lru = a.lru_order + sbase;   // the new order is written from position 0
    if (threadIdx.x == 0) a.lru_head[b] = 0;
    // the first nm free slots become victims (touched from now on); the
    // other free slots keep their order at the front of the new LRU order
#pragma unroll
    for (int j = 0; j < ORD_REGS; ++j) {
      if ((fm[j] >> lane) & 1u) {
        const int r = k + __popc(fm[j] & ((1u << lane) - 1u));
        const int32_t sl = ordv[j];
        if (r < nm) {
          vict[r] = sl;
          hit[sl] = 1;
        } else {
          lru[r - nm] = sl;
        }
      }
      k += __popc(fm[j]);
    }
    __syncthreads();
    // hits and victims take the current time and follow in slot order
    unsigned tm[ORD_REGS];
    int ct = 0;
#pragma unroll
    for (int j = 0; j < ORD_REGS; ++j) {
      const int sl = w * CH + j * 32 + lane;
      tm[j] = __ballot_sync(0xffffffffu, j < NR && sl < a.S && hit[sl]);
      ct += __popc(tm[j]);
    }
    int n_touched;
    k = warp_exscan(ct, scan_tmp, &n_touched) + (n_free - nm);
#pragma unroll
    for (int j = 0; j < ORD_REGS; ++j) {
      if ((tm[j] >> lane) & 1u) {
        const int sl = w * CH + j * 32 + lane;
        lru[k + __popc(tm[j] & ((1u << lane) - 1u))] = sl;
        a.slot_ts[sbase + sl] = a.now;
      }
      k += __popc(tm[j]);
    }
    if (nm > 0) {
      // misses in ascending position order take the victims in order: the
      // i-th smallest miss position gets vict[i]
      const bool by_rank = nW > 0 && L <= nW * 32;
      if (by_rank) {
        const int W = (L + 31) / 32;
        for (int w = threadIdx.x; w < W; w += SW_THREADS) pbm[w] = 0u;
        __syncthreads();
        for (int i = threadIdx.x; i < nm; i += SW_THREADS)
          atomicOr(&pbm[mkey[i] >> 5], 1u << (mkey[i] & 31));
        __syncthreads();
        const int E = (W + SW_THREADS - 1) / SW_THREADS;
        const int lo = threadIdx.x * E, hi = min(W, lo + E);
        int cnt = 0;
        for (int w = lo; w < hi; ++w) cnt += __popc(pbm[w]);
        int tot;
        int k = hs_block_exscan(cnt, scan_tmp, &tot);
        for (int w = lo; w < hi; ++w) { pwp[w] = k; k += __popc(pbm[w]); }
        __syncthreads();
      } else {
        const int nM = pow2_ceil(nm);
        for (int i = nm + threadIdx.x; i < nM; i += SW_THREADS) mkey[i] = INT32_MAX;
        __syncthreads();
        block_bitonic_sort(mkey, nM);
      }
      auto rank_of = [&](int i, int32_t t) -> int {
        return by_rank ? pwp[t >> 5] + __popc(pbm[t >> 5] & ((1u << (t & 31)) - 1u)) : i;
      };
      const int32_t *hbt_row = a.hbt + (int64_t)b * a.hbt_stride;
      uint64_t *desc = a.copy_desc + sbase;
      for (int i = threadIdx.x; i < nm; i += SW_THREADS) {
        const int32_t t = mkey[i];
        const int32_t sl = vict[rank_of(i, t)];
        const int32_t old = a.slot_token[sbase + sl];
        if (old >= 0 && old < a.max_ctx) a.token_slot[cbase + old] = -1;   // not needed now
        a.slot_token[sbase + sl] = t;
        a.token_slot[cbase + t] = sl;
        const int32_t hb = hbt_row[t / a.block_size];
        const int64_t src = (int64_t)hb * a.block_size + t % a.block_size;
        uint64_t copy = ~0ull;
        if (hb >= 0 && src < a.pool_rows)
          copy = ((uint64_t)src << 16) | (uint64_t)sl;   // host row, hot slot
        else
          atomicOr(a.status, HS_STATUS_INDEX);
        desc[i] = copy;
      }
      if (threadIdx.x == 0) a.copy_cnt[b] = nm;      // published for the gather
    }
  }
  __syncthreads();

}

// Arguments of the slot-table pass run inside the gather.
struct TableArgs {
  const int32_t *req_id, *clen, *kv_len, *topk, *token_slot, *copy_cnt;
  int32_t row_lo, n_rows;   // the rows whose entries this launch writes
  int32_t K, max_reqs, S, S_tot, max_ctx;
  int32_t *out, *out_valid;
  uint32_t *status;
};

// Entry e = r * K + j of the slot table: the hot-row index of topk[r][j]
// (-1 for padding, an index error, a refused request or a bad request id).
__device__ __forceinline__ void table_entry(const TableArgs &ta, int64_t e) {
  const int r = (int)(e / ta.K), j = (int)(e - (int64_t)r * ta.K);
  const int32_t b = ta.req_id[r];
  int32_t v = -1;
  if (b < 0 || b >= ta.max_reqs) {
    if (j == 0) {
      if (ta.out_valid) ta.out_valid[r] = 0;
      atomicOr(ta.status, HS_STATUS_INDEX);
    }
  } else {
    const int32_t t = ta.topk[e], n = ta.clen[r], L = ta.kv_len[b];
    if (t >= 0 && t < n) {
      if (t >= L) {
        if (t - L < ta.S_tot - ta.S) v = b * ta.S_tot + ta.S + (t - L);
      } else if (t < ta.max_ctx && ta.copy_cnt[b] >= 0) {
        const int32_t sl = ta.token_slot[(int64_t)b * ta.max_ctx + t];
        if (sl >= 0) v = b * ta.S_tot + sl;
      }
    }
  }
  ta.out[e] = v;
  if (v >= 0 && ta.out_valid) atomicAdd(&ta.out_valid[r], 1);
}

// The copies of the requests of group `group` (req_group, written by
// k_swap_request) and the slot-table entries of rows [row_lo, row_lo + n_rows).
// Chunks of those requests' misses are numbered consecutively (a prefix sum
// over the per-request counts, computed by every block in shared memory) and
// spread over the whole grid, four 16-byte loads in flight per thread; the
// slot table's entries are spread the same way and worked on while the
// loads over the host link are in flight.
__global__ void __launch_bounds__(512) k_swap_gather(const int32_t *__restrict__ copy_cnt,
                                                     const int32_t *__restrict__ req_group,
                                                     int32_t group,
                                                     const uint64_t *__restrict__ copy_desc,
                                                     int32_t max_reqs, int32_t S, int32_t S_tot,
                                                     const uint4 *__restrict__ pool,
                                                     uint4 *__restrict__ hot, TableArgs ta) {
  extern __shared__ int pre[];                     // [max_reqs + 1] chunk offsets
  __shared__ int scan_tmp[33];
  const int tid = threadIdx.x;
  // a programmatic dependent launch of k_swap_request: resident early, it
  // waits here until that kernel has finished and its writes are visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int seg = (max_reqs + (int)blockDim.x - 1) / (int)blockDim.x;
  auto cnt_of = [&](int i) -> int {
    const int c = copy_cnt[i];
    return c > 0 && req_group[i] == group ? c : 0;
  };
  int sum = 0;
  for (int i = tid * seg; i < (tid + 1) * seg && i < max_reqs; ++i) sum += cnt_of(i) * HS_ROW_VEC16;
  {
    int all;
    int acc = hs_block_exscan(sum, scan_tmp, &all);
    for (int i = tid * seg; i < (tid + 1) * seg && i < max_reqs; ++i) {
      pre[i] = acc;
      acc += cnt_of(i) * HS_ROW_VEC16;
    }
    if (tid == 0) pre[max_reqs] = all;
  }
  __syncthreads();
  const int total = pre[max_reqs];
  const int64_t n_entries = (int64_t)ta.n_rows * ta.K, e0 = (int64_t)ta.row_lo * ta.K;
  const int step = gridDim.x * blockDim.x;
  constexpr int TE = 2;                            // table entries per thread per round
  const int g = blockIdx.x * blockDim.x + tid;
  for (int it = 0;; ++it) {
    const int64_t e = (int64_t)g + (int64_t)it * 4 * step;
    const int64_t te = (int64_t)g + (int64_t)it * TE * step;
    if (e >= total && te >= n_entries) break;
    uint4 v[4];
    int64_t dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t k = e + (int64_t)u * step;
      dst[u] = -1;
      if (k < total) {
        int lo = 0, hi = max_reqs;                 // request b with pre[b] <= k < pre[b+1]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (pre[mid] <= k) lo = mid; else hi = mid;
        }
        const int rel = (int)k - pre[lo];
        const int i = rel / HS_ROW_VEC16, c = rel % HS_ROW_VEC16;
        const uint64_t d = copy_desc[(int64_t)lo * S + i];
        if (d != ~0ull) {
          v[u] = pool[(int64_t)(d >> 16) * HS_ROW_VEC16 + c];
          dst[u] = ((int64_t)lo * S_tot + (int64_t)(d & 0xFFFF)) * HS_ROW_VEC16 + c;
        }
      }
    }
    // slot-table entries while the host reads are in flight
#pragma unroll
    for (int u = 0; u < TE; ++u) {
      const int64_t en = te + (int64_t)u * step;
      if (en < n_entries) table_entry(ta, e0 + en);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] >= 0) hot[dst[u]] = v[u];
  }
}

// The follower caches of one hs_swap_apply_plan call.
struct PlanLayers {
  char *hot[HS_MAX_LAYERS];
  const char *pool[HS_MAX_LAYERS];
};

// The leader's latest copy list, repeated for n_layers follower caches: the
// same numbering as k_swap_gather (request, copy, unit of the row), with the
// layer as the outer index. A row is `vec` units of type U (16 or 4 bytes), so
// follower caches may hold rows of another format than the leader's.
template <typename U>
__global__ void __launch_bounds__(256) k_swap_apply(const int32_t *__restrict__ copy_cnt,
                                                    const uint64_t *__restrict__ copy_desc,
                                                    int32_t max_reqs, int32_t S, int32_t S_tot,
                                                    int64_t row_offset, int32_t n_layers,
                                                    int32_t vec,
                                                    const __grid_constant__ PlanLayers pl) {
  extern __shared__ int pre[];                     // [max_reqs + 1] unit offsets
  __shared__ int part[256];
  const int tid = threadIdx.x;
  const int seg = (max_reqs + 255) / 256;
  auto cnt_of = [&](int i) -> int { const int c = copy_cnt[i]; return c > 0 ? c : 0; };
  int sum = 0;
  for (int i = tid * seg; i < (tid + 1) * seg && i < max_reqs; ++i) sum += cnt_of(i) * vec;
  part[tid] = sum;
  __syncthreads();
  if (tid < 32) {
    int v[8], run = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) { v[k] = part[tid * 8 + k]; run += v[k]; }
    int incl = run;
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += o;
    }
    int acc = incl - run;
#pragma unroll
    for (int k = 0; k < 8; ++k) { part[tid * 8 + k] = acc; acc += v[k]; }
  }
  __syncthreads();
  {
    int acc = part[tid];
    for (int i = tid * seg; i < (tid + 1) * seg && i < max_reqs; ++i) {
      pre[i] = acc;
      acc += cnt_of(i) * vec;
    }
    if (tid == 255) pre[max_reqs] = acc;
  }
  __syncthreads();
  const int64_t per_layer = pre[max_reqs];
  const int64_t total = per_layer * n_layers;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + tid; e < total; e += 4 * step) {
    U v[4];
    U *dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t k = e + u * step;
      dst[u] = nullptr;
      if (k < total) {
        const int l = (int)(k / per_layer);
        const int kk = (int)(k - (int64_t)l * per_layer);
        int lo = 0, hi = max_reqs;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (pre[mid] <= kk) lo = mid; else hi = mid;
        }
        const int rel = kk - pre[lo];
        const int i = rel / vec, c = rel - i * vec;
        const uint64_t d = copy_desc[(int64_t)lo * S + i];
        if (d != ~0ull) {
          v[u] = reinterpret_cast<const U *>(pl.pool[l])[(int64_t)(d >> 16) * vec + c];
          dst[u] = reinterpret_cast<U *>(pl.hot[l]) +
                   (row_offset + (int64_t)lo * S_tot + (int64_t)(d & 0xFFFF)) * vec + c;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u]) *dst[u] = v[u];
  }
}

}  // namespace

int hs_swap_plan_launch(hs_buffer *buf, const int32_t *req_id_per_row,
                        const int32_t *row_causal_len, const int32_t *kv_len, const int32_t *topk,
                        int32_t R, int32_t K, int32_t n_groups, const int32_t *group_end,
                        int32_t *out_slot_idx, int32_t *out_valid, int64_t *stats,
                        cudaStream_t stream) {
  SwapArgs a;
  a.req_id = req_id_per_row; a.clen = row_causal_len; a.kv_len = kv_len; a.topk = topk;
  a.R = R; a.K = K;
  a.max_reqs = buf->max_reqs; a.S = buf->S; a.S_tot = buf->S_tot; a.max_ctx = buf->max_ctx;
  a.block_size = buf->block_size; a.hbt_stride = buf->hbt_stride; a.hbt = buf->hbt;
  a.token_slot = buf->token_slot; a.slot_token = buf->slot_token; a.slot_ts = buf->slot_ts;
  a.lru_order = buf->lru_order;
  a.lru_head = buf->lru_head;
  a.pos_mark = buf->pos_mark;
  a.copy_desc = buf->copy_desc;
  a.copy_cnt = buf->copy_cnt;
  a.pool = reinterpret_cast<const uint4 *>(buf->host_pool);
  a.pool_rows = buf->host_pool_rows;
  a.hot = reinterpret_cast<uint4 *>(buf->hot_kv);
  a.stats = stats; a.status = buf->status;
  a.epoch = (uint32_t)buf->clock;
  a.now = buf->clock;
  a.req_group = buf->req_group;
  a.n_groups = n_groups;
  for (int g = 0; g < HS_MAX_GROUPS; ++g) a.group_end[g] = g < n_groups ? group_end[g] : R;

  const size_t smem = swap_smem_bytes(buf->S, buf->max_ctx);
  static bool attr_set[64] = {false};
  if (buf->device >= 64 || !attr_set[buf->device]) {
    HS_CUDA_TRY(cudaFuncSetAttribute(k_swap_request, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)swap_smem_bytes(HS_MAX_SLOTS, RANK_MAX_WORDS * 32)));
    HS_CUDA_TRY(cudaFuncSetAttribute(k_swap_gather, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)((HS_MAX_REQS + 1) * sizeof(int))));
    // the gather takes an SM's leftover beside an attention CTA (one CTA of
    // the attention kernel leaves a few KB of shared memory), so it asks for
    // the same shared-memory carve-out as the attention
    HS_CUDA_TRY(cudaFuncSetAttribute(k_swap_gather, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared));
    if (buf->device < 64) attr_set[buf->device] = true;
  }
  k_swap_request<<<buf->max_reqs, SW_THREADS, smem, stream>>>(a, out_slot_idx, out_valid);
  HS_LAUNCH_CHECK("k_swap_request");
  return HS_OK;
}

int hs_gather_func_attrs(cudaFuncAttributes *attr) {
  HS_CUDA_TRY(cudaFuncGetAttributes(attr, k_swap_gather));
  return HS_OK;
}

int hs_swap_gather_launch(hs_buffer *buf, const int32_t *req_id_per_row,
                          const int32_t *row_causal_len, const int32_t *kv_len,
                          const int32_t *topk, int32_t R, int32_t K, int32_t g, int32_t row_lo,
                          int32_t row_hi, int32_t *out_slot_idx, int32_t *out_valid,
                          int ctas_per_sm, int threads, bool pdl, cudaStream_t stream) {
  static int sms[64] = {0};
  int nsm = (buf->device < 64) ? sms[buf->device] : 0;
  if (nsm == 0) {
    HS_CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, buf->device));
    if (buf->device < 64) sms[buf->device] = nsm;
  }
  (void)R;
  TableArgs ta;
  ta.req_id = req_id_per_row; ta.clen = row_causal_len; ta.kv_len = kv_len; ta.topk = topk;
  ta.token_slot = buf->token_slot; ta.copy_cnt = buf->copy_cnt;
  ta.row_lo = row_lo; ta.n_rows = row_hi - row_lo;
  ta.K = K; ta.max_reqs = buf->max_reqs; ta.S = buf->S; ta.S_tot = buf->S_tot;
  ta.max_ctx = buf->max_ctx;
  ta.out = out_slot_idx; ta.out_valid = out_valid; ta.status = buf->status;
  const size_t gsmem = (size_t)(buf->max_reqs + 1) * sizeof(int);
  if (buf->copy_sms > 0 && buf->copy_sms < nsm) nsm = buf->copy_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nsm * ctas_per_sm));
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = gsmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const uint4 *pool = reinterpret_cast<const uint4 *>(buf->host_pool);
  uint4 *hot = reinterpret_cast<uint4 *>(buf->hot_kv);
  HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_swap_gather, (const int32_t *)buf->copy_cnt,
                                 (const int32_t *)buf->req_group, g,
                                 (const uint64_t *)buf->copy_desc, (int32_t)buf->max_reqs,
                                 (int32_t)buf->S, (int32_t)buf->S_tot, pool, hot, ta));
  HS_LAUNCH_CHECK("k_swap_gather");
  return HS_OK;
}

extern "C" int hs_swap_in(hs_buffer *buf, const int32_t *req_id_per_row,
                          const int32_t *row_causal_len, const int32_t *kv_len,
                          const int32_t *topk, int32_t R, int32_t K, int32_t *out_slot_idx,
                          int32_t *out_valid, int64_t *stats, hs_stream_t stream) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (R < 0 || K < 0 || K > (1 << 20))
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes R=%d K=%d (0..2^20)", R, K);
  if (R > 0 && (!req_id_per_row || !row_causal_len || !kv_len))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL row descriptor");
  if (R > 0 && K > 0 && (!topk || !out_slot_idx))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL topk or out_slot_idx");

  buf->clock += 1;  // the LRU clock advances once per call, even an empty one
  if (R == 0) return HS_OK;
  const int32_t end = R;
  rc = hs_swap_plan_launch(buf, req_id_per_row, row_causal_len, kv_len, topk, R, K, 1, &end,
                           out_slot_idx, out_valid, stats, stream);
  if (rc) return rc;
  // a programmatic dependent launch of k_swap_request: its blocks take the
  // SMs the metadata kernel leaves free and wait until its copy lists are
  // complete
  return hs_swap_gather_launch(buf, req_id_per_row, row_causal_len, kv_len, topk, R, K, 0, 0, R,
                               out_slot_idx, out_valid, 8, 256, true, stream);
}

extern "C" int hs_swap_apply_plan(hs_buffer *buf, int32_t n_layers, void *const *hot_kv,
                                  const void *const *host_pools, int64_t row_offset,
                                  int32_t row_bytes, hs_stream_t stream) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (n_layers < 0 || n_layers > HS_MAX_LAYERS)
    return hs_set_error(HS_ERR_INVALID_ARG, "n_layers %d not in 0..%d", n_layers, HS_MAX_LAYERS);
  if (row_offset < 0) return hs_set_error(HS_ERR_INVALID_ARG, "negative row_offset");
  if (row_bytes < 4 || row_bytes % 4 || row_bytes > (1 << 20))
    return hs_set_error(HS_ERR_INVALID_ARG, "row_bytes %d must be a multiple of 4 in 4..2^20",
                        row_bytes);
  if (n_layers == 0) return HS_OK;
  if (!hot_kv || !host_pools) return hs_set_error(HS_ERR_INVALID_ARG, "NULL layer arrays");
  PlanLayers pl;
  bool wide = row_bytes % 16 == 0;
  for (int l = 0; l < n_layers; ++l) {
    const void *h = nullptr, *p = nullptr;
    if (!hot_kv[l] || !host_pools[l] || ((uintptr_t)hot_kv[l] & 3) || ((uintptr_t)host_pools[l] & 3))
      return hs_set_error(HS_ERR_INVALID_ARG, "hot_kv[%d] / host_pools[%d] NULL or not 4-byte aligned", l, l);
    if (((uintptr_t)hot_kv[l] & 15) || ((uintptr_t)host_pools[l] & 15)) wide = false;
    if ((rc = hs_device_alias(hot_kv[l], &h, "hot_kv[l]", 4))) return rc;
    if ((rc = hs_device_alias(host_pools[l], &p, "host_pools[l]", 4))) return rc;
    pl.hot[l] = reinterpret_cast<char *>(const_cast<void *>(h));
    pl.pool[l] = reinterpret_cast<const char *>(p);
  }
  const int vec = wide ? row_bytes / 16 : row_bytes / 4;
  if ((int64_t)buf->max_reqs * buf->S * vec > INT32_MAX)
    return hs_set_error(HS_ERR_UNSUPPORTED, "max_reqs * slots_per_req * row units exceeds int32");
  static bool attr_set[2][64] = {{false}};
  if (buf->device >= 64 || !attr_set[wide][buf->device]) {
    HS_CUDA_TRY(cudaFuncSetAttribute(wide ? k_swap_apply<uint4> : k_swap_apply<uint32_t>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)((HS_MAX_REQS + 1) * sizeof(int))));
    if (buf->device < 64) attr_set[wide][buf->device] = true;
  }
  int nsm = 0;
  HS_CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, buf->device));
  if (buf->copy_sms > 0 && buf->copy_sms < nsm) nsm = buf->copy_sms;
  const size_t gsmem = (size_t)(buf->max_reqs + 1) * sizeof(int);
  if (wide)
    k_swap_apply<uint4><<<nsm * 8, 256, gsmem, stream>>>(buf->copy_cnt, buf->copy_desc,
                                                         buf->max_reqs, buf->S, buf->S_tot,
                                                         row_offset, n_layers, vec, pl);
  else
    k_swap_apply<uint32_t><<<nsm * 8, 256, gsmem, stream>>>(buf->copy_cnt, buf->copy_desc,
                                                            buf->max_reqs, buf->S, buf->S_tot,
                                                            row_offset, n_layers, vec, pl);
  HS_LAUNCH_CHECK("k_swap_apply");
  return HS_OK;
}
