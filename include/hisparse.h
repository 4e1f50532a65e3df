/*
 * hisparse.h -- C ABI of libhisparse: the decode-step hot path of HiSparse-style
 * hierarchical top-k sparse attention with MTP speculative decoding, for one
 * NVIDIA GB300 (sm_103a).
 *
 * Sources (pages of the hisparse_top_sparse material):
 *   [MTP]  "hiSparse-MTP" (Notion): section 1 (HiSparseCoordinator holds the
 *          device buffer, the host pool, LRU slots, token metadata and an async
 *          stream) and the core state maps (request -> slots, slot -> token
 *          position, position -> host KV location, logical position -> slot).
 *   [KVF]  "投机解码的 KV 流转：prefill 阶段 DFlash 也要吃下整个 prompt"
 *          (shenshijiu.com): sections ④-⑥ and the closing table (greedy verify,
 *          which positions keep target KV, where the next anchor sits).
 *   [VLLM] "vllm 分析(十二) HiSparse 下篇" (devpress.csdn.net): sections
 *          HiSparseCacheHandle.resolve_topk (fully-resident index conversion
 *          versus swap-in) and "数据 back up" (paged host-row arithmetic).
 *
 * Conventions shared by every call
 *   - Every call returns an int status: HS_OK (0) or a negative HS_ERR_* code.
 *     Argument errors are detected on the host and returned at once, with
 *     nothing enqueued; hs_last_error_string() then describes them.
 *   - Every call that takes a stream is asynchronous on that stream (a
 *     cudaStream_t; NULL is the legacy default stream) and only enqueues
 *     kernels. Data errors found on the device (a position beyond a row's
 *     causal length, a request that needs more positions than it has slots)
 *     set bits of a device status word: the buffer's, read with
 *     hs_get_status(), or the caller's word for hs_resolve_topk.
 *   - Pointers named "device" must be device memory (or memory the device can
 *     address) of the current CUDA device. The caller owns every tensor: q,
 *     KV caches, index tables, outputs, logits, the hot KV storage, the pinned
 *     host pool and the block tables. The library owns only the hs_buffer's
 *     metadata (slot maps, timestamps, scratch) which hs_buffer_create
 *     allocates and hs_buffer_destroy frees. No other call allocates.
 *   - bf16 tensors are raw IEEE bfloat16 (uint16) arrays.
 *   - Calls on one hs_buffer must be ordered (one stream, or streams joined
 *     by events): they read and update its slot maps.
 */
#ifndef HISPARSE_H_
#define HISPARSE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *hs_stream_t;

/* Opaque hot-buffer object. */
typedef struct hs_buffer hs_buffer;

enum hs_status_code {
  HS_OK = 0,
  HS_ERR_INVALID_ARG = -1, /* bad pointer, size, alignment or device        */
  HS_ERR_CAPACITY = -2,    /* hs_get_status: a request overflowed its slots */
  HS_ERR_INDEX = -3,       /* hs_get_status: a position was out of range    */
  HS_ERR_CUDA = -4,        /* a CUDA runtime call or a launch failed        */
  HS_ERR_TIMEOUT = -5,     /* reserved: a bounded device wait gave up       */
  HS_ERR_UNSUPPORTED = -6  /* a shape the kernels do not handle             */
};

/* Bits of the device status word. */
#define HS_STATUS_INDEX 1u    /* a top-k position >= the row's causal length,
                                 a negative block-table entry, or a request id
                                 outside the buffer                          */
#define HS_STATUS_CAPACITY 2u /* a request needed more than S positions in one
                                 swap-in, or a commit would pass max_ctx      */
#define HS_STATUS_TIMEOUT 4u  /* a bounded wait inside a kernel gave up (the
                                 kernel wound down; its outputs are invalid) */

#define HS_LATENT_DIM 576 /* q and latent KV row: 512 value dims + 64 rope */
#define HS_VALUE_DIM 512  /* attention values are dims 0..511 of a row     */

#define HS_LOGITS_F32 0
#define HS_LOGITS_BF16 1

/* ------------------------------------------------------------------------ */
/* Hot buffer ([MTP] section 1 and core state maps; [VLLM] HiSparseHotSpec)  */
/* ------------------------------------------------------------------------ */

/*
 * Description of a hot buffer. Request b owns hot rows
 *   b * (slots_per_req + step_slots) + s,
 * where s < slots_per_req are LRU slots and the next step_slots rows hold the
 * KV of the step's own positions kv_len[b] .. kv_len[b] + step_slots - 1
 * (anchor + drafts), which the caller writes before hs_swap_in (they are
 * always hits and never evicted).
 *
 *   max_reqs          number of requests the buffer serves (ids 0..max_reqs-1),
 *                     1 .. 16384
 *   slots_per_req     S, LRU slots per request, 1 .. 8192
 *   step_slots        rows per request per decode step (1 anchor + d drafts),
 *                     1 .. 16; a verify with d drafts needs d + 1 <= step_slots
 *                     (the draft count may not pass this "extra page" space)
 *   max_ctx           positions per request covered by the maps and by the
 *                     host block table (committed KV length never passes it)
 *   block_size        positions per host block (>= 1)
 *   hbt_stride        int32 entries per row of host_block_table
 *                     (>= ceil(max_ctx / block_size))
 *   hot_kv            device bf16 [max_reqs * (S + step_slots)][576]; caller-owned
 *   host_pool         bf16 [host_pool_rows][576] in page-locked host memory the
 *                     device can map (cudaHostAlloc / cudaHostRegister), or in
 *                     device memory; caller-owned
 *   host_pool_rows    rows of host_pool
 *   host_block_table  device int32 [max_reqs][hbt_stride]: the host block that
 *                     holds positions [k*block_size, (k+1)*block_size) of a
 *                     request; the row of position t is
 *                     hbt[b][t / block_size] * block_size + t % block_size
 *                     ([VLLM] 数据 back up, one host page per block)
 */
typedef struct hs_buffer_desc {
  int32_t max_reqs;
  int32_t slots_per_req;
  int32_t step_slots;
  int32_t max_ctx;
  int32_t block_size;
  int32_t hbt_stride;
  void *hot_kv;
  void *host_pool;
  int64_t host_pool_rows;
  const int32_t *host_block_table;
} hs_buffer_desc;

/* Validates desc and allocates the buffer's metadata on the current device:
 * token->slot map [max_reqs][max_ctx], slot->token map and timestamps
 * [max_reqs][S], and per-call scratch; all slots start empty. On success
 * *out receives the buffer. The call synchronises the device. */
int hs_buffer_create(const hs_buffer_desc *desc, hs_buffer **out);

/* Frees the metadata (not the caller's tensors). NULL is accepted. */
int hs_buffer_destroy(hs_buffer *buf);

/* Empties every LRU slot of request req (the state a request has when it is
 * admitted to the decode batch, [MTP] section 3 collect_ready_reqs). */
int hs_request_reset(hs_buffer *buf, int32_t req, hs_stream_t stream);

/* Synchronises stream, returns the buffer's device status bits in *out_bits
 * (HS_STATUS_*) and clears them. */
int hs_get_status(hs_buffer *buf, hs_stream_t stream, uint32_t *out_bits);

/* Copies the buffer's maps to host memory after synchronising stream, for
 * tests and debugging: token_slot int32 [max_reqs][max_ctx], slot_token int32
 * [max_reqs][S], slot_ts int64 [max_reqs][S]; any pointer may be NULL. */
int hs_buffer_dump(hs_buffer *buf, hs_stream_t stream, int32_t *token_slot,
                   int32_t *slot_token, int64_t *slot_ts);

/* Number of swap-in and commit calls made so far (the LRU clock). */
int64_t hs_buffer_clock(const hs_buffer *buf);

/* Limits the copy kernels of hs_swap_in and hs_swap_apply_plan on this
 * buffer to about n_sms SMs' worth of blocks (0, the default: every SM). The
 * host link saturates well before every SM is busy, so a caller that overlaps
 * a swap-in with attention on another stream can leave most SMs to the
 * attention. Takes effect from the next call; n_sms >= 0. */
int hs_buffer_set_copy_sms(hs_buffer *buf, int32_t n_sms);

/* Text of the last error returned on this thread. */
const char *hs_last_error_string(void);

/* ------------------------------------------------------------------------ */
/* a1: fully-resident index conversion ([VLLM] resolve_topk, fully_resident  */
/*     branch: request of the row + block table + top-k -> physical rows)     */
/* ------------------------------------------------------------------------ */

/*
 *   req_id_per_row   device int32 [R]: request (block-table row) of each query row
 *   row_causal_len   device int32 [R]: positions a row may attend (L_b + i + 1
 *                    for row i of request b)
 *   block_table      device int32 [*][bt_stride]: physical block of each
 *                    logical block of a request
 *   topk             device int32 [R][K]: logical positions; < 0 is padding
 *   block_size       positions per logical block
 *   phys_block_stride rows between consecutive physical blocks of the cache
 *   out_idx          device int32 [R][K]:
 *                    block_table[b][t / block_size] * phys_block_stride
 *                    + t % block_size, or -1 for padding and invalid entries
 *   out_valid        device int32 [R] or NULL: non-negative entries per row
 *                    (entries keep their places; no compaction)
 *   status           device uint32 or NULL: HS_STATUS_INDEX is OR-ed in when
 *                    t >= row_causal_len or the block-table entry is negative
 * Requirements: R >= 0, K >= 0, block_size >= 1, phys_block_stride >= 1.
 * The caller guarantees t / block_size < bt_stride for t < row_causal_len.
 */
int hs_resolve_topk(const int32_t *req_id_per_row, const int32_t *row_causal_len,
                    const int32_t *block_table, int32_t bt_stride,
                    const int32_t *topk, int32_t R, int32_t K, int32_t block_size,
                    int32_t phys_block_stride, int32_t *out_idx,
                    int32_t *out_valid, uint32_t *status, hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a2-a5: swap-in for host-backed KV ([VLLM] resolve_topk -> runtime.swap_in; */
/*        [MTP] LRU slots and the position <-> slot maps)                     */
/* ------------------------------------------------------------------------ */

/*
 * For each query row r (request b = req_id_per_row[r], causal length
 * n = row_causal_len[r], committed length L = kv_len[b]) and entry t:
 *   t < 0                 padding                 -> -1
 *   t >= n                index error (status)    -> -1
 *   L <= t < n            step position           -> hot row b*(S+step)+S+(t-L)
 *   t < L                 committed position: made resident, then
 *                                                 -> hot row b*(S+step)+slot
 * Residency, per request over all its rows in the call: hits get timestamp
 * ts := clock (the clock advances by one per call); the distinct missing
 * positions, in ascending order, take the victim slots -- slots holding no
 * position needed in this call -- in ascending (ts, slot) order (empty slots
 * have ts = -1 and come first); the host row of each miss is copied into its
 * slot. A request needing more than S distinct committed positions gets
 * HS_STATUS_CAPACITY, its committed entries come out -1 and its maps are left
 * unchanged.
 *   kv_len        device int32 [max_reqs]: committed length per request
 *                 (0 <= kv_len <= max_ctx)
 *   topk          device int32 [R][K]
 *   out_slot_idx  device int32 [R][K]: rows of hot_kv, for hs_sparse_attn_decode
 *   out_valid     device int32 [R] or NULL
 *   stats         device int64 [2] or NULL: hits and misses of this call are
 *                 ADDED to stats[0] and stats[1]
 * Requirements: R >= 0, K >= 0.
 */
int hs_swap_in(hs_buffer *buf, const int32_t *req_id_per_row,
               const int32_t *row_causal_len, const int32_t *kv_len,
               const int32_t *topk, int32_t R, int32_t K, int32_t *out_slot_idx,
               int32_t *out_valid, int64_t *stats, hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a6: sparse attention over the selected latent rows (the DSA attention that */
/*     consumes resolve_topk / swap_in indices; MLA latent of 576 dims whose  */
/*     first 512 dims are the values)                                         */
/* ------------------------------------------------------------------------ */

/*
 * For each row r, head h:  s_j = scale * <q[r,h,:], kv[idx[r,j],:]> over 576
 * dims;  out[r,h,:] = sum_j softmax(s)_j * kv[idx[r,j], 0:512];
 * lse[r,h] = ln(sum_j exp(s_j)). Entries of idx outside [0, n_kv_rows) are
 * skipped; repeated entries count each time; a row with no valid entry gives
 * out = 0 and lse = -inf. bf16 inputs, fp32 accumulation, bf16 output.
 *   q      device bf16 [R][H][576], 16-byte aligned
 *   kv     device bf16 [n_kv_rows][576], 16-byte aligned (the paged cache for
 *          resolve indices, hot_kv for swap-in indices)
 *   idx    device int32 [R][K]
 *   out    device bf16 [R][H][512], 16-byte aligned
 *   lse    device float [R][H] or NULL
 *   status device uint32 or NULL: HS_STATUS_TIMEOUT is OR-ed in if one of
 *          the kernel's bounded internal waits gives up (never expected)
 * Requirements: R >= 0, 1 <= H <= 1024, K >= 0.
 * Launch: a programmatic dependent launch on `stream`. Its prologue (which
 * reads only q) may start before the previous kernel in the stream has
 * finished, if that kernel lets its dependents start early, as
 * hs_resolve_topk does; idx, kv and the request flags are read only after
 * the previous kernel has finished. So q must not be written by such an
 * early-releasing kernel immediately before this call (no call of this
 * library writes q).
 */
int hs_sparse_attn_decode(const void *q, const void *kv, int64_t n_kv_rows,
                          const int32_t *idx, int32_t R, int32_t H, int32_t K,
                          float scale, void *out, float *lse, uint32_t *status,
                          hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a2-a6 in one call: swap-in and attention of a decode step, with the host  */
/*     reads of later request groups overlapped with the attention of        */
/*     earlier ones ("hiSparse-MTP", section 1: the coordinator's            */
/*     asynchronous copy stream beside the compute stream)                   */
/* ------------------------------------------------------------------------ */

/*
 * Gives exactly the results of
 *   hs_swap_in(buf, req_id_per_row, row_causal_len, kv_len, topk, R, K,
 *              out_slot_idx, out_valid, stats, stream);
 *   hs_sparse_attn_decode(q, hot_kv, max_reqs * (S + step_slots), out_slot_idx,
 *                         R, H, K, scale, out, lse, <buf's status>, stream);
 * (the same slot maps, slot table, counts, hot rows and bit-identical out and
 * lse), with one swap-in on the LRU clock. The rows are split into groups of
 * consecutive rows; a request is swapped in with the group of its first row.
 * The metadata kernel runs once over every row; then the first group's missed
 * rows are copied from the host pool and its rows attended on `stream`, while
 * the copies of the next groups run on a stream of the buffer's own, one
 * group ahead of the attention, which for group g >= 1 runs on further
 * streams of the buffer's own once group g is resident. The copy blocks share
 * each SM with an attention block (a buffer of up to 448 requests; with more,
 * the copies of later groups wait for free SMs and the call is still correct).
 * `stream` waits for all of it before any later work on it starts, so the call
 * is ordered like any other on `stream`, in a CUDA graph capture too. (As for
 * every call that advances the LRU clock, a graph replays the clock value of
 * its capture: the clock is a host counter.)
 *   q, H, scale, out, lse   as hs_sparse_attn_decode (q [R][H][576], out
 *                           [R][H][512]; lse may be NULL)
 *   n_groups       0: the library picks the groups (hs_step_groups); else
 *                  1..8 with group_row_end (host int32 [n_groups]) rising
 *                  strictly from above 0 to R: group g is rows
 *                  [group_row_end[g-1], group_row_end[g])
 *   other arguments as hs_swap_in
 * Status goes to the buffer's status word (hs_get_status): the swap-in's bits
 * and the attention's HS_STATUS_TIMEOUT.
 * Requirements: those of hs_swap_in and hs_sparse_attn_decode. No two calls on
 * the same buffer may be in flight on different streams (the buffer's own
 * streams are shared by its calls).
 */
int hs_swap_in_attn_decode(hs_buffer *buf, const int32_t *req_id_per_row,
                           const int32_t *row_causal_len, const int32_t *kv_len,
                           const int32_t *topk, int32_t R, int32_t K, const void *q, int32_t H,
                           float scale, int32_t n_groups, const int32_t *group_row_end,
                           int32_t *out_slot_idx, int32_t *out_valid, void *out, float *lse,
                           int64_t *stats, hs_stream_t stream);

/*
 * The groups hs_swap_in_attn_decode picks for R rows of H heads on the
 * current device: the first is one wave of the attention kernel (the rows
 * its resident two-SM clusters hold at once); the other rows form at most 7
 * groups of equal size, a whole number of waves, the last taking what is
 * left. Writes n_groups (0 when R = 0) and group_row_end (host int32, room
 * for 8).
 */
int hs_step_groups(int32_t R, int32_t H, int32_t *n_groups, int32_t *group_row_end);

/*
 * Whether, on the current device, one copy block of hs_swap_in_attn_decode's
 * later groups (256 threads) fits on an SM beside one attention CTA: the
 * fullest quarter of the SM's register file (registers are allocated per warp
 * in units of 8 per thread, and a block's warps spread over the SM's four
 * schedulers), the shared memory of both (the copy block's grows with the
 * buffer's max_reqs) and the threads. When it does not, those copies wait
 * for whole SMs and the call runs no faster than hs_swap_in followed by
 * hs_sparse_attn_decode (the overlap that "hiSparse-MTP", section 1, gives
 * the coordinator's asynchronous stream is then lost). Writes *fits (1 or 0);
 * HS_ERR_INVALID_ARG for max_reqs outside 1..16384 or a NULL fits.
 */
int hs_step_overlap_fits(int32_t max_reqs, int32_t *fits);

/* ------------------------------------------------------------------------ */
/* next-3: a batch mixing fully-resident and host-backed requests            */
/*         ("vllm 分析(十二) HiSparse 下篇": the HiSparseResidentSpec and      */
/*          reclaim_resident_blocks sections, the fully_resident flag, and   */
/*          HiSparseCacheHandle.resolve_topk)                                */
/* ------------------------------------------------------------------------ */

/*
 * Releases resident pages when the paged cache runs short of blocks. Scanning
 * requests 0..B-1 and, within each, logical blocks 0 .. n_blocks[b] - 3 (every
 * page but the request's last two, which are still being written), it takes
 * the first `need` entries that are still held (>= 0): each one's physical
 * block id goes to freed[k] in that order and its entry becomes -1. Then
 * fully_resident[b] = 1 if entries 0 .. n_blocks[b] - 1 are all >= 0, else 0.
 * The pages leave the choice among reclaimable pages to a priority rule they
 * do not give; this call takes them in scan order, oldest pages first.
 *   block_table     device int32 [B][stride], updated in place
 *   n_blocks        device int32 [B]: logical blocks each request holds
 *                   (clamped to 0..stride)
 *   need            pages wanted (>= 0)
 *   freed           device int32 [need] or NULL: released block ids, -1 past
 *                   the last release
 *   fully_resident  device int32 [B] or NULL
 *   n_freed         device int32 or NULL: pages released (min(need, held))
 */
int hs_reclaim_resident(int32_t *block_table, int32_t B, int32_t stride,
                        const int32_t *n_blocks, int32_t need, int32_t *freed,
                        int32_t *fully_resident, int32_t *n_freed, hs_stream_t stream);

/*
 * hs_sparse_attn_decode for a batch that mixes both kinds of request: row r
 * reads kv_resident (its indices come from hs_resolve_topk) while its request
 * is fully resident, i.e. fully_resident[row_req[r]] != 0, and kv_hot (its
 * indices come from hs_swap_in) otherwise; each row's entries are valid within
 * its own cache's row count. The pages route a whole batch one way (resident
 * only when every request is); the per-row choice keeps the resident requests
 * off the swap-in path. Output, lse and requirements as hs_sparse_attn_decode.
 *   kv_resident, kv_hot  device bf16 [n_resident][576] / [n_hot][576],
 *                  16-byte aligned; either may be NULL when its count is 0
 *   row_req        device int32 [R]: request of each row, or NULL (the flags
 *                  are then indexed by row)
 *   fully_resident device int32 [n_reqs] (as hs_reclaim_resident writes it),
 *                  or NULL: every row reads kv_resident
 *   status         as hs_sparse_attn_decode; in addition HS_STATUS_INDEX when
 *                  a row's request is outside [0, n_reqs) -- that row then has
 *                  no valid entry
 * hs_sparse_attn_decode(q, kv, n, ...) is this call with kv_resident = kv,
 * n_resident = n and fully_resident = NULL.
 */
int hs_sparse_attn_decode_mixed(const void *q, const void *kv_resident, int64_t n_resident,
                                const void *kv_hot, int64_t n_hot, const int32_t *row_req,
                                const int32_t *fully_resident, int32_t n_reqs,
                                const int32_t *idx, int32_t R, int32_t H, int32_t K,
                                float scale, void *out, float *lse, uint32_t *status,
                                hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* next-1: one swap plan for follower caches ([VLLM] resolve_topk:           */
/*         runtime.apply_plan, produce_plan, plan_row_offset)                */
/* ------------------------------------------------------------------------ */

/*
 * Repeats the copies of buf's latest hs_swap_in or hs_swap_in_attn_decode
 * (the "plan": every missed
 * position's host row and the slot it went to) for n_layers follower caches,
 * e.g. the other layers of the same requests: for each copy (request b, slot
 * s, host row h) and layer l,
 *   hot_kv[l][row_offset + b * (S + step_slots) + s] = host_pools[l][h].
 * The slot table returned by that swap-in indexes every follower cache
 * the same way (plus row_offset). Followers have the leader's geometry (at
 * least row_offset + max_reqs * (S + step_slots) rows in hot_kv[l], host pools
 * paged like the leader's with at least host_pool_rows rows) but their own row
 * size: row_bytes per row, e.g. 1152 for a bf16 latent row like the leader's,
 * or the row of an FP8 / FP4 cache format (next-4: a second kind of cache on
 * the same plan).
 *   hot_kv      host array of n_layers device pointers
 *   host_pools  host array of n_layers pointers to page-locked mapped host
 *               memory (or device memory)
 *   row_offset  rows added to every destination (>= 0)
 *   row_bytes   a multiple of 4 (copies are 16 bytes wide when it is a
 *               multiple of 16 and every pointer is 16-byte aligned, else 4)
 * Call it after the swap-in whose plan it repeats and before the next one
 * (same stream, or ordered). Requirements: 0 <= n_layers <= 64, pointers
 * 4-byte aligned, max_reqs * S * (row units) < 2^31.
 */
int hs_swap_apply_plan(hs_buffer *buf, int32_t n_layers, void *const *hot_kv,
                       const void *const *host_pools, int64_t row_offset, int32_t row_bytes,
                       hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* next-2: page backup of several layers to host ([VLLM] 数据 back up:        */
/*         HiSparseWorker._enqueue_transfers, hisparse_backup_layers)         */
/* ------------------------------------------------------------------------ */

/*
 * For transfer i and layer l, rows src_blocks[l][i] * block_rows + o of
 * src_caches[l] go to rows
 *   (dst_blocks[i] * blocks_per_kv_block + page_offsets[i]) * block_rows + o
 * of dst_caches[l], o = 0 .. block_rows - 1 (each layer's own resident block,
 * one host page shared by the layers). Rows of row_bytes bytes.
 *   src_caches    host array of n_layers device pointers (resident caches)
 *   dst_caches    host array of n_layers pointers to page-locked mapped host
 *                 memory (or device memory)
 *   src_blocks    device int32 [n_layers][n_transfers]
 *   dst_blocks, page_offsets  device int32 [n_transfers]
 *   src_rows, dst_rows        rows in each source / destination cache: a
 *                 transfer reaching outside them (or a negative block) is
 *                 skipped and sets HS_STATUS_INDEX in status (device uint32
 *                 or NULL)
 * Requirements: 0 <= n_layers <= 64, n_transfers >= 0, block_rows >= 1,
 * blocks_per_kv_block >= 1, row_bytes a multiple of 16, pointers 16-byte
 * aligned.
 */
int hs_backup_pages(int32_t n_layers, const void *const *src_caches, void *const *dst_caches,
                    const int32_t *src_blocks, const int32_t *dst_blocks,
                    const int32_t *page_offsets, int32_t n_transfers, int32_t block_rows,
                    int32_t blocks_per_kv_block, int32_t row_bytes, int64_t src_rows,
                    int64_t dst_rows, uint32_t *status, hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* next-4: row backup by slot mapping, and the indexer cache's backup        */
/*         ([VLLM] c4a kv cache 写入: runtime.backup_rows,                    */
/*          compress_hisparse_slot_mapping, hisparse_backup_indexer)          */
/* ------------------------------------------------------------------------ */

/*
 * For every entry i with src_slots[i] >= 0 and dst_slots[i] >= 0 and every
 * layer l: row dst_slots[i] of dst_caches[l] = row src_slots[i] of
 * src_caches[l], token_stride bytes per row (a token's entry is one
 * contiguous run of token_stride bytes on both sides). A negative slot means
 * "no entry" and is skipped; a slot at or past src_rows / dst_rows is skipped
 * and sets HS_STATUS_INDEX in status (device uint32 or NULL). Destination
 * slots are distinct within a call (else which copy lands is unspecified).
 *   src_caches  host array of n_layers device pointers
 *   dst_caches  host array of n_layers pointers to page-locked mapped host
 *               memory (or device memory)
 *   src_slots, dst_slots  device int32 [n]
 * Requirements: 0 <= n_layers <= 64, n >= 0, token_stride a multiple of 4 in
 * 4..2^20, pointers 4-byte aligned (16-byte copies when token_stride and
 * every pointer allow).
 */
int hs_backup_rows(int32_t n_layers, const void *const *src_caches, void *const *dst_caches,
                   const int32_t *src_slots, const int32_t *dst_slots, int32_t n,
                   int32_t token_stride, int64_t src_rows, int64_t dst_rows, uint32_t *status,
                   hs_stream_t stream);

/*
 * hs_backup_rows for the indexer cache, whose host cache stores one entry per
 * compress_ratio tokens in blocks of storage_block_size entries: the host row
 * of entry i is computed from its logical host slot and position,
 *   lbs = storage_block_size * compress_ratio,
 *   dst = (host_slots[i] / lbs) * storage_block_size
 *         + (positions[i] % lbs) / compress_ratio,
 * (-1, skipped, when host_slots[i] or positions[i] is negative), and
 * src_slots[i] < 0 marks a token that wrote no entry.
 *   host_slots, positions  device int32 [n]
 * Requirements as hs_backup_rows, plus storage_block_size >= 1,
 * compress_ratio >= 1.
 */
int hs_backup_indexer(int32_t n_layers, const void *const *src_caches, void *const *dst_caches,
                      const int32_t *src_slots, const int32_t *host_slots,
                      const int32_t *positions, int32_t n, int32_t storage_block_size,
                      int32_t compress_ratio, int32_t token_stride, int64_t src_rows,
                      int64_t dst_rows, uint32_t *status, hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a7-a8: greedy verify and commit of the accepted prefix ([KVF] ④-⑥)       */
/* ------------------------------------------------------------------------ */

/*
 * For batch entry b (request req = req_ids ? req_ids[b] : b, L = kv_len[req]):
 *   pred[i] = argmax_v logits[b][i][v] for i = 0..d (lowest index on ties);
 *     input 0 is the anchor, input i >= 1 is draft i;
 *   m = length of the longest prefix with draft_tokens[b][i] == pred[i];
 *   accept_len[b] = m; next_token[b] = pred[m] (the correction token, or the
 *     bonus token when all d drafts pass);
 *   the KV of inputs 0..m (step_kv[b][0..m], positions L..L+m) is committed:
 *     written to the host pool rows of those positions and placed in LRU
 *     slots taken in ascending (ts, slot) order with nothing protected;
 *     kv_len[req] = L + m + 1. The next token has no KV yet.
 * A request with L + m + 1 > max_ctx gets HS_STATUS_CAPACITY and no commit.
 *   logits        device [B][d+1][V], fp32 (HS_LOGITS_F32) or bf16
 *                 (HS_LOGITS_BF16); finite values
 *   draft_tokens  device int32 [B][d]
 *   step_kv       device bf16 [B][d+1][576]
 *   kv_len        device int32 [max_reqs], updated in place
 *   accept_len, next_token  device int32 [B]
 *   req_ids       device int32 [B] or NULL (identity); distinct request ids.
 *                 A request id out of [0, max_reqs) or repeated within the
 *                 call sets HS_STATUS_INDEX; of a repeated id's entries only
 *                 the first to finish its acceptance commits (which one is
 *                 not specified), the others commit nothing. Every entry
 *                 still gets its accept_len and next_token.
 * Requirements: 1 <= B <= max_reqs, 0 <= d, d + 1 <= step_slots, V >= 1.
 */
int hs_verify_finalize(hs_buffer *buf, const void *logits, int32_t logits_dtype,
                       int32_t B, int32_t d, int32_t V,
                       const int32_t *draft_tokens, const void *step_kv,
                       const int32_t *req_ids, int32_t *kv_len,
                       int32_t *accept_len, int32_t *next_token,
                       hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Greedy acceptance without allocation (no counterpart on the pages)         */
/* ------------------------------------------------------------------------ */

/*
 * The argmax and accepted-prefix half of hs_verify_finalize, with the same
 * accept_len / next_token results, for callers that cannot allocate device
 * memory: code whose device memory is owned by a host framework's allocator,
 * or a serving loop that may not take the synchronisation an allocation can
 * bring. It needs no hs_buffer and commits no KV (the caller does that).
 *   logits, logits_dtype, draft_tokens, accept_len, next_token: as for
 *   hs_verify_finalize ([B][d+1][V] logits, [B][d] drafts, [B] outputs).
 * Scratch: two static device arrays of 65536 int32 (512 KiB) inside the
 * library (per-row argmax, per-request row counts), held by every GPU that
 * loads it until the process exits. Sizes with B * (d + 1) > 65536 return
 * HS_ERR_INVALID_ARG. No cudaMalloc, cudaFree or allocating library routine
 * is called. The first call on a device looks up the arrays' device addresses
 * (cudaGetSymbolAddress) in the device's current context; make that first
 * call before any stream capture. The addresses are kept per device together
 * with the id of that context, and looked up again when a call finds another
 * context current (after cudaDeviceReset, say). Every pointer argument must
 * be memory of the current device. One
 * launch: the last row of each request to finish takes its prefix and puts
 * the request's count back to 0, so nothing carries over between calls, but
 * all calls share the arrays: calls that overlap on the GPU (different
 * streams without ordering) race.
 * Requirements: B >= 1, d >= 0, V >= 1.
 */
int hs_verify_accept_noalloc(const void *logits, int32_t logits_dtype, int32_t B,
                             int32_t d, int32_t V, const int32_t *draft_tokens,
                             int32_t *accept_len, int32_t *next_token,
                             hs_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Measurement helper (no counterpart on the pages)                           */
/* ------------------------------------------------------------------------ */

/* Reads `bytes` (a multiple of 16) from `src` -- e.g. mapped page-locked host
 * memory -- with 16-byte loads on `blocks` x 256 threads and writes one
 * checksum word per block to device uint64 sink[blocks]. Used to measure the
 * host-to-device link bandwidth a zero-copy gather can reach. */
int hs_read_probe(const void *src, size_t bytes, uint64_t *sink, int32_t blocks,
                  hs_stream_t stream);

/* Failure-detection check: one warp runs the attention kernel's bounded
 * mbarrier wait, cut to max_cycles SM cycles (1..2^31), on a phase that
 * nothing completes; when it gives up, HS_STATUS_TIMEOUT is OR-ed into the
 * device uint32 *status, exactly as a wait of hs_sparse_attn_decode that ran
 * out would. Shows that a wait which gives up ends the kernel and leaves the
 * context usable. Returns HS_ERR_INVALID_ARG for a NULL status or a limit
 * out of range. */
int hs_wait_probe(uint32_t *status, int64_t max_cycles, hs_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* HISPARSE_H_ */
