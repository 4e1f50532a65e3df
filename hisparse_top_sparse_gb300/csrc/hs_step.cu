// hs_swap_in_attn_decode: the swap-in and the sparse attention of one decode
// step in one call, with the host reads of later request groups overlapped
// with the attention of earlier ones.
//
// "hiSparse-MTP", section 1 (HiSparseCoordinator.__init__): the coordinator
// owns an asynchronous stream beside the compute stream for its copies.
// "vllm 分析(十二) HiSparse 下篇", HiSparseCacheHandle.resolve_topk: a step's
// rows go through swap_in, then attend over the hot cache with the indices it
// returns. The call keeps that order per request and overlaps across them.
//
// Schedule, rows split into groups (row ranges; a request belongs to the group
// of its first row, so any row order is correct):
//   stream   k_swap_request (every row)  ->  gather of group 0 (every SM, 8
//            blocks each)  ->  attention of group 0
//   side 0   gather of group 1, 2, ... (one block per SM), an event after each
//   side 1/2 attention of group g >= 1 after its gather's event, alternating
//            between two streams so that a group's attention fills the SMs the
//            previous group's last wave leaves idle
// A gather block (256 threads, 54 registers, 144 + 4 * (max_reqs + 1) bytes of
// shared memory) fits on an SM beside one attention CTA (480 threads, at most
// 96 registers, 229,376 bytes; the SM keeps 3 KB of shared memory, and each of
// its four register-file quarters holds four attention warps and two gather
// warps) for up to 448 requests, so the later gathers take no SM away from
// the attention. The caller's stream waits for every side stream before the
// call returns.

#include <algorithm>

#include "hs_internal.cuh"

namespace {

constexpr int STEP_GATHER_THREADS = 256;   // a later group's gather block, one per SM

// Rows [ends[g-1], ends[g]) of the automatic split: the first group one
// attention wave (its copies are the only ones not hidden), the other rows in
// at most HS_MAX_GROUPS - 1 groups of equal size, a whole number of waves
// (the last takes what is left). Small groups keep the copies of the next
// group short, so the attention rarely waits for them.
int auto_groups(int32_t R, int32_t H, int32_t *n, int32_t *ends) {
  int32_t wave = 1;
  int rc = hs_attn_wave_rows(H, &wave);
  if (rc) return rc;
  int g = 0;
  ends[g++] = std::min(R, wave);
  const int64_t rest = (int64_t)R - ends[0];
  if (rest > 0) {
    const int64_t waves = (rest + wave - 1) / wave;
    const int64_t groups = std::min<int64_t>(HS_MAX_GROUPS - 1, waves);
    const int64_t size = (waves + groups - 1) / groups * wave;
    int64_t end = ends[0];
    while (end < R) {
      end = std::min<int64_t>(R, end + size);
      ends[g++] = (int32_t)end;
    }
  }
  *n = g;
  return HS_OK;
}

}  // namespace

extern "C" int hs_step_groups(int32_t R, int32_t H, int32_t *n_groups, int32_t *group_row_end) {
  if (R < 0 || H < 1 || H > 1024 || !n_groups || !group_row_end)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad arguments R=%d H=%d", R, H);
  *n_groups = 0;
  if (R == 0) return HS_OK;
  return auto_groups(R, H, n_groups, group_row_end);
}

extern "C" int hs_step_overlap_fits(int32_t max_reqs, int32_t *fits) {
  if (max_reqs < 1 || max_reqs > HS_MAX_REQS || !fits)
    return hs_set_error(HS_ERR_INVALID_ARG, "max_reqs %d not in 1..%d or NULL fits", max_reqs,
                        HS_MAX_REQS);
  *fits = 0;
  cudaFuncAttributes fa, fg;
  int attn_threads = 0;
  size_t attn_dyn = 0;
  int rc = hs_attn_block_attrs(&fa, &attn_threads, &attn_dyn);
  if (rc) return rc;
  rc = hs_gather_func_attrs(&fg);
  if (rc) return rc;
  int dev = 0, regs_sm = 0, smem_sm = 0, smem_rsv = 0, threads_sm = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev));
  // registers: a warp holds its threads' count rounded up to 8, times 32;
  // a CTA's warps spread over the SM's four schedulers, each with a quarter
  // of the register file, so the fullest quarter holds ceil(warps / 4) of
  // each block
  auto warp_regs = [](int per_thread) { return ((per_thread + 7) / 8) * 8 * 32; };
  const int attn_warps = (attn_threads + 31) / 32, gather_warps = STEP_GATHER_THREADS / 32;
  const long long quarter = (long long)((attn_warps + 3) / 4) * warp_regs(fa.numRegs) +
                            (long long)((gather_warps + 3) / 4) * warp_regs(fg.numRegs);
  const long long smem = (long long)attn_dyn + fa.sharedSizeBytes + smem_rsv +
                         (long long)(max_reqs + 1) * 4 + fg.sharedSizeBytes + smem_rsv;
  *fits = quarter <= regs_sm / 4 && smem <= smem_sm &&
          attn_threads + STEP_GATHER_THREADS <= threads_sm;
  return HS_OK;
}

extern "C" int hs_swap_in_attn_decode(hs_buffer *buf, const int32_t *req_id_per_row,
                                      const int32_t *row_causal_len, const int32_t *kv_len,
                                      const int32_t *topk, int32_t R, int32_t K, const void *q,
                                      int32_t H, float scale, int32_t n_groups,
                                      const int32_t *group_row_end, int32_t *out_slot_idx,
                                      int32_t *out_valid, void *out, float *lse, int64_t *stats,
                                      hs_stream_t stream) {
  int rc = hs_check_buffer(buf);
  if (rc) return rc;
  if (R < 0 || K < 0 || K > (1 << 20) || H < 1 || H > 1024)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes R=%d K=%d (0..2^20) H=%d (1..1024)", R,
                        K, H);
  if (R > 0 && (!req_id_per_row || !row_causal_len || !kv_len || !q || !out))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL row descriptor, q or out");
  if (R > 0 && K > 0 && (!topk || !out_slot_idx))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL topk or out_slot_idx");
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15))
    return hs_set_error(HS_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (!(scale == scale)) return hs_set_error(HS_ERR_INVALID_ARG, "scale is NaN");
  int32_t ends[HS_MAX_GROUPS];
  int G = n_groups;
  if (n_groups < 0 || n_groups > HS_MAX_GROUPS || (n_groups > 0 && !group_row_end))
    return hs_set_error(HS_ERR_INVALID_ARG, "n_groups %d (0..%d) or group_row_end NULL",
                        n_groups, HS_MAX_GROUPS);
  for (int g = 0; g < n_groups; ++g) {
    ends[g] = group_row_end[g];
    if (ends[g] <= (g ? ends[g - 1] : 0) || (g == n_groups - 1 && ends[g] != R))
      return hs_set_error(HS_ERR_INVALID_ARG,
                          "group_row_end must rise strictly from above 0 to R = %d", R);
  }

  buf->clock += 1;  // one swap-in: the LRU clock advances once, as in hs_swap_in
  if (R == 0) return HS_OK;
  if (G == 0) {
    rc = auto_groups(R, H, &G, ends);
    if (rc) return rc;
  }
  rc = hs_swap_plan_launch(buf, req_id_per_row, row_causal_len, kv_len, topk, R, K, G, ends,
                           out_slot_idx, out_valid, stats, stream);
  if (rc) return rc;
  rc = hs_swap_gather_launch(buf, req_id_per_row, row_causal_len, kv_len, topk, R, K, 0, 0,
                             ends[0], out_slot_idx, out_valid, 8, 256, true, stream);
  if (rc) return rc;

  const int64_t n_hot = (int64_t)buf->max_reqs * buf->S_tot;
  auto attend = [&](int g, cudaStream_t st, bool pdl) -> int {
    const int32_t lo = g ? ends[g - 1] : 0, n = ends[g] - lo;
    return hs_attn_launch(static_cast<const char *>(q) + (int64_t)lo * H * HS_ROW_BYTES,
                          buf->hot_kv, n_hot, nullptr, 0, nullptr, nullptr, 0,
                          out_slot_idx ? out_slot_idx + (int64_t)lo * K : nullptr, n, H, K,
                          scale, static_cast<char *>(out) + (int64_t)lo * H * 512 * 2,
                          lse ? lse + (int64_t)lo * H : nullptr, buf->status, pdl, st);
  };
  if (G == 1) {
    // a programmatic dependent launch of the gather: its prologue runs while
    // the gather finishes
    return attend(0, stream, true);
  }
  HS_CUDA_TRY(cudaEventRecord(buf->ev_fork, stream));
  HS_CUDA_TRY(cudaStreamWaitEvent(buf->side[0], buf->ev_fork, 0));
  // from here on every side stream that received work joins `stream` again,
  // also when a later launch fails, so that a stream capture stays whole
  bool used[HS_SIDE_STREAMS] = {true, false, false};
  auto join = [&]() -> int {
    int first = HS_OK;
    for (int s = 0; s < HS_SIDE_STREAMS; ++s) {
      if (!used[s]) continue;
      cudaError_t e = cudaEventRecord(buf->ev_join[s], buf->side[s]);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, buf->ev_join[s], 0);
      if (e != cudaSuccess && first == HS_OK)
        first = hs_set_error(HS_ERR_CUDA, "joining the buffer's streams: %s", cudaGetErrorString(e));
    }
    return first;
  };
  auto fail = [&](int code) -> int {
    join();
    return code;
  };
  for (int g = 1; g < G; ++g) {
    rc = hs_swap_gather_launch(buf, req_id_per_row, row_causal_len, kv_len, topk, R, K, g,
                               ends[g - 1], ends[g], out_slot_idx, out_valid, 1, STEP_GATHER_THREADS, false,
                               buf->side[0]);
    if (rc) return fail(rc);
    const cudaError_t e = cudaEventRecord(buf->ev_gather[g], buf->side[0]);
    if (e != cudaSuccess)
      return fail(hs_set_error(HS_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e)));
  }
  rc = attend(0, stream, true);
  if (rc) return fail(rc);
  for (int g = 1; g < G; ++g) {
    const int s = 1 + (g - 1) % 2;
    used[s] = true;
    const cudaError_t e = cudaStreamWaitEvent(buf->side[s], buf->ev_gather[g], 0);
    if (e != cudaSuccess)
      return fail(hs_set_error(HS_ERR_CUDA, "cudaStreamWaitEvent: %s", cudaGetErrorString(e)));
    rc = attend(g, buf->side[s], false);
    if (rc) return fail(rc);
  }
  return join();
}
