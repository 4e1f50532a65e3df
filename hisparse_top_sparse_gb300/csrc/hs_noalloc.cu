// hs_verify_accept_noalloc: greedy acceptance (the argmax and accepted-prefix
// half of hs_verify_finalize) for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available to it -- a
// plugin inside a host framework whose allocator owns all device memory, or a
// serving loop whose latency budget forbids the implicit synchronisation an
// allocation can cause. Such a caller can still hand over its own logits,
// drafts and output arrays, but cannot create an hs_buffer (that allocates).
//
// The one launch needs scratch: one int32 per verified row (its argmax) and
// one per request (its rows done so far). Both live in file-scope __device__
// arrays of fixed size, which every GPU that loads this library holds until
// the process exits. No call below allocates.

#include <mutex>

#include "hs_internal.cuh"

#define HS_NOALLOC_MAX_ROWS 65536   // B * (d + 1) limit: two int32 arrays, 512 KiB
#define HS_NOALLOC_MAX_DEVICES 64

static __device__ __align__(256) int32_t g_accept_scratch[HS_NOALLOC_MAX_ROWS];
// per request: argmax rows done in the current call (back to 0 at its end)
static __device__ __align__(256) int32_t g_accept_count[HS_NOALLOC_MAX_ROWS];

namespace {

// Device address of g_accept_scratch on each device, looked up once. In host
// code the array's name is only a host-side stand-in; kernels must receive the
// address that cudaGetSymbolAddress returns for the current device.
int32_t *g_scratch_dev[HS_NOALLOC_MAX_DEVICES] = {nullptr};
int32_t *g_count_dev[HS_NOALLOC_MAX_DEVICES] = {nullptr};
std::mutex g_scratch_mu;

int scratch_for_current_device(int32_t **out, int32_t **count) {
  int dev = -1;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= HS_NOALLOC_MAX_DEVICES)
    return hs_set_error(HS_ERR_UNSUPPORTED, "device %d beyond %d", dev, HS_NOALLOC_MAX_DEVICES);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess || !p)
      return hs_set_error(HS_ERR_CUDA, "cudaGetSymbolAddress(g_accept_scratch) failed: %s",
                          cudaGetErrorString(e));
    void *pc = nullptr;
    e = cudaGetSymbolAddress(&pc, g_accept_count);
    if (e != cudaSuccess || !pc)
      return hs_set_error(HS_ERR_CUDA, "cudaGetSymbolAddress(g_accept_count) failed: %s",
                          cudaGetErrorString(e));
    g_scratch_dev[dev] = static_cast<int32_t *>(p);
    g_count_dev[dev] = static_cast<int32_t *>(pc);
  }
  *out = g_scratch_dev[dev];
  *count = g_count_dev[dev];
  return HS_OK;
}

// Block per logits row: argmax with ties to the lowest index into pred[row];
// the request's last row to finish (a count per request) then takes the
// longest agreeing prefix and the next token, and puts the count back to 0.
template <int DTYPE>
__global__ void __launch_bounds__(HS_ARGMAX_THREADS) k_accept(const void *__restrict__ logits,
                                                             int32_t V, int32_t d,
                                                             const int32_t *__restrict__ drafts,
                                                             int32_t *pred, int32_t *count,
                                                             int32_t *__restrict__ accept_len,
                                                             int32_t *__restrict__ next_token) {
  const int64_t row = blockIdx.x;
  const int64_t elem = (DTYPE == HS_LOGITS_F32) ? 4 : 2;
  const int32_t best = hs_row_argmax<DTYPE>(
      reinterpret_cast<const char *>(logits) + row * (int64_t)V * elem, V);
  if (threadIdx.x != 0) return;
  pred[row] = best;
  __threadfence();
  const int64_t b = row / (d + 1);
  if (atomicAdd(&count[b], 1) != d) return;
  __threadfence();   // every row of request b has its pred
  count[b] = 0;
  const int32_t *p = pred + b * (d + 1);
  int m = 0;
  while (m < d && drafts[b * d + m] == __ldcg(p + m)) ++m;
  accept_len[b] = m;
  next_token[b] = __ldcg(p + m);
}

}  // namespace

extern "C" int hs_verify_accept_noalloc(const void *logits, int32_t logits_dtype, int32_t B,
                                        int32_t d, int32_t V, const int32_t *draft_tokens,
                                        int32_t *accept_len, int32_t *next_token,
                                        hs_stream_t stream) {
  if (B < 1 || d < 0 || V < 1)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes B=%d d=%d V=%d", B, d, V);
  if ((int64_t)B * (d + 1) > HS_NOALLOC_MAX_ROWS)
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "B*(d+1) = %lld rows exceeds the static scratch of %d rows",
                        (long long)B * (d + 1), HS_NOALLOC_MAX_ROWS);
  if (logits_dtype != HS_LOGITS_F32 && logits_dtype != HS_LOGITS_BF16)
    return hs_set_error(HS_ERR_INVALID_ARG, "logits_dtype %d", logits_dtype);
  if (!logits || (d > 0 && !draft_tokens) || !accept_len || !next_token)
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL argument");
  int32_t *pred = nullptr, *count = nullptr;
  int rc = scratch_for_current_device(&pred, &count);
  if (rc) return rc;
  const int rows = B * (d + 1);
  if (logits_dtype == HS_LOGITS_F32)
    k_accept<HS_LOGITS_F32><<<rows, HS_ARGMAX_THREADS, 0, stream>>>(logits, V, d, draft_tokens,
                                                                    pred, count, accept_len,
                                                                    next_token);
  else
    k_accept<HS_LOGITS_BF16><<<rows, HS_ARGMAX_THREADS, 0, stream>>>(logits, V, d, draft_tokens,
                                                                     pred, count, accept_len,
                                                                     next_token);
  HS_LAUNCH_CHECK("k_accept");
  return HS_OK;
}
