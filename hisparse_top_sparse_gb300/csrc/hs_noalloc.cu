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

#include <cuda.h>

#include <mutex>

#include "hs_internal.cuh"

#define HS_NOALLOC_MAX_ROWS 65536   // B * (d + 1) limit: two int32 arrays, 512 KiB
#define HS_NOALLOC_MAX_DEVICES 64

static __device__ __align__(256) int32_t g_accept_scratch[HS_NOALLOC_MAX_ROWS];
// per request: argmax rows done in the current call (back to 0 at its end)
static __device__ __align__(256) int32_t g_accept_count[HS_NOALLOC_MAX_ROWS];

namespace {

// Device addresses of the two arrays in each device's current context. In
// host code an array's name is only a host-side stand-in; kernels must
// receive the address that cudaGetSymbolAddress returns with the device
// current. The addresses belong to a context: after cudaDeviceReset the
// device gets a new primary context and the arrays new addresses, so each
// cache entry remembers the unique id of the context it was taken in
// (cuCtxGetId) and is looked up again when the current context's id differs.
struct ScratchEntry {
  unsigned long long ctx_id;
  int32_t *pred;
  int32_t *count;
};
ScratchEntry g_entry[HS_NOALLOC_MAX_DEVICES] = {};
std::mutex g_scratch_mu;

using PFN_ctxGetCurrent = CUresult (*)(CUcontext *);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long *);

// the unique id of the calling thread's current context (0 when unknown)
int current_ctx_id(unsigned long long *id) {
  static PFN_ctxGetCurrent get_current = nullptr;
  static PFN_ctxGetId get_id = nullptr;
  if (!get_current || !get_id) {
    void *f1 = nullptr, *f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || !f1 ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f2)
      return hs_set_error(HS_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId not available");
    get_current = reinterpret_cast<PFN_ctxGetCurrent>(f1);
    get_id = reinterpret_cast<PFN_ctxGetId>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx)
    return hs_set_error(HS_ERR_CUDA, "no current CUDA context");
  if (get_id(ctx, id) != CUDA_SUCCESS)
    return hs_set_error(HS_ERR_CUDA, "cuCtxGetId failed");
  return HS_OK;
}

int lookup_symbols(ScratchEntry *e) {
  void *p = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&p, g_accept_scratch);
  if (err != cudaSuccess || !p)
    return hs_set_error(HS_ERR_CUDA, "cudaGetSymbolAddress(g_accept_scratch) failed: %s",
                        cudaGetErrorString(err));
  void *pc = nullptr;
  err = cudaGetSymbolAddress(&pc, g_accept_count);
  if (err != cudaSuccess || !pc)
    return hs_set_error(HS_ERR_CUDA, "cudaGetSymbolAddress(g_accept_count) failed: %s",
                        cudaGetErrorString(err));
  e->pred = static_cast<int32_t *>(p);
  e->count = static_cast<int32_t *>(pc);
  return HS_OK;
}

int scratch_for_current_device(int32_t **out, int32_t **count) {
  int dev = -1;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= HS_NOALLOC_MAX_DEVICES)
    return hs_set_error(HS_ERR_UNSUPPORTED, "device %d beyond %d", dev, HS_NOALLOC_MAX_DEVICES);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry &e = g_entry[dev];
  unsigned long long id = 0;
  if (current_ctx_id(&id) != HS_OK) {
    // no current context yet: the symbol lookup makes the device's primary
    // context current, then its id can be read
    int rc = lookup_symbols(&e);
    if (rc) return rc;
    rc = current_ctx_id(&id);
    if (rc) return rc;
    e.ctx_id = id;
  } else if (!e.pred || e.ctx_id != id) {
    int rc = lookup_symbols(&e);
    if (rc) return rc;
    e.ctx_id = id;
  }
  *out = e.pred;
  *count = e.count;
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
