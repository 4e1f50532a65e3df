// next-3: reclaim of resident pages ("vllm 分析(十二) HiSparse 下篇",
// section reclaim_resident_blocks: when allocate_slots runs short of blocks the
// coordinator asks HiSparseResidentManager.reclaimable_pages for every
// request's old pages -- all but its last two -- releases the chosen ones with
// release_resident_page, whose table entry becomes null and whose block goes
// back to the pool, and a request with a released page is no longer
// fully_resident).
//
// The block table stays in HBM, so the scan, the release and the new
// fully_resident flags are one small kernel: one block, each thread owning a
// run of requests; a block-wide prefix count ranks the reclaimable pages in
// (request, block) order and the first `need` of them are released.

#include "hs_internal.cuh"

namespace {

constexpr int RT = 1024;

__global__ void __launch_bounds__(RT) k_reclaim(int32_t *__restrict__ bt, int32_t B,
                                                int32_t stride,
                                                const int32_t *__restrict__ n_blocks,
                                                int32_t need, int32_t *__restrict__ freed,
                                                int32_t *__restrict__ fully_resident,
                                                int32_t *__restrict__ n_freed) {
  __shared__ int tmp[33];
  const int E = (B + RT - 1) / RT;
  const int lo = min(B, (int)threadIdx.x * E), hi = min(B, lo + E);
  // pages a reclaim may take: held entries of blocks 0 .. n-3
  int cnt = 0;
  for (int b = lo; b < hi; ++b) {
    const int n = min(max(n_blocks[b], 0), stride);
    const int32_t *row = bt + (int64_t)b * stride;
    for (int i = 0; i < n - 2; ++i) cnt += row[i] >= 0;
  }
  int total;
  int rank = hs_block_exscan(cnt, tmp, &total);
  for (int b = lo; b < hi; ++b) {
    const int n = min(max(n_blocks[b], 0), stride);
    int32_t *row = bt + (int64_t)b * stride;
    bool full = true;
    for (int i = 0; i < n; ++i) {
      int32_t blk = row[i];
      if (i < n - 2 && blk >= 0) {
        if (rank < need) {
          if (freed) freed[rank] = blk;
          row[i] = blk = -1;
        }
        ++rank;
      }
      full &= blk >= 0;
    }
    if (fully_resident) fully_resident[b] = full ? 1 : 0;
  }
  const int done = min(total, need);
  if (freed)
    for (int k = done + (int)threadIdx.x; k < need; k += RT) freed[k] = -1;
  if (n_freed && threadIdx.x == 0) *n_freed = done;
}

}  // namespace

extern "C" int hs_reclaim_resident(int32_t *block_table, int32_t B, int32_t stride,
                                   const int32_t *n_blocks, int32_t need, int32_t *freed,
                                   int32_t *fully_resident, int32_t *n_freed,
                                   hs_stream_t stream) {
  if (B < 0 || stride < 0 || need < 0)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes B=%d stride=%d need=%d", B, stride, need);
  if (B == 0) {
    if (n_freed) HS_CUDA_TRY(cudaMemsetAsync(n_freed, 0, sizeof(int32_t), stream));
    if (freed && need > 0)
      HS_CUDA_TRY(cudaMemsetAsync(freed, 0xff, (size_t)need * sizeof(int32_t), stream));
    return HS_OK;
  }
  if (hs_check_device_ptr(block_table, "block_table", stride == 0) ||
      hs_check_device_ptr(n_blocks, "n_blocks", false) ||
      hs_check_device_ptr(freed, "freed", true) ||
      hs_check_device_ptr(fully_resident, "fully_resident", true) ||
      hs_check_device_ptr(n_freed, "n_freed", true))
    return HS_ERR_INVALID_ARG;
  k_reclaim<<<1, RT, 0, stream>>>(block_table, B, stride, n_blocks, need, freed, fully_resident,
                                  n_freed);
  HS_LAUNCH_CHECK("k_reclaim");
  return HS_OK;
}
