// next-2: backup of whole pages of several layers' device caches to their
// host caches ("vllm 分析(十二) HiSparse 下篇", section 数据 back up:
// HiSparseWorker._enqueue_transfers builds, per transfer, the source rows
// block_id * kernel_block_size + offset of every cache and the destination
// rows host_page * kernel_block_size + offset with host_page =
// destination_block_id * blocks_per_kv_block + destination_page_offset, and
// hisparse_backup_layers copies them device -> host).
//
// One launch copies every (layer, transfer, row) with 16-byte stores into the
// device-mapped page-locked host caches, four loads in flight per thread; the
// row arithmetic is done per chunk in the kernel.

#include "hs_internal.cuh"

namespace {

struct BackupLayers {
  const uint4 *src[HS_MAX_LAYERS];
  uint4 *dst[HS_MAX_LAYERS];
};

__global__ void __launch_bounds__(256) k_backup_pages(const __grid_constant__ BackupLayers bl,
                                                      int32_t n_layers,
                                                      const int32_t *__restrict__ src_blocks,
                                                      const int32_t *__restrict__ dst_blocks,
                                                      const int32_t *__restrict__ page_offsets,
                                                      int32_t n_transfers, int32_t block_rows,
                                                      int32_t blocks_per_kv_block, int32_t row_vec16,
                                                      int64_t src_rows, int64_t dst_rows,
                                                      uint32_t *status) {
  const int64_t per_row = row_vec16;
  const int64_t total = (int64_t)n_layers * n_transfers * block_rows * per_row;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += 4 * step) {
    uint4 v[4];
    uint4 *dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t k = e + u * step;
      dst[u] = nullptr;
      if (k < total) {
        const int64_t rowk = k / per_row;
        const int c = (int)(k - rowk * per_row);
        const int o = (int)(rowk % block_rows);
        const int64_t it = rowk / block_rows;
        const int i = (int)(it % n_transfers);
        const int l = (int)(it / n_transfers);
        const int64_t sb = src_blocks[(int64_t)l * n_transfers + i];
        const int64_t page = (int64_t)dst_blocks[i] * blocks_per_kv_block + page_offsets[i];
        const int64_t sr = sb * block_rows + o, dr = page * block_rows + o;
        if (sb >= 0 && sr < src_rows && dst_blocks[i] >= 0 && page_offsets[i] >= 0 && dr < dst_rows) {
          v[u] = bl.src[l][sr * per_row + c];
          dst[u] = bl.dst[l] + dr * per_row + c;
        } else {
          bad = true;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u]) *dst[u] = v[u];
  }
  if (bad && status) atomicOr(status, HS_STATUS_INDEX);
}

}  // namespace

extern "C" int hs_backup_pages(int32_t n_layers, const void *const *src_caches,
                               void *const *dst_caches, const int32_t *src_blocks,
                               const int32_t *dst_blocks, const int32_t *page_offsets,
                               int32_t n_transfers, int32_t block_rows,
                               int32_t blocks_per_kv_block, int32_t row_bytes, int64_t src_rows,
                               int64_t dst_rows, uint32_t *status, hs_stream_t stream) {
  if (n_layers < 0 || n_layers > HS_MAX_LAYERS)
    return hs_set_error(HS_ERR_INVALID_ARG, "n_layers %d not in 0..%d", n_layers, HS_MAX_LAYERS);
  if (n_transfers < 0 || block_rows < 1 || blocks_per_kv_block < 1 || src_rows < 0 || dst_rows < 0)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes n_transfers=%d block_rows=%d blocks_per_kv_block=%d",
                        n_transfers, block_rows, blocks_per_kv_block);
  if (row_bytes < 16 || row_bytes % 16 || row_bytes > (1 << 20))
    return hs_set_error(HS_ERR_INVALID_ARG, "row_bytes %d must be a multiple of 16 in 16..2^20", row_bytes);
  if (n_layers == 0 || n_transfers == 0) return HS_OK;
  if (!src_caches || !dst_caches || !src_blocks || !dst_blocks || !page_offsets)
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL argument");
  BackupLayers bl;
  int rc;
  for (int l = 0; l < n_layers; ++l) {
    const void *s = nullptr, *d = nullptr;
    if ((rc = hs_device_alias(src_caches[l], &s, "src_caches[l]"))) return rc;
    if ((rc = hs_device_alias(dst_caches[l], &d, "dst_caches[l]"))) return rc;
    bl.src[l] = reinterpret_cast<const uint4 *>(s);
    bl.dst[l] = reinterpret_cast<uint4 *>(const_cast<void *>(d));
  }
  int dev = 0, nsm = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  const int64_t total = (int64_t)n_layers * n_transfers * block_rows * (row_bytes / 16);
  const int64_t want = (total + 4 * 256 - 1) / (4 * 256);
  const int grid = (int)(want < (int64_t)nsm * 8 ? (want > 0 ? want : 1) : (int64_t)nsm * 8);
  k_backup_pages<<<grid, 256, 0, stream>>>(bl, n_layers, src_blocks, dst_blocks, page_offsets,
                                           n_transfers, block_rows, blocks_per_kv_block,
                                           row_bytes / 16, src_rows, dst_rows, status);
  HS_LAUNCH_CHECK("k_backup_pages");
  return HS_OK;
}
