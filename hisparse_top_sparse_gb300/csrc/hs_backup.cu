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

// next-4: the same data movement row by row ("vllm 分析(十二) HiSparse 下篇",
// section c4a kv cache 写入): after the compressor writes a step's entries,
// runtime.backup_rows copies each written row of the cache to its host slot,
// and for the 128-dim indexer cache hisparse_backup_indexer copies token_stride
// bytes per entry to a host cache whose slots are the source slots compressed
// by compress_hisparse_slot_mapping. One kernel serves both: per (layer,
// entry, unit) a 16- or 4-byte copy, the destination slot computed in the
// kernel when a compression ratio is given.

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

struct RowLayers {
  const char *src[HS_MAX_LAYERS];
  char *dst[HS_MAX_LAYERS];
};

// Host row of entry i: dst_slots[i], or with ratio > 0 the compressed slot
// (dst_slots[i] / (sbs * ratio)) * sbs + (positions[i] % (sbs * ratio)) / ratio.
//
// Each row is copied by `tpr` threads of a block (tpr = min(units per row,
// 256), so a block holds rows_per_block = 256 / tpr rows side by side); a
// thread resolves the slots of TB tokens once and then copies its units of
// those TB rows for every layer, TB loads in flight. Tokens without an entry
// cost one slot load.
constexpr int BR_THREADS = 256;
constexpr int BR_TB = 8;

template <typename U>
__global__ void __launch_bounds__(BR_THREADS) k_backup_rows(const __grid_constant__ RowLayers rl,
                                                            int32_t n_layers,
                                                            const int32_t *__restrict__ src_slots,
                                                            const int32_t *__restrict__ dst_slots,
                                                            const int32_t *__restrict__ positions,
                                                            int32_t n, int32_t vec, int32_t tpr,
                                                            int32_t sbs, int32_t ratio,
                                                            int64_t src_rows, int64_t dst_rows,
                                                            uint32_t *status) {
  const int rows_per_block = BR_THREADS / tpr;
  const int c0 = threadIdx.x % tpr, rloc = threadIdx.x / tpr;
  if (rloc >= rows_per_block) return;              // the block's spare threads (no barriers)
  const int64_t row_stride = (int64_t)gridDim.x * rows_per_block;
  const int lbs = sbs * ratio;
  bool bad = false;
  for (int64_t base = (int64_t)blockIdx.x * rows_per_block + rloc; base < n;
       base += row_stride * BR_TB) {
    int64_t so[BR_TB], dof[BR_TB];                 // unit offsets of the rows, -1 = none
#pragma unroll
    for (int t = 0; t < BR_TB; ++t) {
      const int64_t i = base + t * row_stride;
      so[t] = -1;
      dof[t] = 0;
      if (i < n) {
        const int sr = __ldg(src_slots + i);
        int dr = __ldg(dst_slots + i);
        if (ratio > 0) {
          const int p = __ldg(positions + i);
          dr = (dr < 0 || p < 0) ? -1 : (dr / lbs) * sbs + (p % lbs) / ratio;
        }
        if (sr >= 0 && dr >= 0) {
          if (sr < src_rows && dr < dst_rows) {
            so[t] = (int64_t)sr * vec;
            dof[t] = (int64_t)dr * vec;
          } else {
            bad = true;
          }
        }
      }
    }
    for (int l = 0; l < n_layers; ++l) {
      const U *src = reinterpret_cast<const U *>(rl.src[l]);
      U *dst = reinterpret_cast<U *>(rl.dst[l]);
      for (int c = c0; c < vec; c += tpr) {
        U v[BR_TB];
#pragma unroll
        for (int t = 0; t < BR_TB; ++t)
          if (so[t] >= 0) v[t] = src[so[t] + c];
#pragma unroll
        for (int t = 0; t < BR_TB; ++t)
          if (so[t] >= 0) dst[dof[t] + c] = v[t];
      }
    }
  }
  if (bad && status) atomicOr(status, HS_STATUS_INDEX);
}

// Rows whose size (or whose host cache) is not a multiple of 16 bytes: each
// row is cut into the 16-byte-aligned chunks of the destination it overlaps;
// a chunk wholly inside the row is written with one 16-byte store (its four
// words loaded one by one from the source), the partial chunks at the row's
// two ends word by word. Stores over the host link stay mostly 16 bytes wide.
template <int TB>
__global__ void __launch_bounds__(BR_THREADS) k_backup_rows_narrow(
    const __grid_constant__ RowLayers rl, int32_t n_layers, const int32_t *__restrict__ src_slots,
    const int32_t *__restrict__ dst_slots, const int32_t *__restrict__ positions, int32_t n,
    int32_t words, int32_t tpr, int32_t sbs, int32_t ratio, int64_t src_rows, int64_t dst_rows,
    uint32_t *status) {
  const int chunks = (words + 3) / 4 + 1;          // aligned chunks a row can touch
  const int rows_per_block = BR_THREADS / tpr;
  const int c0 = threadIdx.x % tpr, rloc = threadIdx.x / tpr;
  if (rloc >= rows_per_block) return;              // the block's spare threads (no barriers)
  const int64_t row_stride = (int64_t)gridDim.x * rows_per_block;
  const int lbs = sbs * ratio;
  bool bad = false;
  for (int64_t base = (int64_t)blockIdx.x * rows_per_block + rloc; base < n;
       base += row_stride * TB) {
    int64_t so[TB], dof[TB];                       // word offsets of the rows, -1 = none
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const int64_t i = base + t * row_stride;
      so[t] = -1;
      dof[t] = 0;
      if (i < n) {
        const int sr = __ldg(src_slots + i);
        int dr = __ldg(dst_slots + i);
        if (ratio > 0) {
          const int p = __ldg(positions + i);
          dr = (dr < 0 || p < 0) ? -1 : (dr / lbs) * sbs + (p % lbs) / ratio;
        }
        if (sr >= 0 && dr >= 0) {
          if (sr < src_rows && dr < dst_rows) {
            so[t] = (int64_t)sr * words;
            dof[t] = (int64_t)dr * words;
          } else {
            bad = true;
          }
        }
      }
    }
    for (int l = 0; l < n_layers; ++l) {
      const uint32_t *src = reinterpret_cast<const uint32_t *>(rl.src[l]);
      // word index 0 of `dst` is the 16-byte aligned address at or below the
      // cache's start; `mis` words lie between the two
      const int mis = (int)((reinterpret_cast<uintptr_t>(rl.dst[l]) >> 2) & 3);
      uint32_t *dst = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(rl.dst[l]) & ~(uintptr_t)15);
      for (int k = c0; k < chunks; k += tpr) {
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          if (so[t] < 0) continue;
          const int64_t d = dof[t] + mis;          // the row's first word, from dst
          const int64_t c4 = (d & ~(int64_t)3) + 4 * k;
          const int64_t w0 = c4 - d;               // row word at the chunk's start
          if (w0 >= words) continue;
          if (w0 >= 0 && w0 + 4 <= words) {
            const uint32_t *sp = src + so[t] + w0;
            *reinterpret_cast<uint4 *>(dst + c4) = make_uint4(sp[0], sp[1], sp[2], sp[3]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (w0 + e >= 0 && w0 + e < words) dst[c4 + e] = src[so[t] + w0 + e];
          }
        }
      }
    }
  }
  if (bad && status) atomicOr(status, HS_STATUS_INDEX);
}

// Short rows that do not go 16 bytes at a time (token_stride not a multiple
// of 16, or a host cache off 16-byte alignment): a warp takes RUN_EPL * 32
// consecutive entries, compacts the ones with a row to copy (in entry order)
// and works through them 32 at a time. Entries whose host rows are
// consecutive form a run; the run's rows are staged in the warp's shared
// memory as the run's byte image and written out as the 16-byte-aligned
// chunks of host memory they cover, the run's partial first and last chunks
// word by word. A backup of whole blocks (consecutive host rows) is thus
// written in whole lines over the host link; scattered rows are runs of one.
constexpr int RUN_EPL = 4;
constexpr int RUN_WARPS = 4;

__global__ void __launch_bounds__(RUN_WARPS * 32) k_backup_runs(
    const __grid_constant__ RowLayers rl, int32_t n_layers, const int32_t *__restrict__ src_slots,
    const int32_t *__restrict__ dst_slots, const int32_t *__restrict__ positions, int32_t n,
    int32_t words, int32_t sbs, int32_t ratio, int64_t src_rows, int64_t dst_rows,
    uint32_t *status) {
  extern __shared__ uint32_t run_smem[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint32_t *img = run_smem + (size_t)wib * (32 * words + 64);   // 32 rows' image
  int32_t *s_sr = reinterpret_cast<int32_t *>(img + 32 * words);  // their device rows
  int32_t *s_dr = s_sr + 32;                                       // their host rows
  const int lbs = sbs * ratio;
  const int64_t G = 32 * RUN_EPL;
  const int64_t n_groups = ((int64_t)n + G - 1) / G;
  const unsigned lt = (1u << lane) - 1u;
  bool bad = false;
  for (int64_t g = (int64_t)blockIdx.x * RUN_WARPS + wib; g < n_groups;
       g += (int64_t)gridDim.x * RUN_WARPS) {
    int32_t sr[RUN_EPL], dr[RUN_EPL];
    unsigned vm[RUN_EPL];
    int total = 0;
#pragma unroll
    for (int e = 0; e < RUN_EPL; ++e) {
      const int64_t i = g * G + e * 32 + lane;
      bool v = false;
      sr[e] = -1;
      dr[e] = -1;
      if (i < n) {
        sr[e] = __ldg(src_slots + i);
        dr[e] = __ldg(dst_slots + i);
        if (ratio > 0) {
          const int p = __ldg(positions + i);
          dr[e] = (dr[e] < 0 || p < 0) ? -1 : (dr[e] / lbs) * sbs + (p % lbs) / ratio;
        }
        if (sr[e] >= 0 && dr[e] >= 0) {
          if (sr[e] < src_rows && dr[e] < dst_rows) v = true;
          else bad = true;
        }
      }
      vm[e] = __ballot_sync(0xffffffffu, v);
      total += __popc(vm[e]);
    }
    for (int b0 = 0; b0 < total; b0 += 32) {
      const int nb = min(32, total - b0);
      int base = 0;
#pragma unroll
      for (int e = 0; e < RUN_EPL; ++e) {
        if ((vm[e] >> lane) & 1u) {
          const int k = base + __popc(vm[e] & lt) - b0;
          if (k >= 0 && k < 32) { s_sr[k] = sr[e]; s_dr[k] = dr[e]; }
        }
        base += __popc(vm[e]);
      }
      __syncwarp();
      const unsigned rs =
          __ballot_sync(0xffffffffu, lane < nb && (lane == 0 || s_dr[lane] != s_dr[lane - 1] + 1));
      for (int l = 0; l < n_layers; ++l) {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(rl.src[l]);
        for (int w = lane; w < nb * words; w += 32) {
          const int k = w / words;
          img[w] = src[(int64_t)s_sr[k] * words + (w - k * words)];
        }
        __syncwarp();
        // word 0 of `dst` is the 16-byte aligned address at or below the
        // cache's start; `mis` words lie between the two
        const int mis = (int)((reinterpret_cast<uintptr_t>(rl.dst[l]) >> 2) & 3);
        uint32_t *dst = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(rl.dst[l]) & ~(uintptr_t)15);
        unsigned m = rs;
        while (m) {
          const int k0 = __ffs(m) - 1;
          m &= m - 1;
          const int k1 = m ? __ffs(m) - 1 : nb;
          const int64_t d0 = (int64_t)s_dr[k0] * words + mis;    // the run's first host word
          const int64_t d1 = d0 + (int64_t)(k1 - k0) * words;
          const int64_t i0 = (int64_t)k0 * words - d0;           // image index = host word + i0
          for (int64_t c = (d0 >> 2) + lane; c < ((d1 + 3) >> 2); c += 32) {
            const int64_t w0 = 4 * c;
            if (w0 >= d0 && w0 + 4 <= d1) {
              const uint32_t *ip = img + (w0 + i0);
              *reinterpret_cast<uint4 *>(dst + w0) = make_uint4(ip[0], ip[1], ip[2], ip[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (w0 + e >= d0 && w0 + e < d1) dst[w0 + e] = img[w0 + e + i0];
            }
          }
        }
        __syncwarp();
      }
    }
  }
  if (bad && status) atomicOr(status, HS_STATUS_INDEX);
}

int backup_rows_impl(int32_t n_layers, const void *const *src_caches, void *const *dst_caches,
                     const int32_t *src_slots, const int32_t *dst_slots,
                     const int32_t *positions, int32_t n, int32_t sbs, int32_t ratio,
                     int32_t token_stride, int64_t src_rows, int64_t dst_rows, uint32_t *status,
                     hs_stream_t stream) {
  if (n_layers < 0 || n_layers > HS_MAX_LAYERS)
    return hs_set_error(HS_ERR_INVALID_ARG, "n_layers %d not in 0..%d", n_layers, HS_MAX_LAYERS);
  if (n < 0 || src_rows < 0 || dst_rows < 0)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes n=%d src_rows=%lld dst_rows=%lld", n,
                        (long long)src_rows, (long long)dst_rows);
  if (token_stride < 4 || token_stride % 4 || token_stride > (1 << 20))
    return hs_set_error(HS_ERR_INVALID_ARG,
                        "token_stride %d must be a multiple of 4 in 4..2^20", token_stride);
  if (n_layers == 0 || n == 0) return HS_OK;
  if (!src_caches || !dst_caches || !src_slots || !dst_slots || (ratio > 0 && !positions))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL argument");
  RowLayers rl;
  bool wide = token_stride % 16 == 0;
  int rc;
  for (int l = 0; l < n_layers; ++l) {
    const void *sp = nullptr, *dp = nullptr;
    if ((rc = hs_device_alias(src_caches[l], &sp, "src_caches[l]", 4))) return rc;
    if ((rc = hs_device_alias(dst_caches[l], &dp, "dst_caches[l]", 4))) return rc;
    if (((uintptr_t)sp & 15) || ((uintptr_t)dp & 15)) wide = false;
    rl.src[l] = reinterpret_cast<const char *>(sp);
    rl.dst[l] = reinterpret_cast<char *>(const_cast<void *>(dp));
  }
  const int vec = wide ? token_stride / 16 : token_stride / 4;
  // narrow rows of 256 bytes and more go by 16-byte-aligned destination chunks
  // (1152-byte rows at a 4-byte offset: 151 against 129 GB/s over the link);
  // shorter ones a word per thread (132-byte rows: 87 against 65 GB/s)
  const bool chunked = !wide && vec >= 64;
  if (!wide && !chunked) {
    const size_t smem = (size_t)RUN_WARPS * (32 * vec + 64) * sizeof(uint32_t);
    static bool attr_done[64] = {false};
    int dev = 0, nsm = 0;
    HS_CUDA_TRY(cudaGetDevice(&dev));
    HS_CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    if (dev >= 64 || !attr_done[dev]) {
      HS_CUDA_TRY(cudaFuncSetAttribute(k_backup_runs, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)((size_t)RUN_WARPS * (32 * 63 + 64) * sizeof(uint32_t))));
      if (dev < 64) attr_done[dev] = true;
    }
    const int64_t groups = ((int64_t)n + 32 * RUN_EPL - 1) / (32 * RUN_EPL);
    const int64_t want = (groups + RUN_WARPS - 1) / RUN_WARPS;
    const int grid = (int)(want < (int64_t)nsm * 4 ? want : (int64_t)nsm * 4);
    k_backup_runs<<<grid, RUN_WARPS * 32, smem, stream>>>(rl, n_layers, src_slots, dst_slots,
                                                          positions, n, vec, sbs, ratio, src_rows,
                                                          dst_rows, status);
    HS_LAUNCH_CHECK("k_backup_runs");
    return HS_OK;
  }
  const int units = chunked ? vec / 4 + 2 : vec;
  const int tpr = units < BR_THREADS ? units : BR_THREADS;
  const int rows_per_block = BR_THREADS / tpr;
  int dev = 0, nsm = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  const int tb = BR_TB;
  const int64_t want = ((int64_t)n + (int64_t)rows_per_block * tb - 1) / ((int64_t)rows_per_block * tb);
  const int grid = (int)(want < (int64_t)nsm * 8 ? want : (int64_t)nsm * 8);
  if (wide)
    k_backup_rows<uint4><<<grid, BR_THREADS, 0, stream>>>(rl, n_layers, src_slots, dst_slots,
                                                          positions, n, vec, tpr, sbs, ratio,
                                                          src_rows, dst_rows, status);
  else if (chunked)
    k_backup_rows_narrow<BR_TB><<<grid, BR_THREADS, 0, stream>>>(rl, n_layers, src_slots, dst_slots,
                                                                 positions, n, vec, tpr, sbs, ratio,
                                                                 src_rows, dst_rows, status);
  else
    k_backup_rows<uint32_t><<<grid, BR_THREADS, 0, stream>>>(rl, n_layers, src_slots, dst_slots,
                                                             positions, n, vec, tpr, sbs, ratio,
                                                             src_rows, dst_rows, status);
  HS_LAUNCH_CHECK("k_backup_rows");
  return HS_OK;
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

extern "C" int hs_backup_rows(int32_t n_layers, const void *const *src_caches,
                              void *const *dst_caches, const int32_t *src_slots,
                              const int32_t *dst_slots, int32_t n, int32_t token_stride,
                              int64_t src_rows, int64_t dst_rows, uint32_t *status,
                              hs_stream_t stream) {
  return backup_rows_impl(n_layers, src_caches, dst_caches, src_slots, dst_slots, nullptr, n, 0,
                          0, token_stride, src_rows, dst_rows, status, stream);
}

extern "C" int hs_backup_indexer(int32_t n_layers, const void *const *src_caches,
                                 void *const *dst_caches, const int32_t *src_slots,
                                 const int32_t *host_slots, const int32_t *positions, int32_t n,
                                 int32_t storage_block_size, int32_t compress_ratio,
                                 int32_t token_stride, int64_t src_rows, int64_t dst_rows,
                                 uint32_t *status, hs_stream_t stream) {
  if (storage_block_size < 1 || compress_ratio < 1 ||
      (int64_t)storage_block_size * compress_ratio > INT32_MAX)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad storage_block_size %d / compress_ratio %d",
                        storage_block_size, compress_ratio);
  return backup_rows_impl(n_layers, src_caches, dst_caches, src_slots, host_slots, positions, n,
                          storage_block_size, compress_ratio, token_stride, src_rows, dst_rows,
                          status, stream);
}
