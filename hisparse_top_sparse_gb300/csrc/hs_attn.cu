// a6: sparse attention over the selected latent KV rows (decode, one query
// row per (request, input), H heads sharing one 576-dim latent KV row per
// selected position; values are its first 512 dims).
//
// The consumer of resolve_topk / swap_in on the pages is the DSA attention
// backend ("hiSparse-MTP", section 1: init_attention_backend hands the
// coordinator to the DSA backend; "vllm 分析(十二) HiSparse 下篇",
// resolve_topk returns (attention cache, indices[, valid counts])).
//
// Kernel k_attn_mma: one CTA per (query row, group of 64 heads), 8 warps.
//   * Q of the 64 heads (64 x 576 bf16) is staged once in shared memory.
//   * The row's selected KV rows are gathered 64 at a time with 16-byte
//     cp.async into a double-buffered tile (64 x 1152 B); invalid or padding
//     entries are zero-filled and masked to -inf in the scores.
//   * S = Q K^T on bf16 mma.sync tensor-core instructions (fp32 accumulate):
//     warp w computes heads 16*(w%4).. x keys 32*(w/4)..; online softmax in
//     the log2 domain with the running max shared through shared memory.
//   * O += P V: P goes to shared memory as bf16; warp w owns value dims
//     64*w .. 64*w+63 of all 64 heads (128 fp32 accumulators per thread).
//   * Shared-memory rows are XOR-swizzled in 16-byte chunks so that every
//     ldmatrix phase touches 8 distinct bank groups.

#include <math.h>

#include "hs_internal.cuh"

namespace {

constexpr int D = HS_LATENT_DIM;
constexpr int DV = HS_VALUE_DIM;
constexpr int HG = 64;                 // heads per CTA
constexpr int NT = 64;                 // keys per tile
constexpr int ROWB = D * 2;            // 1152 bytes per latent row
constexpr int NCH = ROWB / 16;         // 72 chunks of 16 bytes
constexpr int THREADS = 256;

constexpr int SQ_OFF = 0;
constexpr int SKV_OFF = SQ_OFF + HG * ROWB;          // two tiles
constexpr int SP_OFF = SKV_OFF + 2 * NT * ROWB;      // P tile, 64 x 64 bf16
constexpr int SMAX_OFF = SP_OFF + HG * NT * 2;       // [2][64] float
constexpr int SSUM_OFF = SMAX_OFF + 2 * HG * 4;      // [2][64] float
constexpr int SALPHA_OFF = SSUM_OFF + 2 * HG * 4;    // [64] float
constexpr int SVALID_OFF = SALPHA_OFF + HG * 4;      // [2][64] int
constexpr int SMEM_BYTES = SVALID_OFF + 2 * NT * 4;  // 231,168
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)((chunk & ~7) | ((chunk ^ row) & 7));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(THREADS, 1)
    k_attn_mma(const char *__restrict__ q, const char *__restrict__ kv, int64_t n_kv,
               const int32_t *__restrict__ idx, int32_t H, int32_t K, float scale_log2,
               __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sQ = sbase + SQ_OFF;
  const uint32_t sKV = sbase + SKV_OFF;
  const uint32_t sP = sbase + SP_OFF;
  float *sMax = reinterpret_cast<float *>(smem + SMAX_OFF);
  float *sSum = reinterpret_cast<float *>(smem + SSUM_OFF);
  float *sAlpha = reinterpret_cast<float *>(smem + SALPHA_OFF);
  int *sValid = reinterpret_cast<int *>(smem + SVALID_OFF);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, qd = lane & 3;
  const int n_hg = (H + HG - 1) / HG;
  const int r = blockIdx.x / n_hg;           // head groups of a row are adjacent,
  const int h0 = (blockIdx.x % n_hg) * HG;   // so the row's KV is read once from HBM
  const int mt = warp & 3, nh = warp >> 2;
  const int ntiles = (K + NT - 1) / NT;
  const int32_t *idx_row = idx + (int64_t)r * K;

  // Q of this head group (rows beyond H are zero)
  for (int i = tid; i < HG * NCH; i += THREADS) {
    const int hr = i / NCH, c = i % NCH;
    const int h = h0 + hr;
    const bool v = h < H;
    const char *src = q + (((int64_t)r * H + (v ? h : 0)) * ROWB) + c * 16;
    cp_async16(sQ + hr * ROWB + swz(hr, c) * 16, src, v);
  }
  auto issue_tile = [&](int t, int st) {
    const uint32_t dst0 = sKV + st * NT * ROWB;
    for (int i = tid; i < NT * NCH; i += THREADS) {
      const int kr = i / NCH, c = i % NCH;
      const int j = t * NT + kr;
      const int32_t id = (j < K) ? idx_row[j] : -1;
      const bool v = id >= 0 && id < n_kv;
      if (c == 0) sValid[st * NT + kr] = v;
      const char *src = v ? kv + (int64_t)id * ROWB + c * 16 : q;
      cp_async16(dst0 + kr * ROWB + swz(kr, c) * 16, src, v);
    }
  };
  if (ntiles > 0) issue_tile(0, 0);
  cp_async_commit();

  float o[4][8][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[a][b][c] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    cp_async_wait_all();
    __syncthreads();  // tile t is in; every warp is done with tile t-1
    if (t + 1 < ntiles) issue_tile(t + 1, st ^ 1);
    cp_async_commit();
    const uint32_t tile = sKV + st * NT * ROWB;

    // ---- S = Q K^T: heads 16*mt.., keys 32*nh.. ----
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
    const int arow = 16 * mt + (lane & 15);
#pragma unroll 4
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sQ + arow * ROWB + swz(arow, 2 * kk + (lane >> 4)) * 16, a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int key = 32 * nh + 16 * np + (lane & 7) + ((lane >> 4) << 3);
        const int ch = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tile + key * ROWB + swz(key, ch) * 16, b0, b1, b2, b3);
        mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }

    // ---- online softmax (log2 domain) ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = 32 * nh + 8 * nt + 2 * qd + e;
        const bool v = sValid[st * NT + key] != 0;
        acc[nt][e] = v ? acc[nt][e] * scale_log2 : -INFINITY;
        acc[nt][2 + e] = v ? acc[nt][2 + e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, acc[nt][e]);
        mx1 = fmaxf(mx1, acc[nt][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const int row0 = 16 * mt + g, row1 = row0 + 8;
    if (qd == 0) {
      sMax[nh * HG + row0] = mx0;
      sMax[nh * HG + row1] = mx1;
    }
    __syncthreads();
    const float tm0 = fmaxf(sMax[row0], sMax[HG + row0]);
    const float tm1 = fmaxf(sMax[row1], sMax[HG + row1]);
    const float mn0 = fmaxf(m_run[0], tm0), mn1 = fmaxf(m_run[1], tm1);
    const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m_run[0] - mn0);
    const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m_run[1] - mn1);
    const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
    m_run[0] = mn0;
    m_run[1] = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p00 = exp2f(acc[nt][0] - mu0), p01 = exp2f(acc[nt][1] - mu0);
      const float p10 = exp2f(acc[nt][2] - mu1), p11 = exp2f(acc[nt][3] - mu1);
      ps0 += p00 + p01;
      ps1 += p10 + p11;
      const int chunk = 4 * nh + nt;  // 8 keys per 16-byte chunk
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + row0 * 128 + swz(row0, chunk) * 16 +
                                                       qd * 4),
                   "r"(pack_bf16(p00, p01)));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + row1 * 128 + swz(row1, chunk) * 16 +
                                                       qd * 4),
                   "r"(pack_bf16(p10, p11)));
    }
    l_run[0] = l_run[0] * al0 + ps0;
    l_run[1] = l_run[1] * al1 + ps1;
    if (nh == 0 && qd == 0) {
      sAlpha[row0] = al0;
      sAlpha[row1] = al1;
    }
    __syncthreads();

    // ---- O = O * alpha + P V: value dims 64*warp .. ----
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float x0 = sAlpha[16 * m + g], x1 = sAlpha[16 * m + g + 8];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        o[m][n][0] *= x0; o[m][n][1] *= x0;
        o[m][n][2] *= x1; o[m][n][3] *= x1;
      }
    }
#pragma unroll
    for (int ks = 0; ks < NT / 16; ++ks) {
      uint32_t pa[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int prow = 16 * m + (lane & 15);
        ldsm_x4(sP + prow * 128 + swz(prow, 2 * ks + (lane >> 4)) * 16, pa[m][0], pa[m][1],
                pa[m][2], pa[m][3]);
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = 8 * warp + 2 * np + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tile + key * ROWB + swz(key, ch) * 16, b0, b1, b2, b3);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          mma_bf16(o[m][2 * np], pa[m][0], pa[m][1], pa[m][2], pa[m][3], b0, b1);
          mma_bf16(o[m][2 * np + 1], pa[m][0], pa[m][1], pa[m][2], pa[m][3], b2, b3);
        }
      }
    }
  }
  cp_async_wait_all();

  // ---- epilogue: row sums, output, lse ----
  l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
  l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
  l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
  l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
  if (qd == 0) {
    sSum[nh * HG + 16 * mt + g] = l_run[0];
    sSum[nh * HG + 16 * mt + g + 8] = l_run[1];
    if (nh == 0) {
      sMax[16 * mt + g] = m_run[0];
      sMax[16 * mt + g + 8] = m_run[1];
    }
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < 4; ++m) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = 16 * m + g + 8 * hh;
      const int h = h0 + row;
      if (h >= H) continue;
      const float l = sSum[row] + sSum[HG + row];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16 *orow = out + ((int64_t)r * H + h) * DV + 64 * warp + 2 * qd;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        *reinterpret_cast<uint32_t *>(orow + 8 * n) =
            pack_bf16(o[m][n][2 * hh] * inv, o[m][n][2 * hh + 1] * inv);
      }
    }
  }
  if (lse && tid < HG && h0 + tid < H) {
    const float l = sSum[tid] + sSum[HG + tid];
    lse[(int64_t)r * H + h0 + tid] =
        l > 0.f ? (sMax[tid] + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }
}

}  // namespace

extern "C" int hs_sparse_attn_decode(const void *q, const void *kv, int64_t n_kv_rows,
                                     const int32_t *idx, int32_t R, int32_t H, int32_t K,
                                     float scale, void *out, float *lse, hs_stream_t stream) {
  if (R < 0 || H < 1 || H > 1024 || K < 0 || n_kv_rows < 0)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes R=%d H=%d (1..1024) K=%d n_kv_rows=%lld",
                        R, H, K, (long long)n_kv_rows);
  if (R == 0) return HS_OK;
  if (!q || !out || (K > 0 && (!idx || (!kv && n_kv_rows > 0))))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL q/kv/idx/out");
  if (((uintptr_t)q & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)out & 3))
    return hs_set_error(HS_ERR_INVALID_ARG, "q and kv must be 16-byte aligned, out 4-byte");
  if (!(scale == scale)) return hs_set_error(HS_ERR_INVALID_ARG, "scale is NaN");
  int dev = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  static bool attr_done[64] = {false};
  if (dev >= 64 || !attr_done[dev]) {
    HS_CUDA_TRY(cudaFuncSetAttribute(k_attn_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_BYTES));
    if (dev < 64) attr_done[dev] = true;
  }
  const int64_t blocks = (int64_t)R * ((H + HG - 1) / HG);
  if (blocks > INT32_MAX) return hs_set_error(HS_ERR_UNSUPPORTED, "R*H too large");
  k_attn_mma<<<(unsigned)blocks, THREADS, SMEM_BYTES, stream>>>(
      reinterpret_cast<const char *>(q), reinterpret_cast<const char *>(kv), n_kv_rows, idx, H,
      K, scale * 1.4426950408889634f, reinterpret_cast<__nv_bfloat16 *>(out), lse);
  HS_LAUNCH_CHECK("k_attn_mma");
  return HS_OK;
}
