// a6: sparse attention over the selected latent KV rows (decode: one query row
// per (request, input), H heads sharing one 576-dim latent KV row per selected
// position; values are its first 512 dims).
//
// The consumer of resolve_topk / swap_in on the pages is the DSA attention
// backend ("hiSparse-MTP", section 1: init_attention_backend hands the
// coordinator to the DSA backend; "vllm 分析(十二) HiSparse 下篇",
// resolve_topk returns (attention cache, indices[, valid counts])).
//
// k_attn_umma -- 5th-generation tensor cores (tcgen05) with TMEM accumulators.
//
// Per row, Q (128 heads x 576 bf16 = 147 KB) and O (128 x 512 fp32 = 256 KB,
// all of TMEM) do not fit one SM together with KV tiles. Each row is therefore
// served by two CTAs, c = 0 / 1, each owning value dims [256c, 256c + 256):
//   * O_c (128 x 256 fp32) lives in TMEM columns [0, 256);
//   * Q dims 0..319 live in TMEM columns [256, 416) as the MMA's A operand;
//     Q dims 320..575 live in shared memory (4 x 16 KB, 128-byte swizzle);
//   * S = Q K^T (128 x 32 fp32, all 576 dims -- both CTAs compute it) has
//     three buffers in TMEM columns [416, 512); the softmax overwrites the
//     first 16 columns of its buffer with P (bf16 pairs), which P V then reads
//     from TMEM as its A operand, so a buffer is free again once P V is done;
//   * KV rows are gathered 32 at a time by 16-byte cp.async, each producer
//     thread's copies arriving on the tile's mbarrier as they land
//     (cp.async.mbarrier.arrive). A tile is split by 64-dim swizzle block over
//     two rings: the four blocks of this CTA's value half go to ring B (five
//     16 KB slots), held until P V is done; the other five blocks (the other
//     value half and the rope dims, read by Q K^T only) go to ring A (four
//     20 KB slots), free again as soon as Q K^T is done. A tile is the K-major
//     B operand of Q K^T and, read MN-major from ring B, the B operand of P V.
// Warp roles (384 threads): warps 0-3 softmax + epilogue (thread = head =
// TMEM lane), warps 4-7 gather producers, warps 8-10
// issue Q K^T for tiles t = 0, 1, 2 (mod 3) into three S buffers (one thread
// issues a tcgen05.mma only every ~60-150 cycles, so three chains are kept in
// flight), warp 11 issues P V.
// Online softmax in the log2 domain with lazy rescaling: O is rescaled (in
// TMEM) only when a row's running max grows by more than 2^8.
// Every mbarrier wait is bounded; a wait that gives up sets HS_STATUS_TIMEOUT
// in the caller's status word and the CTA winds down.

#include <math.h>

#include "hs_internal.cuh"

namespace {

constexpr int D = HS_LATENT_DIM;
constexpr int DV = HS_VALUE_DIM;
constexpr int HG = 128;                   // heads per CTA (MMA M)
constexpr int NK = 32;                    // keys per tile (MMA N of Q K^T)
constexpr int ROWB = D * 2;               // 1152
constexpr int NCH = ROWB / 16;            // 72 chunks of 16 B per latent row
constexpr int QT_DIMS = 320;              // Q dims held in TMEM
constexpr int QS_BLOCKS = (D - QT_DIMS) / 64;   // 4 swizzle blocks of Q in SMEM
constexpr int NSB = 3;                    // S buffers = Q K^T chains in flight
constexpr int KV_BLOCKS = D / 64;         // 9 swizzle blocks per KV tile
constexpr int VB_BLOCKS = 4;              // blocks of one value half
constexpr int RA_SLOTS = 4, RB_SLOTS = 5; // ring A (Q K^T only) / ring B (value half)
constexpr int THREADS = 384;
constexpr int NPROD = 128;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int QS_OFF = 0;
constexpr int QS_BYTES = QS_BLOCKS * HG * 128;         // 65536
constexpr int KV_BLOCK_BYTES = NK * 128;               // 4096
constexpr int RA_SLOT_BYTES = (KV_BLOCKS - VB_BLOCKS) * KV_BLOCK_BYTES;   // 20480
constexpr int RB_SLOT_BYTES = VB_BLOCKS * KV_BLOCK_BYTES;                 // 16384
constexpr int RA_OFF = QS_OFF + QS_BYTES;
constexpr int RB_OFF = RA_OFF + RA_SLOTS * RA_SLOT_BYTES;
constexpr int BAR_OFF = RB_OFF + RB_SLOTS * RB_SLOT_BYTES;
constexpr int SMEM_USED = BAR_OFF + 256;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;           // slack for the 1 KB alignment
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t COL_O = 0, COL_Q = 256, COL_S = 416;
static_assert(COL_Q + QT_DIMS / 2 == COL_S && COL_S + NSB * NK == 512, "TMEM column map");

// barriers (8-byte words at BAR_OFF)
enum { B_FULL = 0, B_EMPTYA = B_FULL + RA_SLOTS, B_EMPTYB = B_EMPTYA + RA_SLOTS,
       B_SFULL = B_EMPTYB + RB_SLOTS, B_SFREE = B_SFULL + NSB, B_PFULL = B_SFREE + NSB,
       B_OFULL = B_PFULL + NSB, B_COUNT = B_OFULL + 1 };
static_assert(B_COUNT * 8 + 8 <= 256, "barrier area");

// Shared-memory address of swizzle block a (0..8) of a tile whose ring A /
// ring B slots start at ra / rb, for the CTA owning value half c: blocks
// 4c..4c+3 are in ring B, the others in ring A in ascending order.
__device__ __forceinline__ uint32_t kv_block(uint32_t ra, uint32_t rb, int c, int a) {
  if ((a >> 2) == c && a < 8) return rb + (uint32_t)(a & 3) * KV_BLOCK_BYTES;
  const int pa = (c == 0) ? a - 4 : (a == 8 ? 4 : a);
  return ra + (uint32_t)pa * KV_BLOCK_BYTES;
}

constexpr int WAIT_LIMIT = 1 << 24;

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
  // kind::f16 instruction descriptor: D fp32, A and B bf16, A K-major
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t IDESC_QK = idesc_bf16(128, NK, 0);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, 1);

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// Bounded wait for the phase of the given parity: gives up (false) after
// about 2^31 SM cycles (~1 s) or WAIT_LIMIT polls, whichever comes first.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  for (int i = 0; i < WAIT_LIMIT; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > (1ll << 31)) break;
  }
  return false;
}

// The same wait taken by a whole warp, with one verdict for every lane (the
// warp then issues warp-collective tcgen05 loads and stores).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, bar_wait(bar, parity));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

#define TMEM_LD32(taddr, r)                                                                    \
  asm volatile(                                                                                \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"    \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),         \
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),         \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),         \
        "=r"(r[31])                                                                            \
      : "r"(taddr))
#define TMEM_ST32(taddr, r)                                                                    \
  asm volatile(                                                                                \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"  \
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),         \
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),       \
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),   \
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),   \
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]))
#define TMEM_ST16(taddr, r)                                                                    \
  asm volatile(                                                                                \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
      "%13,%14,%15,%16};\n" ::"r"(taddr),                                                     \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),  \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),       \
      "r"(r[15]))
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// 2^x with the PTX approximate base-2 exponential (flushes subnormal results)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(THREADS, 1)
    k_attn_umma(const char *__restrict__ q, const char *__restrict__ kv, int64_t n_kv,
                const int32_t *__restrict__ idx, int32_t H, int32_t K, float scale_log2,
                __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, uint32_t *status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm);
  const uint32_t bars = sbase + BAR_OFF;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + BAR_OFF + B_COUNT * 8);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_hg = (H + HG - 1) / HG;
  const int c = blockIdx.x & 1;                     // value half
  const int rg = blockIdx.x >> 1;
  const int r = rg / n_hg;
  const int h0 = (rg % n_hg) * HG;
  const int T = (K + NK - 1) / NK;
  const int32_t *idx_row = idx + (int64_t)r * K;

  if (tid == 0) {
    for (int s = 0; s < RA_SLOTS; ++s) {
      bar_init(bar(B_FULL + s), NPROD);
      bar_init(bar(B_EMPTYA + s), 1);
    }
    for (int s = 0; s < RB_SLOTS; ++s) bar_init(bar(B_EMPTYB + s), 1);
    for (int b = 0; b < NSB; ++b) {
      bar_init(bar(B_SFULL + b), 1);
      bar_init(bar(B_SFREE + b), 1);
      bar_init(bar(B_PFULL + b), 4);
    }
    bar_init(bar(B_OFULL), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
        (uint32_t)__cvta_generic_to_shared(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }

  // Q dims 320..575 -> SMEM (four 64-dim swizzle blocks), all threads
  for (int i = tid; i < HG * QS_BLOCKS * 8; i += THREADS) {
    const int hr = i / (QS_BLOCKS * 8), rem = i % (QS_BLOCKS * 8);
    const int j = rem / 8, cc = rem % 8;
    const int h = h0 + hr;
    const bool v = h < H;
    const char *src = v ? q + ((int64_t)r * H + h) * ROWB + (QT_DIMS + 64 * j) * 2 + cc * 16 : q;
    cp_async16(sbase + QS_OFF + j * (HG * 128) + sw128(hr, cc), src, v);
  }
  cp_async_commit();

  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // Q dims 0..319 -> TMEM columns [256, 416): lane = head, column j holds
    // dims 2j, 2j+1
    const int h = h0 + tid;
    const uint4 *qrow = reinterpret_cast<const uint4 *>(q + ((int64_t)r * H + (h < H ? h : 0)) * ROWB);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int part = 0; part < QT_DIMS / 64; ++part) {
      uint32_t v[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint4 w = make_uint4(0, 0, 0, 0);
        if (h < H) w = qrow[part * 8 + k];
        v[4 * k] = w.x; v[4 * k + 1] = w.y; v[4 * k + 2] = w.z; v[4 * k + 3] = w.w;
      }
      TMEM_ST32(lane_base + COL_Q + part * 32, v);
    }
    tmem_wait_st();
  }
  cp_async_wait<0>();
  fence_proxy_async();
  fence_before();
  __syncthreads();
  fence_after();

  bool timed_out = false;

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------ gather producers ----
    const int p = tid - 128;          // 0..127
    const int key = p >> 2;           // 32 keys per tile, 4 threads per key
    const int sub = p & 3;            // chunks sub, sub+4, ..., 18 per thread
    // this thread's key index for tiles t and t+1 is loaded two tiles ahead so
    // the index load never sits between a stage becoming free and its refill
    auto load_id = [&](int t) -> int32_t {
      const int j = t * NK + key;
      return (t < T && j < K) ? __ldg(idx_row + j) : -1;
    };
    int32_t id0 = load_id(0), id1 = load_id(1);
    for (int t = 0; t < T && !timed_out; ++t) {
      const int sa = t % RA_SLOTS, sbv = t % RB_SLOTS;
      const int32_t id = id0;
      id0 = id1;
      id1 = load_id(t + 2);
      if (t >= RA_SLOTS && !bar_wait(bar(B_EMPTYA + sa), ((t / RA_SLOTS) - 1) & 1)) {
        timed_out = true;
        break;
      }
      if (t >= RB_SLOTS && !bar_wait(bar(B_EMPTYB + sbv), ((t / RB_SLOTS) - 1) & 1)) {
        timed_out = true;
        break;
      }
      const bool v = id >= 0 && id < n_kv;
      const char *src = kv + (v ? (int64_t)id * ROWB : 0);
      const uint32_t ra = sbase + RA_OFF + sa * RA_SLOT_BYTES;
      const uint32_t rb = sbase + RB_OFF + sbv * RB_SLOT_BYTES;
      // copy k of this thread is chunk sub + 4k: swizzle block k / 2, chunk
      // sub + 4 (k & 1) within the block's 128-byte row
#pragma unroll
      for (int k = 0; k < NCH / 4; ++k) {
        const int ch = sub + 4 * k;
        cp_async16(kv_block(ra, rb, c, k >> 1) + sw128(key, ch & 7), v ? src + ch * 16 : q, v);
      }
      // the tile's barrier gets this thread's arrival when its copies land
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(
                       bar(B_FULL + sa))
                   : "memory");
    }
    cp_async_wait<0>();
  } else if (warp >= 8 && warp < 8 + NSB) {
    // ------------------------------------------ Q K^T issuers (3 warps) ----
    // warp 8 + b issues tiles t = b, b + 3, ... into S buffer b, so three
    // 36-instruction chains are in flight at once
    if (lane == 0) {
      const uint32_t qs0 = sbase + QS_OFF;
      const int sb = warp - 8;
      bool ok = true;
      for (int t = sb; t < T && ok; t += NSB) {
        const int sa = t % RA_SLOTS;
        ok = bar_wait(bar(B_FULL + sa), (t / RA_SLOTS) & 1);
        if (ok && t >= NSB) ok = bar_wait(bar(B_SFREE + sb), ((t / NSB) - 1) & 1);
        if (!ok) break;
        fence_after();
        fence_proxy_async();   // the tile was written by cp.async (generic proxy)
        const uint32_t ra = sbase + RA_OFF + sa * RA_SLOT_BYTES;
        const uint32_t rb = sbase + RB_OFF + (t % RB_SLOTS) * RB_SLOT_BYTES;
        const uint32_t sd = tmem + COL_S + sb * NK;
#pragma unroll
        for (int kk = 0; kk < QT_DIMS / 16; ++kk)
          mma_ts(sd, tmem + COL_Q + kk * 8,
                 sdesc(kv_block(ra, rb, c, kk >> 2) + (kk & 3) * 32, 16, 1024), IDESC_QK, kk > 0);
#pragma unroll
        for (int kk = QT_DIMS / 16; kk < D / 16; ++kk) {
          const int qk = kk - QT_DIMS / 16;
          mma_ss(sd, sdesc(qs0 + (qk >> 2) * (HG * 128) + (qk & 3) * 32, 16, 1024),
                 sdesc(kv_block(ra, rb, c, kk >> 2) + (kk & 3) * 32, 16, 1024), IDESC_QK, 1);
        }
        mma_commit(bar(B_SFULL + sb));
        mma_commit(bar(B_EMPTYA + sa));   // ring A slot: Q K^T was its last reader
      }
      timed_out = !ok;
    }
  } else if (warp == 8 + NSB) {
    // --------------------------------------------------- P V issuer ----
    if (lane == 0) {
      bool ok = true;
      for (int u = 0; u < T && ok; ++u) {
        const int sb = u % NSB, sbv = u % RB_SLOTS;
        ok = bar_wait(bar(B_PFULL + sb), (u / NSB) & 1);
        if (!ok) break;
        fence_after();
        const uint32_t vbase = sbase + RB_OFF + sbv * RB_SLOT_BYTES;
#pragma unroll
        for (int ks = 0; ks < NK / 16; ++ks)
          mma_ts(tmem + COL_O, tmem + COL_S + sb * NK + ks * 8,
                 sdesc(vbase + ks * 2048, KV_BLOCK_BYTES, 1024), IDESC_PV, (u > 0 || ks > 0));
        mma_commit(bar(B_SFREE + sb));    // S/P buffer may take tile u + 3
        mma_commit(bar(B_EMPTYB + sbv));  // ring B slot may take tile u + 5
      }
      if (ok && T > 0) mma_commit(bar(B_OFULL));
      timed_out = !ok;
    }
  } else {
    // ---------------------------------------------- softmax (warps 0-3) ----
    const int hrow = tid;                          // head row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    // index of key `lane` of tile t, loaded a tile ahead
    auto load_id = [&](int t) -> int32_t {
      return (t < T && t * NK + lane < K) ? __ldg(idx_row + t * NK + lane) : -1;
    };
    int32_t my_id = load_id(0);
    for (int t = 0; t < T; ++t) {
      const int sb = t % NSB;
      if (!warp_wait(bar(B_SFULL + sb), (t / NSB) & 1)) { timed_out = true; break; }
      fence_after();
      uint32_t sr[NK];
      TMEM_LD32(lane_base + COL_S + sb * NK, sr);
      tmem_wait_ld();

      // invalid keys -> -inf in place (warp-uniform skip when all are valid)
      const uint32_t vmask = __ballot_sync(0xffffffffu, my_id >= 0 && my_id < n_kv);
      my_id = load_id(t + 1);
      if (vmask != 0xffffffffu) {
#pragma unroll
        for (int k = 0; k < NK; ++k)
          if (!((vmask >> k) & 1u)) sr[k] = 0xff800000u;
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < NK; ++k) mx[k & 3] = fmaxf(mx[k & 3], __uint_as_float(sr[k]));
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
      // lazy rescale: only when the running max grows by more than 8 (log2)
      const bool grow = mt > m_used + 8.0f;
      const bool need_o = grow && m_used != -INFINITY;
      if (__any_sync(0xffffffffu, need_o)) {
        // O must hold every PV issued so far before it is rescaled
        if (t >= 1 && !warp_wait(bar(B_SFREE + (t - 1) % NSB), ((t - 1) / NSB) & 1)) {
          timed_out = true;
          break;
        }
        fence_after();
        const float alpha = need_o ? ex2(m_used - mt) : 1.0f;
#pragma unroll 1
        for (int part = 0; part < 256 / 32; ++part) {
          uint32_t o[32];
          TMEM_LD32(lane_base + COL_O + part * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          TMEM_ST32(lane_base + COL_O + part * 32, o);
        }
        tmem_wait_st();
        if (need_o) l *= alpha;
      }
      if (grow) m_used = mt;

      // P = exp2(s * scale - m) as bf16 over the first 16 columns of the same
      // buffer (P V reads it from TMEM as its A operand)
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < NK / 2; ++k) {
        const float a = ex2(fmaf(__uint_as_float(sr[2 * k]), scale_log2, -mu));
        const float b = ex2(fmaf(__uint_as_float(sr[2 * k + 1]), scale_log2, -mu));
        ps[k & 3] += a + b;
        sr[k] = pack_bf16(a, b);          // in place: pair k of P
      }
      l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      TMEM_ST16(lane_base + COL_S + sb * NK, sr);
      tmem_wait_st();
      fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(bar(B_PFULL + sb));
    }

    // ---------------------------------------------------------- epilogue --
    const int h = h0 + hrow;
    if (!timed_out && T > 0 && !warp_wait(bar(B_OFULL), 0)) timed_out = true;
    fence_after();
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    __nv_bfloat16 *orow = out + ((int64_t)r * H + (h < H ? h : 0)) * DV + 256 * c;
#pragma unroll 1
    for (int part = 0; part < 256 / 32; ++part) {
      uint32_t o[32];
      if (T > 0 && !timed_out) {
        TMEM_LD32(lane_base + COL_O + part * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0u;
      }
      if (h < H) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow + part * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_uint4(pack_bf16(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                              pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                              pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                              pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
      }
    }
    if (lse && c == 0 && h < H)
      lse[(int64_t)r * H + h] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }

  if (timed_out && status) atomicOr(status, 4u);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
  }
}

}  // namespace

extern "C" int hs_sparse_attn_decode(const void *q, const void *kv, int64_t n_kv_rows,
                                     const int32_t *idx, int32_t R, int32_t H, int32_t K,
                                     float scale, void *out, float *lse, uint32_t *status,
                                     hs_stream_t stream) {
  if (R < 0 || H < 1 || H > 1024 || K < 0 || n_kv_rows < 0)
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes R=%d H=%d (1..1024) K=%d n_kv_rows=%lld",
                        R, H, K, (long long)n_kv_rows);
  if (R == 0) return HS_OK;
  if (!q || !out || (K > 0 && (!idx || (!kv && n_kv_rows > 0))))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL q/kv/idx/out");
  if (((uintptr_t)q & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)out & 15))
    return hs_set_error(HS_ERR_INVALID_ARG, "q, kv and out must be 16-byte aligned");
  if (!(scale == scale)) return hs_set_error(HS_ERR_INVALID_ARG, "scale is NaN");
  int dev = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  static bool attr_done[64] = {false};
  if (dev >= 64 || !attr_done[dev]) {
    HS_CUDA_TRY(cudaFuncSetAttribute(k_attn_umma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_ALLOC));
    if (dev < 64) attr_done[dev] = true;
  }
  const int64_t blocks = (int64_t)R * ((H + HG - 1) / HG) * 2;
  if (blocks > INT32_MAX) return hs_set_error(HS_ERR_UNSUPPORTED, "R*H too large");
  k_attn_umma<<<(unsigned)blocks, THREADS, SMEM_ALLOC, stream>>>(
      reinterpret_cast<const char *>(q), reinterpret_cast<const char *>(kv), n_kv_rows, idx, H,
      K, scale * 1.4426950408889634f, reinterpret_cast<__nv_bfloat16 *>(out), lse, status);
  HS_LAUNCH_CHECK("k_attn_umma");
  return HS_OK;
}
