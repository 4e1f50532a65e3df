// a6: sparse attention over the selected latent KV rows (decode: one query row
// per (request, input), H heads sharing one 576-dim latent KV row per selected
// position; values are its first 512 dims).
//
// The consumer of resolve_topk / swap_in on the pages is the DSA attention
// backend ("hiSparse-MTP", section 1: init_attention_backend hands the
// coordinator to the DSA backend; "vllm 分析(十二) HiSparse 下篇",
// resolve_topk returns (attention cache, indices[, valid counts])).
//
// k_attn_pair -- 5th-generation tensor cores (tcgen05) with TMEM accumulators,
// one two-CTA cluster per (query row, group of 128 heads).
//
// Per row, Q (128 heads x 576 bf16 = 147 KB) and O (128 x 512 fp32 = 256 KB,
// all of TMEM) do not fit one SM together with KV tiles, so the row's work is
// split over the two CTAs of a cluster, c = 0 / 1:
//   * CTA c owns value dims [256c, 256c + 256): O_c (128 x 256 fp32) lives in
//     its TMEM columns [0, 256);
//   * the selected keys come in tiles of 32; CTA c computes S = Q K^T (all 576
//     dims) and the softmax numerators P only for its own tiles t = c, c + 2,
//     ...; Q dims 0..383 sit in TMEM columns [256, 448) as the MMA's A
//     operand, dims 384..575 in shared memory (3 x 16 KB, 128-byte swizzle);
//     S has two 32-column TMEM buffers [448, 512), and the softmax writes P
//     (bf16 pairs) over the first 16 columns of its buffer;
//   * P of an own tile goes to the CTA's own P V (read from TMEM) and to the
//     peer's P V (read from shared memory): each softmax warp stages its 32
//     rows in this CTA's shared memory and sends them with one 2 KB bulk
//     copy into the peer's; the peer's P V commit arrives back on this CTA's
//     mbarrier (tcgen05.commit multicast), freeing both buffers (one
//     staging and one receiving buffer per CTA: the next own tile's P waits
//     for the peer's P V of the previous one);
//   * the KV rows of an own tile are gathered whole (16-byte cp.async, each
//     producer thread's copies arriving on the tile's mbarrier as they land):
//     the four 64-dim swizzle blocks of this CTA's value half into ring VO
//     (4 slots), the other five into ring A (3 slots, each freed once its
//     Q K^T is done); of a peer tile only this CTA's value half is
//     gathered, into ring VP (2 slots), and two own tiles later than it
//     would be in tile order: its rows are read only once the peer's P has
//     come, so a VP slot is held about 1.3 us instead of 3;
//   * both CTAs use one softmax reference per head: the larger of their first
//     tiles' maxima, agreed through distributed shared memory before any P is
//     made, so every P of the row is on one scale and O is never rescaled. A
//     later tile whose maximum exceeds the reference by more than 2^30 marks
//     the row, and the pair then runs the row again with the exact maximum
//     (exchanged at the end of the first pass) as the reference. The row sum
//     l is the sum of both CTAs' partial sums.
// Warp roles (480 threads): warps 0-3 softmax, P exchange and epilogue (thread
// = head = TMEM lane), warps 4-11 gather producers (eight threads per key, one
// 16-byte chunk of each 64-dim block per thread), warps 12-13 issue Q K^T for
// own tiles into S buffers 0 / 1, warp 14 issues P V for every tile. The
// gathers and the P V walk the tiles pair by pair with the CTA's own tile
// first (CTA 1 takes tile 2k + 1 before 2k): the peer's P comes through
// distributed shared memory about half a microsecond after the CTA's own P
// of the same pair, and an own tile queued behind it would hold its ring
// slots that much longer.
// The kernel is a programmatic dependent launch: its prologue (barriers, TMEM,
// Q) overlaps the previous kernel (hs_resolve_topk releases it at entry), and
// it reads the indices and request flags after griddepcontrol.wait.
// Every mbarrier wait is bounded; a wait that gives up sets HS_STATUS_TIMEOUT
// in the caller's status word and the CTA winds down.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "hs_internal.cuh"

namespace {

constexpr int D = HS_LATENT_DIM;
constexpr int DV = HS_VALUE_DIM;
constexpr int HG = 128;                   // heads per cluster (MMA M)
constexpr int NK = 32;                    // keys per tile (MMA N of Q K^T)
constexpr int ROWB = D * 2;               // 1152
constexpr int NCH = ROWB / 16;            // 72 chunks of 16 B per latent row
constexpr int QT_DIMS = 384;              // Q dims held in TMEM
constexpr int QS_BLOCKS = (D - QT_DIMS) / 64;   // 3 swizzle blocks of Q in SMEM
constexpr int NSB = 2;                    // S / P buffers (own tiles)
constexpr int VB_BLOCKS = 4;              // swizzle blocks of one value half
constexpr int RA_SLOTS = 3, VO_SLOTS = 4, VP_SLOTS = 2, XP_SLOTS = 1;
constexpr int PEER_LAG = 2;               // own tiles gathered ahead of the peer tiles
constexpr int THREADS = 480;
// Registers per thread, at most: a swap-in gather block (256 threads, 56
// registers each) must fit beside one attention CTA in each of the SM's four
// register-file quarters (16 K registers; four attention warps and two gather
// warps share one) so that the one-call step overlaps its copies with the
// attention. 4 x 96 x 32 + 2 x 56 x 32 = 15,872; at 98 (rounded to 104) it
// no longer fits and the copies wait for whole SMs.
#define ATTN_MAX_REGS 96
static_assert(THREADS * ATTN_MAX_REGS <= 65536, "register budget");
constexpr int NPROD = 256;
constexpr float REF_SLACK = 30.0f;        // P <= 2^30 on the shared reference

// shared memory (offsets from a 1024-byte aligned base)
constexpr int KV_BLOCK_BYTES = NK * 128;                    // 4096
constexpr int QS_OFF = 0;
constexpr int QS_BYTES = QS_BLOCKS * HG * 128;              // 49152
constexpr int RA_SLOT_BYTES = (D / 64 - VB_BLOCKS) * KV_BLOCK_BYTES;   // 20480
constexpr int V_SLOT_BYTES = VB_BLOCKS * KV_BLOCK_BYTES;              // 16384
constexpr int P_SLOT_BYTES = HG * NK * 2;                   // 8192: 128 rows x 64 B, 64-byte swizzle
constexpr int RA_OFF = QS_OFF + QS_BYTES;
constexpr int VO_OFF = RA_OFF + RA_SLOTS * RA_SLOT_BYTES;
constexpr int XS_OFF = VO_OFF + VO_SLOTS * V_SLOT_BYTES;    // own P staged for the bulk copy
constexpr int XP_OFF = XS_OFF + XP_SLOTS * P_SLOT_BYTES;    // the peer's P
constexpr int VP_OFF = XP_OFF + XP_SLOTS * P_SLOT_BYTES;
constexpr int XMAX_OFF = VP_OFF + VP_SLOTS * V_SLOT_BYTES;  // peer's first-tile maxima
constexpr int XEND_OFF = XMAX_OFF + HG * 4;                 // peer's (l or mark, max) per pass
constexpr int BAR_OFF = XEND_OFF + 2 * HG * 8;
constexpr int SMEM_USED = BAR_OFF + 512;
// 1 KB of slack to align the base to 1024 bytes (the 128-byte swizzled tiles
// need it) at run time; declaring the alignment instead gave slower code. The
// SM keeps 3 KB of shared memory beside one CTA for a small kernel (the
// swap-in gather).
constexpr int SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
static_assert(RA_OFF % 1024 == 0 && VO_OFF % 1024 == 0 && VP_OFF % 1024 == 0 &&
                  XS_OFF % 1024 == 0 && XP_OFF % 1024 == 0, "slot alignment");

// TMEM columns
constexpr uint32_t COL_O = 0, COL_Q = 256, COL_S = 448;
static_assert(COL_Q + QT_DIMS / 2 == COL_S && COL_S + NSB * NK == 512, "TMEM column map");

// barriers (8-byte words at BAR_OFF)
enum {
  B_FULLA = 0,                        // own tile landed (NPROD arrivals)
  B_EMPTYA = B_FULLA + RA_SLOTS,      // ring A slot: Q K^T done
  B_EMPTYVO = B_EMPTYA + RA_SLOTS,    // ring VO slot: own P V done
  B_FULLVP = B_EMPTYVO + VO_SLOTS,    // peer tile's value half landed (NPROD arrivals)
  B_EMPTYVP = B_FULLVP + VP_SLOTS,    // ring VP slot: P V done
  B_SFULL = B_EMPTYVP + VP_SLOTS,     // S ready
  B_SFREE = B_SFULL + NSB,            // own P V done with the S / P buffer
  B_PFULL = B_SFREE + NSB,            // P in TMEM (4 softmax warps)
  B_XPFULL = B_PFULL + NSB,           // the peer's P landed here (1 arrival + bytes)
  B_XPFREE = B_XPFULL + XP_SLOTS,     // the peer is done with our P in its slot
  B_XMAX = B_XPFREE + XP_SLOTS,       // the peer's first-tile maxima landed
  B_XEND = B_XMAX + 1,                // the peer's end-of-pass figures (one per pass)
  B_VOTE = B_XEND + 2,                // the four softmax warps have voted for a second pass
  B_DECIDE = B_VOTE + 1,              // softmax -> other roles: second pass or not
  B_OFULL = B_DECIDE + 1,             // all P V of a pass done (one per pass)
  B_QLOAD = B_OFULL + 2,              // Q landed (9 x 16 KB by tensor copies)
  B_QSTAGED = B_QLOAD + 1,            // Q dims 0..383 are in TMEM (4 softmax warps)
  B_COUNT = B_QSTAGED + 1
};
static_assert(B_COUNT * 8 + 16 <= 512, "barrier area");
// O staged for the epilogue's stores: four 16 KB blocks over ring A and the
// start of ring VO (free once the last P V is done)
constexpr int O_STG_OFF = RA_OFF;
static_assert(O_STG_OFF + 4 * HG * 128 <= XS_OFF, "O staging");

constexpr int WAIT_LIMIT = 1 << 24;

// Shared-memory address of swizzle block a (0..8) of an own tile whose ring A
// / ring VO slots start at ra / rv, for the CTA owning value half c: blocks
// 4c..4c+3 are in ring VO, the others in ring A in ascending order.
__device__ __forceinline__ uint32_t kv_block(uint32_t ra, uint32_t rv, int c, int a) {
  if ((a >> 2) == c && a < 8) return rv + (uint32_t)(a & 3) * KV_BLOCK_BYTES;
  const int pa = (c == 0) ? a - 4 : (a == 8 ? 4 : a);
  return ra + (uint32_t)pa * KV_BLOCK_BYTES;
}

// Staging place of Q block a (dims 64a..64a+63, a < 6) before it moves into
// TMEM: slots 1-2 of ring A (two blocks), slots 1-3 of ring VO (three
// blocks), the two P buffers (one block). Slot 0 of rings A and VO and all of
// ring VP are left for the first tiles, which are gathered meanwhile.
__host__ __device__ constexpr uint32_t q_stage_off(int a) {
  return a < 2 ? RA_OFF + RA_SLOT_BYTES + a * (HG * 128)
               : a < 5 ? VO_OFF + V_SLOT_BYTES + (a - 2) * (HG * 128) : XS_OFF;
}
static_assert(q_stage_off(1) + HG * 128 <= RA_OFF + RA_SLOTS * RA_SLOT_BYTES &&
                  q_stage_off(4) + HG * 128 == XS_OFF && XS_OFF + HG * 128 == VP_OFF &&
                  q_stage_off(0) % 1024 == 0 && q_stage_off(1) % 1024 == 0 &&
                  q_stage_off(2) % 1024 == 0 && q_stage_off(5) % 1024 == 0 && RA_SLOTS == 3 &&
                  VO_SLOTS == 4 && XP_SLOTS == 1,
              "Q staging map");

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ uint64_t sdesc64(uint32_t addr) {
  // the same for K-major rows of 64 bytes, 64-byte swizzle: 8-row groups of
  // 512 bytes
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(512 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)4 << 61);
}
// byte offset of 16-byte chunk j (keys 8j..8j+7) of row `row` in a P slot
__device__ __forceinline__ uint32_t sw64(uint32_t row, uint32_t j) {
  return row * 64 + ((j ^ ((row >> 1) & 3)) << 4);
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
  // kind::f16 instruction descriptor: D fp32, A and B bf16, A K-major
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t IDESC_QK = idesc_bf16(128, NK, 0);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, 1);

// MMA issue: a warp elects one lane once (elect_one), and that lane issues a
// whole group of MMAs and commits with the single-thread helpers below. One
// lane issuing a straight run keeps the tensor pipe fed (~16 cycles per
// M=128, N=32, K=16 MMA); an elect.sync around every MMA costs ~80 cycles
// each, which then bounds Q K^T.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\nselp.u32 %0, 1, 0, e;\n}\n" : "=r"(e));
  return e != 0;
}
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
// commits (the issuing lane); the multicast form's arrival lands at the same
// offset in the CTAs of `mask`
__device__ __forceinline__ void mma_commit_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n" ::"r"(bar), "h"(mask)
      : "memory");
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
// max_cycles SM cycles or WAIT_LIMIT polls, whichever comes first.
__device__ __forceinline__ bool bar_wait_n(uint32_t bar, uint32_t parity, long long max_cycles) {
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
    if (clock64() - t0 > max_cycles) break;
  }
  return false;
}
// the kernel's waits: about 2^31 SM cycles (~1 s)
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  return bar_wait_n(bar, parity, 1ll << 31);
}

// The same wait taken by a whole warp, with one answer for every lane (the
// warp then issues warp-collective tcgen05 loads and stores).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, bar_wait(bar, parity));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
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


// ---- cluster helpers --------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// named barrier `id` over the first `n` threads of the CTA (whole warps)
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
// the cluster barrier in two halves: arrive (this thread's earlier writes
// released) and wait (the other CTA's writes before its arrival acquired)
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}
// 8 / 4 bytes into the peer's shared memory; the peer's mbarrier `rbar`
// counts the bytes when they land
__device__ __forceinline__ void st_async_v2(uint32_t addr, uint32_t a, uint32_t b, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];\n" ::"r"(addr),
      "r"(a), "r"(b), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];\n" ::"r"(addr),
               "r"(v), "r"(rbar)
               : "memory");
}
// `bytes` of this CTA's shared memory into the peer's, counted by the peer's
// mbarrier `rbar` when they land (both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                             uint32_t rbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          dst),
      "r"(src), "r"(bytes), "r"(rbar)
      : "memory");
}
// this thread's arrival plus the bytes still to come in the current phase
__device__ __forceinline__ void arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// bounded wait on a barrier that the peer CTA completes (cluster-scope acquire)
__device__ __forceinline__ bool bar_wait_cluster(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  for (int i = 0; i < WAIT_LIMIT; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > (1ll << 31)) break;
  }
  return false;
}
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, bar_wait_cluster(bar, parity));
}

__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(ATTN_MAX_REGS)
    k_attn_pair(const __grid_constant__ CUtensorMap tmap_q,
                const char *__restrict__ q,
                const char *__restrict__ kv_res, int64_t n_res, const char *__restrict__ kv_hot,
                int64_t n_hot, const int32_t *__restrict__ row_req,
                const int32_t *__restrict__ fully_resident, int32_t n_reqs,
                const int32_t *__restrict__ idx, int32_t H, int32_t K, float scale_log2,
                __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, uint32_t *status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm);
  const uint32_t bars = sbase + BAR_OFF;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + BAR_OFF + B_COUNT * 8);
  volatile uint32_t *s_redo = tmem_slot + 1;
  volatile uint32_t *s_last = tmem_slot + 2;   // the last pass run (0 or 1)
  volatile uint32_t *s_fail = tmem_slot + 3;   // a wait of warps 0-7 gave up
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 12 + NSB && lane == 0)
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
  const int c = (int)cluster_rank();                // value half; own tiles t = c mod 2
  const uint32_t peer = (uint32_t)(c ^ 1);
  const int n_hg = (H + HG - 1) / HG;
  const int rg = blockIdx.x >> 1;
  const int r = rg / n_hg;
  const int h0 = (rg % n_hg) * HG;
  const int T = (K + NK - 1) / NK;
  const int n_own = T > c ? (T - c + 1) / 2 : 0;
  const int n_peer = T - n_own;
  const int32_t *idx_row = idx + (int64_t)r * K;
  // Position i of the tile sequence that the gathers and the P V issuer walk:
  // every pair of tiles with this CTA's own tile first (CTA 1 swaps the
  // pairs), so that an own tile's P V never waits behind the peer's P.
  auto tile_at = [&](int i) -> int {
    return (c == 1 && i < T && (i ^ 1) < T) ? (i ^ 1) : i;
  };

  if (warp == 1) {
    // one barrier per lane: its arrival count
    static_assert(B_COUNT <= 32, "one lane per barrier");
    if (lane < B_COUNT) {
      const int i = lane;
      const bool prod = (i >= B_FULLA && i < B_FULLA + RA_SLOTS) || (i >= B_FULLVP && i < B_FULLVP + VP_SLOTS);
      const bool four = (i >= B_PFULL && i < B_PFULL + NSB) || i == B_VOTE;
      bar_init(bar(i), prod ? NPROD : four ? 4 : 1);
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (lane == 0) {
      *s_redo = 0u;
      *s_last = 0u;
      *s_fail = 0u;
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
        (uint32_t)__cvta_generic_to_shared(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }

  // This CTA's barriers and TMEM exist: the CTA proceeds at once, and it
  // arrives on the cluster barrier, whose wait the warps that write into the
  // peer CTA (softmax and P V issuer) take before their first remote write.
  // The other warps take it just before the closing cluster barrier.
  fence_before();
  __syncthreads();
  fence_after();
  cluster_arrive();
  const uint32_t tmem = *tmem_slot;
  // Q by nine tensor copies of 128 heads x 64 dims (16 KB, 128-byte swizzle,
  // rows past H filled with zeros), all issued by this CTA into its own
  // shared memory: dims 384..575 land in SMEM as the MMA's A operand, dims
  // 0..383 in a staging area over the (still empty) slots 1 and 2 of ring
  // A, 1 to 3 of ring VO and the P buffers, from where one lane moves them
  // into TMEM. Slot 0 of rings A and VO and ring VP stay free, so the first
  // own and the first peer tiles are gathered while Q comes in.
  // The copies are issued by the P V issuer warp, whose first MMA waits for
  // the first P anyway: issuing them can stall the issuing thread for
  // microseconds while the other CTAs of the wave load their Q.
  if (warp == 12 + NSB && lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    arrive_expect_tx(bar(B_QLOAD), 9 * HG * 128);
    for (int a = 0; a < D / 64; ++a) {
      const uint32_t dst = a < 6 ? sbase + q_stage_off(a) : sbase + QS_OFF + (a - 6) * (HG * 128);
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
          "l"(reinterpret_cast<uint64_t>(&tmap_q)), "r"(64 * a), "r"(h0), "r"(r), "r"(bar(B_QLOAD))
          : "memory");
    }
  }
  bool timed_out = false;
  int own_sent = 0;        // own tiles whose P went to the peer (softmax warps)
  if (warp == 0) {
    // staged Q dims 0..383 -> TMEM columns [256, 448), the layout the Q K^T
    // MMAs read their A operand in: one 128-row x 32-byte tensor-memory copy
    // per 16-dim slice (the slice the MMA would read from shared memory),
    // issued by one lane; their completion (B_QSTAGED) frees the staging
    // slots for KV tiles and lets the Q K^T issuers start
    if (!warp_wait(bar(B_QLOAD), 0)) timed_out = true;
    fence_after();
    if (elect_one()) {
#pragma unroll 1
      for (int kk = 0; kk < QT_DIMS / 16; ++kk)
        asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;\n" ::"r"(tmem + COL_Q + kk * 8),
                     "l"(sdesc(sbase + q_stage_off(kk >> 2) + (kk & 3) * 32, 16, 1024))
                     : "memory");
      mma_commit(bar(B_QSTAGED));
    }
    __syncwarp();
  }

  // Up to here the kernel has read only q. It is launched as a programmatic
  // dependent of the kernel before it (hs_resolve_topk lets it start at once),
  // so that its prologue overlaps that kernel: the indices and the request
  // flags are read only after that kernel has finished.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // the row's cache: the paged resident cache while its request is fully
  // resident, else the hot buffer its swap-in indices address
  // (a request id outside [0, n_reqs) leaves the row without a valid entry)
  const int32_t req = fully_resident ? (row_req ? __ldg(row_req + r) : r) : 0;
  const bool req_ok = !fully_resident || (req >= 0 && req < n_reqs);
  const bool hot = req_ok && fully_resident && __ldg(fully_resident + req) == 0;
  const char *kv = hot ? kv_hot : kv_res;
  const int64_t n_kv = !req_ok ? 0 : hot ? n_hot : n_res;
  if (!req_ok && status && tid == 0 && c == 0) atomicOr(status, HS_STATUS_INDEX);


  if (warp >= 4 && warp < 12) {
    // ------------------------------------------------ gather producers ----
    const int p = tid - 128;          // 0..255
    const int key = p >> 3;           // 32 keys per tile, 8 threads per key
    const int sub = p & 7;            // chunk sub of every 64-dim block
    auto load_id = [&](int t) -> int32_t {
      const int j = t * NK + key;
      return (t < T && j < K) ? __ldg(idx_row + j) : -1;
    };
    int ig = 0, jg = 0;               // own / peer tiles issued, over both passes
    for (int pass = 0; pass < 2 && !timed_out; ++pass) {
      if (pass == 1) {
        if (!bar_wait(bar(B_DECIDE), 0)) { timed_out = true; break; }
        if (!*s_redo) break;
      }
      // gather order: the own tiles run up to PEER_LAG + 1 ahead of the
      // peer tiles, whose value halves are read only once the peer's P has
      // come, so that a ring VP slot is taken only shortly before its use
      int na = 0, nb = 0;             // own / peer tiles of this pass taken
      int la = 0, lb = 0;             // the same two steps ahead (index prefetch)
      auto step = [&](int &a, int &b) -> int {
        if (a < n_own && (b >= n_peer || a < b + PEER_LAG + 1)) return 2 * (a++) + c;
        if (b < n_peer) return 2 * (b++) + (1 - c);
        return T;
      };
      const int t0 = step(la, lb);
      const int t1 = step(la, lb);
      int32_t id0 = load_id(t0), id1 = load_id(t1);
      for (int i = 0; i < T; ++i) {
        const int t = step(na, nb);
        const int32_t id = id0;
        id0 = id1;
        id1 = load_id(step(la, lb));
        const bool v = id >= 0 && id < n_kv;
        const char *src = kv + (v ? (int64_t)id * ROWB : 0);
        if ((t & 1) == c) {
          const int sa = ig % RA_SLOTS, so = ig % VO_SLOTS;
          // slots 1 and 2 hold staged Q until it is in TMEM
          if (ig == 1 && !bar_wait(bar(B_QSTAGED), 0)) {
            timed_out = true;
            break;
          }
          if (ig >= RA_SLOTS && !bar_wait(bar(B_EMPTYA + sa), ((ig / RA_SLOTS) - 1) & 1)) {
            timed_out = true;
            break;
          }
          if (ig >= VO_SLOTS && !bar_wait(bar(B_EMPTYVO + so), ((ig / VO_SLOTS) - 1) & 1)) {
            timed_out = true;
            break;
          }
          const uint32_t ra = sbase + RA_OFF + sa * RA_SLOT_BYTES;
          const uint32_t rv = sbase + VO_OFF + so * V_SLOT_BYTES;
          // copy k of this thread is chunk sub + 4k: swizzle block k / 2,
          // chunk sub + 4 (k & 1) within the block's 128-byte row
#pragma unroll
          for (int k = 0; k < NCH / 8; ++k) {
            const int ch = sub + 8 * k;
            cp_async16(kv_block(ra, rv, c, k) + sw128(key, sub), v ? src + ch * 16 : q, v);
          }
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar(B_FULLA + sa))
                       : "memory");
          ++ig;
        } else {
          const int sp = jg % VP_SLOTS;
          if (jg >= VP_SLOTS && !bar_wait(bar(B_EMPTYVP + sp), ((jg / VP_SLOTS) - 1) & 1)) {
            timed_out = true;
            break;
          }
          const uint32_t rv = sbase + VP_OFF + sp * V_SLOT_BYTES;
          // only this CTA's value half: copies k = 8c .. 8c + 7 of the 18
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int ch = 32 * c + sub + 8 * k;
            cp_async16(rv + k * KV_BLOCK_BYTES + sw128(key, sub), v ? src + ch * 16 : q, v);
          }
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar(B_FULLVP + sp))
                       : "memory");
          ++jg;
        }
      }
    }
    cp_async_wait<0>();
  } else if (warp >= 12 && warp < 12 + NSB) {
    // ------------------------------------- Q K^T issuers (own tiles) ----
    // warp 12 + b issues own tiles ig = b, b + 2, ... into S buffer b
    {
      const uint32_t qs0 = sbase + QS_OFF;
      const int b = warp - 12;
      bool ok = warp_wait(bar(B_QSTAGED), 0);   // Q dims 0..383 in TMEM
      fence_after();
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          ok = warp_wait(bar(B_DECIDE), 0);
          if (!ok || !*s_redo) break;
        }
        for (int il = 0; il < n_own && ok; ++il) {
          const int ig = pass * n_own + il;
          if (ig % NSB != b) continue;
          const int sa = ig % RA_SLOTS;
          ok = warp_wait(bar(B_FULLA + sa), (ig / RA_SLOTS) & 1);
          if (ok && ig >= NSB) ok = warp_wait(bar(B_SFREE + b), ((ig / NSB) - 1) & 1);
          if (!ok) break;
          fence_after();
          fence_proxy_async();   // the tile was written by cp.async (generic proxy)
          const uint32_t ra = sbase + RA_OFF + sa * RA_SLOT_BYTES;
          const uint32_t rv = sbase + VO_OFF + (ig % VO_SLOTS) * V_SLOT_BYTES;
          const uint32_t sd = tmem + COL_S + b * NK;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < QT_DIMS / 16; ++kk)
              mma_ts(sd, tmem + COL_Q + kk * 8,
                     sdesc(kv_block(ra, rv, c, kk >> 2) + (kk & 3) * 32, 16, 1024), IDESC_QK, kk > 0);
#pragma unroll
            for (int kk = QT_DIMS / 16; kk < D / 16; ++kk) {
              const int qk = kk - QT_DIMS / 16;
              mma_ss(sd, sdesc(qs0 + (qk >> 2) * (HG * 128) + (qk & 3) * 32, 16, 1024),
                     sdesc(kv_block(ra, rv, c, kk >> 2) + (kk & 3) * 32, 16, 1024), IDESC_QK, 1);
            }
            mma_commit(bar(B_SFULL + b));
            mma_commit(bar(B_EMPTYA + sa));   // ring A slot: Q K^T was its last reader
          }
          __syncwarp();
        }
      }
      timed_out = !ok;
    }
  } else if (warp == 12 + NSB) {
    // ------------------------- P V issuer (every tile, own tile of a pair first) ----
    __syncwarp();
    cluster_wait();                                // the peer's barriers exist
    {
      bool ok = true;
      int ig = 0, jg = 0;
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          ok = warp_wait(bar(B_DECIDE), 0);
          if (!ok || !*s_redo) break;
        }
        for (int i = 0; i < T && ok; ++i) {
          const int t = tile_at(i);
          if ((t & 1) == c) {
            const int sb = ig % NSB, so = ig % VO_SLOTS;
            ok = warp_wait(bar(B_PFULL + sb), (ig / NSB) & 1);
            if (!ok) break;
            fence_after();
            const uint32_t vb = sbase + VO_OFF + so * V_SLOT_BYTES;
            if (elect_one()) {
#pragma unroll
              for (int ks = 0; ks < NK / 16; ++ks)
                mma_ts(tmem + COL_O, tmem + COL_S + sb * NK + ks * 8,
                       sdesc(vb + ks * 2048, KV_BLOCK_BYTES, 1024), IDESC_PV, (i > 0 || ks > 0));
              mma_commit(bar(B_SFREE + sb));    // S / P buffer may take own tile ig + 2
              mma_commit(bar(B_EMPTYVO + so));
            }
            __syncwarp();
            ++ig;
          } else {
            const int sp = jg % VP_SLOTS, xs = jg % XP_SLOTS;
            ok = warp_wait(bar(B_FULLVP + sp), (jg / VP_SLOTS) & 1);
            if (ok) {
              if (lane == 0) arrive_expect_tx(bar(B_XPFULL + xs), HG * 64);
              __syncwarp();
              ok = warp_wait_cluster(bar(B_XPFULL + xs), (jg / XP_SLOTS) & 1);
            }
            if (!ok) break;
            fence_after();
            fence_proxy_async();   // V by cp.async, P by a bulk copy
            const uint32_t vb = sbase + VP_OFF + sp * V_SLOT_BYTES;
            if (elect_one()) {
#pragma unroll
              for (int ks = 0; ks < NK / 16; ++ks)
                mma_ss(tmem + COL_O, sdesc64(sbase + XP_OFF + xs * P_SLOT_BYTES + ks * 32),
                       sdesc(vb + ks * 2048, KV_BLOCK_BYTES, 1024), IDESC_PV, (i > 0 || ks > 0));
              mma_commit(bar(B_EMPTYVP + sp));
              mma_commit_multicast(bar(B_XPFREE + xs), (uint16_t)(1u << peer));   // the peer may refill
            }
            __syncwarp();
            ++jg;
          }
        }
        if (ok && T > 0) {
          if (elect_one()) mma_commit(bar(B_OFULL + pass));
          __syncwarp();
        }
      }
      timed_out = !ok;
    }
  } else if (warp < 4) {
    // -------------------------------- softmax + P exchange (warps 0-3) ----
    __syncwarp();
    cluster_wait();                                // the peer's barriers exist
    const int hrow = tid;                          // head row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t peer_xp = peer_addr(sbase + XP_OFF, peer) + (uint32_t)warp * 32 * 64;
    float ref = 0.f, l = 0.f, l_peer = 0.f, m_ex = -INFINITY;
    bool flag = false, ref_unset = false, decided = false;
    int ig = 0, last_pass = 0;
    auto load_id = [&](int t) -> int32_t {
      return (t < T && t * NK + lane < K) ? __ldg(idx_row + t * NK + lane) : -1;
    };
    // the peer's first-tile maxima, taken once
    auto agree_ref = [&](float mt) -> bool {
      st_async_b32(peer_addr(sbase + XMAX_OFF, peer) + hrow * 4, __float_as_uint(mt),
                   peer_addr(bar(B_XMAX), peer));
      if (!warp_wait_cluster(bar(B_XMAX), 0)) return false;
      const float pm = reinterpret_cast<volatile float *>(sm + XMAX_OFF)[hrow];
      ref = fmaxf(mt, pm);
      if (ref == -INFINITY) {   // neither first tile has a valid key
        ref = 0.f;
        ref_unset = true;
      }
      return true;
    };
    if (tid == 0) arrive_expect_tx(bar(B_XMAX), HG * 4);
    for (int pass = 0; pass < 2 && !timed_out; ++pass) {
      if (tid == 0) arrive_expect_tx(bar(B_XEND + pass), HG * 8);
      int32_t my_id = load_id(c);
      for (int il = 0; il < n_own; ++il, ++ig) {
        const int t = 2 * il + c;
        const int sb = ig % NSB;
        if (!warp_wait(bar(B_SFULL + sb), (ig / NSB) & 1)) { timed_out = true; break; }
        fence_after();
        uint32_t sr[NK];
        TMEM_LD32(lane_base + COL_S + sb * NK, sr);
        tmem_wait_ld();

        // invalid keys -> -inf in place (warp-uniform skip when all are valid)
        const uint32_t vmask = __ballot_sync(0xffffffffu, my_id >= 0 && my_id < n_kv);
        my_id = load_id(t + 2);
        if (vmask != 0xffffffffu) {
#pragma unroll
          for (int k = 0; k < NK; ++k)
            if (!((vmask >> k) & 1u)) sr[k] = 0xff800000u;
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < NK; ++k) mx[k & 3] = fmaxf(mx[k & 3], __uint_as_float(sr[k]));
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
        if (pass == 0) {
          m_ex = fmaxf(m_ex, mt);
          if (il == 0 && !agree_ref(mt)) { timed_out = true; break; }
          if (ref_unset ? (mt != -INFINITY) : (mt > ref + REF_SLACK)) flag = true;
        }

        // P = exp2(s * scale - ref) as bf16 pairs over the first 16 columns
        // of the S buffer (P V reads it from TMEM as its A operand)
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < NK / 2; ++k) {
          const float a = ex2(fmaf(__uint_as_float(sr[2 * k]), scale_log2, -ref));
          const float b = ex2(fmaf(__uint_as_float(sr[2 * k + 1]), scale_log2, -ref));
          ps[k & 3] += a + b;
          sr[k] = pack_bf16(a, b);          // in place: pair k of P
        }
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        TMEM_ST16(lane_base + COL_S + sb * NK, sr);
        tmem_wait_st();
        fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(bar(B_PFULL + sb));

        // the same P to the peer, into slot ig % XP_SLOTS of its P buffer
        // (64-byte swizzled K-major rows, the A operand layout of its P V):
        // staged in this CTA's slot of the same number, then one 2 KB bulk
        // copy per warp. The peer's P V commit on a slot (XPFREE) means that
        // the copy out of the staging slot has landed as well.
        const int xs = ig % XP_SLOTS;
        if (ig >= XP_SLOTS && !warp_wait_cluster(bar(B_XPFREE + xs), ((ig / XP_SLOTS) - 1) & 1)) {
          timed_out = true;
          break;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(sm + XS_OFF + xs * P_SLOT_BYTES + sw64(hrow, j)) =
              make_uint4(sr[4 * j], sr[4 * j + 1], sr[4 * j + 2], sr[4 * j + 3]);
        fence_proxy_async();     // the bulk copy reads through the async proxy
        __syncwarp();
        if (lane == 0)
          bulk_to_peer(peer_xp + xs * P_SLOT_BYTES,
                       sbase + XS_OFF + xs * P_SLOT_BYTES + warp * 32 * 64, 32 * 64,
                       peer_addr(bar(B_XPFULL + xs), peer));
      }
      if (timed_out) break;
      if (pass == 0 && n_own == 0 && !agree_ref(-INFINITY)) { timed_out = true; break; }

      // end of pass: (l, running max, flag) to the peer, the peer's back
      // l < 0 carries a mark for a second pass (only the first pass marks)
      st_async_v2(peer_addr(sbase + XEND_OFF + pass * HG * 8, peer) + hrow * 8,
                  __float_as_uint(pass == 0 && flag ? -1.f : l), __float_as_uint(m_ex),
                  peer_addr(bar(B_XEND + pass), peer));
      if (!warp_wait_cluster(bar(B_XEND + pass), 0)) { timed_out = true; break; }
      const volatile uint32_t *pe =
          reinterpret_cast<const volatile uint32_t *>(sm + XEND_OFF + pass * HG * 8) + hrow * 2;
      l_peer = __uint_as_float(pe[0]);
      const float m_peer = __uint_as_float(pe[1]);
      const bool f_peer = pass == 0 && l_peer < 0.f;
      last_pass = pass;
      if (pass == 1) break;
      // second pass iff any head of either CTA was marked
      if (__any_sync(0xffffffffu, flag || f_peer) && lane == 0) atomicOr((uint32_t *)s_redo, 1u);
      __syncwarp();
      if (lane == 0) bar_arrive(bar(B_VOTE));
      if (!warp_wait(bar(B_VOTE), 0)) { timed_out = true; break; }
      const bool redo = *s_redo != 0u;
      if (tid == 0) bar_arrive(bar(B_DECIDE));
      decided = true;
      if (!redo) break;
      ref = fmaxf(m_ex, m_peer);
      if (ref == -INFINITY) ref = 0.f;
      l = 0.f;
    }
    if (!decided && tid == 0) bar_arrive(bar(B_DECIDE));   // lets the other roles wind down

    // 1 / l of the head for the epilogue (the first-tile maxima's slot is
    // free: the reference was agreed in the first pass)
    const int h = h0 + hrow;
    const float lt = l + l_peer;
    reinterpret_cast<volatile float *>(sm + XMAX_OFF)[hrow] = lt > 0.f ? 1.0f / lt : 0.f;
    if (lse && c == 0 && h < H)
      lse[(int64_t)r * H + h] = lt > 0.f ? (ref + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
    if (tid == 0) *s_last = (uint32_t)last_pass;
    own_sent = ig;
  }

  // ------------------------------------------------------------ epilogue ----
  // Warps 0-7 (two per TMEM lane quarter, 128 columns each) read O once the
  // last P V is done, scale it by 1 / l, write it as bf16 into four 128-byte
  // swizzled 16 KB blocks over the free ring A, and each half (four warps)
  // copies its two blocks to the output with coalesced 16-byte stores (rows
  // past H skipped). A tensor store instead kept the CTA ~1 us waiting for
  // the copy to read shared memory; these stores drain after the CTA.
  if (warp < 8) {
    if (timed_out) atomicOr((uint32_t *)s_fail, 1u);
    named_bar_sync(1, 256);             // 1 / l, the pass count and failures are in place
    bool ok = *s_fail == 0u && T > 0;
    if (ok) {
      ok = warp_wait(bar(B_OFULL + *s_last), 0);
      if (!ok) timed_out = true;
    }
    fence_after();
    const int q4 = warp & 3, half = warp >> 2;
    const int row = q4 * 32 + lane;
    const float inv = ok ? reinterpret_cast<volatile float *>(sm + XMAX_OFF)[row] : 0.f;
    const uint32_t lane_q = tmem + ((uint32_t)(q4 * 32) << 16);
#pragma unroll 1
    for (int pp = 0; pp < 4; pp += 2) {
      const int p0 = half * 4 + pp;
      uint32_t o[2][32];
      if (ok) {
        TMEM_LD32(lane_q + COL_O + p0 * 32, o[0]);
        TMEM_LD32(lane_q + COL_O + (p0 + 1) * 32, o[1]);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[0][k] = o[1][k] = 0u;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int part = p0 + u;
        unsigned char *blk = sm + O_STG_OFF + (part >> 1) * (HG * 128) + row * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = (part & 1) * 4 + k;
          *reinterpret_cast<uint4 *>(blk + ((j ^ (row & 7)) << 4)) =
              make_uint4(pack_bf16(__uint_as_float(o[u][8 * k]) * inv, __uint_as_float(o[u][8 * k + 1]) * inv),
                         pack_bf16(__uint_as_float(o[u][8 * k + 2]) * inv, __uint_as_float(o[u][8 * k + 3]) * inv),
                         pack_bf16(__uint_as_float(o[u][8 * k + 4]) * inv, __uint_as_float(o[u][8 * k + 5]) * inv),
                         pack_bf16(__uint_as_float(o[u][8 * k + 6]) * inv, __uint_as_float(o[u][8 * k + 7]) * inv));
        }
      }
    }
    // each half (four warps) copies its two blocks out as soon as it has
    // written them: lane l of a warp takes 16-byte chunk l & 7 of block
    // 2 half + ((l >> 3) & 1) of row 8 it + 2 w + (l >> 4), so one warp
    // store writes two whole 256-byte row segments; nothing waits for the
    // stores, and the shared memory is free once it has been read
    if (half == 0)
      named_bar_sync(2, 128);
    else
      named_bar_sync(3, 128);
    {
      const int wq = warp & 3, b = 2 * half + ((lane >> 3) & 1), j = lane & 7;
      const unsigned char *src = sm + O_STG_OFF + b * (HG * 128);
      __nv_bfloat16 *dst_row = out + ((int64_t)r * H + h0) * DV + 256 * c + 64 * b + 8 * j;
#pragma unroll 4
      for (int it = 0; it < HG / 8; ++it) {
        const int row = 8 * it + 2 * wq + (lane >> 4);
        const uint4 v = *reinterpret_cast<const uint4 *>(src + row * 128 + ((j ^ (row & 7)) << 4));
        if (h0 + row < H) *reinterpret_cast<uint4 *>(dst_row + (int64_t)row * DV) = v;
      }
    }
    if (tid == 0) {
      // every P sent must have been consumed by the peer (its multicast
      // commit arrives here) before this CTA's shared memory goes away
      if (!timed_out) {
        for (int xs = 0; xs < XP_SLOTS; ++xs) {
          const int uses = own_sent > xs ? (own_sent - xs + XP_SLOTS - 1) / XP_SLOTS : 0;
          if (uses > 0 && !bar_wait_cluster(bar(B_XPFREE + xs), (uses - 1) & 1)) timed_out = true;
        }
      }
    }
  }

  if (timed_out && status) atomicOr(status, HS_STATUS_TIMEOUT);
  __syncwarp();
  if (warp >= 4 && warp < 12 + NSB) cluster_wait();   // the opening barrier's wait
  fence_before();
  cluster_sync();          // the peer writes into this CTA's shared memory until here
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
  }
}

}  // namespace

// A wait that runs out: one warp takes the kernel's bounded wait, cut to
// max_cycles, on an mbarrier phase that nothing completes, and reports
// HS_STATUS_TIMEOUT the way k_attn_pair does.
__global__ void k_wait_probe(uint32_t *status, long long max_cycles) {
  __shared__ uint64_t probe_bar;
  const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&probe_bar);
  if (threadIdx.x == 0) bar_init(bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, bar_wait_n(bar, 0, max_cycles));
  if (!ok && threadIdx.x == 0) atomicOr(status, HS_STATUS_TIMEOUT);
}

extern "C" int hs_wait_probe(uint32_t *status, int64_t max_cycles, hs_stream_t stream) {
  if (!status) return hs_set_error(HS_ERR_INVALID_ARG, "NULL status");
  if (max_cycles < 1 || max_cycles > (1ll << 31))
    return hs_set_error(HS_ERR_INVALID_ARG, "max_cycles %lld not in 1..2^31", (long long)max_cycles);
  k_wait_probe<<<1, 32, 0, stream>>>(status, (long long)max_cycles);
  HS_LAUNCH_CHECK("k_wait_probe");
  return HS_OK;
}

static int set_attn_attributes() {
  int dev = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  static bool attr_done[64] = {false};
  if (dev >= 64 || !attr_done[dev]) {
    HS_CUDA_TRY(cudaFuncSetAttribute(k_attn_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_ALLOC));
    if (dev < 64) attr_done[dev] = true;
  }
  return HS_OK;
}

int hs_attn_block_attrs(cudaFuncAttributes *attr, int *threads, size_t *dyn_smem) {
  int rc = set_attn_attributes();
  if (rc) return rc;
  HS_CUDA_TRY(cudaFuncGetAttributes(attr, k_attn_pair));
  *threads = THREADS;
  *dyn_smem = SMEM_ALLOC;
  return HS_OK;
}

int hs_attn_wave_rows(int32_t H, int32_t *rows) {
  int rc = set_attn_attributes();
  if (rc) return rc;
  int dev = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  static int clusters[64] = {0};
  int n = dev < 64 ? clusters[dev] : 0;
  if (n == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    HS_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, k_attn_pair, &cfg));
    if (n < 1) n = 1;
    if (dev < 64) clusters[dev] = n;
  }
  const int per_row = (H + HG - 1) / HG;
  *rows = n / per_row > 0 ? n / per_row : 1;
  return HS_OK;
}

extern "C" int hs_sparse_attn_decode_mixed(const void *q, const void *kv_resident,
                                           int64_t n_resident, const void *kv_hot, int64_t n_hot,
                                           const int32_t *row_req, const int32_t *fully_resident,
                                           int32_t n_reqs, const int32_t *idx, int32_t R,
                                           int32_t H, int32_t K,
                                           float scale, void *out, float *lse, uint32_t *status,
                                           hs_stream_t stream) {
  return hs_attn_launch(q, kv_resident, n_resident, kv_hot, n_hot, row_req, fully_resident,
                        n_reqs, idx, R, H, K, scale, out, lse, status, true, stream);
}

int hs_attn_launch(const void *q, const void *kv_resident, int64_t n_resident, const void *kv_hot,
                   int64_t n_hot, const int32_t *row_req, const int32_t *fully_resident,
                   int32_t n_reqs, const int32_t *idx, int32_t R, int32_t H, int32_t K,
                   float scale, void *out, float *lse, uint32_t *status, bool pdl,
                   cudaStream_t stream) {
  if (R < 0 || H < 1 || H > 1024 || K < 0 || n_resident < 0 || n_hot < 0 ||
      (fully_resident && n_reqs < 0))
    return hs_set_error(HS_ERR_INVALID_ARG, "bad sizes R=%d H=%d (1..1024) K=%d n_kv=%lld/%lld",
                        R, H, K, (long long)n_resident, (long long)n_hot);
  if (R == 0) return HS_OK;
  if (!q || !out ||
      (K > 0 && (!idx || (!kv_resident && n_resident > 0) || (!kv_hot && n_hot > 0))))
    return hs_set_error(HS_ERR_INVALID_ARG, "NULL q/kv/idx/out");
  if (((uintptr_t)q & 15) || ((uintptr_t)kv_resident & 15) || ((uintptr_t)kv_hot & 15) ||
      ((uintptr_t)out & 15))
    return hs_set_error(HS_ERR_INVALID_ARG, "q, kv and out must be 16-byte aligned");
  if (!(scale == scale)) return hs_set_error(HS_ERR_INVALID_ARG, "scale is NaN");
  int rc = set_attn_attributes();
  if (rc) return rc;
  const int64_t blocks = (int64_t)R * ((H + HG - 1) / HG) * 2;
  if (blocks > INT32_MAX) return hs_set_error(HS_ERR_UNSUPPORTED, "R*H too large");
  // q as a [R][H][576] bf16 tensor for the prologue's tensor copies
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult qr;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess || !fn)
      return hs_set_error(HS_ERR_CUDA, "cuTensorMapEncodeTiled not available");
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  alignas(64) CUtensorMap tmap;
  const cuuint64_t gdim[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)R};
  const cuuint64_t gstride[2] = {(cuuint64_t)ROWB, (cuuint64_t)H * ROWB};
  const cuuint32_t box[3] = {64, HG, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult er = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), gdim,
                             gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (er != CUDA_SUCCESS) return hs_set_error(HS_ERR_CUDA, "tensor map of q failed (%d)", (int)er);
  // a programmatic dependent launch: the prologue (barriers, TMEM, Q) may
  // run while the previous kernel in the stream finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  HS_CUDA_TRY(cudaLaunchKernelEx(
      &cfg, k_attn_pair, tmap, reinterpret_cast<const char *>(q),
      reinterpret_cast<const char *>(kv_resident), n_resident,
      reinterpret_cast<const char *>(kv_hot), n_hot, row_req, fully_resident, n_reqs, idx, H, K,
      scale * 1.4426950408889634f, reinterpret_cast<__nv_bfloat16 *>(out), lse, status));
  HS_LAUNCH_CHECK("k_attn_pair");
  return HS_OK;
}

extern "C" int hs_sparse_attn_decode(const void *q, const void *kv, int64_t n_kv_rows,
                                     const int32_t *idx, int32_t R, int32_t H, int32_t K,
                                     float scale, void *out, float *lse, uint32_t *status,
                                     hs_stream_t stream) {
  return hs_sparse_attn_decode_mixed(q, kv, n_kv_rows, nullptr, 0, nullptr, nullptr, 0, idx, R,
                                     H, K, scale, out, lse, status, stream);
}
