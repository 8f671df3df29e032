// Tree attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Same computation as the CUDA-core kernel in attn.cu ("Tree Verification",
// "Tree Attention"; "Build the tree attention mask that verifies a draft tree
// in one pass", "The mask."): every (node, query head) row of a GQA group
// attends to the whole cached prefix with no mask and then to the tree nodes
// in its ancestor row.  The pages only say that a FlashAttention-style kernel
// may take the tree part as a parent array expanded per tile; the design here
// is built for sm_103a:
//
//  * rows: the G query heads x N nodes of one KV head are packed into 128-row
//    MMA tiles (row = node * G + g), so every K/V byte fetched from HBM feeds
//    up to 256 query rows (two M tiles); one TMA box per M tile loads Q;
//  * keys: the paged cache ([num_blocks, Hkv, block_size, 128] bf16) is read by
//    TMA, one box per (block, 64-column half), into 128B-swizzled K-major tiles
//    of 64 keys; the tree K/V ([B, N, Hkv, 128]) is one more 64-key tile whose
//    rows beyond N are zero-filled by TMA;
//  * S = Q K^T and O += P V run as tcgen05.mma kind::f16 (bf16 in, fp32 in
//    TMEM): S_m uses 64 TMEM columns, O_m 128 columns per M tile;
//  * softmax: one thread per row reads its S row from TMEM, applies no mask on
//    prefix tiles except the ragged tail (key position < L) and the ancestor
//    bit test on the tree tile, keeps a lazily rescaled running max (O is
//    rescaled in TMEM only when the max grows by more than 2^8), writes P as
//    bf16 into a swizzled shared-memory tile, and finally normalises O;
//  * roles: warp 0 issues TMA, warp 1 (one lane) issues MMAs and owns TMEM,
//    one warpgroup per M tile runs the softmax and the epilogue; stages are
//    handed over with mbarriers (TMA transaction counts and tcgen05.commit);
//  * work split: the persistent grid walks the balanced tile plan of
//    attn_common.cuh; split units write float32 partials for the combine.
//
// Every mbarrier wait is bounded (2 s); on timeout the CTA raises
// TV_DEV_TIMEOUT in the status word, drains its own TMA loads, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "attn_tc.h"
#include "rope_math.cuh"

#ifdef TV_TC_TRACE
// Development aid: clock64 stamps of pipeline events of CTA 0, one slot per
// (event, tile).  Not part of the product build.
namespace tv { namespace trace {
constexpr int kEvents = 32, kTiles = 512;
__device__ unsigned long long g_trace[kEvents][kTiles];
// per CTA: globaltimer at entry, exit; segments; first unit; last epilogue
// start, end; total epilogue ns
__device__ unsigned long long g_cta_time[1024][8];
__device__ unsigned long long g_epi[1024][8];  // row 0: ns per route (complete, direct, publish, publish + merge), counts
}}  // namespace tv::trace
#define TV_TRACE(ev, tile) \
  do { if (blockIdx.x == 0 && (tile) < tv::trace::kTiles) tv::trace::g_trace[ev][tile] = clock64(); } while (0)
#define TV_TRACE_CTA(k)                                                                                  \
  do {                                                                                                    \
    if (threadIdx.x == 0 && blockIdx.x < 1024) {                                                          \
      unsigned long long t_;                                                                              \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                              \
      tv::trace::g_cta_time[blockIdx.x][k] = t_;                                                          \
    }                                                                                                     \
  } while (0)
#define TV_TRACE_ROW0(k, v)                                                  \
  do {                                                                      \
    if (row == 0 && blockIdx.x < 1024) tv::trace::g_cta_time[blockIdx.x][k] = (v); \
  } while (0)
#else
#define TV_TRACE(ev, tile) do { } while (0)
#define TV_TRACE_CTA(k) do { } while (0)
#define TV_TRACE_ROW0(k, v) do { } while (0)
#endif

namespace tv {

namespace {

constexpr int kD = 128;                          // head dim of this kernel
constexpr int kBlk = kTcBlk;                     // keys per tile (64)
constexpr int kKVHalfBytes = kBlk * 128;         // 64 rows x 128 B
constexpr int kKVTileBytes = 2 * kKVHalfBytes;   // one K (or V) tile
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;        // log2 units

// M query tiles of 128 rows per CTA.  TMEM columns (fp32 cells):
//   S_m: 64 (one 64-key score tile; P_m, bf16 pairs, overwrites its first 32)
//   Q_m: 64 (128 bf16 per row, the A operand of S = Q K^T)
//   O_m: 128 (fp32 accumulator)
// Shared memory holds only the K/V stage ring.
template <int M>
struct Cfg {
  static constexpr int kStages = (M == 1) ? 3 : 6;
  static constexpr int kCtasPerSm = (M == 1) ? 2 : 1;
  // warp 0: TMA; warps 1..M: one MMA issuer per M tile (a single thread
  // issues at most about one MMA per 70 cycles, so each tile gets its own);
  // then one softmax warpgroup per M tile.
  static constexpr int kSoftmaxWarp0 = 1 + M;
  static constexpr int kThreads = 32 * (1 + M + 4 * M);
  static constexpr uint32_t kTmemCols = (M == 1) ? 256 : 512;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kKVTileBytes;
  static constexpr int kBytes = kOffV + kStages * kKVTileBytes;
  static constexpr int kSmem = kBytes + 1024;        // slack for 1024-byte alignment
  static constexpr uint32_t col_s(int m) { return m * 64; }
  static constexpr uint32_t col_q(int m) { return M * 64 + m * 64; }
  static constexpr uint32_t col_o(int m) { return 128 * M + m * 128; }
};

struct Bars {
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t peer_full[8];  // CTA pairs: the odd CTA's half of a tile has landed (even CTA's copy)
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t s_free[2];
  uint64_t q_full;
  uint64_t sh_stat, sh_read;  // shared units (two-M-tile kernel): M tile 1's part posted / read
  uint64_t tail_sync;         // tail rows (two-M-tile kernel): the four producer warps' end-of-unit exchange
  uint64_t drain[4];          // one per MMA-issuing thread: its products have completed (after an abort)
  uint64_t q0s_full, cp_done;  // staged Q (two-M-tile kernel): the next unit's Q_0 has landed / been copied to TMEM
  uint64_t q1_free, q1_full;   //   ... this unit's last S_1 has completed / the next unit's Q_1 has landed
  uint64_t merge_full[2][4];   //   ... the other piece's rows of warp q of M tile m have landed (end-of-slice merge)
  uint32_t tmem_base;
  int abort;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#ifdef TV_TEST_HOOKS
// Development builds only (-DTV_TEST_HOOKS; the product library has none of
// these variables): a test shortens the wait limit and has CTA 0's TMA
// producers skip the loads (and the arrival) of one ring tile, so that the
// bounded waits run out and the timeout exit is exercised without a fault;
// or it keeps the epilogue warps of some TMEM quarters off the direct merge,
// so that the warps of one M tile take different merge routes; or it makes
// the first pair of tail warps sleep before each of its tiles, so that it
// falls behind the other pair.
__device__ unsigned long long g_test_timeout_ns = kTimeoutNs;
__device__ int g_test_withhold = -1;      // ring index of CTA 0 left without loads
__device__ int g_test_publish_warps = 0;  // bit q: warps of TMEM quarter q never merge directly
__device__ unsigned long long g_test_tail_delay_ns = 0;  // sleep of tail pair 0 before each tile
__device__ __forceinline__ unsigned long long timeout_ns() { return *(volatile unsigned long long*)&g_test_timeout_ns; }
__device__ __forceinline__ bool test_withhold(uint32_t g) {
  return blockIdx.x == 0 && (int)g == *(volatile int*)&g_test_withhold;
}
__device__ __forceinline__ bool test_no_direct(int rl) {
  return (*(volatile int*)&g_test_publish_warps >> (rl >> 5)) & 1;
}
__device__ __forceinline__ void test_tail_delay(int pair) {
  const unsigned long long d = *(volatile unsigned long long*)&g_test_tail_delay_ns;
  if (pair != 0 || d == 0) return;
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < d);
}
#else
__device__ __forceinline__ unsigned long long timeout_ns() { return kTimeoutNs; }
__device__ __forceinline__ bool test_withhold(uint32_t) { return false; }
__device__ __forceinline__ bool test_no_direct(int) { return false; }
__device__ __forceinline__ void test_tail_delay(int) {}
#endif

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity (one thread); false on timeout,
// or on another role's abort when honor_abort is set.
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, Bars* bars, int32_t* status, bool honor_abort = true) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (honor_abort && *(volatile int*)&bars->abort) return false;
      if (globaltimer() - t0 > timeout_ns()) {
        *(volatile int*)&bars->abort = 1;
        if (status) atomicOr(status, TV_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// The same wait for a whole warp: every lane polls and all lanes leave
// together with the same answer (warp-collective tcgen05 ops follow).
__device__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, Bars* bars, int32_t* status) {
  bool done = mbar_test(bar, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (!done) done = mbar_test(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((it & 255u) == 0) {
      bool stop = *(volatile int*)&bars->abort != 0 || globaltimer() - t0 > timeout_ns();
      if (__any_sync(0xffffffffu, stop)) {
        if ((threadIdx.x & 31) == 0 && !*(volatile int*)&bars->abort) {
          *(volatile int*)&bars->abort = 1;
          if (status) atomicOr(status, TV_DEV_TIMEOUT);
        }
        return false;
      }
    }
  }
}

// Cache-hinted 2-D load: the prefix K/V stream is read once, so its lines
// are marked first to leave L2 (keeping Q rows, ancestor rows and the
// partials of split units resident while the stream passes through).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_2d_stream(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
      "[%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Instruction descriptor, kind::f16: bf16 x bf16 -> f32, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Matrix descriptors as two 32-bit words: the low word carries the start
// address (>> 4) and the leading offset, so a K step is one 32-bit add.
__host__ __device__ constexpr uint32_t desc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);  // SBO, version 1, SWIZZLE_128B
}
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo & 0x3FFFFu) >> 4) << 16);
}

// O/S += A(TMEM) B(smem); the accumulate flag is a literal.
template <bool kAcc>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t b_hi, uint32_t idesc) {
  if constexpr (kAcc)
    asm volatile(
        "{\n\t.reg .b64 bd;\n\tmov.b64 bd, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, 1;\n\t}" ::"r"(d),
        "r"(a), "r"(b_lo), "r"(b_hi), "r"(idesc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .b64 bd;\n\tmov.b64 bd, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, 0;\n\t}" ::"r"(d),
        "r"(a), "r"(b_lo), "r"(b_hi), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// After an abort: the issuing thread waits (bounded) until every MMA it has
// issued has completed, so that no product still writes TMEM or reads a
// stage when the CTA frees TMEM and exits.
__device__ __forceinline__ void mma_drain(Bars& bars, int i) {
  mma_commit(&bars.drain[i]);
  mbar_wait(&bars.drain[i], 0, &bars, nullptr, false);
}

#define TV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define TV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : TV_R8(0), TV_R8(8), TV_R8(16), TV_R8(24)
      : "r"(taddr));
}

// 16 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : TV_R8(0), TV_R8(8)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      TV_W8(0), TV_W8(8), TV_W8(16), TV_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of a 64-entry row.
__device__ __forceinline__ float row_max64(const float (&v)[64]) {
  float a[22];
#pragma unroll
  for (int i = 0; i < 21; ++i) a[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[21] = v[63];
  float b[8];
#pragma unroll
  for (int i = 0; i < 7; ++i) b[i] = max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[7] = a[21];
  return max3(max3(b[0], b[1], b[2]), max3(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
}

// (e0, e1) = 2^(s0 * sc - m), 2^(s1 * sc - m) with one packed FMA; sc2/negm2 hold
// (sc, sc) and (-m, -m).
__device__ __forceinline__ void exp2_pair(float s0, float s1, uint64_t sc2, uint64_t negm2, float& e0, float& e1) {
  asm("{\n\t.reg .b64 s2, t2;\n\t.reg .f32 t0, t1;\n\t"
      "mov.b64 s2, {%2, %3};\n\t"
      "fma.rn.f32x2 t2, s2, %4, %5;\n\t"
      "mov.b64 {t0, t1}, t2;\n\t"
      "ex2.approx.ftz.f32 %0, t0;\n\t"
      "ex2.approx.ftz.f32 %1, t1;\n\t}"
      : "=f"(e0), "=f"(e1)
      : "f"(s0), "f"(s1), "l"(sc2), "l"(negm2));
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float sum_f32x2(uint64_t a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return lo + hi;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------ fused RoPE of Q

// Position of a row from its ancestor row: L + depth with depth = popcount - 1
// (the row holds the node and its ancestors); an absent node (row 0) has none.
__device__ __forceinline__ int row_pos(uint64_t mrow, int L) { return mrow ? L + __popcll(mrow) - 1 : -1; }

// Rotate-half RoPE of one whole bf16 query row (q[c] = elements 8c .. 8c+7) at
// position pos, with the float32 arithmetic and bf16 rounding of
// tv_rope_apply, so the rotated row has the same bits.  The G consecutive
// lanes holding the G heads of one node share the position: lane j of the
// group loads the cosines and sines of frequencies [j * 64 / G, (j+1) * 64 / G)
// of the table row and the others read them by shuffles (every lane of the
// warp takes part).  pos outside [0, max_pos) leaves the row as it is (-1:
// an absent node; otherwise TV_DEV_BAD_POSITION).
template <int G>
__device__ __forceinline__ void rope_row_group(uint4 (&q)[16], const float* __restrict__ cs, int pos, int max_pos,
                                               int32_t* status, int lane) {
  constexpr int kPer = 64 / G;
  static_assert(kPer % 4 == 0, "whole float4 table loads per lane");
  const int j = lane % G, base = lane - j;
  const bool inb = pos >= 0 && pos < max_pos;
  if (pos >= max_pos && j == 0 && status) atomicOr(status, TV_DEV_BAD_POSITION);
  float c[kPer], sn[kPer];
#pragma unroll
  for (int v = 0; v < kPer; ++v) c[v] = sn[v] = 0.f;
  if (inb) {
    const float4* c4 = reinterpret_cast<const float4*>(cs + (int64_t)pos * kD + j * kPer);
    const float4* s4 = reinterpret_cast<const float4*>(cs + (int64_t)pos * kD + kD / 2 + j * kPer);
#pragma unroll
    for (int v = 0; v < kPer / 4; ++v) {
      const float4 a = __ldg(c4 + v), b = __ldg(s4 + v);
      c[4 * v] = a.x; c[4 * v + 1] = a.y; c[4 * v + 2] = a.z; c[4 * v + 3] = a.w;
      sn[4 * v] = b.x; sn[4 * v + 1] = b.y; sn[4 * v + 2] = b.z; sn[4 * v + 3] = b.w;
    }
  }
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const uint32_t lo[4] = {q[ch].x, q[ch].y, q[ch].z, q[ch].w};
    const uint32_t hi[4] = {q[ch + 8].x, q[ch + 8].y, q[ch + 8].z, q[ch + 8].w};
    uint32_t olo[4], ohi[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int k0 = 8 * ch + 2 * w, k1 = k0 + 1;
      const float c0 = __shfl_sync(0xffffffffu, c[k0 % kPer], base + k0 / kPer);
      const float s0 = __shfl_sync(0xffffffffu, sn[k0 % kPer], base + k0 / kPer);
      const float c1 = __shfl_sync(0xffffffffu, c[k1 % kPer], base + k1 / kPer);
      const float s1 = __shfl_sync(0xffffffffu, sn[k1 % kPer], base + k1 / kPer);
      float y1a, y2a, y1b, y2b;
      rope_pair(__uint_as_float(lo[w] << 16), __uint_as_float(hi[w] << 16), c0, s0, y1a, y2a);
      rope_pair(__uint_as_float(lo[w] & 0xffff0000u), __uint_as_float(hi[w] & 0xffff0000u), c1, s1, y1b, y2b);
      olo[w] = pack_bf16(y1a, y1b);
      ohi[w] = pack_bf16(y2a, y2b);
    }
    if (inb) {
      q[ch] = make_uint4(olo[0], olo[1], olo[2], olo[3]);
      q[ch + 8] = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
    }
  }
}

// The G of the launch (4, 8 or 16: the fused path needs whole power-of-two
// lane groups of at least four).
__device__ __forceinline__ void rope_row(uint4 (&q)[16], const AttnParams& p, int pos, int32_t* status, int lane) {
  switch (p.G) {
    case 4: rope_row_group<4>(q, p.rope_cs, pos, p.rope_max_pos, status, lane); break;
    case 8: rope_row_group<8>(q, p.rope_cs, pos, p.rope_max_pos, status, lane); break;
    default: rope_row_group<16>(q, p.rope_cs, pos, p.rope_max_pos, status, lane); break;
  }
}

// ---------------------------------------------------------------- work walk

// This CTA's slice of the tile sequence and the unit holding its first tile.
struct SlicePlan {
  int T, t0, t1;
  int us0;  // first (virtual) tile of unit u0
  int u0;
  int P;    // slices the plan is cut into (CTAs from P on have no work)
  int c;    // this CTA's slice (its CTA index, or its CTA pair's index)
};

// Fewest tiles a slice gets: a small plan goes to fewer CTAs rather than
// cutting every unit into many pieces whose merge costs more than it saves.
#ifndef TV_MIN_SLICE_TILES
#define TV_MIN_SLICE_TILES 12
#endif

// Tiles of every unit of request b, virtual ones included.
__device__ __forceinline__ int unit_tiles(const AttnParams& p, int b) {
  return (clamp_len(p, b) + kBlk - 1) / kBlk + 1 + p.unit_cost;
}

// Warp-collective.  The units of request b are consecutive and all have
// unit_tiles(b) tiles, so the tile prefix sums are taken over requests.
__device__ void plan_slice(const AttnParams& p, int lane, SlicePlan& sp, int c) {
  const int64_t upb = (int64_t)p.Hkv * p.RG;
  long long tot = 0;
  for (int b = lane; b < p.B; b += 32) tot += unit_tiles(p, b);
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const int T = (int)(tot * upb);  // the host bounds the plan below 2^31 tiles
  int P = (T + TV_MIN_SLICE_TILES - 1) / TV_MIN_SLICE_TILES;
  P = P < 1 ? 1 : (P > p.P ? p.P : P);
  const int t0 = c < P ? (int)cta_start(c, T, P) : T, t1 = c < P ? (int)cta_start(c + 1, T, P) : T;
  int u0 = p.U, us0 = T;
  if (t0 < t1) {
    long long carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      const int nt = b < p.B ? unit_tiles(p, b) : 0;
      const long long n = (long long)nt * upb;
      long long incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && carry + incl > t0);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const long long start = __shfl_sync(0xffffffffu, carry + incl - n, src);
        const int ntb = __shfl_sync(0xffffffffu, nt, src);
        const int k = (int)((t0 - start) / ntb);
        u0 = (int)((base + src) * upb + k);
        us0 = (int)(start + (long long)k * ntb);
        break;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0) {
    sp.c = c;
    sp.T = T;
    sp.P = P;
    sp.t0 = t0;
    sp.t1 = t1;
    sp.u0 = u0;
    sp.us0 = us0;
  }
}

struct Segment {
  int u, a, e, n;  // unit, local real tiles [a, e) of its n real tiles
  int b, kvh, rg, L;
  int real_start;  // index of the unit's first real tile in the plan
};

struct Walk {
  int t0, t1, us;
  int u;
  __device__ explicit Walk(const SlicePlan& sp) : t0(sp.t0), t1(sp.t1), us(sp.us0), u(sp.u0) {}
  // Next unit with real tiles in this CTA's slice (units whose slice part is
  // only their virtual cost tiles are skipped).
  __device__ bool next(const AttnParams& p, Segment& s) {
    while (u < p.U && us < t1) {
      int b, kvh, rg;
      unit_coords(p, u, b, kvh, rg);
      const int L = clamp_len(p, b);
      const int rs = us + p.unit_cost, ue = rs + (L + kBlk - 1) / kBlk + 1;  // real tiles [rs, ue)
      const int a = max(t0, rs), e = min(t1, ue);
      const int uu = u++;
      us = ue;
      if (a >= e) continue;
      s.u = uu;
      s.a = a - rs;
      s.e = e - rs;
      s.n = ue - rs;
      s.real_start = rs;
      s.b = b;
      s.kvh = kvh;
      s.rg = rg;
      s.L = L;
      return true;
    }
    return false;
  }
};

// ---------------------------------------------------------------- output of a finished segment

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* ptr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}

// The pieces of a split unit: CTAs c0..c1 whose slice is not empty.  Each
// wrote its normalised partial rows and log2-sum-exp to slot 0 of its two
// slots, except c0 when the unit began after the start of its slice (slot 1).
struct Pieces {
  int T, P, c0, c1;
  int self;  // this CTA's slice
  bool c0_slot1;
  __device__ Pieces(const SlicePlan& sp, int real_start, int n_real) : T(sp.T), P(sp.P), self(sp.c) {
    c0 = (int)cta_of(real_start, T, P);
    c1 = (int)cta_of(real_start + n_real - 1, T, P);
    c0_slot1 = cta_start(c0, T, P) < real_start;
  }
  __device__ bool present(int c) const { return T >= P || cta_start(c, T, P) < cta_start(c + 1, T, P); }
  __device__ int64_t slot(int c) const { return (int64_t)c * 2 + ((c == c0 && c0_slot1) ? 1 : 0); }
};

// Both merge routes below take the same arithmetic in the same order (pieces
// c0..c1, the finishing CTA's piece as the float32 values it would publish),
// so the merged row does not depend on which piece finished last.

// (mx, z): maximum and normaliser of the pieces' log2-sum-exps; with kSelf the
// piece of CTA `self` is self_lse instead of its published value.
template <bool kSelf>
__device__ __forceinline__ void piece_stats(const AttnParams& p, const Pieces& pc, int self, float self_lse, int row,
                                            float& mx, float& z) {
  mx = -INFINITY;
  for (int c = pc.c0; c <= pc.c1; ++c)
    if (pc.present(c)) mx = fmaxf(mx, (kSelf && c == self) ? self_lse : __ldcg(p.part_lse + pc.slot(c) * p.RPG + row));
  z = 0.f;
  for (int c = pc.c0; c <= pc.c1; ++c)
    if (pc.present(c))
      z += exp2f(((kSelf && c == self) ? self_lse : __ldcg(p.part_lse + pc.slot(c) * p.RPG + row)) - mx);
}

// acc += sum over pieces of 2^(lse_c - mx) / z * O_c[row][col0 .. col0 + 15]
// (with kSelf, CTA self's columns are selfv).
template <bool kSelf>
__device__ __forceinline__ void accum_pieces(float (&acc)[16], const AttnParams& p, const Pieces& pc, int self,
                                             const float (&selfv)[16], float self_lse, int row, int col0, float mx,
                                             float zinv) {
  for (int c = pc.c0; c <= pc.c1; ++c) {
    if (!pc.present(c)) continue;
    const int64_t sr = pc.slot(c) * p.RPG + row;
    if (kSelf && c == self) {
      const float w = exp2f(self_lse - mx) * zinv;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = fmaf(w, selfv[j], acc[j]);
      continue;
    }
    const float w = exp2f(__ldcg(p.part_lse + sr) - mx) * zinv;
    const float4* src = reinterpret_cast<const float4*>(p.part_o + sr * kD + col0);
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldcg(src + j);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[4 * j] = fmaf(w, v[j].x, acc[4 * j]);
      acc[4 * j + 1] = fmaf(w, v[j].y, acc[4 * j + 1]);
      acc[4 * j + 2] = fmaf(w, v[j].z, acc[4 * j + 2]);
      acc[4 * j + 3] = fmaf(w, v[j].w, acc[4 * j + 3]);
    }
  }
}

// 16 columns of an output row (dst 32-byte aligned: a row is 256 bytes and
// the columns start at a multiple of 16).  kWide: one 32-byte store, which
// halves the store transactions of a warp writing 32 rows at once (measured
// faster in the two-M-tile kernel without tail rows, slower in the others,
// whose code it changes); else two 16-byte stores.
template <bool kWide = false>
__device__ __forceinline__ void store_bf16_16(__nv_bfloat16* dst, const float (&acc)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = pack_bf16(acc[2 * j], acc[2 * j + 1]);
  if constexpr (kWide) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Writes this thread's row of a finished segment; warp-collective (reads the
// row's O accumulator, 128 TMEM columns at tO, 16 at a time).  O / l and its log2-sum-exp
// m + log2 l are exact for this CTA's share of the unit's keys.
//  * whole unit in this slice: O / l straight to the output;
//  * split unit, every other piece already published (the arrival counter
//    already holds all other real tiles): merge here, from TMEM and the
//    others' partials;
//  * otherwise publish the partial, count this piece's tiles in, and merge
//    from memory if that completed the count (a piece that finished in the
//    meantime saw the count short and left the merge to this one).
// Merge of a split unit's row when the K/V stage ring is idle (the slice's
// last segment): every other piece's row is copied into shared memory by
// cp.async -- with two pieces the other's whole row at once, else a 32-column
// quarter of all pieces at a time: one memory round trip per batch and no
// registers held for the loads -- and combined with this CTA's O from TMEM in
// piece order, with the same float32 arithmetic as the other merge routes.
// A 16 KB slot holds one quarter of one piece (slot = quarter with two
// pieces, else piece index k = c - c0 < np <= kStagePieces): row rl, 16-byte
// chunk j at slot * 16384 + rl * 128 + ((j ^ (rl & 7)) * 16), so eight
// consecutive rows hit eight different bank groups.  Warp-collective (TMEM
// reads); `active` lanes merge their row.
constexpr int kStagePieces = 4;
constexpr int kStageBytes = kStagePieces * 16384;
static_assert(3 * kKVTileBytes * 2 >= kStageBytes, "the single-M-tile ring holds the staging slots");

__device__ __forceinline__ void staged_merge(const AttnParams& p, const Pieces& pc, float lse2, float inv, int row,
                                             int rl, int64_t orow, uint32_t tO, uint8_t* stage, bool active) {
  constexpr float kLn2 = 0.69314718055994530942f;
  const int self = pc.self;
  const int np = pc.c1 - pc.c0 + 1;
  float lse[kStagePieces], w[kStagePieces];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kStagePieces; ++k) {
    const int c = pc.c0 + k;
    lse[k] = 0.f;
    if (k < np) {
      lse[k] = (c == self) ? lse2 : (active ? __ldcg(p.part_lse + pc.slot(c) * p.RPG + row) : 0.f);
      mx = fmaxf(mx, lse[k]);
    }
  }
  float z = 0.f;
#pragma unroll
  for (int k = 0; k < kStagePieces; ++k)
    if (k < np) z += exp2f(lse[k] - mx);
  const float zinv = 1.f / z;
#pragma unroll
  for (int k = 0; k < kStagePieces; ++k) w[k] = exp2f(lse[k] - mx) * zinv;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  const uint32_t sbase = smem_u32(stage);
  // quarter qq of piece c into slot `sl`
  auto issue = [&](int c, int qq, int sl) {
    const float* src = p.part_o + (pc.slot(c) * p.RPG + row) * kD + qq * 32;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sbase + sl * 16384 + rl * 128 + ((j ^ (rl & 7)) << 4)),
                   "l"(src + 4 * j)
                   : "memory");
  };
  // two pieces: the other piece's whole row goes in at once (quarter qq in slot qq)
  const bool whole = np == 2;
  if (whole) {
    if (active)
      for (int qq = 0; qq < kD / 32; ++qq) issue(self == pc.c0 ? pc.c1 : pc.c0, qq, qq);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }
#pragma unroll 1
  for (int qq = 0; qq < kD / 32; ++qq) {
    if (!whole) {
      if (active) {
#pragma unroll
        for (int k = 0; k < kStagePieces; ++k) {
          const int c = pc.c0 + k;
          if (k < np && c != self) issue(c, qq, k);
        }
      }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    }
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(tO + qq * 32, r);
    tmem_ld_wait();
    if (!active) continue;
    float acc[32];
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int k = 0; k < kStagePieces; ++k) {
        const int c = pc.c0 + k;
        if (k >= np) continue;
        float4 v;
        if (c == self) {
          v = make_float4(__uint_as_float(r[4 * g4]) * inv, __uint_as_float(r[4 * g4 + 1]) * inv,
                          __uint_as_float(r[4 * g4 + 2]) * inv, __uint_as_float(r[4 * g4 + 3]) * inv);
        } else {
          v = *reinterpret_cast<const float4*>(stage + (whole ? qq : k) * 16384 + rl * 128 + ((g4 ^ (rl & 7)) << 4));
        }
        a0 = fmaf(w[k], v.x, a0);
        a1 = fmaf(w[k], v.y, a1);
        a2 = fmaf(w[k], v.z, a2);
        a3 = fmaf(w[k], v.w, a3);
      }
      acc[4 * g4] = a0;
      acc[4 * g4 + 1] = a1;
      acc[4 * g4 + 2] = a2;
      acc[4 * g4 + 3] = a3;
    }
    uint4* dst = reinterpret_cast<uint4*>(out + orow * kD + qq * 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 v;
      v.x = pack_bf16(acc[8 * j + 0], acc[8 * j + 1]);
      v.y = pack_bf16(acc[8 * j + 2], acc[8 * j + 3]);
      v.z = pack_bf16(acc[8 * j + 4], acc[8 * j + 5]);
      v.w = pack_bf16(acc[8 * j + 6], acc[8 * j + 7]);
      dst[j] = v;
    }
  }
  __syncwarp();
  if (active && p.lse) p.lse[orow] = (mx + log2f(z)) * kLn2;
}

// Direct merge of a split unit's row with exactly one other piece, at the
// slice's last segment of the two-M-tile kernel: the other piece's row is
// copied by cp.async into the idle K/V ring (16-byte chunk k of row r at
// (k * 128 + (r & 127)) * 16, so a warp's 32 rows read 512 consecutive bytes)
// while its log2-sum-exp loads, then combined with this CTA's O from TMEM in
// piece order with the arithmetic of piece_stats / accum_pieces, so the row
// matches the other merge routes bit for bit.  Warp-collective (TMEM reads);
// `active` lanes merge their row.
// kWide (the staged-Q two-M-tile kernel): each warp's 32 rows of the other
// piece come by TMA (pm: four 4 KB boxes of 32 columns x 32 rows,
// 128B-swizzled, on the warp's own barrier `mbar`) instead of 32 16-byte
// cp.async requests per thread, which the load/store unit took about 9,000
// cycles to issue; rows are then read swizzled (4 wavefronts per warp access,
// the minimum for 512 bytes).  Each warp takes this route on its own rows'
// arrival counts, so no warp waits for a copy another warp issues.
template <bool kWide>
__device__ __forceinline__ void staged_pair_merge(const AttnParams& p, const Pieces& pc, float lse2, float inv,
                                                  int row, int rl, int64_t orow, uint32_t tO, uint8_t* stage,
                                                  bool active, const CUtensorMap* pm, uint64_t* mbar) {
  constexpr float kLn2 = 0.69314718055994530942f;
  const bool self_first = pc.self == pc.c0;
  const int64_t so = pc.slot(self_first ? pc.c1 : pc.c0) * p.RPG + row;
  const uint32_t dst = smem_u32(stage) + rl * 16;
  float lo = 0.f;
  if constexpr (kWide) {
    if ((rl & 31) == 0) {
      const int y = (int)so;  // the warp's first row in the partials
      mbar_expect_tx(mbar, 32 * kD * 4);
#pragma unroll
      for (int k = 0; k < kD / 32; ++k) tma_2d(smem_u32(stage) + k * 16384 + rl * 128, pm, 32 * k, y, mbar);
    }
    if (active) lo = __ldcg(p.part_lse + so);
  } else {
    if (active) {
      const float* src = p.part_o + so * kD;
#pragma unroll
      for (int j = 0; j < kD / 4; ++j)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + j * 2048), "l"(src + 4 * j) : "memory");
      lo = __ldcg(p.part_lse + so);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const float l0 = self_first ? lse2 : lo, l1 = self_first ? lo : lse2;
  float mx = -INFINITY;
  mx = fmaxf(mx, l0);
  mx = fmaxf(mx, l1);
  float z = 0.f;
  z += exp2f(l0 - mx);
  z += exp2f(l1 - mx);
  const float zinv = 1.f / z;
  const float w0 = exp2f(l0 - mx) * zinv, w1 = exp2f(l1 - mx) * zinv;
  if constexpr (kWide) {
    // bounded; the copy is waited for even after another role's abort, so
    // that it has landed before the CTA exits
    const unsigned long long t0 = globaltimer();
    bool landed = mbar_test(mbar, 0);
    while (!landed) {
      landed = mbar_test(mbar, 0);
      if (!landed && globaltimer() - t0 > timeout_ns()) {
        if (p.status) atomicOr(p.status, TV_DEV_TIMEOUT);
        break;
      }
    }
  } else {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  const uint8_t* srow = stage + rl * 16;
#pragma unroll 1
  for (int c = 0; c < kD; c += 16) {
    uint32_t r[16];
    __syncwarp();
    tmem_ld16(tO + c, r);
    tmem_ld_wait();
    if (!active) continue;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q4 = (c >> 2) + j;  // float4 chunk of the row
      const float4 o = kWide ? *reinterpret_cast<const float4*>(stage + (q4 >> 3) * 16384 + rl * 128 +
                                                                 (((q4 & 7) ^ (rl & 7)) << 4))
                             : *reinterpret_cast<const float4*>(srow + q4 * 2048);
      const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mine = __uint_as_float(r[4 * j + e]) * inv;
        const float a = fmaf(w0, self_first ? mine : ov[e], 0.f);
        acc[4 * j + e] = fmaf(w1, self_first ? ov[e] : mine, a);
      }
    }
    store_bf16_16<kWide>(out + orow * kD + c, acc);
  }
  __syncwarp();
  if (active && p.lse) p.lse[orow] = (mx + log2f(z)) * kLn2;
}

// kStage: 0 no staging; 1 merges at the slice's last segment may stage
// through `stage` (staged_merge); 2 only a direct merge with one other piece
// stages (staged_pair_merge).
template <int kStage, bool kWide = false>
__device__ __forceinline__ int finish_row_impl(const AttnParams& p, const SlicePlan& sp, const Segment& s, int row,
                                               bool valid_row, int64_t orow, uint32_t tO, float m_run, float l,
                                               uint8_t* stage, const CUtensorMap* pm = nullptr,
                                               uint64_t* mbar = nullptr) {
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  constexpr float kLn2 = 0.69314718055994530942f;
  const float inv = l > 0.f ? 1.f / l : 0.f;  // no key at all (empty prefix, absent node): zero row
  const float lse2 = m_run + log2f(l);
  const bool complete = (s.a == 0 && s.e == s.n);
  const Pieces pc(sp, s.real_start, s.n);
  const int self = pc.self;
  uint32_t* ctr = p.arrive + (int64_t)pc.c0 * p.RPG + row;
  const uint32_t mine = (uint32_t)(s.e - s.a);
  bool direct = false;
  float mx = lse2, z = 1.f;
  const int rl = row & 127;
  const bool staged = kStage == 1 && stage != nullptr && !complete && pc.c1 - pc.c0 < kStagePieces && pc.T >= pc.P;
  if (!complete && valid_row && p.direct_merge && !test_no_direct(rl))
    direct = ld_acquire_u32(ctr) + mine == (uint32_t)s.n;
  if constexpr (kStage == 1) {
    if (staged && __all_sync(0xffffffffu, direct || !valid_row) && __any_sync(0xffffffffu, direct)) {
      staged_merge(p, pc, lse2, inv, row, rl, orow, tO, stage, valid_row);
      if (valid_row) *ctr = 0;  // every other piece has arrived: leave the counter at zero
      return 1;
    }
  }
  if constexpr (kStage == 2) {
    const bool pair = stage != nullptr && pc.c1 - pc.c0 == 1 && pc.T >= pc.P;
    if (pair && __all_sync(0xffffffffu, direct || !valid_row) && __any_sync(0xffffffffu, direct)) {
      staged_pair_merge<kWide>(p, pc, lse2, inv, row, rl, orow, tO, stage, valid_row, pm, mbar);
      if (valid_row) *ctr = 0;
      return 1;
    }
  }
  if (staged) direct = false;  // a mixed warp publishes; its last arriver merges below
  if (direct) piece_stats<true>(p, pc, self, lse2, row, mx, z);
  const float zinv = 1.f / z;
  const int64_t srow = pc.slot(self) * p.RPG + row;
#pragma unroll 1
  for (int c = 0; c < kD; c += 16) {
    uint32_t r[16];
    __syncwarp();
    tmem_ld16(tO + c, r);
    tmem_ld_wait();
    if (!valid_row) continue;
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]) * inv;
    if (complete) {
      store_bf16_16<kWide>(out + orow * kD + c, v);
    } else if (direct) {
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.f;
      accum_pieces<true>(acc, p, pc, self, v, lse2, row, c, mx, zinv);
      store_bf16_16<kWide>(out + orow * kD + c, acc);
    } else {
      float4* dst = reinterpret_cast<float4*>(p.part_o + srow * kD + c);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
  __syncwarp();
  if (complete || direct) {
    if (valid_row && p.lse) p.lse[orow] = (mx + log2f(z)) * kLn2;
    if (direct && valid_row) *ctr = 0;
    return complete ? 0 : 1;
  }
  if constexpr (kStage == 1) {
    if (staged) {
      bool last = false;
      if (valid_row) {
        p.part_lse[srow] = lse2;
        last = atom_add_acq_rel(ctr, mine) + mine == (uint32_t)s.n;
      }
      if (__any_sync(0xffffffffu, last)) {
        staged_merge(p, pc, lse2, inv, row, rl, orow, tO, stage, last);
        if (last) *ctr = 0;
        return last ? 3 : 2;
      }
      return 2;
    }
  }
  if (!valid_row) return 0;
  p.part_lse[srow] = lse2;
  if (atom_add_acq_rel(ctr, mine) + mine != (uint32_t)s.n) return 2;
  // every piece is published: merge from memory
  piece_stats<false>(p, pc, -1, 0.f, row, mx, z);
  const float zinv2 = 1.f / z;
#pragma unroll 1
  for (int c = 0; c < kD; c += 16) {
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    accum_pieces<false>(acc, p, pc, -1, acc, 0.f, row, c, mx, zinv2);
    store_bf16_16<kWide>(out + orow * kD + c, acc);
  }
  if (p.lse) p.lse[orow] = (mx + log2f(z)) * kLn2;
  *ctr = 0;
  return 3;
}

// kStage (as in finish_row_impl): how merges at the slice's last segment may
// stage through `stage`.
template <int kStage, bool kWide = false>
__device__ __forceinline__ void finish_row(const AttnParams& p, const SlicePlan& sp, const Segment& s, int row,
                                           bool valid_row, int64_t orow, uint32_t tO, float m_run, float l,
                                           uint8_t* stage, const CUtensorMap* pm = nullptr,
                                           uint64_t* mbar = nullptr) {
#ifdef TV_TC_TRACE
  const unsigned long long t_in = globaltimer();
  TV_TRACE_ROW0(4, t_in);
#endif
#ifdef TV_TC_TRACE
  const int route =
#endif
  finish_row_impl<kStage, kWide>(p, sp, s, row, valid_row, orow, tO, m_run, l, stage, pm, mbar);
#ifdef TV_TC_TRACE
  const unsigned long long t_out = globaltimer();
  TV_TRACE_ROW0(5, t_out);
  if (row == 0 && blockIdx.x < 1024) {
    tv::trace::g_cta_time[blockIdx.x][6] += t_out - t_in;
    tv::trace::g_epi[blockIdx.x][route] += t_out - t_in;
    tv::trace::g_epi[blockIdx.x][4 + route] += 1;
  }
#endif
}


struct TcMaps {
  CUtensorMap kc, vc, kt, vt;
  CUtensorMap qm;  // Q [B * N][Hq][D] in boxes of 64 columns x G heads x 128 / G nodes (128 rows of a unit)
  CUtensorMap pm;  // float32 partials [2 P RPG][D] in boxes of 32 columns x 32 rows (one warp's rows)
};

// TMA producer (warp 0): streams every tile of the CTA's slice into the
// K/V stage ring, one box per (cache block, 64-column half).
// With kProducers > 1 the boxes of every tile are dealt round-robin to that
// many warps (one warp issues a TMA box only about every 150 cycles, so a
// single warp cannot keep a two-M-tile CTA fed); producer 0 posts the stage's
// byte count.
template <int kStages, int kProducers = 1>
__device__ __forceinline__ void run_producer(const AttnParams& p, const SlicePlan& sp, const TcMaps& maps, Bars& bars,
                                             uint32_t sK, uint32_t sV, int lane, int32_t* status, int prod = 0) {
    // ------------------------------------------------------------ TMA producer
    // The producer shares its sub-partition with busy softmax warps, so the
    // tile loop is kept short: each lane's box (K or V, column half,
    // sub-block, its offset in the stage) is fixed for the whole slice, and
    // block arithmetic uses shifts when the block size is a power of two.
    const int bs = p.block_size;
    const int lbs = (bs & (bs - 1)) == 0 ? __ffs(bs) - 1 : -1;  // log2(bs) for a power of two
    const int br = bs < kBlk ? bs : kBlk;  // rows per TMA box
    const int nsub = kBlk / br;
    const int64_t rows_total = (int64_t)p.num_blocks * p.Hkv * bs;
    const uint64_t pol = policy_evict_first();
    // box j < 4 * nsub: sub-box j / 4, column half (j / 2) % 2, K (even j) or V
    // (odd j); this warp issues the boxes j = lane * kProducers + prod
    const int j = lane * kProducers + prod;
    const int sub = (j >> 2) < nsub ? (j >> 2) : 0;
    const int h = (j >> 1) & 1;
    const bool is_v = j & 1;
    const bool has_box = j < 4 * nsub;
    const uint32_t dst_base = (is_v ? sV : sK) + h * kKVHalfBytes + sub * br * 128;
    const CUtensorMap* map = is_v ? &maps.vc : &maps.kc;
    const CUtensorMap* tmap = is_v ? &maps.vt : &maps.kt;
    auto div_bs = [&](int x) { return lbs >= 0 ? x >> lbs : x / bs; };
    uint32_t g = 0;
    bool ok = true;
    Walk walk(sp);
    Segment s;
    while (ok && walk.next(p, s)) {
      // Block-table entries of this unit are read in 32-entry windows, one
      // coalesced load per window, the next window requested a window ahead,
      // so no TMA issue waits on a dependent global load.
      {
        // warm L2 with this unit's query rows and ancestor rows: the softmax
        // warps read them when the consumer side reaches the unit, a few
        // tiles from now
        const int rows = p.R - s.rg * p.RPG < p.RPG ? p.R - s.rg * p.RPG : p.RPG;
        const char* qb = static_cast<const char*>(p.q);
        for (int r = lane * kProducers + prod; r < rows; r += 32 * kProducers) {
          const int ur = s.rg * p.RPG + r;
          const int64_t orow = ((int64_t)s.b * p.N + ur / p.G) * p.Hq + s.kvh * p.G + ur % p.G;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + orow * (kD * 2)));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + orow * (kD * 2) + 128));
        }
        if (lane == 0 && prod == 0)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.mask + (int64_t)s.b * p.mask_bstride));
      }
      const int nb = div_bs(s.L + bs - 1);  // valid table entries of request b
      const int32_t* trow = p.block_table + (int64_t)s.b * p.max_blocks;
      const int64_t head_row = (int64_t)s.kvh * bs;
      const int last_pos = s.L > 0 ? (s.L - 1) / br * br : 0;  // ragged tail: finite rows, weight 0
      int w0 = div_bs(s.a * kBlk);  // first entry held in `cur`
      int32_t cur = (w0 + lane < nb) ? __ldg(trow + w0 + lane) : 0;
      int32_t nxt = (w0 + 32 + lane < nb) ? __ldg(trow + w0 + 32 + lane) : 0;
      for (int t = s.a; t < s.e && ok; ++t, ++g) {
        const int stage = g % kStages;
        const uint32_t use = g / kStages;
        const bool tree_tile = (t == s.n - 1);
        if (!tree_tile && div_bs(t * kBlk) >= w0 + 32) {
          w0 += 32;
          cur = nxt;
          nxt = (w0 + 32 + lane < nb) ? __ldg(trow + w0 + 32 + lane) : 0;
        }
        int pos = t * kBlk + sub * br;
        if (pos >= s.L) pos = last_pos;
        const int bi = div_bs(pos);
        const int rel = bi - w0;
        const int32_t from_cur = __shfl_sync(0xffffffffu, cur, rel & 31);
        const int32_t from_nxt = __shfl_sync(0xffffffffu, nxt, rel & 31);
        const int64_t blk = rel < 32 ? from_cur : from_nxt;
        if (use > 0) ok = mbar_wait_warp(&bars.kv_empty[stage], (use - 1) & 1, &bars, status);
        if (!ok) break;
        if (test_withhold(g)) continue;  // development builds only
        if (prod == 0 && lane == 0) { TV_TRACE(0, g); mbar_expect_tx(&bars.kv_full[stage], 2 * kKVTileBytes); }
        __syncwarp();
        const uint32_t dst = dst_base + stage * kKVTileBytes;
        if (tree_tile) {
          if (j < 4) tma_4d(dst, tmap, h * 64, s.kvh, 0, s.b, &bars.kv_full[stage]);
        } else if (has_box) {
          int64_t y = blk * p.Hkv * bs + head_row + (pos - bi * bs);
          if (blk < 0 || blk >= p.num_blocks) {  // out of range: TMA fills zeros
            y = rows_total;
            if (status) atomicOr(status, TV_DEV_BAD_BLOCK);
          }
          tma_2d_stream(dst, map, h * 64, (int)y, &bars.kv_full[stage], pol);
        }
        __syncwarp();
        if (prod == 0 && lane == 0) TV_TRACE(31, g);
      }
      if (ok && s.a == 0 && s.e < s.n) {
        // This slice holds the head of a split unit and finishes it last (the
        // other pieces start their slices with it), merging their published
        // partials in its epilogue: pull them into L2 while the last tiles run.
        const Pieces pc(sp, s.real_start, s.n);
        const int64_t bytes = (int64_t)p.RPG * kD * 4;
        for (int c = pc.c0 + 1; c <= pc.c1; ++c) {
          if (!pc.present(c)) continue;
          const char* po = reinterpret_cast<const char*>(p.part_o + pc.slot(c) * p.RPG * kD);
          for (int64_t off = (int64_t)(prod * 32 + lane) * 128; off < bytes; off += kProducers * 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(po + off));
          const char* pl = reinterpret_cast<const char*>(p.part_lse + pc.slot(c) * p.RPG);
          for (int off = (prod * 32 + lane) * 128; off < p.RPG * 4; off += kProducers * 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(pl + off));
        }
      }
    }
    // drain: every load this warp issued has landed before the CTA exits
    if (lane == 0) {
      const uint32_t first = g > (uint32_t)kStages ? g - kStages : 0;
      for (uint32_t i = first; i < g; ++i)
        mbar_wait(&bars.kv_full[i % kStages], (i / kStages) & 1, &bars, nullptr, false);
    }
}

// ---------------------------------------------------------------- the kernel

template <int M, bool kRope>
__global__ void __launch_bounds__(Cfg<M>::kThreads, Cfg<M>::kCtasPerSm)
    attn_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TcMaps maps, int32_t* status) {
  using C = Cfg<M>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sK = base + C::kOffK, sV = base + C::kOffV;

  TV_TRACE_CTA(0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __shared__ SlicePlan sp;
  if (warp == 0) plan_slice(p, lane, sp, blockIdx.x);
  __syncthreads();
  if (sp.t0 >= sp.t1) return;  // empty slice: uniform exit before any setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], M);  // one commit per MMA issuer
    }
    for (int m = 0; m < M; ++m) {
      mbar_init(&bars.s_full[m], 1);
      mbar_init(&bars.p_full[m], 128);
      mbar_init(&bars.o_done[m], 1);
    }
    mbar_init(&bars.q_full, 128 * M);
    for (int i = 0; i < 4; ++i) mbar_init(&bars.drain[i], 1);
    bars.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == 0) {
    run_producer<C::kStages>(p, sp, maps, bars, sK, sV, lane, status);
  } else if (warp >= 1 && warp < 1 + M) {
    // ------------------------------------------------------------ MMA issuer of M tile m
    // Per tile g: O_m += P_m(g-1) V(g-1), then S_m(g) = Q_m K(g)^T.  The
    // tensor pipe runs them in issue order, so S_m(g) overwrites the TMEM
    // columns holding P_m(g-1) only after that P has been consumed, and the
    // commit that signals S_m(g) also covers O_m's update by tile g-1.
    const int m = warp - 1;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, kBlk, false);
      constexpr uint32_t idO = idesc_bf16(128, kD, true);
      constexpr uint32_t hi = desc_hi(1024);
      const uint32_t dS = tmem + C::col_s(m), dO = tmem + C::col_o(m), aQ = tmem + C::col_q(m);
      uint32_t g = 0;
      int seg_i = 0;
      bool ok = true;
      Walk walk(sp);
      Segment s;
      auto issue_pv = [&](int stage, bool accumulate) {
        const uint32_t lo = desc_lo(sV + stage * kKVTileBytes, kKVHalfBytes);  // MN-major V: LBO = next 64 columns
        if (accumulate) mma_ts<true>(dO, dS, lo, hi, idO);
        else mma_ts<false>(dO, dS, lo, hi, idO);
#pragma unroll
        for (int kk = 1; kk < kBlk / 16; ++kk) mma_ts<true>(dO, dS + kk * 8, lo + kk * (2048 >> 4), hi, idO);
        mma_commit(&bars.o_done[m]);
      };
      auto issue_s = [&](int stage) {
        const uint32_t lo = desc_lo(sK + stage * kKVTileBytes, 0);
        mma_ts<false>(dS, aQ, lo, hi, idS);
#pragma unroll
        for (int kk = 1; kk < kD / 16; ++kk)
          mma_ts<true>(dS, aQ + kk * 8, lo + (kk / 4) * (kKVHalfBytes >> 4) + (kk % 4) * 2, hi, idS);
        mma_commit(&bars.s_full[m]);
      };
      while (ok && walk.next(p, s)) {
        const int n_seg = s.e - s.a;
        ok = mbar_wait(&bars.q_full, seg_i & 1, &bars, status);
        if (!ok) break;
        fence_after();
        for (int k = 0; k < n_seg && ok; ++k, ++g) {
          const int stage = g % C::kStages;
          ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
          if (!ok) break;
          if (m == 0) TV_TRACE(1, g);
          if (k > 0) {
            ok = mbar_wait(&bars.p_full[m], (g - 1) & 1, &bars, status);
            if (!ok) break;
            fence_after();
            issue_pv((g - 1) % C::kStages, k > 1);
            mma_commit(&bars.kv_empty[(g - 1) % C::kStages]);
            TV_TRACE(4 + m, g - 1);
          }
          issue_s(stage);
          TV_TRACE(2 + m, g);
        }
        if (!ok) break;
        ok = mbar_wait(&bars.p_full[m], (g - 1) & 1, &bars, status);
        if (!ok) break;
        fence_after();
        issue_pv((g - 1) % C::kStages, n_seg > 1);
        mma_commit(&bars.kv_empty[(g - 1) % C::kStages]);
        TV_TRACE(4 + m, g - 1);
        ++seg_i;
      }
      if (!ok) mma_drain(bars, m);
    }
    __syncwarp();
  } else if (warp >= C::kSoftmaxWarp0 && warp < C::kSoftmaxWarp0 + 4 * M) {
    // ------------------------------------------------------------ softmax / epilogue
    const int m = (warp - C::kSoftmaxWarp0) / 4;
    const int quarter = warp % 4;         // TMEM lanes 32*quarter .. +31
    const int rl = quarter * 32 + lane;   // row within the M tile = TMEM lane
    const int row = m * 128 + rl;         // row within the unit
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = lane_addr + C::col_s(m);
    const uint32_t tQ = lane_addr + C::col_q(m);
    const uint32_t tO = lane_addr + C::col_o(m);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    uint32_t g = 0;
    bool ok = true;
    Walk walk(sp);
    Segment s;
    while (ok && walk.next(p, s)) {
      const int unit_row = s.rg * p.RPG + row;  // row within the (b, kv head) group
      const bool valid_row = unit_row < p.R;
      const int node = valid_row ? unit_row / p.G : 0;
      const int head_in_group = unit_row % p.G;
      const int64_t orow = ((int64_t)s.b * p.N + node) * p.Hq + s.kvh * p.G + head_in_group;
      const uint64_t mrow = valid_row ? p.mask[(int64_t)s.b * p.mask_bstride + node] : 1ull;
      // this row of Q into TMEM (the previous unit's MMAs are complete: its
      // epilogue waited for the last O update)
      if constexpr (kRope) {
        // the whole row, rotated at the node's position, then into TMEM
        const uint4* src = reinterpret_cast<const uint4*>(q + orow * kD);
        uint4 qr[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) qr[c] = valid_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        rope_row(qr, p, valid_row ? row_pos(mrow, s.L) : -1, status, lane);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = qr[c * 8 + j];
            r[4 * j] = v.x; r[4 * j + 1] = v.y; r[4 * j + 2] = v.z; r[4 * j + 3] = v.w;
          }
          tmem_st32(tQ + c * 32, r);
        }
        tmem_st_wait();
        fence_before();
        mbar_arrive(&bars.q_full);
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(q + orow * kD);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = valid_row ? __ldg(src + c * 8 + j) : make_uint4(0, 0, 0, 0);
            r[4 * j] = v.x; r[4 * j + 1] = v.y; r[4 * j + 2] = v.z; r[4 * j + 3] = v.w;
          }
          tmem_st32(tQ + c * 32, r);
        }
        tmem_st_wait();
        fence_before();
        mbar_arrive(&bars.q_full);
      }
      float m_run = -INFINITY, l = 0.f;
      const int n_seg = s.e - s.a;
      for (int k = 0; k < n_seg; ++k, ++g) {
        const int t = s.a + k;
        ok = mbar_wait_warp(&bars.s_full[m], g & 1, &bars, status);
        if (!ok) break;
        fence_after();
        if (rl == 0) TV_TRACE(6 + 4 * m, g);
        float sv[kBlk];
        {
          uint32_t r[32];
          tmem_ld32(tS, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(r[c]);
          tmem_ld32(tS + 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[32 + c] = __uint_as_float(r[c]);
        }
        if (rl == 0) TV_TRACE(7 + 4 * m, g);
        if (t == s.n - 1) {
#pragma unroll
          for (int c = 0; c < kBlk; ++c)
            if (!(c < p.N && ((mrow >> c) & 1ull))) sv[c] = -INFINITY;
        } else {
          const int lim = s.L - t * kBlk;  // keys [0, lim) of this tile are in the prefix
          if (lim < kBlk) {
#pragma unroll
            for (int c = 0; c < kBlk; ++c)
              if (c >= lim) sv[c] = -INFINITY;
          }
        }
        float mx = row_max64(sv);
        mx *= p.scale_log2;  // scale > 0: max of scaled = scaled max
        const float m_new = fmaxf(m_run, mx);
        const bool grow = m_new > m_run + kRescaleThreshold;
        // O_m already holds tiles < g (the S_m(g) commit covered them)
        if (k > 0 && __any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? exp2f(m_run - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < kD; c += 32) {
            uint32_t r[32];
            tmem_ld32(tO + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tmem_st32(tO + c, r);
          }
        }
        if (grow) {
          l *= exp2f(m_run - m_new);
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t sc2 = pack_f32x2(p.scale_log2, p.scale_log2), negm2 = pack_f32x2(-m_use, -m_use);
        uint64_t acc0 = 0, acc1 = 0;  // two packed (f32, f32) partial sums
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < kBlk / 2; ++c) {
          float e0, e1;
          exp2_pair(sv[2 * c], sv[2 * c + 1], sc2, negm2, e0, e1);
          if (c & 1) acc1 = add_f32x2(acc1, pack_f32x2(e0, e1)); else acc0 = add_f32x2(acc0, pack_f32x2(e0, e1));
          pk[c] = pack_bf16(e0, e1);
        }
        l += sum_f32x2(add_f32x2(acc0, acc1));
        tmem_st32(tS, pk);  // P_m(g) over the first 32 columns of S_m
        tmem_st_wait();
        fence_before();
        mbar_arrive(&bars.p_full[m]);
        if (rl == 0) TV_TRACE(9 + 4 * m, g);
      }
      if (!ok) break;
      // epilogue: O / l for this unit's rows
      ok = mbar_wait_warp(&bars.o_done[m], (g - 1) & 1, &bars, status);
      if (!ok) break;
      fence_after();
      Walk ahead = walk;
      Segment s_ahead;
      // after the slice's last tile the K/V ring is idle: merges stage through it
      uint8_t* stage = ahead.next(p, s_ahead) ? nullptr : smem_raw + (base - raw) + C::kOffK;
      finish_row<1>(p, sp, s, row, valid_row, orow, tO, m_run, l, stage);
      fence_before();
    }
  }

  TV_TRACE_CTA(1);
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------- tail rows of the two-M-tile kernel
//
// When a (request, KV head) has R = G * N rows just above the 256 that two
// 128-row M tiles hold (the long-context shape: 33 nodes x 8 heads = 264), a
// second row group would stream the unit's whole K/V a second time for a few
// rows, and a third M tile costs as much tensor time as a full one and does
// not fit in TMEM.  The rows 256 .. R - 1 (at most kTailRows) are instead
// computed from the K/V tiles already in the stage ring by warps of their
// own (kTW tail warps), with warp-level bf16 MMAs (mma.sync m16n8k16, fp32
// accumulation) in transposed form, so that the tail rows sit on the MMA's
// 8-wide N side and nothing is padded:
//   S^T [16 keys x 8 rows]  = K[16 keys x 128] Q_tail^T
//   O_w^T [128 x 8 rows]   += V[16 keys x 128]^T P^T
// Two tail warps share each tile, 32 keys each; with four tail warps the two
// pairs take alternate tiles of the ring, so that each warp pays the per-tile
// costs (barrier wait, row maxima across lanes, proxy fence and release)
// once per two tiles.  Every warp keeps its own running maximum and sum over
// the keys it saw; the parts are merged once per unit, in warp order, and the
// rows are written (or, for a split unit, published and merged) with the
// same arithmetic as the other rows' memory merge.  A tail warp frees a stage with its own arrival on the
// stage's empty barrier once its reads of the stage are done, so the ring
// waits for the tail as it waits for the P V products; the tail warps lag the
// TMA stream by at most the ring's depth and never hold up a TMA issue.
//
// These MMAs share the SM's tensor pipe with the tcgen05 products: while
// those run, one sub-partition completes a warp-level MMA only every 40-70
// cycles (measured), so the tail is spread over as many sub-partitions as
// the launch allows -- four tail warps, one per sub-partition, when one TMA
// warp can issue a tile's boxes (block size >= 32: at most 8 boxes), else two.
constexpr int kTailRows = 8;

template <int kTW>
struct TailSmem {
  float m[kTW][kTailRows];                      // per warp at the unit's end: running maximum (log2)
  float l[kTW][kTailRows];                      //   ... and the sum of its keys' weights
  float o[kTW][kTailRows][kD];                  //   ... and its unnormalised rows
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// d += A[16 x 16] B[16 x 8], bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Transpose of an 8x8 matrix of 16-bit elements held as one 32-bit fragment
// per lane (row lane / 4, columns 2 (lane % 4), + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// One tail warp's share of the tail rows of the unit in progress.  Lane
// (g = lane / 4, t = lane % 4) holds, in MMA fragment order: Q of tail row g
// (the B operand of S^T: d = 16 ks + 2t, +1 and + 8, + 9), and the scores,
// weights and O^T entries of tail rows 2t and 2t + 1 for keys (or head
// dimensions) g and g + 8 of each 16-wide block.
struct TailRowsState {
  uint32_t qb[8][2];
  uint64_t mr[2];  // ancestor rows of tail rows 2t, 2t + 1
  float m_run[2], l[2];
  float o[8][4];   // O^T block mb: (d 16mb + g, row 2t), (.., row 2t + 1), (d 16mb + g + 8, row 2t), (.., 2t + 1)
};

// Loads Q of the segment's tail rows (rotated here when Q arrives unrotated)
// and the tail rows' ancestor rows, and clears the running state.
template <bool kRope>
__device__ __forceinline__ void tail_begin(const AttnParams& p, const Segment& s, TailRowsState& ts, int lane,
                                           int32_t* status) {
  const int g = lane >> 2, tq = lane & 3;
  const int ur = kTcMaxRows + g;  // unit row of this lane's Q operand column
  const bool v = ur < p.R;
  const int node = v ? ur / p.G : 0;
  const int64_t orow = ((int64_t)s.b * p.N + node) * p.Hq + s.kvh * p.G + ur % p.G;
  const uint32_t* src = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(p.q) + orow * kD);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    ts.qb[ks][0] = v ? __ldg(src + 8 * ks + tq) : 0u;
    ts.qb[ks][1] = v ? __ldg(src + 8 * ks + tq + 4) : 0u;
  }
  const unsigned long long* mrows =
      reinterpret_cast<const unsigned long long*>(p.mask) + (int64_t)s.b * p.mask_bstride;
  if constexpr (kRope) {
    // rotate-half at the node's position with tv_rope_apply's float32
    // arithmetic and bf16 rounding: element d pairs with d + 64, i.e. word
    // ks with word ks + 4 of the same lane
    const int pos = v ? row_pos(__ldg(mrows + node), s.L) : -1;
    if (pos >= p.rope_max_pos && tq == 0 && status) atomicOr(status, TV_DEV_BAD_POSITION);
    if (pos >= 0 && pos < p.rope_max_pos) {
      const float* cs = p.rope_cs + (int64_t)pos * kD;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int wd = 0; wd < 2; ++wd) {
          const int k0 = 16 * ks + 2 * tq + 8 * wd;  // frequency of the word's low element
          const uint32_t lo = ts.qb[ks][wd], hi = ts.qb[ks + 4][wd];
          float a0, b0, a1, b1;
          rope_pair(__uint_as_float(lo << 16), __uint_as_float(hi << 16), __ldg(cs + k0), __ldg(cs + kD / 2 + k0), a0,
                    b0);
          rope_pair(__uint_as_float(lo & 0xffff0000u), __uint_as_float(hi & 0xffff0000u), __ldg(cs + k0 + 1),
                    __ldg(cs + kD / 2 + k0 + 1), a1, b1);
          ts.qb[ks][wd] = pack_bf16(a0, a1);
          ts.qb[ks + 4][wd] = pack_bf16(b0, b1);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = kTcMaxRows + 2 * tq + j;
    ts.mr[j] = r < p.R ? __ldg(mrows + r / p.G) : 0ull;
    ts.m_run[j] = -INFINITY;
    ts.l[j] = 0.f;
  }
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int e = 0; e < 4; ++e) ts.o[mb][e] = 0.f;
}

// Tile t of the segment from the stage at kb (K) / vb (V): S^T of this
// warp's 32 keys (half h of the tile), online softmax over them,
// O^T += V^T P^T.
constexpr int kTailSplit = 2;  // tail warps per tile
__device__ __forceinline__ void tail_tile(const AttnParams& p, const Segment& s, int t, uint32_t kb, uint32_t vb,
                                          TailRowsState& ts, int h, int lane) {
  constexpr int kTailKeys = kBlk / kTailSplit;  // keys of a tile per tail warp
  constexpr int kNB = kTailKeys / 16;           // 16-key blocks per tail warp
  static_assert(kNB >= 1 && kNB * 16 * kTailSplit == kBlk, "whole 16-key blocks per tail warp");
  const int w = h;
  const int g = lane >> 2, tq = lane & 3, i8 = lane >> 3;
  // S^T per 16-key block: A = K rows x 16 head dims per step, by ldmatrix:
  // matrices (keys 0-7 | 8-15) x (dims 0-7 | 8-15) of the step, lane
  // i8 * 8 + r addressing row r of matrix i8; four accumulators per block
  // (steps ks, ks + 4 chained) so that MMA latency overlaps
  float sv[kNB][4];
  {
    float acc[kNB][4][4];
#pragma unroll
    for (int kb2 = 0; kb2 < kNB; ++kb2)
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[kb2][c][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int kb2 = 0; kb2 < kNB; ++kb2) {
        const int key = kTailKeys * w + 16 * kb2 + (lane & 7) + 8 * (i8 & 1);
        uint32_t a[4];
        ldsm_x4(kb + key * 128 + (ks >> 2) * kKVHalfBytes + (((2 * (ks & 3) + (i8 >> 1)) ^ (key & 7)) << 4), a);
        mma_m16n8k16(acc[kb2][ks & 3], a, ts.qb[ks][0], ts.qb[ks][1]);
      }
    }
#pragma unroll
    for (int kb2 = 0; kb2 < kNB; ++kb2)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        sv[kb2][e] = (acc[kb2][0][e] + acc[kb2][1][e]) + (acc[kb2][2][e] + acc[kb2][3][e]);
  }
  // sv[kb2]: (key k, row 2t), (k, 2t + 1), (k + 8, 2t), (k + 8, 2t + 1), k = 32w + 16 kb2 + g
#pragma unroll
  for (int kb2 = 0; kb2 < kNB; ++kb2) {
    const int k0 = kTailKeys * w + 16 * kb2 + g, k1 = k0 + 8;
    if (t == s.n - 1) {
      if (!(k0 < p.N && ((ts.mr[0] >> k0) & 1ull))) sv[kb2][0] = -INFINITY;
      if (!(k0 < p.N && ((ts.mr[1] >> k0) & 1ull))) sv[kb2][1] = -INFINITY;
      if (!(k1 < p.N && ((ts.mr[0] >> k1) & 1ull))) sv[kb2][2] = -INFINITY;
      if (!(k1 < p.N && ((ts.mr[1] >> k1) & 1ull))) sv[kb2][3] = -INFINITY;
    } else {
      const int lim = s.L - t * kBlk;
      if (k0 >= lim) sv[kb2][0] = sv[kb2][1] = -INFINITY;
      if (k1 >= lim) sv[kb2][2] = sv[kb2][3] = -INFINITY;
    }
  }
  float mx[2] = {fmaxf(sv[0][0], sv[0][2]), fmaxf(sv[0][1], sv[0][3])};
#pragma unroll
  for (int kb2 = 1; kb2 < kNB; ++kb2) {
    mx[0] = fmaxf(mx[0], fmaxf(sv[kb2][0], sv[kb2][2]));
    mx[1] = fmaxf(mx[1], fmaxf(sv[kb2][1], sv[kb2][3]));
  }
  // The weights are first taken against the running maxima as they stand,
  // while the tile's row maxima are reduced across lanes beside them; only
  // when some row of the warp has no maximum yet, or its maximum grows past
  // the rescale threshold, are they taken again after the update below --
  // the same values as updating first, with the cross-lane reduction off
  // the path from the scores to the P V products.
  float pv[kNB][4];
#pragma unroll
  for (int kb2 = 0; kb2 < kNB; ++kb2)
#pragma unroll
    for (int e = 0; e < 4; ++e) pv[kb2][e] = fast_exp2(fmaf(sv[kb2][e], p.scale_log2, -ts.m_run[e & 1]));
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
    mx[j] *= p.scale_log2;
  }
  const bool redo = ts.m_run[0] == -INFINITY || ts.m_run[1] == -INFINITY ||
                    mx[0] > ts.m_run[0] + kRescaleThreshold || mx[1] > ts.m_run[1] + kRescaleThreshold;
  if (__any_sync(0xffffffffu, redo)) {
    float m_use[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float m_new = fmaxf(ts.m_run[j], mx[j]);
      if (m_new > ts.m_run[j] + kRescaleThreshold) {
        const float al = exp2f(ts.m_run[j] - m_new);
        ts.l[j] *= al;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          ts.o[mb][j] *= al;
          ts.o[mb][2 + j] *= al;
        }
        ts.m_run[j] = m_new;
      }
      m_use[j] = ts.m_run[j] == -INFINITY ? 0.f : ts.m_run[j];
    }
#pragma unroll
    for (int kb2 = 0; kb2 < kNB; ++kb2)
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[kb2][e] = fast_exp2(fmaf(sv[kb2][e], p.scale_log2, -m_use[e & 1]));
  }
  {
    float l0 = pv[0][0] + pv[0][2], l1 = pv[0][1] + pv[0][3];
#pragma unroll
    for (int kb2 = 1; kb2 < kNB; ++kb2) {
      l0 += pv[kb2][0] + pv[kb2][2];
      l1 += pv[kb2][1] + pv[kb2][3];
    }
    ts.l[0] += l0;
    ts.l[1] += l1;
  }
  // P^T as the B operand of O^T: the weights of (key g | g + 8, rows 2t,
  // 2t + 1), packed as bf16 pairs, are 8x8 fragments of P[key][row];
  // movmatrix transposes them in registers to P[row g][keys 2t, 2t + 1]
  // (resp. 8 + 2t, 9 + 2t), the B fragment layout
  uint32_t bp[kNB][2];
#pragma unroll
  for (int kb2 = 0; kb2 < kNB; ++kb2) {
    bp[kb2][0] = movmatrix_trans(pack_bf16(pv[kb2][0], pv[kb2][1]));
    bp[kb2][1] = movmatrix_trans(pack_bf16(pv[kb2][2], pv[kb2][3]));
  }
  // O^T: A = V^T (16 head dims x 16 keys) by transposing ldmatrix of the V
  // rows: matrices (dims 0-7 | 8-15) x (keys 0-7 | 8-15)
#pragma unroll
  for (int kb2 = 0; kb2 < kNB; ++kb2) {
    const int key = kTailKeys * w + 16 * kb2 + (lane & 7) + 8 * (i8 >> 1);
    const uint32_t row = vb + key * 128;
    const int sw = key & 7;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      uint32_t a[4];
      ldsm_x4_trans(row + (mb >> 2) * kKVHalfBytes + (((2 * (mb & 3) + (i8 & 1)) ^ sw) << 4), a);
      mma_m16n8k16(ts.o[mb], a, bp[kb2][0], bp[kb2][1]);
    }
  }
}

// End of a segment: the tail warps' parts are merged (warp order) and the
// tail rows written; a split unit publishes its part and the piece that
// completes the rows' arrival counts merges them from memory, with the
// arithmetic of the other rows' memory merge.  Collective over the tail
// warps (two passes of the tail_sync barrier).
template <int kTW>
__device__ __forceinline__ bool tail_end(const AttnParams& p, const SlicePlan& sp, const Segment& s, TailRowsState& ts,
                                         TailSmem<kTW>* sm, Bars& bars, uint32_t& tb, int w, int lane,
                                         int32_t* status) {
  constexpr float kLn2 = 0.69314718055994530942f;
  constexpr int kThreadsPerRow = 64 / kTailRows;  // the merge runs on tail warps 0 and 1
  constexpr int kCols = kD / kThreadsPerRow;      // head dims per thread in the merge
  static_assert(kCols == 16, "the merge below handles 16 head dims per thread");
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) ts.l[j] += __shfl_xor_sync(0xffffffffu, ts.l[j], off);
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      sm->m[w][2 * tq + j] = ts.m_run[j];
      sm->l[w][2 * tq + j] = ts.l[j];
    }
  }
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int e = 0; e < 4; ++e) sm->o[w][2 * tq + (e & 1)][16 * mb + g + 8 * (e >> 1)] = ts.o[mb][e];
  mbar_arrive(&bars.tail_sync);
  if (!mbar_wait_warp(&bars.tail_sync, tb & 1, &bars, status)) return false;
  ++tb;
  if (w >= 2) {  // the scratch is read by tail warps 0 and 1 only
    mbar_arrive(&bars.tail_sync);
    const bool ok = mbar_wait_warp(&bars.tail_sync, tb & 1, &bars, status);
    ++tb;
    return ok;
  }
  // thread i of tail warps 0 and 1: tail row i / 8, head dims (i % 8) * 16 .. + 15
  const int i = w * 32 + lane;
  const int r = i / kThreadsPerRow, d0 = (i % kThreadsPerRow) * kCols;
  const int ur = kTcMaxRows + r;
  float M = -INFINITY;
#pragma unroll
  for (int q = 0; q < kTW; ++q) M = fmaxf(M, sm->m[q][r]);
  float a[kTW], l = 0.f;
#pragma unroll
  for (int q = 0; q < kTW; ++q) {
    a[q] = M == -INFINITY ? 0.f : exp2f(sm->m[q][r] - M);
    l = fmaf(a[q], sm->l[q][r], l);
  }
  float v[kCols];
#pragma unroll
  for (int j = 0; j < kCols; ++j) {
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kTW; ++q) acc = fmaf(a[q], sm->o[q][r][d0 + j], acc);
    v[j] = acc;
  }
  // the scratch may be reused once every tail thread has read it
  mbar_arrive(&bars.tail_sync);
  const float inv = l > 0.f ? 1.f / l : 0.f;  // no key at all: zero row
#pragma unroll
  for (int j = 0; j < kCols; ++j) v[j] *= inv;
  const float lse2 = M + log2f(l);
  const bool valid = ur < p.R;
  const int node = valid ? ur / p.G : 0;
  const int64_t orow = ((int64_t)s.b * p.N + node) * p.Hq + s.kvh * p.G + ur % p.G;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  const bool lead = (lane % kThreadsPerRow) == 0;
  if (s.a == 0 && s.e == s.n) {
    if (valid) {
      store_bf16_16(out + orow * kD + d0, v);
      if (lead && p.lse) p.lse[orow] = lse2 * kLn2;
    }
  } else {
    const Pieces pc(sp, s.real_start, s.n);
    const uint32_t mine = (uint32_t)(s.e - s.a);
    const int64_t srow = pc.slot(pc.self) * p.RPG + ur;
    if (valid) {
      float4* dst = reinterpret_cast<float4*>(p.part_o + srow * kD + d0);
#pragma unroll
      for (int j = 0; j < kCols / 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      if (lead) p.part_lse[srow] = lse2;
    }
    __threadfence();
    __syncwarp();
    bool last = false;
    uint32_t* ctr = p.arrive + (int64_t)pc.c0 * p.RPG + ur;
    if (valid && lead) last = atom_add_acq_rel(ctr, mine) + mine == (uint32_t)s.n;
    last = __shfl_sync(0xffffffffu, last, lane & ~(kThreadsPerRow - 1));
    if (last) {
      __threadfence();
      float mx, z;
      piece_stats<false>(p, pc, -1, 0.f, ur, mx, z);
      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.f;
      accum_pieces<false>(acc, p, pc, -1, acc, 0.f, ur, d0, mx, 1.f / z);
      store_bf16_16(out + orow * kD + d0, acc);
      if (lead && p.lse) p.lse[orow] = (mx + log2f(z)) * kLn2;
      if (lead) *ctr = 0;  // every piece has arrived: leave the counter at zero
    }
  }
  const bool ok = mbar_wait_warp(&bars.tail_sync, tb & 1, &bars, status);
  ++tb;
  return ok;
}

// A tail warp's loop: every tile of the CTA's slice, in ring order, after
// the TMA producers' loads land; the stage is freed after the warp's reads.
template <int kStages, bool kRope, int kTW>
__device__ __forceinline__ void run_tail(const AttnParams& p, const SlicePlan& sp, Bars& bars, uint32_t sK, uint32_t sV,
                                         TailSmem<kTW>* tsm, int w, int lane, int32_t* status) {
  uint32_t g = 0, tb = 0;
  bool ok = true;
  Walk walk(sp);
  Segment s;
  TailRowsState ts;
  constexpr int kRR = kTW / kTailSplit;  // tail warp pairs, taking tiles in turn
  const int pair = w / kTailSplit;
  while (ok && walk.next(p, s)) {
    tail_begin<kRope>(p, s, ts, lane, status);
    for (int t = s.a; t < s.e; ++t, ++g) {
      if ((int)(g % kRR) != pair) continue;  // the other pair's tile
      const int stage = g % kStages;
      ok = mbar_wait_warp(&bars.kv_full[stage], (g / kStages) & 1, &bars, status);
      if (!ok) break;
      test_tail_delay(pair);
      tail_tile(p, s, t, sK + stage * kKVTileBytes, sV + stage * kKVTileBytes, ts, w % kTailSplit, lane);
      // the stage was read through the generic proxy (ldmatrix) and the next
      // TMA load writes it through the async proxy: order the reads first
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.kv_empty[stage]);
    }
    if (!ok) break;
    ok = tail_end<kTW>(p, sp, s, ts, tsm, bars, tb, w, lane, status);
  }
}

// ---------------------------------------------------------------- two M tiles (up to 256 rows)
//
// Every operand placement is chosen so that no single resource is on the
// critical path of a 64-key tile (about 1400 cycles of HBM time per SM):
//  * four MMA-issuing warps (S_0, S_1, O_0 += P_0 V, O_1 += P_1 V), because one
//    thread issues at most one tcgen05.mma about every 70 cycles;
//  * P_m has its own TMEM columns, so S_m(g+1) is computed while the softmax
//    of tile g runs;
//  * TMEM (512 columns) holds S_0 S_1 P_0 P_1 Q_0 O_0 O_1 = 64+64+32+32+64+128+128;
//    Q_1 therefore stays in shared memory (S_1 = Q_1 K^T reads both operands
//    from shared memory), which keeps shared-memory traffic near 128 KB per tile.
template <int kTailW, bool kQS = false>
struct PairCfgT {
  // Five K/V stages (measured 1-3 % faster than six on the 64-request and
  // long-context shapes); the shared memory left holds the tail rows'
  // end-of-unit scratch.
  static constexpr int kStages = 5;
  // Warps 0-3 issue TMA, 4-7 issue MMAs (S_0, S_1, PV_0, PV_1), 8-15 are the
  // two softmax warpgroups: warp w runs on sub-partition w % 4, so each
  // sub-partition carries one producer, one issuer and two softmax warps.
  // With two tail warps (kTailW = 2), warps 0-1 issue TMA and 2-3 compute the
  // tail rows; with four, warps 0-3 compute the tail rows, warp 6 issues both
  // P V products and warp 7 issues TMA.
  static_assert(kTailW == 0 || kTailW == 2 || kTailW == 4, "0, 2 or 4 tail warps");
  static constexpr int kProducers = kTailW == 4 ? 1 : 4 - kTailW;
  static constexpr int kThreads = 32 * 16;
  static constexpr int kAllocWarp = 4;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kKVTileBytes;
  static constexpr int kOffQ1 = kOffV + kStages * kKVTileBytes;  // 2 halves x 128 rows x 128 B
  static constexpr int kOffTail = kOffQ1 + 2 * 128 * 128;
  // kQS: the next unit's Q_0 is staged here by TMA (32 KB, 128B-swizzled)
  static constexpr int kOffQ0S = kOffTail + (kTailW ? (int)sizeof(TailSmem<kTailW>) : 0);
  static constexpr int kBytes = kOffQ0S + (kQS ? 128 * kD * 2 : 0);
  static constexpr int kSmem = kBytes + 1024;
  static constexpr uint32_t col_s(int m) { return m * 64; }
  static constexpr uint32_t col_p(int m) { return 128 + m * 32; }
  static constexpr uint32_t kColQ0 = 192;
  static constexpr uint32_t col_o(int m) { return 256 + m * 128; }
  static constexpr int kSoftmaxWarp0 = 8;
};
using PairCfg = PairCfgT<0>;
static_assert(PairCfgT<4>::kSmem <= 227 * 1024 - 1024, "the tail variant fits the opt-in shared memory");
static_assert(PairCfgT<0, true>::kSmem <= 227 * 1024 - 1024, "the staged-Q variant fits the opt-in shared memory");
static_assert(PairCfgT<0, true>::kOffQ0S % 1024 == 0, "the Q_0 staging tile is 1024-byte aligned (128B swizzle)");
static_assert(PairCfgT<4>::kStages * kKVTileBytes >= 128 * kD * 4, "each half of the pair ring holds one M tile's rows");
static_assert(PairCfg::kStages * kKVTileBytes >= 128 * kD * 4, "each half of the pair ring holds one M tile's rows");

// The unit is the last row group of a (request, KV head) with at most 128
// rows left, so one M tile holds all its rows.
__device__ __forceinline__ bool shared_unit(const AttnParams& p, const Segment& s) {
  return p.R - s.rg * p.RPG <= 128;
}

// kSkip: a shared unit (shared_unit) has its rows in both M tiles, and the
// key tiles go to the M tile sh_owner names, each M tile with its own running
// max and sum; at the unit's end M tile 1 posts its (max, sum) through shared
// memory, and M tile 0 merges M tile 1's accumulator into its own (same TMEM
// lanes; a part without keys adds nothing) and finishes the rows.  The
// per-M-tile barriers (s_full/s_free/p_full/o_done) then count that M tile's
// products, not the ring's tiles.
//
// kSplitKeys: the two M tiles take the even and the odd key tiles.  On the
// 264-row shape (33 nodes, G = 8) that measured slower than M tile 0 taking
// every tile (0.715 against 0.690 ms): its shared units are bound by the
// second read of their K/V, not by one M tile's chain.  So M tile 0 computes
// shared units alone and M tile 1's part is empty.
constexpr bool kSplitKeys = false;
__device__ __forceinline__ int sh_owner(int t) { return kSplitKeys ? (t & 1) : 0; }
template <bool kRope, bool kSkip, int kTailW, bool kStagedQ>
__global__ void __launch_bounds__(PairCfg::kThreads, 1)
    attn_tc_pair_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TcMaps maps, int32_t* status) {
  // kQS (kStagedQ, where the variant allows it): after a CTA's first unit,
  // each unit's Q reaches its operand slots
  // through the S issuers instead of the softmax warps: Q_0 is staged in
  // shared memory by TMA during the previous unit and copied into TMEM with
  // tcgen05.cp just before the unit's first S_0 products (the same thread
  // issued the previous unit's S_0, so the copy follows them in the pipe);
  // Q_1 is loaded by TMA into its tile once the previous unit's last S_1 has
  // completed.  The softmax warps then only write the finished unit's rows at
  // a boundary.
  constexpr bool kQS = kStagedQ && !kRope && !kSkip && kTailW == 0;
  using C = PairCfgT<kTailW, kQS>;
  static_assert(!(kSkip && kTailW), "tail rows replace the second row group");
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ float s_sh[kSkip ? 256 : 1];  // shared units: M tile 1's running max and sum per row
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sK = base + C::kOffK, sV = base + C::kOffV, sQ1 = base + C::kOffQ1;
  uint8_t* gQ1 = smem_raw + (base - raw) + C::kOffQ1;

  TV_TRACE_CTA(0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __shared__ SlicePlan sp;
  if (warp == 0) plan_slice(p, lane, sp, blockIdx.x);
  __syncthreads();
  if (sp.t0 >= sp.t1) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], kTailW ? 2 + kTailSplit : 2);  // one commit per P V product (+ the tile's tail warps)
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(&bars.s_full[m], 1);
      mbar_init(&bars.s_free[m], 128);
      mbar_init(&bars.p_full[m], 128);
      mbar_init(&bars.o_done[m], 1);
    }
    mbar_init(&bars.q_full, 256);
    mbar_init(&bars.sh_stat, 128);
    mbar_init(&bars.sh_read, 128);
    mbar_init(&bars.tail_sync, 32 * (kTailW ? kTailW : 1));
    for (int i = 0; i < 4; ++i) mbar_init(&bars.drain[i], 1);
    mbar_init(&bars.q0s_full, 1);
    mbar_init(&bars.cp_done, 1);
    mbar_init(&bars.q1_free, 1);
    mbar_init(&bars.q1_full, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&bars.merge_full[i / 4][i % 4], 1);
    bars.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == C::kAllocWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars.tmem_base;
  constexpr uint32_t hi = desc_hi(1024);

  if (warp < 4) {
    if constexpr (kTailW > 0) {
      // the first 4 - kTailW warps issue every TMA box (none with four tail
      // warps: warp 7 does), the others compute the tail rows
      if (warp < 4 - kTailW) {
        run_producer<C::kStages, C::kProducers>(p, sp, maps, bars, sK, sV, lane, status, warp);
      } else {
        auto* tsm = reinterpret_cast<TailSmem<kTailW>*>(smem_raw + (base - raw) + C::kOffTail);
        run_tail<C::kStages, kRope, kTailW>(p, sp, bars, sK, sV, tsm, warp - (4 - kTailW), lane, status);
      }
    } else {
      run_producer<C::kStages, C::kProducers>(p, sp, maps, bars, sK, sV, lane, status, warp);
    }
  } else if (kTailW == 4 && warp == 7) {
    run_producer<C::kStages, 1>(p, sp, maps, bars, sK, sV, lane, status, 0);
  } else if (kTailW == 4 && warp == 6) {
    // ------------------------------------------------------------ O_0 += P_0 V, then O_1 += P_1 V
    if (lane == 0) {
      constexpr uint32_t idO = idesc_bf16(128, kD, true);
      uint32_t g = 0;
      bool ok = true;
      Walk walk(sp);
      Segment s;
      while (ok && walk.next(p, s)) {
        for (int t = s.a; t < s.e && ok; ++t, ++g) {
          const int stage = g % C::kStages;
          ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
          const uint32_t vlo = desc_lo(sV + stage * kKVTileBytes, kKVHalfBytes);
          for (int m = 0; m < 2 && ok; ++m) {
            ok = mbar_wait(&bars.p_full[m], g & 1, &bars, status);
            if (!ok) break;
            fence_after();
            const uint32_t dO = tmem + C::col_o(m), aP = tmem + C::col_p(m);
            if (t > s.a) mma_ts<true>(dO, aP, vlo, hi, idO);
            else mma_ts<false>(dO, aP, vlo, hi, idO);
#pragma unroll
            for (int kk = 1; kk < kBlk / 16; ++kk) mma_ts<true>(dO, aP + kk * 8, vlo + kk * (2048 >> 4), hi, idO);
            mma_commit(&bars.o_done[m]);
            mma_commit(&bars.kv_empty[stage]);
          }
          if (ok) TV_TRACE(4, g);
        }
      }
      if (!ok) mma_drain(bars, 2);
    }
    __syncwarp();
  } else if (warp == 4 || warp == 5) {
    // ------------------------------------------------------------ S_m = Q_m K^T issuer
    const int m = warp - 4;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, kBlk, false);
      const uint32_t dS = tmem + C::col_s(m);
      uint32_t g = 0, g1 = 0;  // tiles of the ring; with kSkip, S products of this M tile
      uint32_t& gm = kSkip ? g1 : g;
      int seg_i = 0;
      bool ok = true;
      Walk walk(sp);
      Segment s;
      // kQS: Q loads this thread issued (and whether the last is still in flight)
      uint32_t nq = 0;
      bool q_pending = false;
      const uint32_t sQ0S = base + C::kOffQ0S;
      // the Q rows of M tile m of unit sg by TMA: two boxes of 64 columns
      auto load_q = [&](const Segment& sg, uint32_t dst, uint64_t* bar) {
        mbar_expect_tx(bar, 128 * kD * 2);
        const int y = sg.kvh * p.G, z = sg.b * p.N + (sg.rg * p.RPG + m * 128) / p.G;
        tma_3d(dst, &maps.qm, 0, y, z, bar);
        tma_3d(dst + 16384, &maps.qm, 64, y, z, bar);
        ++nq;
        q_pending = true;
      };
      while (ok && walk.next(p, s)) {
        Segment sn;
        bool hn = false;
        if constexpr (kQS) {
          Walk wn = walk;
          hn = wn.next(p, sn);
        }
        if (!kQS || seg_i == 0) {
          ok = mbar_wait(&bars.q_full, seg_i & 1, &bars, status);
          if (!ok) break;
          fence_after();
          if (kQS && m == 0 && hn) load_q(sn, sQ0S, &bars.q0s_full);  // the staging tile is free
        } else if (m == 1) {
          ok = mbar_wait(&bars.q1_full, (seg_i - 1) & 1, &bars, status);
          if (!ok) break;
          q_pending = false;
        }
        const bool sh = kSkip && shared_unit(p, s);
        if (m == 0) TV_TRACE(3, g);
        for (int t = s.a; t < s.e && ok; ++t, ++g) {
          if (sh && sh_owner(t) != m) continue;  // the other M tile's tile
          const int stage = g % C::kStages;
          ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
          if (m == 0) TV_TRACE(29, g);
          if (ok && gm > 0) ok = mbar_wait(&bars.s_free[m], (gm - 1) & 1, &bars, status);
          if (!ok) break;
          fence_after();
          if (m == 0) TV_TRACE(30, g);
          const uint32_t blo = desc_lo(sK + stage * kKVTileBytes, 0);
          if (kQS && m == 0 && seg_i > 0 && t == s.a) {
            // the previous unit's S_0 products have completed (its last S_0
            // was read): copy this unit's staged Q_0 into TMEM; the S_0
            // products below follow the copies in this thread's pipe order
            ok = mbar_wait(&bars.q0s_full, (seg_i - 1) & 1, &bars, status);
            if (!ok) break;
            q_pending = false;
            const uint32_t qlo = desc_lo(sQ0S, 0);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) {
              const uint64_t d = ((uint64_t)hi << 32) | (qlo + (k / 4) * (16384 >> 4) + (k % 4) * 2);
              asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(tmem + C::kColQ0 + k * 8), "l"(d)
                           : "memory");
            }
            mma_commit(&bars.cp_done);
          }
          if (m == 0) {
            const uint32_t aQ = tmem + C::kColQ0;
            mma_ts<false>(dS, aQ, blo, hi, idS);
#pragma unroll
            for (int kk = 1; kk < kD / 16; ++kk)
              mma_ts<true>(dS, aQ + kk * 8, blo + (kk / 4) * (kKVHalfBytes >> 4) + (kk % 4) * 2, hi, idS);
          } else {
            const uint32_t alo = desc_lo(sQ1, 0);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint64_t a = ((uint64_t)hi << 32) | (alo + (kk / 4) * (16384 >> 4) + (kk % 4) * 2);
              const uint64_t b = ((uint64_t)hi << 32) | (blo + (kk / 4) * (kKVHalfBytes >> 4) + (kk % 4) * 2);
              mma_bf16(dS, a, b, idS, kk > 0);
            }
          }
          mma_commit(&bars.s_full[m]);
          if constexpr (kSkip) ++g1;
          if (m == 0) TV_TRACE(2, g);
          if (kQS && m == 0 && seg_i > 0 && t == s.a && hn) {
            // once the copies have read the staging tile, stage the next unit's Q_0
            ok = mbar_wait(&bars.cp_done, (seg_i - 1) & 1, &bars, status);
            if (!ok) break;
            load_q(sn, sQ0S, &bars.q0s_full);
          }
        }
        if (ok && kQS && m == 1 && hn) {
          // the Q_1 tile is free once this unit's last S_1 has completed
          mma_commit(&bars.q1_free);
          ok = mbar_wait(&bars.q1_free, seg_i & 1, &bars, status);
          if (ok) load_q(sn, sQ1, &bars.q1_full);
        }
        ++seg_i;
      }
      if (!ok) mma_drain(bars, m);
      // a Q load still in flight lands before the CTA exits
      if (q_pending) mbar_wait(m == 0 ? &bars.q0s_full : &bars.q1_full, (nq - 1) & 1, &bars, nullptr, false);
    }
    __syncwarp();
  } else if (warp == 6 || warp == 7) {
    // ------------------------------------------------------------ O_m += P_m V issuer
    const int m = warp - 6;
    if (lane == 0) {
      constexpr uint32_t idO = idesc_bf16(128, kD, true);
      const uint32_t dO = tmem + C::col_o(m), aP = tmem + C::col_p(m);
      uint32_t g = 0, g1 = 0;  // tiles of the ring; with kSkip, P.V products of this M tile
      uint32_t& gm = kSkip ? g1 : g;
      bool ok = true;
      Walk walk(sp);
      Segment s;
      while (ok && walk.next(p, s)) {
        const bool sh = kSkip && shared_unit(p, s);
        bool started = false;  // with kSkip: this M tile has a product in this unit
        for (int t = s.a; t < s.e && ok; ++t, ++g) {
          const int stage = g % C::kStages;
          if (sh && sh_owner(t) != m) {  // the other M tile's tile: release this share once it has landed
            ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
            if (!ok) break;
            mma_commit(&bars.kv_empty[stage]);
            continue;
          }
          ok = mbar_wait(&bars.p_full[m], gm & 1, &bars, status);
          if (ok) ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
          if (!ok) break;
          fence_after();
          const uint32_t vlo = desc_lo(sV + stage * kKVTileBytes, kKVHalfBytes);
          if (kSkip ? started : t > s.a) mma_ts<true>(dO, aP, vlo, hi, idO);
          else mma_ts<false>(dO, aP, vlo, hi, idO);
          started = true;
#pragma unroll
          for (int kk = 1; kk < kBlk / 16; ++kk) mma_ts<true>(dO, aP + kk * 8, vlo + kk * (2048 >> 4), hi, idO);
          mma_commit(&bars.o_done[m]);
          mma_commit(&bars.kv_empty[stage]);
          if constexpr (kSkip) ++g1;
          if (m == 0) TV_TRACE(4, g);
        }
      }
      if (!ok) mma_drain(bars, 2 + m);
    }
    __syncwarp();
  } else if (warp >= C::kSoftmaxWarp0 && warp < C::kSoftmaxWarp0 + 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int m = (warp - C::kSoftmaxWarp0) / 4;
    const int quarter = warp % 4;
    const int rl = quarter * 32 + lane;
    const int row = m * 128 + rl;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = lane_addr + C::col_s(m), tP = lane_addr + C::col_p(m), tO = lane_addr + C::col_o(m);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    uint32_t g = 0, g1 = 0;  // tiles of the ring; with kSkip, tiles this M tile computed
    uint32_t& gm = kSkip ? g1 : g;
    uint32_t useg = 0, shi = 0;  // with kSkip: units of the slice walked so far; shared units
    bool ok = true;
    Walk walk(sp);
    Segment s;
#ifdef TV_TC_TRACE
    int n_segs_traced = 0;
#endif
    // Row identity of this thread inside a unit, and the unit's Q row and
    // ancestor row (the producer warps have already pulled both into L2).
    struct RowOf {
      bool valid;
      int node;
      int64_t orow;
    };
    auto row_of = [&](const Segment& sg) {
      RowOf r;
      const int unit_row = sg.rg * p.RPG + ((kSkip && shared_unit(p, sg)) ? rl : row);
      r.valid = unit_row < p.R;
      r.node = r.valid ? unit_row / p.G : 0;
      r.orow = ((int64_t)sg.b * p.N + r.node) * p.Hq + sg.kvh * p.G + unit_row % p.G;
      return r;
    };
    uint4 qreg[16];
    uint64_t mrow_next = 1ull;
    auto fetch_q = [&](const Segment& sg) {
      const RowOf r = row_of(sg);
      const uint4* src = reinterpret_cast<const uint4*>(q + r.orow * kD);
#pragma unroll
      for (int c = 0; c < 16; ++c) qreg[c] = r.valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      mrow_next = r.valid ? __ldg(reinterpret_cast<const unsigned long long*>(p.mask) +
                                  (int64_t)sg.b * p.mask_bstride + r.node)
                          : 1ull;
      if constexpr (kRope) rope_row(qreg, p, r.valid ? row_pos(mrow_next, sg.L) : -1, status, lane);
    };
    // Q row into its operand slot: M tile 0 into TMEM, M tile 1 into the
    // swizzled shared tile; then tell the S issuers.
    auto place_q = [&]() {
      if (m == 0) {
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            r[4 * j] = qreg[c * 8 + j].x; r[4 * j + 1] = qreg[c * 8 + j].y;
            r[4 * j + 2] = qreg[c * 8 + j].z; r[4 * j + 3] = qreg[c * 8 + j].w;
          }
          tmem_st32(lane_addr + C::kColQ0 + c * 32, r);
        }
        tmem_st_wait();
        fence_before();
      } else {
        uint8_t* rowp = gQ1 + (rl / 8) * 1024 + (rl % 8) * 128;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(rowp + (c / 8) * 16384 + (((c % 8) ^ (rl % 8)) * 16)) = qreg[c];
        fence_proxy_async();
      }
      mbar_arrive(&bars.q_full);
    };
    bool have = walk.next(p, s);
    if (have) {
      fetch_q(s);
      place_q();
    }
    while (ok && have) {
#ifdef TV_TC_TRACE
      if (threadIdx.x == C::kSoftmaxWarp0 * 32 && blockIdx.x < 1024) {
        if (n_segs_traced == 0) tv::trace::g_cta_time[blockIdx.x][3] = s.u;
        tv::trace::g_cta_time[blockIdx.x][2] = ++n_segs_traced;
      }
#endif
      const bool sh = kSkip && shared_unit(p, s);
      const RowOf rid = row_of(s);
      const bool valid_row = rid.valid;
      const int64_t orow = rid.orow;
      const uint64_t mrow = mrow_next;
      float m_run = -INFINITY, l = 0.f;
      const int n_seg = s.e - s.a;
      int kk = 0;  // with kSkip: tiles this M tile computed in this unit
      for (int k = 0; k < n_seg; ++k, ++g) {
        const int t = s.a + k;
        if (sh && sh_owner(t) != m) continue;  // the other M tile's tile
        ok = mbar_wait_warp(&bars.s_full[m], gm & 1, &bars, status);
        if (!ok) break;
        fence_after();
        if (rl == 0) TV_TRACE(6 + 4 * m, g);
        float sv[kBlk];
        {
          uint32_t r[32];
          tmem_ld32(tS, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(r[c]);
          tmem_ld32(tS + 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[32 + c] = __uint_as_float(r[c]);
        }
        fence_before();
        mbar_arrive(&bars.s_free[m]);  // the next S_m may be computed now
        if (rl == 0) TV_TRACE(7 + 4 * m, g);
        if (t == s.n - 1) {
#pragma unroll
          for (int c = 0; c < kBlk; ++c)
            if (!(c < p.N && ((mrow >> c) & 1ull))) sv[c] = -INFINITY;
        } else {
          const int lim = s.L - t * kBlk;
          if (lim < kBlk) {
#pragma unroll
            for (int c = 0; c < kBlk; ++c)
              if (c >= lim) sv[c] = -INFINITY;
          }
        }
        float mx = row_max64(sv);
        mx *= p.scale_log2;
        const float m_new = fmaxf(m_run, mx);
        const bool grow = m_new > m_run + kRescaleThreshold;
        const float m_use = grow ? m_new : ((m_run == -INFINITY) ? 0.f : m_run);
        const uint64_t sc2 = pack_f32x2(p.scale_log2, p.scale_log2), negm2 = pack_f32x2(-m_use, -m_use);
        uint64_t acc0 = 0, acc1 = 0;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < kBlk / 2; ++c) {
          float e0, e1;
          exp2_pair(sv[2 * c], sv[2 * c + 1], sc2, negm2, e0, e1);
          if (c & 1) acc1 = add_f32x2(acc1, pack_f32x2(e0, e1)); else acc0 = add_f32x2(acc0, pack_f32x2(e0, e1));
          pk[c] = pack_bf16(e0, e1);
        }
        const float sum0 = sum_f32x2(add_f32x2(acc0, acc1)), sum1 = 0.f;
        if ((kSkip ? kk : k) > 0) {
          // P_m(g-1) consumed and O_m holds tiles < g
          ok = mbar_wait_warp(&bars.o_done[m], (gm - 1) & 1, &bars, status);
          if (!ok) break;
          fence_after();
          if (__any_sync(0xffffffffu, grow)) {
            const float alpha = grow ? exp2f(m_run - m_new) : 1.f;
#pragma unroll 1
            for (int c = 0; c < kD; c += 32) {
              uint32_t r[32];
              tmem_ld32(tO + c, r);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
              tmem_st32(tO + c, r);
            }
          }
        }
        if (grow) {
          l *= exp2f(m_run - m_new);
          m_run = m_new;
        }
        l += sum0 + sum1;
        tmem_st32(tP, pk);
        tmem_st_wait();
        fence_before();
        mbar_arrive(&bars.p_full[m]);
        if (rl == 0) TV_TRACE(9 + 4 * m, g);
        if constexpr (kSkip) {
          ++kk;
          ++g1;
        }
      }
      if (!ok) break;
      if (sh) {  // this unit's query phase completes before the next unit's arrivals go out
        ok = mbar_wait_warp(&bars.q_full, useg & 1, &bars, status);
        if (!ok) break;
      }
      // The next unit's Q goes in first (its S_m MMAs then run during this
      // epilogue): this unit's S_m MMAs have all completed -- the softmax has
      // read every S_m tile -- and its rows are warm in L2.
      Segment s_next;
      const bool have_next = walk.next(p, s_next);
      if (have_next) {
        if constexpr (kQS) {
          // the S issuers bring the next unit's Q in; only its ancestor row here
          const RowOf r = row_of(s_next);
          mrow_next = r.valid ? __ldg(reinterpret_cast<const unsigned long long*>(p.mask) +
                                      (int64_t)s_next.b * p.mask_bstride + r.node)
                              : 1ull;
        } else {
          fetch_q(s_next);
          place_q();
        }
      }
      if (m == 0 && rl == 0) TV_TRACE(15, g - 1);
      if (!sh || kk > 0) {
        ok = mbar_wait_warp(&bars.o_done[m], (gm - 1) & 1, &bars, status);
        if (!ok) break;
        fence_after();
      }
      if constexpr (kSkip) {
        if (sh) {
          if (m == 1) {  // post this M tile's (max, sum); its accumulator stays until M tile 0 has read it
            s_sh[rl] = m_run;
            s_sh[128 + rl] = kk > 0 ? l : 0.f;
            fence_before();
            mbar_arrive(&bars.sh_stat);
            ok = mbar_wait_warp(&bars.sh_read, shi & 1, &bars, status);
            if (!ok) break;
            ++shi;
            ++useg;
            s = s_next;
            have = have_next;
            continue;
          }
          ok = mbar_wait_warp(&bars.sh_stat, shi & 1, &bars, status);
          if (!ok) break;
          fence_after();
          ++shi;
          // O = O_0 2^(m_0 - m) + O_1 2^(m_1 - m), l likewise, m = max (a part
          // without keys -- no tile, or every key masked -- adds nothing)
          const float m1v = s_sh[rl], l1v = s_sh[128 + rl];
          const bool h0 = kk > 0 && l > 0.f, h1 = l1v > 0.f;
          const float mm = h0 ? (h1 ? fmaxf(m_run, m1v) : m_run) : (h1 ? m1v : m_run);
          const float a0 = h0 ? exp2f(m_run - mm) : 0.f, a1 = h1 ? exp2f(m1v - mm) : 0.f;
          const uint32_t tO1 = lane_addr + C::col_o(1);
#pragma unroll 1
          for (int c = 0; c < kD; c += 32) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tO + c, r0);
            tmem_ld32(tO1 + c, r1);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              r0[j] = __float_as_uint((h0 ? __uint_as_float(r0[j]) * a0 : 0.f) +
                                      (h1 ? __uint_as_float(r1[j]) * a1 : 0.f));
            tmem_st32(tO + c, r0);
          }
          tmem_st_wait();
          l = (h0 ? l * a0 : 0.f) + (h1 ? l1v * a1 : 0.f);
          m_run = mm;
          fence_before();
          mbar_arrive(&bars.sh_read);  // M tile 1's accumulator is free again
        }
      }
      // After the slice's last tile the K/V ring goes idle once both M tiles'
      // last P.V products have completed (the last stage's empty barrier
      // counts one commit from each O issuer, and each commit covers that
      // issuer's earlier products; the S products completed before their
      // softmax) and the tail warps have read their last tiles: with four
      // tail warps the two pairs take tiles in turn, so the other pair's last
      // tile is the one before, whose stage may still be read after the last
      // tile's is released (no stage is loaded again, so each of these
      // barriers has completed at most the phase waited for).  A direct
      // merge with one other piece then stages that piece's rows through the
      // ring, M tile m in its own 64 KB (the K half of the ring for m = 0,
      // the V half for 1).
      uint8_t* stage = nullptr;
      if (!have_next) {
        constexpr int kLastTiles = kTailW ? kTailW / kTailSplit : 1;  // tail warp pairs taking tiles in turn
        for (int j = 1; j <= kLastTiles && j <= (int)g && ok; ++j)
          ok = mbar_wait_warp(&bars.kv_empty[(g - j) % C::kStages], ((g - j) / C::kStages) & 1, &bars, status);
        if (!ok) break;
        fence_after();
        stage = smem_raw + (base - raw) + (m == 0 ? C::kOffK : C::kOffV);
      }
      if (m == 0 && rl == 0) TV_TRACE(14, g - 1);
      finish_row<2, kQS>(p, sp, s, row, valid_row, orow, tO, m_run, l, stage, &maps.pm,
                         &bars.merge_full[m][rl >> 5]);
      fence_before();
      if (m == 0 && rl == 0) TV_TRACE(5, g - 1);
      if constexpr (kSkip) ++useg;
      s = s_next;
      have = have_next;
    }
  }

  TV_TRACE_CTA(1);
  fence_before();
  __syncthreads();
  if (warp == C::kAllocWarp) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2), up to 256 rows
//
// Two SMs share every unit of up to 256 rows: the rows are split 128 / 128
// between the pair's CTAs (each keeps its rows' S, P, Q and O in its own
// TMEM), and every MMA is one tcgen05.mma.cta_group::2 with M = 256 issued
// by the even CTA.  The B operand of an MMA is split between the two CTAs'
// shared memory along N, so each SM loads half of every K/V tile from HBM:
//   S = Q K^T   (N = 64 keys):       this CTA holds keys 32r .. 32r + 31;
//   O += P V    (N = 128 head dims): this CTA holds head dims 64r .. 64r + 63.
// Per row an SM then has 512 TMEM columns for 128 rows instead of 256, which
// holds two sets of S, P and O: two softmax warpgroups take the even and the
// odd key tiles of a unit, each with its own running max, sum and O, merged
// at the unit's end.  The S product of the next tile is computed while the
// softmax of the current one runs, and each warpgroup has two tiles' time
// for its softmax.  TMEM columns: S_A 0-63, S_B 64-127, P_A 128-159,
// P_B 160-191, Q 192-255 (the A operand of S, "TS" form), O_A 256-383,
// O_B 384-511.
//
// Barriers: each CTA's loads complete on its own kv_full barrier; the odd
// CTA forwards that completion to the even CTA's peer_full barrier, so the
// issuing thread knows both halves of a tile have landed.  MMA completions
// are committed to both CTAs' barriers at once (multicast); the softmax
// warps of both CTAs arrive on the even CTA's s_free / p_full / q_full
// barriers (one arrival per warp, through the cluster's shared memory).
struct DuoCfg {
  static constexpr int kStages = 8;
  static constexpr int kKHalfBytes = 32 * 128;  // 32 keys x 64 head dims
  static constexpr int kKBytes = 2 * kKHalfBytes;
  static constexpr int kVBytes = kBlk * 128;     // 64 keys x 64 head dims
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  static constexpr int kBytes = kOffV + kStages * kVBytes;
  static constexpr int kSmem = kBytes + 1024;
  // warps 0-3: TMA (boxes dealt round-robin: one warp issues a box only
  // about every 150 cycles and then stalls); warps 4 / 5: S_A / S_B issuers
  // (even CTA), warp 4 of the odd CTA forwards its loads' completion; warp
  // 6: P V issuer (even CTA) and TMEM allocation; warp 7 idle; warps 8-11 /
  // 12-15: softmax warpgroups A (even tiles) / B (odd tiles).
  static constexpr int kThreads = 32 * 16;
  static constexpr int kProducers = 4;
  static constexpr int kAllocWarp = 6;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t col_s(int x) { return x * 64; }
  static constexpr uint32_t col_p(int x) { return 128 + x * 32; }
  static constexpr uint32_t kColQ = 192;
  static constexpr uint32_t col_o(int x) { return 256 + x * 128; }
  static constexpr int kSoftmaxWarp0 = 8;
};
static_assert(DuoCfg::kStages * DuoCfg::kKBytes >= 128 * kD * 4, "the K ring holds one M tile's staged rows");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Arrival on the even CTA's copy of a barrier (remote for the odd CTA).  The
// remote arrival is relaxed: a release at cluster scope stalls the arriving
// warp for about a thousand cycles, and the operations it would order have
// completed already (tcgen05.wait::ld / ::st precede every such arrival, and
// the MMAs that consume the data are issued after it is observed).
__device__ __forceinline__ void mbar_arrive_leader(uint64_t* bar, uint32_t rank) {
  if (rank == 0) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
  } else {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(smem_u32(bar)));
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
  }
}

__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait for barriers that other CTAs of the cluster arrive on.
__device__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, Bars* bars, int32_t* status) {
  if (mbar_test_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_cluster(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*(volatile int*)&bars->abort) return false;
      if (globaltimer() - t0 > timeout_ns()) {
        *(volatile int*)&bars->abort = 1;
        if (status) atomicOr(status, TV_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void mma2(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}

// Completion of the issuing thread's earlier MMAs, signalled on the barrier
// at this offset in both CTAs of the pair.
__device__ __forceinline__ void mma_commit2(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// mma_drain for the pair's MMA issuer (the commit arrives on both CTAs'
// copies of the barrier; the issuer waits on its own).
__device__ __forceinline__ void mma_drain2(Bars& bars, int i) {
  mma_commit2(&bars.drain[i]);
  mbar_wait(&bars.drain[i], 0, &bars, nullptr, false);
}

struct DuoMaps {
  CUtensorMap kc, vc, kt, vt;  // K boxes of 32 (or block_size) rows, V boxes of 64 (or block_size) rows
};

// TMA producer of one CTA of the pair: this CTA's 32 keys (both head-dim
// halves) and this CTA's head-dim half of all 64 keys of every tile.  The
// producer shares its sub-partition with busy softmax warps, so the tile loop
// is kept short: each lane's box (which half, which sub-block, its offset in
// the tile and in the stage) is fixed for the whole slice, and block
// arithmetic uses shifts when the block size is a power of two.
template <int kStages, int kProducers>
__device__ __forceinline__ void duo_producer(const AttnParams& p, const SlicePlan& sp, const DuoMaps& maps, Bars& bars,
                                             uint32_t sK, uint32_t sV, uint32_t rank, int lane, int32_t* status,
                                             int prod) {
  using C = DuoCfg;
  const int bs = p.block_size;
  const int lbs = (bs & (bs - 1)) == 0 ? __ffs(bs) - 1 : -1;  // log2(bs) for a power of two
  const int brk = bs < 32 ? bs : 32, nk = 32 / brk;        // K boxes per head-dim half
  const int brv = bs < kBlk ? bs : kBlk, nv = kBlk / brv;  // V boxes
  const int64_t rows_total = (int64_t)p.num_blocks * p.Hkv * bs;
  const uint64_t pol = policy_evict_first();
  // this lane's box j (j < 2 nk: K, half j / nk, sub-box j % nk; then V
  // sub-box j - 2 nk): dealt round-robin over the producer warps
  const int j = lane * kProducers + prod;
  const bool is_k = j < 2 * nk;
  const bool has_box = j < 2 * nk + nv;
  const int sub = is_k ? j % nk : j - 2 * nk;
  const int h = is_k ? j / nk : (int)rank;
  const int br = is_k ? brk : brv;
  const int off = is_k ? (int)rank * 32 + sub * brk : sub * brv;  // key offset of the box in the tile
  const uint32_t dst_off = is_k ? (uint32_t)(h * C::kKHalfBytes + sub * brk * 128) : (uint32_t)(sub * brv * 128);
  const uint32_t dst_base = is_k ? sK : sV;
  const uint32_t dst_stride = is_k ? C::kKBytes : C::kVBytes;
  const CUtensorMap* map = is_k ? &maps.kc : &maps.vc;
  auto div_bs = [&](int x) { return lbs >= 0 ? x >> lbs : x / bs; };
  uint32_t g = 0;
  bool ok = true;
  Walk walk(sp);
  Segment s;
  while (ok && walk.next(p, s)) {
    {
      const int rows = p.R - s.rg * p.RPG < p.RPG ? p.R - s.rg * p.RPG : p.RPG;
      const char* qb = static_cast<const char*>(p.q);
      for (int r = lane * kProducers + prod; r < 128; r += 32 * kProducers) {
        const int ur = s.rg * p.RPG + (int)rank * 128 + r;
        if (ur - s.rg * p.RPG >= rows) break;
        const int64_t orow = ((int64_t)s.b * p.N + ur / p.G) * p.Hq + s.kvh * p.G + ur % p.G;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + orow * (kD * 2)));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + orow * (kD * 2) + 128));
      }
      if (lane == 0 && prod == 0)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.mask + (int64_t)s.b * p.mask_bstride));
    }
    const int nb = div_bs(s.L + bs - 1);
    const int32_t* trow = p.block_table + (int64_t)s.b * p.max_blocks;
    const int64_t head_row = (int64_t)s.kvh * bs;  // row of (block 0, this KV head) over Hkv * bs rows per block
    const int last_pos = s.L > 0 ? (s.L - 1) / br * br : 0;  // ragged tail: finite rows, weight 0
    int w0 = div_bs(s.a * kBlk);
    int32_t cur = (w0 + lane < nb) ? __ldg(trow + w0 + lane) : 0;
    int32_t nxt = (w0 + 32 + lane < nb) ? __ldg(trow + w0 + 32 + lane) : 0;
    for (int t = s.a; t < s.e && ok; ++t, ++g) {
      const int stage = g % kStages;
      const uint32_t use = g / kStages;
      const bool tree_tile = (t == s.n - 1);
      if (!tree_tile && div_bs(t * kBlk) >= w0 + 32) {
        w0 += 32;
        cur = nxt;
        nxt = (w0 + 32 + lane < nb) ? __ldg(trow + w0 + 32 + lane) : 0;
      }
      int pos = t * kBlk + off;
      if (pos >= s.L) pos = last_pos;
      const int bi = div_bs(pos);
      const int rel = bi - w0;
      const int32_t from_cur = __shfl_sync(0xffffffffu, cur, rel & 31);
      const int32_t from_nxt = __shfl_sync(0xffffffffu, nxt, rel & 31);
      const int64_t blk = rel < 32 ? from_cur : from_nxt;
      if (use > 0) ok = mbar_wait_warp(&bars.kv_empty[stage], (use - 1) & 1, &bars, status);
      if (!ok) break;
      if (lane == 0 && prod == 0) mbar_expect_tx(&bars.kv_full[stage], C::kKBytes + C::kVBytes);
      __syncwarp();
      if (tree_tile) {
        const uint32_t dk = sK + stage * C::kKBytes, dv = sV + stage * C::kVBytes;
        if (j < 2)
          tma_4d(j == 0 ? dk : dk + C::kKHalfBytes, &maps.kt, 64 * j, s.kvh, (int)rank * 32, s.b, &bars.kv_full[stage]);
        else if (j == 2)
          tma_4d(dv, &maps.vt, 64 * (int)rank, s.kvh, 0, s.b, &bars.kv_full[stage]);
      } else if (has_box) {
        int64_t y = blk * p.Hkv * bs + head_row + (pos - bi * bs);
        if (blk < 0 || blk >= p.num_blocks) {
          y = rows_total;
          if (status) atomicOr(status, TV_DEV_BAD_BLOCK);
        }
        tma_2d_stream(dst_base + stage * dst_stride + dst_off, map, h * 64, (int)y, &bars.kv_full[stage], pol);
      }
      __syncwarp();
    }
  }
  // drain: every load this warp issued has landed before it exits
  if (lane == 0) {
    const uint32_t first = g > (uint32_t)kStages ? g - kStages : 0;
    for (uint32_t i = first; i < g; ++i)
      mbar_wait(&bars.kv_full[i % kStages], (i / kStages) & 1, &bars, nullptr, false);
  }
}

template <bool kRope>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DuoCfg::kThreads, 1)
    attn_tc_duo_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ DuoMaps maps, int32_t* status) {
  using C = DuoCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ float s_sh[256];  // warpgroup B's running max and sum per row at a unit's end
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sK = base + C::kOffK, sV = base + C::kOffV;
  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __shared__ SlicePlan sp;
  if (warp == 0) plan_slice(p, lane, sp, blockIdx.x / 2);
  __syncthreads();
  if (sp.t0 >= sp.t1) return;  // both CTAs of the pair have the same (empty) slice
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.peer_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.s_free[x], 8);
      mbar_init(&bars.p_full[x], 8);
      mbar_init(&bars.o_done[x], 1);
    }
    mbar_init(&bars.q_full, 8);
    mbar_init(&bars.sh_stat, 4);
    mbar_init(&bars.sh_read, 4);
    for (int i = 0; i < 4; ++i) mbar_init(&bars.drain[i], 1);
    bars.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == C::kAllocWarp) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  fence_before();
  // both CTAs' barriers are initialised (and their TMEM allocated) before any
  // remote arrival or multicast commit
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  fence_after();
  const uint32_t tmem = bars.tmem_base;
  constexpr uint32_t hi = desc_hi(1024);

  if (warp < C::kProducers) {
    duo_producer<C::kStages, C::kProducers>(p, sp, maps, bars, sK, sV, rank, lane, status, warp);
  } else if (warp == 4 && rank == 1) {
    if (lane == 0) {
      // forwarder: this CTA's half of tile g has landed -> the even CTA's peer_full
      uint32_t g = 0;
      bool ok = true;
      Walk walk(sp);
      Segment s;
      while (ok && walk.next(p, s)) {
        for (int t = s.a; t < s.e && ok; ++t, ++g) {
          const int stage = g % C::kStages;
          ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
          if (ok) mbar_arrive_leader(&bars.peer_full[stage], 1);
        }
      }
    }
    __syncwarp();
  } else if ((warp == 4 || warp == 5) && rank == 0) {
    if (lane == 0) {
      // S_X = Q K^T for the tiles of warpgroup X (warp 4: the even tiles of a
      // unit, warp 5: the odd ones)
      const int x = warp - 4;
      constexpr uint32_t idS = idesc_bf16(256, kBlk, false);
      uint32_t g = 0, uses = 0;
      int seg_i = 0;
      bool ok = true;
      Walk walk(sp);
      Segment s;
      while (ok && walk.next(p, s)) {
        ok = mbar_wait_cl(&bars.q_full, seg_i & 1, &bars, status);
        if (!ok) break;
        fence_after();
        for (int t = s.a; t < s.e && ok; ++t, ++g) {
          if (((t - s.a) & 1) != x) continue;
          const int stage = g % C::kStages;
          ok = mbar_wait(&bars.kv_full[stage], (g / C::kStages) & 1, &bars, status);
          if (ok) ok = mbar_wait_cl(&bars.peer_full[stage], (g / C::kStages) & 1, &bars, status);
          if (ok && uses > 0) ok = mbar_wait_cl(&bars.s_free[x], (uses - 1) & 1, &bars, status);
          if (!ok) break;
          fence_after();
          const uint32_t blo = desc_lo(sK + stage * C::kKBytes, 0);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t b = ((uint64_t)hi << 32) | (blo + (kk / 4) * (C::kKHalfBytes >> 4) + (kk % 4) * 2);
            mma2(tmem + C::col_s(x), tmem + C::kColQ + kk * 8, b, idS, kk > 0);
          }
          mma_commit2(&bars.s_full[x]);
          ++uses;
        }
        ++seg_i;
      }
      if (!ok) mma_drain2(bars, x);
    }
    __syncwarp();
  } else if (warp == 6) {
    if (lane == 0 && rank == 0) {
      // O_X += P_X V
      constexpr uint32_t idO = idesc_bf16(256, kD, true);
      uint32_t g = 0, uses[2] = {0, 0};
      bool ok = true;
      Walk walk(sp);
      Segment s;
      while (ok && walk.next(p, s)) {
        for (int t = s.a; t < s.e && ok; ++t, ++g) {
          const int k = t - s.a, x = k & 1;
          const int stage = g % C::kStages;
          ok = mbar_wait_cl(&bars.p_full[x], uses[x] & 1, &bars, status);
          if (!ok) break;
          fence_after();
          const uint32_t vlo = desc_lo(sV + stage * C::kVBytes, 0);
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk)
            mma2(tmem + C::col_o(x), tmem + C::col_p(x) + kk * 8, ((uint64_t)hi << 32) | (vlo + kk * (2048 >> 4)), idO,
                 k >= 2 || kk > 0);
          mma_commit2(&bars.o_done[x]);
          mma_commit2(&bars.kv_empty[stage]);
          ++uses[x];
        }
      }
      if (!ok) mma_drain2(bars, 2);
    }
    __syncwarp();
  } else if (warp >= C::kSoftmaxWarp0 && warp < C::kSoftmaxWarp0 + 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int x = (warp - C::kSoftmaxWarp0) / 4;  // 0: warpgroup A (even tiles), 1: B (odd tiles)
    const int quarter = warp % 4;
    const int rl = quarter * 32 + lane;
    const int row = (int)rank * 128 + rl;  // row within the unit
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = lane_addr + C::col_s(x), tP = lane_addr + C::col_p(x), tO = lane_addr + C::col_o(x);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    uint32_t g = 0, uses = 0, useg = 0;
    bool ok = true;
    Walk walk(sp);
    Segment s;
    struct RowOf {
      bool valid;
      int node;
      int64_t orow;
    };
    auto row_of = [&](const Segment& sg) {
      RowOf r;
      const int unit_row = sg.rg * p.RPG + row;
      r.valid = unit_row < p.R;
      r.node = r.valid ? unit_row / p.G : 0;
      r.orow = ((int64_t)sg.b * p.N + r.node) * p.Hq + sg.kvh * p.G + unit_row % p.G;
      return r;
    };
    // Q rows of a unit into TMEM (warpgroup A), then the even CTA's q_full
    auto place_q = [&](const Segment& sg) {
      const RowOf r = row_of(sg);
      const uint4* src = reinterpret_cast<const uint4*>(q + r.orow * kD);
      uint4 qr[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) qr[c] = r.valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      if constexpr (kRope) {
        const uint64_t mrow = r.valid ? __ldg(reinterpret_cast<const unsigned long long*>(p.mask) +
                                              (int64_t)sg.b * p.mask_bstride + r.node)
                                      : 1ull;
        rope_row(qr, p, r.valid ? row_pos(mrow, sg.L) : -1, status, lane);
      }
#pragma unroll
      for (int c = 0; c < kD / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[4 * j] = qr[c * 8 + j].x; v[4 * j + 1] = qr[c * 8 + j].y;
          v[4 * j + 2] = qr[c * 8 + j].z; v[4 * j + 3] = qr[c * 8 + j].w;
        }
        tmem_st32(lane_addr + C::kColQ + c * 32, v);
      }
      tmem_st_wait();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_leader(&bars.q_full, rank);
    };
    bool have = walk.next(p, s);
    if (have && x == 0) place_q(s);
    while (ok && have) {
      const RowOf rid = row_of(s);
      const uint64_t mrow = rid.valid ? __ldg(reinterpret_cast<const unsigned long long*>(p.mask) +
                                              (int64_t)s.b * p.mask_bstride + rid.node)
                                      : 1ull;
      float m_run = -INFINITY, l = 0.f;
      const int n_seg = s.e - s.a;
      int mine = 0;  // tiles of this unit this warpgroup computed
      for (int k = x; k < n_seg; k += 2) {
        const int t = s.a + k;
        ok = mbar_wait_warp(&bars.s_full[x], uses & 1, &bars, status);
        if (!ok) break;
        fence_after();
        float sv[kBlk];
        {
          uint32_t r[32];
          tmem_ld32(tS, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(r[c]);
          tmem_ld32(tS + 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[32 + c] = __uint_as_float(r[c]);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_leader(&bars.s_free[x], rank);  // the next S_X may be computed now
        if (t == s.n - 1) {
#pragma unroll
          for (int c = 0; c < kBlk; ++c)
            if (!(c < p.N && ((mrow >> c) & 1ull))) sv[c] = -INFINITY;
        } else {
          const int lim = s.L - t * kBlk;
          if (lim < kBlk) {
#pragma unroll
            for (int c = 0; c < kBlk; ++c)
              if (c >= lim) sv[c] = -INFINITY;
          }
        }
        float mx = row_max64(sv);
        mx *= p.scale_log2;
        const float m_new = fmaxf(m_run, mx);
        const bool grow = m_new > m_run + kRescaleThreshold;
        const float m_use = grow ? m_new : ((m_run == -INFINITY) ? 0.f : m_run);
        const uint64_t sc2 = pack_f32x2(p.scale_log2, p.scale_log2), negm2 = pack_f32x2(-m_use, -m_use);
        uint64_t acc0 = 0, acc1 = 0;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < kBlk / 2; ++c) {
          float e0, e1;
          exp2_pair(sv[2 * c], sv[2 * c + 1], sc2, negm2, e0, e1);
          if (c & 1) acc1 = add_f32x2(acc1, pack_f32x2(e0, e1)); else acc0 = add_f32x2(acc0, pack_f32x2(e0, e1));
          pk[c] = pack_bf16(e0, e1);
        }
        const float sum = sum_f32x2(add_f32x2(acc0, acc1));
        if (mine > 0) {
          // P_X of this warpgroup's previous tile consumed; O_X holds it
          ok = mbar_wait_warp(&bars.o_done[x], (uses - 1) & 1, &bars, status);
          if (!ok) break;
          fence_after();
          if (__any_sync(0xffffffffu, grow)) {
            const float alpha = grow ? exp2f(m_run - m_new) : 1.f;
#pragma unroll 1
            for (int c = 0; c < kD; c += 32) {
              uint32_t r[32];
              tmem_ld32(tO + c, r);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
              tmem_st32(tO + c, r);
            }
          }
        }
        if (grow) {
          l *= exp2f(m_run - m_new);
          m_run = m_new;
        }
        l += sum;
        tmem_st32(tP, pk);
        tmem_st_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_leader(&bars.p_full[x], rank);
        ++uses;
        ++mine;
      }
      if (!ok) break;
      g += n_seg;
      Segment s_next;
      const bool have_next = walk.next(p, s_next);
      if (x == 1) {
        // warpgroup B: post (max, sum) once its last P V has completed; its
        // accumulator stays until warpgroup A has merged it
        if (mine > 0) {
          ok = mbar_wait_warp(&bars.o_done[1], (uses - 1) & 1, &bars, status);
          if (!ok) break;
        }
        s_sh[rl] = m_run;
        s_sh[128 + rl] = mine > 0 ? l : 0.f;
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.sh_stat);
        ok = mbar_wait_warp(&bars.sh_read, useg & 1, &bars, status);
        if (!ok) break;
      } else {
        ok = mbar_wait_warp(&bars.o_done[0], (uses - 1) & 1, &bars, status);
        if (ok) ok = mbar_wait_warp(&bars.sh_stat, useg & 1, &bars, status);
        if (!ok) break;
        fence_after();
        // every S product of this unit has been read (ours, and B's before
        // it posted): the next unit's Q goes in, so its S products run
        // during this epilogue
        if (have_next) place_q(s_next);
        // O = O_A 2^(m_A - m) + O_B 2^(m_B - m), l likewise (a part without
        // keys adds nothing)
        const float m1v = s_sh[rl], l1v = s_sh[128 + rl];
        const bool h0 = l > 0.f, h1 = l1v > 0.f;
        if (h1) {
          const float mm = h0 ? fmaxf(m_run, m1v) : m1v;
          const float a0 = h0 ? exp2f(m_run - mm) : 0.f, a1 = exp2f(m1v - mm);
          const uint32_t tO1 = lane_addr + C::col_o(1);
#pragma unroll 1
          for (int c = 0; c < kD; c += 32) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tO + c, r0);
            tmem_ld32(tO1 + c, r1);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              r0[j] = __float_as_uint((h0 ? __uint_as_float(r0[j]) * a0 : 0.f) + __uint_as_float(r1[j]) * a1);
            tmem_st32(tO + c, r0);
          }
          tmem_st_wait();
          l = (h0 ? l * a0 : 0.f) + l1v * a1;
          m_run = mm;
        } else {
          // B had no key: its columns are not read (warp-uniform skip of the loads only)
          __syncwarp();
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.sh_read);  // O_B may be overwritten now
        // after the slice's last tile the ring goes idle once the last P V
        // product has completed: a direct merge stages through the K ring
        uint8_t* stage = nullptr;
        if (!have_next) {
          ok = mbar_wait_warp(&bars.kv_empty[(g - 1) % C::kStages], ((g - 1) / C::kStages) & 1, &bars, status);
          if (!ok) break;
          fence_after();
          stage = smem_raw + (base - raw) + C::kOffK;
        }
        finish_row<2>(p, sp, s, row, rid.valid, rid.orow, tO, m_run, l, stage);
        fence_before();
      }
      ++useg;
      s = s_next;
      have = have_next;
    }
  }

  fence_before();
  // no CTA of the pair leaves (or frees TMEM) while the other's MMAs may read it
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp == C::kAllocWarp) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encoder(EncodeTiled* fn) {
  static std::once_flag once;
  static EncodeTiled cached = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiled>(f);
  });
  if (!cached) return fail(TV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorName(err));
  *fn = cached;
  return TV_OK;
}

int encode(EncodeTiled fn, CUtensorMap* map, const void* ptr, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box, const char* what,
           CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, type, rank, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return TV_OK;
}

template <int M, bool kRope>
int launch_m(const AttnParams& p, const TcMaps& maps, int32_t* status, cudaStream_t stream) {
  using C = Cfg<M>;
  cudaError_t e =
      cudaFuncSetAttribute(attn_tc_kernel<M, kRope>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_tc_kernel)");
  attn_tc_kernel<M, kRope><<<p.P, C::kThreads, C::kSmem, stream>>>(p, maps, status);
  TV_LAUNCH_CHECK("attn_tc_kernel");
  return TV_OK;
}

template <bool kRope, bool kSkip, int kTailW, bool kStagedQ = false>
int launch_pair(const AttnParams& p, const TcMaps& maps, int32_t* status, cudaStream_t stream) {
  constexpr int smem = PairCfgT<kTailW, kStagedQ && !kRope && !kSkip && kTailW == 0>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_pair_kernel<kRope, kSkip, kTailW, kStagedQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_tc_pair_kernel)");
  attn_tc_pair_kernel<kRope, kSkip, kTailW, kStagedQ><<<p.P, PairCfg::kThreads, smem, stream>>>(p, maps, status);
  TV_LAUNCH_CHECK("attn_tc_pair_kernel");
  return TV_OK;
}

template <bool kRope>
int launch_duo(const AttnParams& p, const DuoMaps& maps, int32_t* status, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_tc_duo_kernel<kRope>, cudaFuncAttributeMaxDynamicSharedMemorySize, DuoCfg::kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_tc_duo_kernel)");
  attn_tc_duo_kernel<kRope><<<2 * p.P, DuoCfg::kThreads, DuoCfg::kSmem, stream>>>(p, maps, status);
  TV_LAUNCH_CHECK("attn_tc_duo_kernel");
  return TV_OK;
}

}  // namespace

int tc_duo_pairs(const DeviceInfo& dev) {
  // CTA pairs resident at once (one per SM pair the GPCs can place), cached per device
  static std::mutex mu;
  static int cached[64] = {};
  if (dev.device < 0 || dev.device >= 64) return dev.sm_count / 2;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev.device]) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(DuoCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = DuoCfg::kSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(attn_tc_duo_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DuoCfg::kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, attn_tc_duo_kernel<false>, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = dev.sm_count / 2;
    }
    cached[dev.device] = n;
  }
  return cached[dev.device];
}

const char* tc_unsupported_reason(const DeviceInfo& dev, int dtype, int head_dim, int rows, int G, int block_size,
                                  bool rope) {
  if (rope && G != 4 && G != 8 && G != 16) return "Q rotated while loading needs Hq/Hkv in {4, 8, 16}";
  if (dev.cc_major != 10) return "device is not sm_10x";
  if (dtype != TV_BF16) return "dtype is not bf16";
  if (head_dim != kD) return "head_dim is not 128";
  if (rows > 2 * kTcMaxRows) return "(Hq/Hkv)*N exceeds 512";
  if (G < 1 || 128 % G) return "Hq/Hkv does not divide 128";
  if (block_size % 16 || !(kBlk % block_size == 0 || block_size % kBlk == 0))
    return "block_size is not a multiple of 16 that divides or is divisible by 64";
  // dynamic ring + barriers + the shared-unit statistics + the slice plan
  if (dev.max_smem_optin < (size_t)PairCfgT<4>::kSmem + sizeof(Bars) + 256 * sizeof(float) + 64)
    return "not enough opt-in shared memory";
  return nullptr;
}

bool tc_supported(const DeviceInfo& dev, int dtype, int head_dim, int rows, int G, int block_size, bool rope) {
  return tc_unsupported_reason(dev, dtype, head_dim, rows, G, block_size, rope) == nullptr;
}

int tc_rows_per_unit(int rows) {
  if (rows <= 128) return 128;
  if (rows <= kTcMaxRows) return kTcMaxRows;
  // up to kTailRows rows past the two M tiles: one unit holds them all (tail rows)
  return rows <= kTcMaxRows + kTailRows ? rows : kTcMaxRows;
}

int tc_ctas_per_sm(int rows) { return rows <= 128 ? Cfg<1>::kCtasPerSm : 1; }

// Virtual tiles charged per unit: measured cost of finishing one unit and
// starting the next, in units of one 64-key tile of the steady state (chosen
// by sweeping: 3 for one M tile; 6 for two -- 3 to 8 swept on the 64-request,
// dynamic and ragged workloads once Q reached the operand slots through the
// S issuers, 6 best on all three; every two-M-tile variant takes the same
// value, so that the fused-RoPE and separate paths split units alike and give
// the same bits).
#ifndef TV_UNIT_COST_M1
#define TV_UNIT_COST_M1 3
#endif
#ifndef TV_UNIT_COST_M2
#define TV_UNIT_COST_M2 6
#endif

int tc_unit_cost(int rows_per_unit) { return rows_per_unit <= 128 ? TV_UNIT_COST_M1 : TV_UNIT_COST_M2; }

#ifdef TV_TC_TRACE
extern "C" int tv_debug_trace(void* dst, size_t bytes) {
  const size_t n = sizeof(trace::g_trace) < bytes ? sizeof(trace::g_trace) : bytes;
  return cudaMemcpyFromSymbol(dst, trace::g_trace, n) == cudaSuccess ? 0 : -1;
}
extern "C" int tv_debug_epi_times(void* dst, size_t bytes) {
  const size_t n = sizeof(trace::g_epi) < bytes ? sizeof(trace::g_epi) : bytes;
  return cudaMemcpyFromSymbol(dst, trace::g_epi, n) == cudaSuccess ? 0 : -1;
}
extern "C" int tv_debug_cta_times(void* dst, size_t bytes) {
  const size_t n = sizeof(trace::g_cta_time) < bytes ? sizeof(trace::g_cta_time) : bytes;
  return cudaMemcpyFromSymbol(dst, trace::g_cta_time, n) == cudaSuccess ? 0 : -1;
}
#endif

int launch_attn_tc(const AttnParams& p, int32_t* status, cudaStream_t stream, bool duo) {
  EncodeTiled fn;
  int st = get_encoder(&fn);
  if (st) return st;
  TcMaps maps;
  const cuuint64_t row_bytes = (cuuint64_t)kD * 2;
  const int br = p.block_size < kBlk ? p.block_size : kBlk;
  {
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.num_blocks * p.Hkv * p.block_size};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, (cuuint32_t)br};
    if ((st = encode(fn, &maps.kc, p.k_cache, 2, dims, strides, box, "k_cache"))) return st;
    if ((st = encode(fn, &maps.vc, p.v_cache, 2, dims, strides, box, "v_cache"))) return st;
  }
  {
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)p.Hkv, (cuuint64_t)p.N, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {row_bytes, row_bytes * p.Hkv, row_bytes * p.Hkv * p.N};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kBlk, 1};
    if ((st = encode(fn, &maps.kt, p.k_tree, 4, dims, strides, box, "k_tree"))) return st;
    if ((st = encode(fn, &maps.vt, p.v_tree, 4, dims, strides, box, "v_tree"))) return st;
  }
  if (p.RPG <= 128)
    return p.rope_cs ? launch_m<1, true>(p, maps, status, stream) : launch_m<1, false>(p, maps, status, stream);
  {
    // Q as [B * N][Hq][D]: one box is 128 consecutive rows (node, head) of a
    // unit's M tile, 64 columns wide (G divides 128)
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.Hq, (cuuint64_t)p.B * p.N};
    cuuint64_t strides[2] = {row_bytes, row_bytes * p.Hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.G, (cuuint32_t)(128 / p.G)};
    if ((st = encode(fn, &maps.qm, p.q, 3, dims, strides, box, "q"))) return st;
  }
  {
    // the float32 partials [2 P RPG][D]: one box is 32 rows x 32 columns
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)2 * p.P * p.RPG};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
    cuuint32_t box[2] = {32, 32};
    if ((st = encode(fn, &maps.pm, p.part_o, 2, dims, strides, box, "partials", CU_TENSOR_MAP_DATA_TYPE_FLOAT32)))
      return st;
  }
  if (duo) {
    // one unit of up to 256 rows on a CTA pair: half of every K/V tile per SM
    DuoMaps dm;
    const int brk = p.block_size < 32 ? p.block_size : 32, brv = p.block_size < kBlk ? p.block_size : kBlk;
    {
      cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.num_blocks * p.Hkv * p.block_size};
      cuuint64_t strides[1] = {row_bytes};
      cuuint32_t bk[2] = {64, (cuuint32_t)brk}, bv[2] = {64, (cuuint32_t)brv};
      if ((st = encode(fn, &dm.kc, p.k_cache, 2, dims, strides, bk, "k_cache"))) return st;
      if ((st = encode(fn, &dm.vc, p.v_cache, 2, dims, strides, bv, "v_cache"))) return st;
    }
    {
      cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)p.Hkv, (cuuint64_t)p.N, (cuuint64_t)p.B};
      cuuint64_t strides[3] = {row_bytes, row_bytes * p.Hkv, row_bytes * p.Hkv * p.N};
      cuuint32_t bk[4] = {64, 1, 32, 1}, bv[4] = {64, 1, (cuuint32_t)kBlk, 1};
      if ((st = encode(fn, &dm.kt, p.k_tree, 4, dims, strides, bk, "k_tree"))) return st;
      if ((st = encode(fn, &dm.vt, p.v_tree, 4, dims, strides, bv, "v_tree"))) return st;
    }
    return p.rope_cs ? launch_duo<true>(p, dm, status, stream) : launch_duo<false>(p, dm, status, stream);
  }
  // rows past the two M tiles computed beside them (tc_rows_per_unit gave the unit all R rows)
  // (four tail warps when one TMA warp issues a tile's boxes: at most 8)
  if (p.RPG > kTcMaxRows && p.block_size >= 32)
    return p.rope_cs ? launch_pair<true, false, 4>(p, maps, status, stream)
                     : launch_pair<false, false, 4>(p, maps, status, stream);
  if (p.RPG > kTcMaxRows)
    return p.rope_cs ? launch_pair<true, false, 2>(p, maps, status, stream)
                     : launch_pair<false, false, 2>(p, maps, status, stream);
  if (p.rope_cs) return launch_pair<true, false, 0>(p, maps, status, stream);
  // a last row group of at most 128 rows leaves M tile 1 idle: skip it
  const int tail = p.R % p.RPG;
  if (p.R > p.RPG && tail > 0 && tail <= 128) return launch_pair<false, true, 0>(p, maps, status, stream);
  // Q staged by the S issuers pays off at unit boundaries: with no more units
  // than CTAs every slice holds one or two segments, and the variant with the
  // softmax warps placing Q measured faster there (16 requests of the 64-node
  // tree: 0.119 against 0.104 ms; 32 requests: 0.137 against 0.142 ms; the
  // two give the same bits)
  return p.U > p.P ? launch_pair<false, false, 0, true>(p, maps, status, stream)
                   : launch_pair<false, false, 0, false>(p, maps, status, stream);
}

}  // namespace tv

#ifdef TV_TEST_HOOKS
// Development builds only: sets the wait limit of the tensor-core kernels and
// the ring tile of CTA 0 whose TMA loads are withheld (-1: none).  Not part of
// the product library's interface.
extern "C" int tv_test_set_hooks(unsigned long long timeout_ns, int withhold_tile) {
  if (cudaMemcpyToSymbol(tv::g_test_timeout_ns, &timeout_ns, sizeof(timeout_ns)) != cudaSuccess) return -6;
  if (cudaMemcpyToSymbol(tv::g_test_withhold, &withhold_tile, sizeof(withhold_tile)) != cudaSuccess) return -6;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -6;
}

// Development builds only: warps of the TMEM quarters in `mask` (bit q for
// lanes 32 q .. 32 q + 31 of every M tile) publish their rows of a split unit
// instead of merging them directly; 0 restores the normal routes.
extern "C" int tv_test_set_publish_warps(int mask) {
  if (cudaMemcpyToSymbol(tv::g_test_publish_warps, &mask, sizeof(mask)) != cudaSuccess) return -6;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -6;
}

// Development builds only: the first pair of tail warps sleeps delay_ns
// (about; 0: not at all) after each of its tiles has landed and before it
// reads the tile.
extern "C" int tv_test_set_tail_delay(unsigned long long delay_ns) {
  if (cudaMemcpyToSymbol(tv::g_test_tail_delay_ns, &delay_ns, sizeof(delay_ns)) != cudaSuccess) return -6;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -6;
}
#endif
