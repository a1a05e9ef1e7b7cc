// Grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators) for experts
// with many routed rows (prefill-sized batches).
//
// "Who Says Elephants Can't Run", section 3 / Figure 1: one launch computes every expert's
// sub-matrix product; section 4: dequantization fused into the GEMM; optimized I2F with the
// interleaved INT4 word.  "Specter", method step 5: tokens grouped per expert form a GEMM.
//
// Orientation (swap-AB): D[128 output channels x N rows] = W^T[128 x K] . Xp^T[K x N].
//   * A operand = dequantized weights, written by dequant warps straight into tensor memory
//     (tcgen05.st), never through shared memory: shared-memory bandwidth is left to the
//     activation operand.
//   * B operand = up to 160 consecutive rows (128 for 16-bit weights) of the expert's segment
//     of Xp, TMA-loaded with 128-byte swizzle (K-major), so the MMA reads it through a
//     shared-memory descriptor.
//   * D = fp32 accumulator in tensor memory, double-buffered so the epilogue of one tile
//     overlaps the mainloop of the next.
//
// Warp roles (one CTA per SM, persistent over tiles):
//   warps 0-7    epilogue: warp w reads TMEM lanes 32*(w%4).. and every other 32-column chunk
//                of the tile's columns; scale / activation, global stores;
//   warp 8       activation copies: TMA of the tile's activation block into the activation ring;
//   warp 9       MMA issuer (one thread);
//   warps 10-21  dequant, three groups of four warps; group g converts the K blocks with
//                index = g (mod 3), so each weight stage and each A stage always belongs to the
//                same group.  Warp w owns TMEM lanes 32*(w%4).. (one output channel per lane);
//                it reads that channel's packed words from shared memory, converts them with
//                the magic-number I2F (and the group-128 scale) and stores the 16-bit pairs into
//                the A stage;
//   warp 22      weight copies: TMA of the packed weight block into the weight ring, and a
//                rolling L2 prefetch of the weight blocks ahead of them.
// Tiles are 128 output channels x up to 160 routed rows (an expert with up to 160 rows is one
// tile).  TMEM columns: [0,320) two 160-column accumulators, [320,512) three 64-column A stages.
//
// Synchronisation per 128-wide K block (stage s = block index mod 3 in every ring): the weight
// copy completes `wfull[s]`; the dequant group waits on it and on `sfree[s]` (the MMAs that last
// read the A stage are done), fills the A stage, releases the weight stage (`wfree[s]`), waits
// for the block's activation copy (`bfull[s]`) and arrives on `ready[s]`; the MMA thread waits on
// `ready[s]` alone, issues eight MMAs and commits once to `sfree[s]`, which frees the activation
// stage and the A stage.  Weights and activations travel in separate rings with their own copy
// warps, so a block's dequant starts when its weights land, not when its (five times larger)
// activation block does, and the single MMA thread does one wait and one commit per block.
// A K block of 128 keeps 512-640 tensor cycles of work queued behind each wait/commit pair.
// (16-bit weights: no dequant; the MMA thread waits on both copies and `sfree` frees both stages.)
//
// Every wait on an mbarrier is bounded (about two seconds); on expiry the CTA records an
// error code in a device word, stops issuing work, drains its own asynchronous copies and
// MMAs, frees its tensor memory and returns.  The kernel is launched with programmatic stream
// serialization: its first act is to wait for the previous kernel in the stream (pdl_enter).
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "moe_internal.cuh"

namespace moe {

__device__ int g_moe_device_error = 0;

// CTA pairs for the quantized GEMM (moe_set_gemm_pairs); off by default: measured on GB300 the
// pairs are correct (bit-identical to single CTAs) but slower -- Phi FC1 1.73 vs 1.27 ms, encdec
// FC1 64 vs 52 us -- because each K block's readiness must cross to the other CTA (about
// 1-2 k cycles through the relay), more than the three A stages can hide
std::atomic<bool> g_tc_pairs{false};

int set_gemm_pairs(int on) { return g_tc_pairs.exchange(on != 0) ? 1 : 0; }

MOE_DEFINE_CHECK_WORD(gemm_tc)

namespace {

constexpr int kEpiWarps = 8;        // epilogue warps (two per TMEM lane quarter)
constexpr int kDqGroups = 3;        // dequant warp groups (each: 4 warps covering 128 lanes)
constexpr int kProdWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1, kDqWarp0 = kEpiWarps + 2;
constexpr int kWProdWarp = kDqWarp0 + 4 * kDqGroups;   // weight copies and their L2 prefetch
constexpr int kThreads = (kWProdWarp + 1) * 32;
constexpr int kBM = 128;          // output channels per tile (MMA M)
constexpr int kBNMax = 160;       // rows per tile at most (MMA N upper bound)
constexpr int kBK = 128;          // K per pipeline stage
constexpr int kAStages = 3;       // TMEM A stages (quantized weights), one per dequant group
// Every fill of a weight stage or an A stage must go to the same dequant group.  A group waits on
// its stage's barriers by phase parity, which cannot tell "one phase ahead" from "complete":
// with groups taking K blocks round-robin over a stage count they do not divide, the group of
// fill it + kStages could reach the barrier while fill it (another group's) was still in flight
// -- TMA completions of different stages are not ordered -- and pass the wait at once.
static_assert(kAStages % kDqGroups == 0, "each A stage must belong to one dequant group");
static_assert(kBNMax % 32 == 0 && kBNMax <= 256, "tile rows: whole 32-column epilogue chunks, MMA N <= 256");
constexpr int kMaxE = 256;
constexpr uint32_t kTmemCols = 512;
// Tile geometry.  Quantized weights: up to 160 rows per tile, so an expert with up to 160 routed
// rows is one tile (a second, nearly empty tile would repeat the whole dequant of its weights);
// tensor memory holds two 160-column accumulators and three 64-column A stages.  16-bit weights
// (A from shared memory, 32 KB per stage) keep 128 rows.
template <int BITS> struct TB {
  static constexpr int kBN = BITS == 16 ? 128 : kBNMax;   // rows per tile
  static constexpr int kBHalf = kBN * 64 * 2;             // one 64-wide swizzle atom column block
  static constexpr int kBBytes = 2 * kBHalf;              // activation stage
  static constexpr uint32_t kACol0 = 2 * kBN;             // A stages after the two accumulators
};
static_assert(2 * kBNMax + kAStages * 64 <= 512, "tensor memory: accumulators + A stages");
constexpr uint32_t kAStageCols = kBK / 2;    // 64 columns of 16-bit pairs
constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s at 2 GHz

enum : int { kErrTimeoutFull = 1, kErrTimeoutFree = 2, kErrTimeoutReady = 3, kErrTimeoutD = 4, kErrTimeoutDrain = 5 };

// 4/8-bit: packed words, dequantized into TMEM.  A stage holds 128 channel rows of kRowBytes
// (64 B INT4, 128 B INT8), copied with the swizzle of that width, so 16-byte piece j of row r
// sits at piece j ^ ((r * kRowBytes / 128) & (kRowBytes / 16 - 1)): the dequant warps (lane =
// row) read a piece of eight consecutive rows per quarter-warp without bank conflicts, where the
// plain layout put 4 (INT4) or 8 (INT8) of them on the same banks.  16-bit: the weights are
// the A operand as they are, TMA-loaded with the same 128-byte swizzle as the activations and
// read by the MMA from shared memory (no dequant work); a stage is then 64 KB, so three stages.
template <int BITS> struct WB {
  static constexpr int kWordsPerRow = kBK * BITS / 32;    // u32 words per channel per stage
  static constexpr int kRowBytes = kWordsPerRow * 4;
  static constexpr int kSwzMask = kRowBytes / 16 - 1;
  static constexpr int kBytes = kBM * kWordsPerRow * 4;   // weight stage bytes
  // weight and activation rings have as many stages as there are A stages, so stage s of every
  // ring holds the same K block and one MMA commit frees all three
  static constexpr int kWStages = kAStages;
  static constexpr int kBStages = kAStages;
};
static_assert(WB<4>::kWStages % kDqGroups == 0 && WB<8>::kWStages % kDqGroups == 0, "weight stages per group");
static_assert(WB<4>::kRowBytes == 64 && WB<8>::kRowBytes == 128 && WB<16>::kSwzMask == 15,
              "swizzled weight rows: 64-byte (INT4) and 128-byte (INT8) copies");

// Activation tensor maps with boxes of 32, 64, ... kBNMax rows: a tile copies the smallest box
// that covers its rows, so an expert's last, partial tile does not pull up to 128 rows of the
// next expert through shared memory (the MMA, sized to the tile's rows, never reads them).
struct XMaps {
  CUtensorMap box[kBNMax / 32];
};

struct TcParams {
  const int32_t *offsets;
  const uint16_t *scales;
  void *out;
  int R, E, K, N, group, act, out_dtype, ncb, swiglu;
  const int32_t *row_dest;   // fused top-1 un-permute (see GemmArgs), or nullptr
  const float *row_gate;
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t su32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)), "r"(bytes) : "memory");
}
// A waiting thread is suspended in hardware until the phase completes (or the hint, 1 ms, runs
// out) instead of re-issuing the test: the compute warps waiting on their stages would otherwise
// take issue slots from the single-thread MMA and copy loops on their SM sub-partitions.
template <bool CL = false>
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  if constexpr (CL)   // barriers the other CTA of a pair arrives on (remote arrivals, multicast commits)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, 1000000;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
  return ok != 0;
}
// Bounded wait: false if the CTA aborted or this wait expired (then the abort flag is set).
template <bool CL = false>
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, volatile int *abort_flag, int code) {
  if (mbar_try<CL>(b, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try<CL>(b, parity)) return true;
    if ((it & 7) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kTimeoutCycles) {
        *abort_flag = 1;
        atomicExch(&g_moe_device_error, code);
        return false;
      }
    }
  }
}

// ---- CTA pairs (clusters of two): addresses in the peer CTA, remote arrivals, cluster barrier
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(su32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

// Bring a weight box into L2 ahead of its shared-memory copy (no barrier, no shared memory).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(su32(bar))
               : "memory");
}
// pairs: completion of the pair's MMAs issued so far, signalled on `bar` in both CTAs / in this one
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
          su32(bar)),
      "h"(both)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_local(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(su32(bar))
               : "memory");
}

// A from shared memory (16-bit weights)
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The eight MMAs of one 128-wide K block (A from tensor memory), in one statement: the first
// accumulates only when `acc` is set, the others always; MMA j reads A columns a + 8j and the
// B descriptor advanced by j's start offset (16-byte units: 2 per 16-wide step inside a 64-wide
// swizzle atom column, half16 to the next column block).  The offsets are added to the low word
// only: the start-address field cannot carry (shared addresses stay below 256 KB).
#define MOE_TC_MMA_KBLOCK(GROUP)                                                                                  \
  asm volatile(                                                                                                   \
      "{\n .reg .pred p, t;\n .reg .b32 a1, bl1;\n .reg .b64 bd;\n"                                            \
      " setp.ne.b32 p, %5, 0;\n setp.eq.b32 t, %5, %5;\n"                                                       \
      " mov.b64 bd, {%2, %3};\n tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [%1], bd, %4, p;\n"             \
      " add.u32 a1, %1, 8;\n add.u32 bl1, %2, 2;\n mov.b64 bd, {bl1, %3};\n"                                  \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      " add.u32 a1, %1, 16;\n add.u32 bl1, %2, 4;\n mov.b64 bd, {bl1, %3};\n"                                 \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      " add.u32 a1, %1, 24;\n add.u32 bl1, %2, 6;\n mov.b64 bd, {bl1, %3};\n"                                 \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      " add.u32 a1, %1, 32;\n add.u32 bl1, %2, %6;\n mov.b64 bd, {bl1, %3};\n"                                \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      " add.u32 a1, %1, 40;\n add.u32 bl1, %2, %7;\n mov.b64 bd, {bl1, %3};\n"                                \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      " add.u32 a1, %1, 48;\n add.u32 bl1, %2, %8;\n mov.b64 bd, {bl1, %3};\n"                                \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      " add.u32 a1, %1, 56;\n add.u32 bl1, %2, %9;\n mov.b64 bd, {bl1, %3};\n"                                \
      " tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], bd, %4, t;\n"                                     \
      "}\n" ::"r"(d), "r"(a), "r"(bl), "r"(bh), "r"(idesc), "r"(acc), "n"(HALF16), "n"(HALF16 + 2), "n"(HALF16 + 4), \
      "n"(HALF16 + 6)                                                                                             \
      : "memory")
template <int HALF16, bool PAIR>
__device__ __forceinline__ void tc_mma_kblock_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  const uint32_t bl = uint32_t(b), bh = uint32_t(b >> 32);
  if constexpr (PAIR) MOE_TC_MMA_KBLOCK("2");   // M = 256: A rows and B columns from both CTAs of the pair
  else MOE_TC_MMA_KBLOCK("1");
}
#undef MOE_TC_MMA_KBLOCK
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);          // start address
  d |= uint64_t(1) << 16;                          // leading byte offset (unused with swizzle)
  d |= uint64_t(1024 >> 4) << 32;                  // stride byte offset
  d |= uint64_t(1) << 46;                          // descriptor version
  d |= uint64_t(2) << 61;                          // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: fp32 D, A/B f16 (0) or bf16 (1), both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int is_bf16, int M, int N) {
  return (1u << 4) | (uint32_t(is_bf16) << 7) | (uint32_t(is_bf16) << 10) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

template <typename T> __device__ __forceinline__ float ldscale(const uint16_t *s, int64_t i) {
  const uint16_t b = s[i];
  if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half(b));
  else return __bfloat162float(__ushort_as_bfloat16(b));
}

struct Tile {
  int e, row0, nrows, cb;
};

__device__ __forceinline__ Tile decode_tile(int tile, const int *s_tstart, const int *s_off, int E, int ncb,
                                            int bn) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tstart[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  Tile t;
  t.e = lo;
  const int in_e = tile - s_tstart[lo];
  const int tt = in_e / ncb;
  t.cb = in_e - tt * ncb;
  t.row0 = s_off[lo] + tt * bn;
  t.nrows = min(bn, s_off[lo + 1] - t.row0);
  return t;
}

template <typename OT> __device__ __forceinline__ void store_typed(void *out, int64_t i, float v) {
  static_cast<OT *>(out)[i] = from_f32<OT>(v);
}

// Epilogue of one tile for one warp: TMEM lanes 32q.. (output channel rows), tile columns
// [c_lo, c_hi) (routed rows).  SwiGLU tiles hold 64 gate rows then the 64 matching up rows;
// the up quarters hand their values to the gate quarters through shared memory.
template <typename T, typename OT>
__device__ __forceinline__ void epilogue_cols(const TcParams &p, const Tile &t, uint32_t tmem_d, int q, int lane,
                                              int c_lo, int c_hi, int c_step, float *xbuf, int bar_id) {
  const int r = q * 32 + lane;
  int ch;
  if (p.swiglu) ch = r < kBM / 2 ? t.cb * (kBM / 2) + r : (p.N >> 1) + t.cb * (kBM / 2) + (r - kBM / 2);
  else ch = t.cb * kBM + r;
  const float sc = (p.group == 0 && p.scales) ? ldscale<T>(p.scales, int64_t(t.e) * p.N + ch) : 1.0f;
  const int Nout = p.swiglu ? (p.N >> 1) : p.N;
  for (int c0 = c_lo; c0 < c_hi; c0 += c_step) {
    float v[32];
    tc_ld32(tmem_d + (uint32_t(q * 32) << 16) + uint32_t(c0), v);
    const int nvalid = min(32, t.nrows - c0);
    if (p.swiglu) {
      if (q >= 2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) xbuf[j * 64 + (r - 64)] = v[j] * sc;
      }
      asm volatile("bar.sync %0, 128;\n" ::"r"(bar_id) : "memory");
      if (q < 2) {
        OT *o = static_cast<OT *>(p.out) + int64_t(t.row0 + c0) * Nout + t.cb * (kBM / 2) + r;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {   // two SiLUs per paired-fp32 evaluation
          float g0 = v[j] * sc, g1 = v[j + 1] * sc;
          act_silu2(g0, g1);
          if (j < nvalid) o[int64_t(j) * Nout] = from_f32<OT>(g0 * xbuf[j * 64 + r]);
          if (j + 1 < nvalid) o[int64_t(j + 1) * Nout] = from_f32<OT>(g1 * xbuf[(j + 1) * 64 + r]);
        }
      }
      asm volatile("bar.sync %0, 128;\n" ::"r"(bar_id) : "memory");
    } else if (p.row_dest) {   // top-1 un-permute: row j goes to its token's row, times its gate
      int dl = 0;
      float gl = 0.f;
      if (lane < nvalid) {
        dl = p.row_dest[t.row0 + c0 + lane];
        gl = p.row_gate[dl];
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int dj = __shfl_sync(0xffffffffu, dl, j);
        const float gj = __shfl_sync(0xffffffffu, gl, j);
        if (j < nvalid) static_cast<OT *>(p.out)[int64_t(dj) * Nout + ch] = from_f32<OT>((v[j] * sc) * gj);
      }
    } else {
      OT *o = static_cast<OT *>(p.out) + int64_t(t.row0 + c0) * Nout + ch;
      if (p.act == MOE_ACT_GELU) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {   // two GELUs per paired-fp32 evaluation
          float g0 = v[j] * sc, g1 = v[j + 1] * sc;
          act_gelu2(g0, g1);
          if (j < nvalid) o[int64_t(j) * Nout] = from_f32<OT>(g0);
          if (j + 1 < nvalid) o[int64_t(j + 1) * Nout] = from_f32<OT>(g1);
        }
      } else if (p.act == MOE_ACT_RELU) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) o[int64_t(j) * Nout] = from_f32<OT>(act_relu(v[j] * sc));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) o[int64_t(j) * Nout] = from_f32<OT>(v[j] * sc);
      }
    }
  }
}

// PAIR: the kernel runs in clusters of two CTAs (CTA pairs, tcgen05 cta_group::2).  A pair tile
// is 256 output channels x up to 160 rows: each CTA dequantizes its 128 channels into its own
// tensor memory and copies its half of the tile's rows (rows [n/2 * rank, n/2 * rank + n/2) of
// the MMA's N = n) into its own shared memory; the rank-0 CTA issues M = 256 MMAs that read both
// CTAs' operands and commits to both CTAs' barriers.  Each SM then moves half the activation bytes
// per MMA FLOP through its shared memory.  The rank-1 CTA's dequant groups arrive on its own
// `ready`; one thread of it (the idle MMA warp's) relays each completed phase to rank 0's
// `ready`, and its epilogue warps arrive on rank 0's `d_empty`.
template <typename T, int BITS, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ XMaps maps_x, const __grid_constant__ CUtensorMap map_w,
                   const TcParams p) {
  pdl_enter();   // see launch_pdl
  static_assert(!PAIR || BITS != 16, "pairs take quantized weights");
  constexpr int kWBytes = WB<BITS>::kBytes;
  constexpr int kWords = WB<BITS>::kWordsPerRow;
  constexpr int kWS = WB<BITS>::kWStages, kBS = WB<BITS>::kBStages;
  constexpr int kBN = TB<BITS>::kBN;
  constexpr int kBRows = PAIR ? kBN / 2 : kBN;          // activation rows a CTA holds per tile
  constexpr int kBHalf = kBRows * 64 * 2, kBBytes = 2 * kBHalf;
  constexpr int kBoxUnit = PAIR ? 16 : 32;               // rows of activation box i: kBoxUnit (i + 1)
  constexpr uint32_t kACol0 = TB<BITS>::kACol0;
  constexpr bool CL = PAIR;                              // waits that see the peer's arrivals
  extern __shared__ __align__(1024) uint8_t dsmem[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
  uint8_t *sB = base;                                   // kBS x kBBytes (two 1024-aligned K halves)
  uint8_t *sW = sB + kBS * kBBytes;                     // kWS x kWBytes
  float *sX = reinterpret_cast<float *>(sW + kWS * kWBytes);  // SwiGLU exchange: 2 halves x 32 x 64 fp32
  uint64_t *bar = reinterpret_cast<uint64_t *>(sX + 2 * 32 * 64);
  // wfull/wfree: weight ring; bfull: activation ring; ready: TMEM A stages; sfree: the MMAs of
  // stage s are done (frees the activation stage, the A stage and, for 16-bit weights, the weight
  // stage)
  static_assert(kWS == kAStages && kBS == kAStages, "one stage index for every ring");
  uint64_t *wfull = bar, *wfree = wfull + kWS, *bfull = wfree + kWS, *ready = bfull + kBS, *sfree = ready + kAStages;
  uint64_t *d_full = sfree + kAStages, *d_empty = d_full + 2, *drain = d_empty + 2;
  int *s_tstart = reinterpret_cast<int *>(drain + 1);
  int *s_off = s_tstart + kMaxE + 1;
  int *scratch = s_off + kMaxE + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(scratch + 32);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E;
  // pairs: tiles are dealt per pair; this CTA's 128-channel block of a pair tile by its rank
  const int prank = PAIR ? int(cluster_rank()) : 0;
  const int ncbx = PAIR ? p.ncb / 2 : p.ncb;
  const int tile0 = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int tstride = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
  auto get_tile = [&](int tile) {
    Tile t = decode_tile(tile, s_tstart, s_off, E, ncbx, kBN);
    if constexpr (PAIR) t.cb = 2 * t.cb + prank;
    return t;
  };

  // ---- setup: barriers, TMEM, tile table
  if (tid == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wfree[s], 4);   // the dequant group's 4 warps (quantized weights)
      mbar_init(&bfull[s], 1);
      mbar_init(&ready[s], PAIR && prank == 0 ? 5 : 4);   // + the peer's relayed phase
      mbar_init(&sfree[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&d_full[s], 1);
      mbar_init(&d_empty[s], PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    if constexpr (PAIR) {   // one warp of each CTA of the pair
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(tmem_slot)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::);
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(tmem_slot)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
    }
  }
  int cnt = 0;
  // checked build: unusable offsets leave the kernel without tiles (nothing is read or written)
  const bool off_ok = p.offsets == nullptr || offsets_usable(p.offsets, E, p.R, [] { check_fail(kCheckOffsets); });
  if (tid < E && off_ok) {   // no offsets array: one expert owning all R rows
    const int o0 = p.offsets ? p.offsets[tid] : 0, o1 = p.offsets ? p.offsets[tid + 1] : p.R;
    cnt = ((o1 - o0 + kBN - 1) / kBN) * ncbx;
    s_off[tid] = o0;
    if (tid == E - 1) s_off[E] = o1;
  }
  int start = 0;
  const int total_tiles = block_exclusive_scan(cnt, &start, scratch);  // contains __syncthreads
  if (tid < E) s_tstart[tid] = start;
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();   // both CTAs' barriers initialised before any remote arrival
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t ready_r0 = PAIR ? map_to_rank(ready, 0) : 0u;     // rank 0's barriers, cluster addresses
  const uint32_t d_empty_r0 = PAIR ? map_to_rank(d_empty, 0) : 0u;
  const int nkb = p.K / kBK;
  const int is_bf16 = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
  // the drain of a copy ring: every issued fill has landed before the CTA may exit (2 bits per
  // stage: 0 = never filled, else the parity of its last fill + 1)
  // (pairs: also every release of a stage the rank-0 CTA's commits send here has arrived)
  auto drain_ring = [&](uint64_t *fullb, uint64_t *freeb, int nst, uint32_t issued) {
    for (int s = 0; s < nst; ++s)
      if ((issued >> (2 * s)) & 3u) {
        volatile int never = 0;
        mbar_wait(&fullb[s], ((issued >> (2 * s)) & 3u) - 1, &never, kErrTimeoutDrain);
        if (freeb != nullptr) mbar_wait<CL>(&freeb[s], ((issued >> (2 * s)) & 3u) - 1, &never, kErrTimeoutDrain);
      }
  };

  if (warp == kProdWarp) {
    // ------------------------------------------------ activation copies (TMA)
    if (lane == 0) {
      uint32_t it = 0, issued = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total_tiles; tile += tstride) {
        const Tile t = get_tile(tile);
        // pairs: the MMA's N columns (rows of the tile) split in halves, this CTA copies its half
        const int crows = PAIR ? ((t.nrows + 15) & ~15) >> 1 : t.nrows;
        const int brow = t.row0 + prank * crows;
        const int nb = (crows + kBoxUnit - 1) / kBoxUnit;   // box units covering the CTA's rows
        const CUtensorMap *mx = &maps_x.box[nb - 1];
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kBS;
          if (!mbar_wait<CL>(&sfree[s], ((it / kBS) & 1) ^ 1, abort_flag, kErrTimeoutFree)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&bfull[s], uint32_t(nb) * kBoxUnit * 128 * 2);
          tma_load_2d(sB + s * kBBytes, mx, kb * kBK, brow, &bfull[s]);
          tma_load_2d(sB + s * kBBytes + kBHalf, mx, kb * kBK + 64, brow, &bfull[s]);
          issued = (issued & ~(3u << (2 * s))) | ((((it / kBS) & 1) + 1) << (2 * s));
        }
      }
      drain_ring(bfull, PAIR ? sfree : nullptr, kBS, issued);
    }
  } else if (warp == kWProdWarp) {
    // ------------------------------------------------ weight copies (TMA) + L2 prefetch
    if (lane == 0) {
      // rolling L2 prefetch of the weight blocks kPrefetch K blocks ahead of the stage copies (into
      // the CTA's next tile), so a stage copy waits on L2 rather than DRAM
      constexpr int kPrefetch = 8;
      int pf_tile = tile0, pf_kb = 0, pf_A = 0, pf_B = 0;
      auto pf_rows = [&]() {
        const Tile tn = get_tile(pf_tile);
        pf_A = tn.e * p.N + (p.swiglu ? tn.cb * (kBM / 2) : tn.cb * kBM);
        pf_B = p.swiglu ? tn.e * p.N + (p.N >> 1) + tn.cb * (kBM / 2) : pf_A + kBM / 2;
      };
      auto pf_step = [&]() {   // prefetch the block at the cursor, then advance it
        if (pf_tile >= total_tiles) return;
        if constexpr (BITS == 16) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_prefetch_2d(&map_w, pf_kb * kBK + 64 * h, pf_A);
            tma_prefetch_2d(&map_w, pf_kb * kBK + 64 * h, pf_B);
          }
        } else {
          tma_prefetch_2d(&map_w, pf_kb * kWords, pf_A);
          tma_prefetch_2d(&map_w, pf_kb * kWords, pf_B);
        }
        if (++pf_kb == nkb) {
          pf_kb = 0;
          pf_tile += tstride;
          if (pf_tile < total_tiles) pf_rows();
        }
      };
      if (pf_tile < total_tiles) pf_rows();
      for (int i = 0; i < kPrefetch; ++i) pf_step();
      uint32_t it = 0, issued = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total_tiles; tile += tstride) {
        const Tile t = get_tile(tile);
        const int rowA = t.e * p.N + (p.swiglu ? t.cb * (kBM / 2) : t.cb * kBM);
        const int rowB = p.swiglu ? t.e * p.N + (p.N >> 1) + t.cb * (kBM / 2) : rowA + kBM / 2;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kWS;
          if (!mbar_wait(BITS == 16 ? &sfree[s] : &wfree[s], ((it / kWS) & 1) ^ 1, abort_flag, kErrTimeoutFree)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&wfull[s], kWBytes);
          if constexpr (BITS == 16) {   // K halves of 16 KB; rows 0-63 (rowA..) then 64-127 (rowB..)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tma_load_2d(sW + s * kWBytes + h * kBHalf, &map_w, kb * kBK + 64 * h, rowA, &wfull[s]);
              tma_load_2d(sW + s * kWBytes + h * kBHalf + kBHalf / 2, &map_w, kb * kBK + 64 * h, rowB, &wfull[s]);
            }
          } else {
            tma_load_2d(sW + s * kWBytes, &map_w, kb * kWords, rowA, &wfull[s]);
            tma_load_2d(sW + s * kWBytes + kWBytes / 2, &map_w, kb * kWords, rowB, &wfull[s]);
          }
          issued = (issued & ~(3u << (2 * s))) | ((((it / kWS) & 1) + 1) << (2 * s));
          pf_step();
        }
      }
      drain_ring(wfull, nullptr, kWS, issued);
    }
  } else if (warp == kMmaWarp && PAIR && prank == 1) {
    // ------------------------------------------------ pairs, rank 1: relay of `ready` to rank 0
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total_tiles; tile += tstride) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kAStages;
          if (!mbar_wait(&ready[s], (it / kAStages) & 1, abort_flag, kErrTimeoutReady)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(ready_r0 + uint32_t(s) * 8u);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer (pairs: rank 0 issues for both CTAs)
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total_tiles; tile += tstride, ++tcount) {
        const Tile t = get_tile(tile);
        const int n = (t.nrows + 15) & ~15;
        const uint32_t idesc = idesc_f16(is_bf16, PAIR ? 2 * kBM : kBM, n);
        const int db = tcount & 1;
        if (!mbar_wait<CL>(&d_empty[db], ((tcount >> 1) & 1) ^ 1, abort_flag, kErrTimeoutD)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(db * kBN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kAStages;
          const uint32_t par = (it / kAStages) & 1;
          // 16-bit weights: both copies landed; quantized: the dequant group signals `ready` once
          // its A stage is filled and it has seen the block's activation copy land
          if (!(BITS == 16 ? mbar_wait(&wfull[s], par, abort_flag, kErrTimeoutFull) &&
                                 mbar_wait(&bfull[s], par, abort_flag, kErrTimeoutFull)
                           : mbar_wait<CL>(&ready[s], par, abort_flag, kErrTimeoutReady))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd0 = sw128_desc(su32(sB + s * kBBytes));
          if constexpr (BITS == 16) {
            // descriptor of the stage built once; MMA j adds its start offset (16-byte units, no
            // carry out of the 14-bit field: shared addresses stay below 256 KB)
            const uint64_t ad0 = sw128_desc(su32(sW + s * kWBytes));
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j) {
              const uint64_t off = uint64_t(((j >> 2) * kBHalf + (j & 3) * 32) >> 4);
              tc_mma_ss(d_tmem, ad0 + off, bd0 + off, idesc, (kb | j) != 0);
            }
          } else {
            static_assert(kBK == 128, "tc_mma_kblock_ts issues the eight MMAs of a 128-wide K block");
            tc_mma_kblock_ts<kBHalf / 16, PAIR>(d_tmem, tmem + kACol0 + uint32_t(s) * kAStageCols, bd0, idesc,
                                                uint32_t(kb));
          }
          if constexpr (PAIR) tc_commit_pair(&sfree[s]);
          else tc_commit(&sfree[s]);
        }
        if (ok) {
          if constexpr (PAIR) tc_commit_pair(&d_full[db]);
          else tc_commit(&d_full[db]);
        }
      }
      // drain: all issued MMAs complete before TMEM is released (and, with pairs, before the
      // cluster barrier that lets the other CTA exit)
      if constexpr (PAIR) tc_commit_pair_local(drain);
      else tc_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, kErrTimeoutDrain);
    }
  } else if (warp >= kDqWarp0) {
    if constexpr (BITS != 16) {   // 16-bit weights need no conversion: these warps idle
    // ------------------------------------------------ dequant -> TMEM A stages
    const int q = warp & 3;                  // TMEM lane quarter
    const int grp = (warp - kDqWarp0) >> 2;  // converts K blocks kb with kb % kDqGroups == grp
    const int r = q * 32 + lane;             // A row (channel within the tile)
    const int swz = ((r * WB<BITS>::kRowBytes) >> 7) & WB<BITS>::kSwzMask;   // this row's piece swizzle
    uint32_t it = 0;
    bool ok = true;
    for (int tile = tile0; ok && tile < total_tiles; tile += tstride) {
      const Tile t = get_tile(tile);
      int ch;
      if (p.swiglu) ch = r < kBM / 2 ? t.cb * (kBM / 2) + r : (p.N >> 1) + t.cb * (kBM / 2) + (r - kBM / 2);
      else ch = t.cb * kBM + r;
      const int G = p.group == 0 ? 1 : p.K / p.group;
      const uint16_t *srow = p.scales + int64_t(t.e) * G * p.N + ch;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        if ((it % kDqGroups) != uint32_t(grp)) continue;
        const int sw = it % kWS, sa = it % kAStages;   // the same index: every ring has kAStages stages
        uint32_t s2 = 0;
        if (p.group != 0) {  // one scale per 128-wide K block (group 128)
          const uint16_t sb = srow[int64_t((kb * kBK) / p.group) * p.N];
          s2 = uint32_t(sb) | (uint32_t(sb) << 16);
        }
        // the block's weights have landed, and the MMAs that read this A stage last are done
        if (!mbar_wait(&wfull[sw], (it / kWS) & 1, abort_flag, kErrTimeoutFull) ||
            !mbar_wait<CL>(&sfree[sa], ((it / kAStages) & 1) ^ 1, abort_flag, kErrTimeoutFree)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t *wp = sW + sw * kWBytes + r * (kWords * 4);
        const uint32_t ta = tmem + (uint32_t(q * 32) << 16) + kACol0 + uint32_t(sa) * kAStageCols;
#pragma unroll
        for (int c = 0; c < 4; ++c) {   // 32-wide quarters of the K block: 16 columns of pairs each
          uint32_t pr[16];
          if constexpr (BITS != 8) {   // 4-bit (16-bit never reaches the dequant warps): one piece
            const uint4 w = *reinterpret_cast<const uint4 *>(wp + 16 * (c ^ swz));
            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t hh[4];
              i2f_int4(words[i], hh, T());
#pragma unroll
              for (int j = 0; j < 4; ++j) pr[4 * i + j] = hh[j];
            }
          } else {                     // 8-bit: two pieces
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const uint4 w = *reinterpret_cast<const uint4 *>(wp + 16 * ((2 * c + v) ^ swz));
              const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t hh[2];
                i2f_int8(words[i], hh, T());
                pr[8 * v + 2 * i] = hh[0];
                pr[8 * v + 2 * i + 1] = hh[1];
              }
            }
          }
          if (p.group != 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) pr[j] = scale_pair(pr[j], s2, T());
          }
          tc_st16(ta + uint32_t(16 * c), pr);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wfree[sw]);   // the block's weights are in registers / TMEM now
        tc_wait_st();
        tc_fence_before();
        // the MMA thread waits on `ready` alone: the group also waits for the block's activation copy
        if (!mbar_wait(&bfull[sa], (it / kAStages) & 1, abort_flag, kErrTimeoutFull)) {
          ok = false;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[sa]);
      }
    }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 0-7)
    const int q = warp & 3;
    const int half = warp >> 2;   // tile columns: 32-wide chunks 2 c + half
    uint32_t tcount = 0;
    for (int tile = tile0; tile < total_tiles; tile += tstride, ++tcount) {
      const Tile t = get_tile(tile);
      const int db = tcount & 1;
      if (!mbar_wait<CL>(&d_full[db], (tcount >> 1) & 1, abort_flag, kErrTimeoutD)) break;
      tc_fence_after();
      const int c_lo = 32 * half, c_hi = t.nrows;
      const uint32_t tmem_d = tmem + uint32_t(db * kBN);
      float *xbuf = sX + half * (32 * 64);
      if (c_lo < c_hi) {
        if (p.out_dtype == MOE_F32) epilogue_cols<T, float>(p, t, tmem_d, q, lane, c_lo, c_hi, 64, xbuf, 1 + half);
        else if (p.out_dtype == MOE_F16) epilogue_cols<T, __half>(p, t, tmem_d, q, lane, c_lo, c_hi, 64, xbuf, 1 + half);
        else epilogue_cols<T, __nv_bfloat16>(p, t, tmem_d, q, lane, c_lo, c_hi, 64, xbuf, 1 + half);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster(d_empty_r0 + uint32_t(db) * 8u);   // rank 0 issues the MMAs
        else mbar_arrive(&d_empty[db]);
      }
    }
  }

  // ---- teardown: everyone done (pairs: in both CTAs), release tensor memory
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

size_t smem_bytes(int bits, bool pair) {
  const size_t wbytes = bits == 4 ? WB<4>::kBytes : (bits == 8 ? WB<8>::kBytes : WB<16>::kBytes);
  const int ws = bits == 4 ? WB<4>::kWStages : (bits == 8 ? WB<8>::kWStages : WB<16>::kWStages);
  const int bs = bits == 4 ? WB<4>::kBStages : (bits == 8 ? WB<8>::kBStages : WB<16>::kBStages);
  const size_t bbytes = (bits == 16 ? TB<16>::kBBytes : TB<4>::kBBytes) / (pair ? 2 : 1);
  return 1024 /*align slack*/ + bs * bbytes + ws * wbytes + 2 * 32 * 64 * 4 + (2 * ws + 2 * bs + 2 * kAStages + 5) * 8 +
         (2 * (kMaxE + 1) + 32 + 2) * 4;
}
static_assert(1024 + WB<4>::kBStages * TB<4>::kBBytes + WB<4>::kWStages * WB<4>::kBytes + 2 * 32 * 64 * 4 +
                      (2 * WB<4>::kWStages + 2 * WB<4>::kBStages + 2 * kAStages + 5) * 8 + (2 * (kMaxE + 1) + 34) * 4 <=
                  232448,
              "INT4 shared memory");
static_assert(1024 + WB<8>::kBStages * TB<8>::kBBytes + WB<8>::kWStages * WB<8>::kBytes + 2 * 32 * 64 * 4 +
                      (2 * WB<8>::kWStages + 2 * WB<8>::kBStages + 2 * kAStages + 5) * 8 + (2 * (kMaxE + 1) + 34) * 4 <=
                  232448,
              "INT8 shared memory");
static_assert(1024 + WB<16>::kBStages * TB<16>::kBBytes + WB<16>::kWStages * WB<16>::kBytes + 2 * 32 * 64 * 4 +
                      (2 * WB<16>::kWStages + 2 * WB<16>::kBStages + 2 * kAStages + 5) * 8 + (2 * (kMaxE + 1) + 34) * 4 <=
                  232448,
              "16-bit shared memory");

// Pairs the device can run at once (0 if the pair kernel cannot be placed), per instance and
// device; also sets the pair kernel's shared-memory opt-in, which the query needs.
template <typename T, int BITS> int max_pairs(size_t smem, int dev) {
  static std::atomic<int> c[64];   // 0 = not asked yet, else pairs + 1
  int v = c[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    v = 1;
    if (cudaFuncSetAttribute(gemm_tc_kernel<T, BITS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * unsigned(num_sms()));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<T, BITS, true>, &cfg) == cudaSuccess) v = n + 1;
    }
    cudaGetLastError();   // a refused query leaves no error behind: the single-CTA kernel runs
    c[dev].store(v, std::memory_order_relaxed);
  }
  return v - 1;
}

template <typename T, int BITS, bool PAIR>
int launch_typed(const GemmArgs &g, cudaStream_t st, int dev, int pairs_max) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  XMaps mx{};
  CUtensorMap mw;
  constexpr int kUnit = PAIR ? 16 : 32;   // box heights: a CTA's rows of a tile, in these units
  for (int i = 0; i < TB<BITS>::kBN / 32; ++i) {   // box i: 64 columns (one 128-byte swizzle atom) x kUnit (i + 1) rows
    const cuuint64_t dims[2] = {cuuint64_t(g.K), cuuint64_t(g.R)};
    const cuuint64_t strides[1] = {cuuint64_t(g.K) * 2};
    const cuuint32_t box[2] = {64u, cuuint32_t(kUnit * (i + 1))};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = enc(&mx.box[i], std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           2, const_cast<void *>(g.a), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ERR_CUDA, "activation tensor map encode failed (%d)", int(r));
  }
  if constexpr (BITS == 16) {   // (E*N, K) 16-bit rows, 64 x 64 boxes with the activations' swizzle
    const cuuint64_t dims[2] = {cuuint64_t(g.K), cuuint64_t(int64_t(g.E) * g.N)};
    const cuuint64_t strides[1] = {cuuint64_t(g.K) * 2};
    const cuuint32_t box[2] = {64u, cuuint32_t(kBM / 2)};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = enc(&mw, std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           2, const_cast<void *>(g.w), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ERR_CUDA, "weight tensor map encode failed (%d)", int(r));
  } else {
    const int words_per_row = g.K * BITS / 32;
    const cuuint64_t dims[2] = {cuuint64_t(words_per_row), cuuint64_t(int64_t(g.E) * g.N)};
    const cuuint64_t strides[1] = {cuuint64_t(words_per_row) * 4};
    const cuuint32_t box[2] = {cuuint32_t(WB<BITS>::kWordsPerRow), cuuint32_t(kBM / 2)};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(g.w), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           WB<BITS>::kRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ERR_CUDA, "weight tensor map encode failed (%d)", int(r));
  }
  TcParams tp{};
  tp.row_dest = g.row_dest;
  tp.row_gate = g.row_gate;
  tp.offsets = g.offsets;
  tp.scales = static_cast<const uint16_t *>(g.scales);
  tp.out = g.out;
  tp.R = int(g.R);
  tp.E = g.E;
  tp.K = g.K;
  tp.N = g.N;
  tp.group = g.group;
  tp.act = g.act;
  tp.out_dtype = g.out_dtype;
  tp.swiglu = g.act == MOE_ACT_SWIGLU ? 1 : 0;
  tp.ncb = g.N / kBM;  // SwiGLU: 64 gate + 64 up channels per 128-channel block, the same count
  const size_t smem = smem_bytes(BITS, PAIR);
  // tiles upper bound: (row tiles) x channel blocks (pairs: x channel-block pairs)
  const int64_t row_tiles = std::min<int64_t>(g.E, g.R) + cdiv(g.R, TB<BITS>::kBN);
  if constexpr (PAIR) {   // the opt-in was set by max_pairs
    const int64_t tiles = row_tiles * (tp.ncb / 2);
    const int pairs = int(std::max<int64_t>(1, std::min<int64_t>(tiles, pairs_max)));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * unsigned(pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaLaunchKernelEx(&cfg, gemm_tc_kernel<T, BITS, true>, mx, mw, tp);
    return check_launch("grouped_gemm_tc (pairs)");
  } else {
    // the shared-memory opt-in is a per-device attribute of the kernel: set once per device
    static std::atomic<bool> attr_set[64];   // one per instance (template) and device
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
      if (cudaFuncSetAttribute(gemm_tc_kernel<T, BITS, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(smem)) != cudaSuccess)
        return check_launch("gemm_tc attribute");
      attr_set[dev].store(true, std::memory_order_relaxed);
    }
    const int64_t tiles = row_tiles * tp.ncb;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(tiles, num_sms())));
    launch_pdl(gemm_tc_kernel<T, BITS, false>, dim3(grid), dim3(kThreads), smem, st, mx, mw, tp);
    return check_launch("grouped_gemm_tc");
  }
}

// Pairs take 4- and 8-bit weights whose channel blocks come in pairs, on devices that can place
// them; everything else runs on single CTAs.
template <typename T, int BITS> int launch_tc(const GemmArgs &g, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("gemm_tc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(MOE_ERR_UNSUPPORTED, "gemm_tc: device index %d >= 64", dev);
  if constexpr (BITS != 16) {
    if (g_tc_pairs && (g.N / kBM) % 2 == 0) {
      const int pm = max_pairs<T, BITS>(smem_bytes(BITS, true), dev);
      if (pm > 0) return launch_typed<T, BITS, true>(g, st, dev, pm);
    }
  }
  return launch_typed<T, BITS, false>(g, st, dev, 0);
}

}  // namespace

bool tc_shape_ok(int64_t E, int64_t K, int64_t N, int bits, int group, int act) {
  if (bits != 4 && bits != 8 && bits != 16) return false;
  if (bits == 16 && group != 0) return false;
  if (K % kBK != 0) return false;
  if (act == MOE_ACT_SWIGLU) {
    if ((N / 2) % (kBM / 2) != 0) return false;
  } else if (N % kBM != 0) {
    return false;
  }
  if (group != 0 && group % kBK != 0) return false;
  return E * N < (int64_t(1) << 31);
}

bool tc_supported(const GemmArgs &g) {
  return (g.offsets != nullptr || g.E == 1) && tc_shape_ok(g.E, g.K, g.N, g.bits, g.group, g.act);
}

int launch_gemm_tc(const GemmArgs &g, cudaStream_t st) {
  if (g.R == 0) return MOE_OK;
  const bool bf = g.a_dtype == MOE_BF16;
  if (g.bits == 4) return bf ? launch_tc<__nv_bfloat16, 4>(g, st) : launch_tc<__half, 4>(g, st);
  if (g.bits == 8) return bf ? launch_tc<__nv_bfloat16, 8>(g, st) : launch_tc<__half, 8>(g, st);
  return bf ? launch_tc<__nv_bfloat16, 16>(g, st) : launch_tc<__half, 16>(g, st);
}

int read_device_error(cudaStream_t st, int *out) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return check_launch("device error read");
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_moe_device_error, sizeof(int)) != cudaSuccess) return check_launch("device error read");
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_moe_device_error, &zero, sizeof(int)) != cudaSuccess) return check_launch("device error reset");
  *out = v;
  return MOE_OK;
}

}  // namespace moe
