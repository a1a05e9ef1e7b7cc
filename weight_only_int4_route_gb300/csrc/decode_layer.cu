// The whole MoE layer of a decode step in one kernel launch.
//
// "Specter" summary page, technical novelty and method step (5): the draft model runs every
// expert sub-computation of a step in a single fused launch, tokens grouped per expert so that
// the per-token GEMVs over fine-grained expert matrices become small GEMMs, then scattered back.
// "Who Says Elephants Can't Run", section 3 workflow: gating, sort by expert id, grouped GEMM
// with dequantization fused (optimized I2F, interleaved INT4 word), un-permute with
// expert_scale; Figure 1: experts without rows load no weights.
//
// One persistent launch (one block per SM) runs, for T <= 32 tokens: router + top-k, the
// counting sort, FC1 (+ activation), FC2, the 16-bit shared expert (two GEMMs) and the combine.
//
// Block = 8 consumer warps + 1 producer warp.  The producer streams the weights of one work unit
// after another into a ring of 16 KB stages with 2-D TMA copies (plus the unit's activation rows
// and scales with 1-D bulk copies); the consumers convert and multiply each stage as it lands and
// hand it back.  A unit is 128 output channels of one matrix over its K range (or one K split of
// it): for the routed experts one row chunk of up to 8 routed rows, for the shared expert all T
// tokens.  Units form one sequence ordered by their dependencies,
//
//   shared FC1 -> routed FC1 -> routed FC2 (K splits) -> shared FC2 (K splits),
//
// dealt over kQ queues; each block takes the next unit of its queue with one atomic.  Before it
// copies a unit's activation rows the producer waits (bounded) until the units that write them
// are done: routed FC1 on the routing tables, a routed FC2 unit on every FC1 unit of its row
// chunk, shared FC2 on every shared FC1 unit.  A unit only waits on units earlier in the sequence
// and is only taken by a running block, so the waits cannot form a cycle.  Completion is
// published with release fences and acquire-release atomics; waiters read counts with relaxed
// loads and acquire once they see them reached (one polling warp per block and flag).
//
// The router runs first, one block per token, all 8 consumer warps over slices of d (weights
// staged in shared memory with every piece in flight); the block that finishes the last token
// sorts the rows by expert id (stable counting sort by one warp, R = T*k <= 256) and publishes
// the tables.  After the last unit the consumers run the combine (token x 256 columns per warp).
// The last block to leave resets the control words for the next launch on the same workspace.
//
// Every wait is bounded (about a second); on expiry a code goes to this file's device error
// word, an abort flag makes every other wait give up, and the launch returns with incomplete
// outputs (moe_device_error reports it).
#include <cuda.h>

#include <algorithm>
#include <cmath>

#include "moe_internal.cuh"

namespace moe {

namespace {
__device__ int g_decode_error = 0;
}

int decode_error_take(int *out) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int)) != cudaSuccess) return check_launch("decode error read");
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int)) != cudaSuccess) return check_launch("decode error reset");
  }
  if (*out == 0) *out = v;
  return MOE_OK;
}

namespace {

constexpr int kCW = 8;                        // consumer warps
constexpr int kThr = (kCW + 1) * 32;          // + the producer warp
constexpr int kProd = kCW;                    // producer warp index
constexpr int kStages = 9;                    // ring stages
constexpr int kWB = 16384;                    // weight bytes of a stage
constexpr int kX16 = 144;                     // activation row stride, 16-bit stages (64 elements + pad)
constexpr int kX4 = 528;                      // activation row stride, 4-bit stages (256 elements + pad)
constexpr int kXB = 32 * kX16;                // activation area of a stage (>= 8 * kX4)
constexpr int kSB = 512;                      // scale area of a stage
constexpr int kSlot = (kWB + kXB + kSB + 1023) / 1024 * 1024;
static_assert(8 * kX4 <= kXB, "activation area");
constexpr int kRingBytes = kStages * kSlot;
constexpr int kCombCols = 256;                // columns per combine unit
constexpr long long kTimeout = 2000000000LL;  // ~1 s of clock64 at 2 GHz

// Work units are dealt over kQ queues (queue q holds units q, q + kQ, ...; block b takes from
// queue b % kQ) and the completion counts that many blocks bump are kept kQ-fold (a waiter sums
// them), so no single word takes every block's atomics.
constexpr int kQ = 8;
constexpr int kLine = 32;   // words per cache line
enum : int {
  cGrab = 0,                  // + kLine q: next position in queue q
  cRouteTok = kQ * kLine,     // tokens whose top-k is written
  cReady = cRouteTok + kLine, // routing tables published (polled: a line of its own)
  cRC = cReady + kLine,       // row chunks
  cAbort = cRC + kLine,       // a wait expired: every other wait gives up
  cExit = cAbort + kLine,     // blocks that have left
  cFc2 = cExit + kLine,       // + kLine q: routed FC2 units done (queue q's share)
  cSh1 = cFc2 + kQ * kLine,   // + kLine q: shared FC1 units done
  cSh2 = cSh1 + kQ * kLine,   // + kLine q: shared FC2 units done
  cFc1 = cSh2 + kQ * kLine,   // + kLine rc: FC1 units done of row chunk rc
};
// waited-on flags, as indices of the per-block wait table
enum : int { fReady = 0, fSh1 = 1, fFc2 = 2, fSh2 = 3, fFc1 = 4 };
enum : int { kErrRoute = 11, kErrFc1 = 12, kErrSh1 = 13, kErrFc2 = 14, kErrRing = 15 };
enum : int { kSh1 = 0, kFc1 = 1, kFc2 = 2, kSh2 = 3, kEnd = 4 };

struct DLP {
  const uint16_t *x;          // (T, d) activations
  const void *wr;             // (d, E) router weights, fp32 or 16-bit
  const float *bias;          // (E) or nullptr
  const uint16_t *s1;         // FC1 scales (E, G1, F1)
  const uint16_t *s2;         // FC2 scales (E, G2, d)
  void *out;                  // (T, d)
  int32_t *ids;               // (T, k)
  float *gate;                // (T, k)
  int32_t *offsets;           // (E + 1)
  int32_t *perm, *inv;        // (R)
  uint16_t *h;                // (R, F) FC1 output, expert-sorted rows
  float *ypart;               // (S2, R, d) FC2 partial sums
  uint16_t *hs;               // (T, Fs) shared FC1 output
  float *yspart;              // (S3, T, d) shared FC2 partial sums
  int4 *rctab;                // row chunks: (expert, first row, rows, 0)
  int32_t *ctrl;              // control words
  int T, d, F, E, k, Fs;
  int act, group, renorm, router_f32;
  int S2, CH2;                // FC2 K splits, 128-wide chunks per split
  int S3, CH3;                // shared FC2 K splits, 64-wide slices per split
  int rcmax;                  // row-chunk table capacity
};

struct Maps {
  CUtensorMap w1, w2, sgu, sd;   // weights
  CUtensorMap s1, s2;            // group-128 scales (grouped weights only)
};

// stage description, written by the producer before the stage's copies
struct Meta {
  int kind, s, nst;           // unit kind, stage index within the unit, stages of the unit
  int e, row0, nrows;         // routed: expert and rows; shared: 0, 0, T
  int cb, kbase, nchunk;      // channel block; first K element of the stage; 4-bit: 128-chunks present
  int rc, split;              // row chunk (routed); K split (FC2 / shared FC2)
  int pad;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t su32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ int ld_relaxed(const int *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;\n" ::: "memory"); }
__device__ __forceinline__ int atom_add_acq_rel(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded mbarrier wait: false if it expired (the abort flag is then raised) or the launch aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, int *ctrl) {
  if (mbar_try(b, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(b, parity)) return true;
    if ((it & 255) == 0) {
      if (ld_relaxed(ctrl + cAbort)) return false;
      if (clock64() - t0 > kTimeout) {
        atomicExch(&g_decode_error, kErrRing);
        st_release(ctrl + cAbort, 1);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, a multiple of 16 bytes)
__device__ __forceinline__ void bulk_1d(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void cp16_cg(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kCW * 32) : "memory"); }

template <typename T> __device__ __forceinline__ float h2f(uint16_t b) {
  if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half(b));
  else return __bfloat162float(__ushort_as_bfloat16(b));
}
template <typename T> __device__ __forceinline__ uint16_t f2h(float v) {
  if constexpr (std::is_same<T, __half>::value) return __half_as_ushort(__float2half_rn(v));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ uint4 lds128(const unsigned char *p) { return *reinterpret_cast<const uint4 *>(p); }

// ---------------------------------------------------------------- waits on other blocks

// Per-block wait table in shared memory: for each waited-on flag the largest count any warp of
// the block has seen, and whether a warp is polling it in global memory.
struct WaitTab {
  int *seen;
  int *poll;
};

// Sum of a count kept in n parts kLine words apart (relaxed loads, in flight together).
__device__ __forceinline__ int ld_sum(const int *p, int n) {
  int v[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) v[q] = q < n ? ld_relaxed(p + q * kLine) : 0;
  int s = 0;
#pragma unroll
  for (int q = 0; q < kQ; ++q) s += v[q];
  return s;
}

// Bounded wait (one lane) until the count at p (n parts) reaches target; then acquire.  False if
// it expired or the launch aborted.
__device__ __forceinline__ bool wait_count(int *ctrl, const WaitTab &W, int fi, const int *p, int n, int target,
                                           int code) {
  volatile int *seen = W.seen + fi;
  if (*seen < target) {
    const long long t0 = clock64();
    unsigned pause = 64;
    for (;;) {
      if (*(volatile int *)(W.poll + fi) == 0 && atomicCAS(W.poll + fi, 0, 1) == 0) {   // poll for the block
        const int v = ld_sum(p, n);
        atomicMax(W.seen + fi, v);
        atomicExch(W.poll + fi, 0);
        if (v >= target) break;
        if (ld_relaxed(ctrl + cAbort)) return false;
        __nanosleep(pause);
        pause = pause < 256 ? pause * 2 : 256;
      } else {
        __nanosleep(256);
      }
      if (*seen >= target) break;
      if (clock64() - t0 > kTimeout) {
        atomicExch(&g_decode_error, code);
        st_release(ctrl + cAbort, 1);
        return false;
      }
    }
  }
  (void)ld_sum(p, n);
  fence_acq_rel();
  return true;
}

// ---------------------------------------------------------------- router and sort

// Router of one token by the 8 consumer warps: warp w sums rows [w d/8, (w+1) d/8) of d in
// sub-chunks staged in its part of the ring (weights and x copied with every 16-byte piece in
// flight, two sub-chunks in turn), lanes over experts; the 8 partial sums per expert are added in
// warp order by warp 0, which takes the top-k and the softmax.
template <typename T>
__device__ void route_token(const DLP &P, int t, int warp, int lane, unsigned char *ring, float *red) {
  const int E = P.E, wb = P.router_f32 ? 4 : 2;
  const int rows_w = P.d / kCW, m0 = warp * rows_w;
  constexpr int kArea = (kRingBytes - (kCW + 1) * 256 * 4) / kCW / 1024 * 1024;
  constexpr int kHalf = kArea / 2;
  unsigned char *area = ring + warp * kArea;
  int sub = 8;   // rows per sub-chunk: weights + x of a sub-chunk fit half the warp's area
  while (sub * 2 <= rows_w && (sub * 2) * (E * wb + 2) <= kHalf) sub *= 2;
  const int nsub = rows_w / sub;
  auto stage = [&](int i, int buf) {
    unsigned char *dst = area + buf * kHalf;
    const int wbytes = sub * E * wb;
    const unsigned char *ws = static_cast<const unsigned char *>(P.wr) + int64_t(m0 + i * sub) * E * wb;
    for (int o = lane * 16; o < wbytes; o += 512) cp16_cg(su32(dst + o), ws + o);
    const unsigned char *xs = reinterpret_cast<const unsigned char *>(P.x + int64_t(t) * P.d + m0 + i * sub);
    for (int o = lane * 16; o < sub * 2; o += 512) cp16_cg(su32(dst + wbytes + o), xs + o);
    cp_commit();
  };
  // E <= 32: lane = (row phase, expert) with EP >= E lanes per row, rows strided by 32 / EP;
  // E > 32: lanes over experts, NJ slots each
  int EP = 1;
  while (EP < E && EP < 32) EP *= 2;
  const int RPH = 32 / EP, le = lane % EP, rp = lane / EP;
  const int NJ = (E + 31) / 32;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  auto wval = [&](const unsigned char *src, int idx) -> float {
    return P.router_f32 ? reinterpret_cast<const float *>(src)[idx] : h2f<T>(reinterpret_cast<const uint16_t *>(src)[idx]);
  };
  stage(0, 0);
  for (int i = 0; i < nsub; ++i) {
    if (i + 1 < nsub) stage(i + 1, (i + 1) & 1);
    else cp_commit();
    cp_wait<1>();
    __syncwarp();
    const unsigned char *src = area + (i & 1) * kHalf;
    const uint16_t *xs = reinterpret_cast<const uint16_t *>(src + sub * E * wb);
    if (E <= 32) {
      if (le < E) {
#pragma unroll 4
        for (int m = rp; m < sub; m += RPH) acc[0] = fmaf(h2f<T>(xs[m]), wval(src, m * E + le), acc[0]);
      }
    } else if (NJ <= 2) {
#pragma unroll 4
      for (int m = 0; m < sub; ++m) {
        const float xm = h2f<T>(xs[m]);
        acc[0] = fmaf(xm, wval(src, m * E + lane), acc[0]);
        if (lane + 32 < E) acc[1] = fmaf(xm, wval(src, m * E + lane + 32), acc[1]);
      }
    } else {
      for (int m = 0; m < sub; ++m) {
        const float xm = h2f<T>(xs[m]);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < NJ && lane + 32 * j < E) acc[j] = fmaf(xm, wval(src, m * E + lane + 32 * j), acc[j]);
      }
    }
    __syncwarp();   // the buffer is free for the sub-chunk after next
  }
  if (E <= 32) {   // sum the row phases (fixed order: a butterfly over the phase lanes)
    for (int o = EP; o < 32; o <<= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
    if (lane < E) red[warp * 256 + lane] = acc[0];
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < NJ && lane + 32 * j < E) red[warp * 256 + lane + 32 * j] = acc[j];
  }
  consumers_sync();
  if (warp == 0) {
    float *lg = red + kCW * 256;
    for (int e = lane; e < E; e += 32) {
      float v = 0.f;
      for (int w = 0; w < kCW; ++w) v += red[w * 256 + e];
      lg[e] = v + (P.bias ? P.bias[e] : 0.f);
    }
    __syncwarp();
    topk_softmax_warp(lg, E, P.k, P.renorm, P.ids + t * P.k, P.gate + t * P.k);
  }
}

// Stable counting sort of the R = T*k rows by expert id (one warp), expert offsets, the
// inverse permutation and the row-chunk table (chunks of at most 8 rows per expert).  Counts by
// shared-memory atomics; within each batch of 32 rows a row's rank among the earlier rows of its
// expert comes from a per-expert lane mask (rows are taken in batch order, so the order is
// stable in the flat row index).
__device__ void sort_rows(const DLP &P, int lane, int *sc) {
  int *cnt = sc, *off = sc + 256, *run = sc + 512, *rcs = sc + 768;
  unsigned *msk = reinterpret_cast<unsigned *>(sc + 1024);
  const int E = P.E, R = P.T * P.k;
  for (int e = lane; e < 256; e += 32) {
    cnt[e] = 0;
    run[e] = 0;
    msk[e] = 0u;
  }
  int ide[8];   // R <= 256: every id loaded once, the loads in flight together
#pragma unroll
  for (int b = 0; b < 8; ++b) ide[b] = b * 32 + lane < R ? __ldcg(P.ids + b * 32 + lane) : -1;
  __syncwarp();
#pragma unroll
  for (int b = 0; b < 8; ++b)
    if (ide[b] >= 0) atomicAdd(cnt + ide[b], 1);
  __syncwarp();
  int c8[8], r8[8], sc_rows = 0, sc_rc = 0;   // lane owns experts 8 lane .. 8 lane + 7
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    c8[i] = e < E ? cnt[e] : 0;
    r8[i] = (c8[i] + 7) / 8;
    sc_rows += c8[i];
    sc_rc += r8[i];
  }
  int incl_rows = sc_rows, incl_rc = sc_rc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, incl_rows, o), b = __shfl_up_sync(0xffffffffu, incl_rc, o);
    if (lane >= o) {
      incl_rows += a;
      incl_rc += b;
    }
  }
  int base_rows = incl_rows - sc_rows, base_rc = incl_rc - sc_rc;
  const int total_rc = __shfl_sync(0xffffffffu, incl_rc, 31);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    if (e < E) {
      off[e] = base_rows;
      rcs[e] = base_rc;
      P.offsets[e] = base_rows;
    }
    base_rows += c8[i];
    base_rc += r8[i];
  }
  if (lane == 0) P.offsets[E] = R;
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    if (b * 32 >= R) break;
    const int f = b * 32 + lane;
    const int e = ide[b];
    if (e >= 0) atomicOr(msk + e, 1u << lane);
    __syncwarp();
    unsigned m = 0u;
    if (e >= 0) {
      m = msk[e];
      const int pos = off[e] + run[e] + __popc(m & lt);
      P.perm[pos] = f;
      P.inv[f] = pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) {   // one lane per expert of the batch
      run[e] += __popc(m);
      msk[e] = 0u;
    }
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    if (e < E)
      for (int q = 0; q < r8[i]; ++q) P.rctab[rcs[e] + q] = make_int4(e, off[e] + 8 * q, min(8, c8[i] - 8 * q), 0);
  }
  if (lane == 0) P.ctrl[cRC] = total_rc;
}

// ---------------------------------------------------------------- stage compute

// 4-bit stage (routed FC1 / FC2): 128 channels x two 128-wide K chunks, as two boxes of 64 rows
// x 128 bytes (the two chunks side by side) written by the TMA with the 128-byte swizzle (16-byte
// piece j of row r at piece j ^ (r % 8)).  Lane (g, t) of warp w takes A rows g and g + 8 from
// box rows 8w + perm(g) (perm = 0,4,1,5,2,6,3,7: the two rows a quarter-warp reads fall in
// different halves of the swizzle, so its eight 16-byte reads hit eight bank groups), piece
// 4c + t of chunk c: 32 reduction elements, converted with the magic-number I2F.  The two
// chunks are two independent MMA chains, interleaved.  Group scales: [box][chunk][64].
__device__ __forceinline__ int row_perm(int g) { return (g >> 1) | ((g & 1) << 2); }

template <typename T, bool GROUPED>
__device__ __forceinline__ void stage_int4(const unsigned char *slot, const Meta &m, bool swiglu, int warp, int lane,
                                           float (&acc)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const int pg = row_perm(g);
  // (box, row in box) of A rows g and g + 8
  int bA, rA, bB, rB;
  if (swiglu) {
    bA = 0;
    bB = 1;
    rA = rB = 8 * warp + pg;
  } else {
    bA = bB = warp >> 2;
    rA = 16 * (warp & 3) + pg;
    rB = rA + 8;
  }
  const bool two = m.nchunk > 1;
  const unsigned char *xb = slot + kWB;
  const uint16_t *sc = reinterpret_cast<const uint16_t *>(slot + kWB + kXB);
  uint4 wa[2], wb[2], xv[2][4];
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    const int cc = ch == 0 ? 0 : (two ? 1 : 0);   // a one-chunk stage runs chain 1 on chunk 0 and drops it
    const int j = 4 * cc + t;
    wa[ch] = lds128(slot + bA * 8192 + rA * 128 + ((j ^ (rA & 7)) << 4));
    wb[ch] = lds128(slot + bB * 8192 + rB * 128 + ((j ^ (rB & 7)) << 4));
#pragma unroll
    for (int v = 0; v < 4; ++v) xv[ch][v] = lds128(xb + g * kX4 + cc * 256 + 64 * t + 16 * v);
  }
  float tmp[2][4];
#pragma unroll
  for (int ch = 0; ch < 2; ++ch)
#pragma unroll
    for (int i = 0; i < 4; ++i) tmp[ch][i] = 0.f;
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    uint32_t ha[2][4], hb[2][4];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      i2f_int4((&wa[ch].x)[wi], ha[ch], T());
      i2f_int4((&wb[ch].x)[wi], hb[ch], T());
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int st = wi * 2 + kk;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const uint32_t a[4] = {ha[ch][2 * kk], hb[ch][2 * kk], ha[ch][2 * kk + 1], hb[ch][2 * kk + 1]};
        const uint4 &xq = xv[ch][st >> 1];
        mma16816(tmp[ch], a, (st & 1) ? xq.z : xq.x, (st & 1) ? xq.w : xq.y, T());
      }
    }
  }
  if constexpr (GROUPED) {   // group-128 scale on each chunk's fp32 sum, chunks in order
    const int iA = bA * 128 + (rA & 63), iB = bB * 128 + (rB & 63);
    const float cA0 = h2f<T>(sc[iA]), cB0 = h2f<T>(sc[iB]);
    acc[0] = fmaf(tmp[0][0], cA0, acc[0]);
    acc[1] = fmaf(tmp[0][1], cA0, acc[1]);
    acc[2] = fmaf(tmp[0][2], cB0, acc[2]);
    acc[3] = fmaf(tmp[0][3], cB0, acc[3]);
    if (two) {
      const float cA1 = h2f<T>(sc[iA + 64]), cB1 = h2f<T>(sc[iB + 64]);
      acc[0] = fmaf(tmp[1][0], cA1, acc[0]);
      acc[1] = fmaf(tmp[1][1], cA1, acc[1]);
      acc[2] = fmaf(tmp[1][2], cB1, acc[2]);
      acc[3] = fmaf(tmp[1][3], cB1, acc[3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += two ? tmp[0][i] + tmp[1][i] : tmp[0][i];
  }
}

// 16-bit stage (shared expert): 64 reduction elements per row, rows of 128 bytes written by the
// TMA with the 128-byte swizzle (16-byte piece j of row r at piece j ^ (r % 8)); lane t takes
// elements [16t, 16t + 16) of the slice: pieces 2t and 2t + 1.
template <typename T, int NTS>
__device__ __forceinline__ void stage_w16(const unsigned char *slot, bool swiglu, int warp, int lane,
                                          float (&acc)[NTS][4]) {
  const int g = lane >> 2, t = lane & 3;
  int rA, rB;
  if (swiglu) {
    rA = 8 * warp + g;
    rB = 64 + 8 * warp + g;
  } else {
    rA = 16 * warp + g;
    rB = 16 * warp + 8 + g;
  }
  auto piece = [&](int r, int j) -> uint4 {
    const unsigned char *box = slot + (r >> 6) * 8192;
    const int rr = r & 63;
    return lds128(box + rr * 128 + ((j ^ (rr & 7)) << 4));
  };
  const uint4 a0 = piece(rA, 2 * t), a1 = piece(rA, 2 * t + 1), b0 = piece(rB, 2 * t), b1 = piece(rB, 2 * t + 1);
  const uint32_t wA[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t wB[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
  for (int n = 0; n < NTS; ++n) {
    const unsigned char *xr = slot + kWB + (n * 8 + g) * kX16 + 32 * t;
    const uint4 x0 = lds128(xr), x1 = lds128(xr + 16);
    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int st = 0; st < 4; ++st) {
      const uint32_t a[4] = {wA[2 * st], wB[2 * st], wA[2 * st + 1], wB[2 * st + 1]};
      mma16816(acc[n], a, xw[2 * st], xw[2 * st + 1], T());
    }
  }
}

// ---------------------------------------------------------------- the kernel

template <typename AT, bool GROUPED, int NTS>
__global__ void __launch_bounds__(kThr, 1) decode_layer_kernel(const __grid_constant__ Maps M, const DLP P) {
  extern __shared__ __align__(1024) unsigned char dl_smem[];
  unsigned char *ring = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dl_smem) + 1023) & ~uintptr_t(1023));
  Meta *meta = reinterpret_cast<Meta *>(ring + kRingBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(meta + kStages);
  uint64_t *empty = full + kStages;
  WaitTab W;
  W.seen = reinterpret_cast<int *>(empty + kStages);
  W.poll = W.seen + fFc1 + P.rcmax;
  __shared__ int s_flag;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  int *ctrl = P.ctrl;
  const int T = P.T, d = P.d, F = P.F, k = P.k, R = T * k;
  const bool swiglu = P.act == MOE_ACT_SWIGLU;
  const int F1 = swiglu ? 2 * F : F;
  const int G1 = P.group == 0 ? 1 : d / 128, G2 = P.group == 0 ? 1 : F / 128;
  const int qb = blockIdx.x % kQ;   // this block's queue
  // units of each kind (routed ones depend on the row-chunk count RC, known after routing)
  const int Us1 = P.Fs > 0 ? P.Fs / 64 : 0;             // 64 hidden channels each
  const int NB1 = swiglu ? F / 64 : F / 128;             // FC1 channel blocks per row chunk
  const int NB2 = d / 128;                               // FC2 channel blocks
  const int Us2 = P.Fs > 0 ? NB2 * P.S3 : 0;

  for (int i = threadIdx.x; i < 2 * (fFc1 + P.rcmax); i += kThr) W.seen[i] = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  // ---------------------------------------------------------- router: block b routes token b
  if (blockIdx.x < unsigned(T)) {
    if (warp < kCW) {
      float *red = reinterpret_cast<float *>(ring + kRingBytes - (kCW + 1) * 256 * 4);
      route_token<AT>(P, blockIdx.x, warp, lane, ring, red);
      if (warp == 0) {
        fence_acq_rel();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel(ctrl + cRouteTok, 1) == T - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {   // the last token: sort the rows and publish the tables
          fence_acq_rel();
          sort_rows(P, lane, reinterpret_cast<int *>(ring));
          fence_acq_rel();
          __syncwarp();
          if (lane == 0) st_release(ctrl + cReady, 1);
        }
      }
    }
    __syncthreads();   // the ring is free for the weight stream
  }

  int RC = -1;
  if (warp == kProd) {
    // ---------------------------------------------------------- producer
    // lane 0 takes units, waits and writes the stage descriptions; the copies of a stage are
    // issued by several lanes at once (weight boxes, scale boxes, activation rows)
    // the tensor maps in use into the descriptor cache ahead of their first use
    const CUtensorMap *pm = lane == 0 ? &M.w1 : lane == 1 ? &M.w2 : (lane == 2 && P.Fs > 0) ? &M.sgu
                          : (lane == 3 && P.Fs > 0) ? &M.sd : (lane == 4 && GROUPED) ? &M.s1 : (lane == 5 && GROUPED) ? &M.s2
                          : nullptr;
    if (pm != nullptr) asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(pm)) : "memory");
    uint32_t it = 0;
    bool ok = true;
    while (ok) {
      Meta mt{};
      int tok = 0;   // routed FC1: token of this lane's row (lane < 8)
      if (lane == 0) {
        int u = qb + kQ * atomicAdd(ctrl + cGrab + kLine * qb, 1);
        if (u < Us1) {
          mt.kind = kSh1;
          mt.cb = u;
          mt.nst = d / 64;
          mt.nrows = T;
        } else {
          u -= Us1;
          if (RC < 0) {
            if (!wait_count(ctrl, W, fReady, ctrl + cReady, 1, 1, kErrRoute)) mt.kind = -1;
            else RC = __ldcg(ctrl + cRC);
          }
          if (mt.kind == 0) {
            const int Uf1 = RC * NB1, Uf2 = RC * NB2 * P.S2;
            if (u < Uf1) {
              mt.kind = kFc1;
              mt.rc = u / NB1;
              mt.cb = u % NB1;
              mt.nst = (d / 128 + 1) / 2;
            } else if ((u -= Uf1) < Uf2) {
              mt.kind = kFc2;
              mt.rc = u / (NB2 * P.S2);
              const int rem = u % (NB2 * P.S2);
              mt.split = rem / NB2;
              mt.cb = rem % NB2;
              mt.nst = (P.CH2 + 1) / 2;
            } else if ((u -= Uf2) < Us2) {
              mt.kind = kSh2;
              mt.split = u / NB2;
              mt.cb = u % NB2;
              mt.nst = P.CH3;
              mt.nrows = T;
            } else {
              mt.kind = kEnd;
            }
            if (mt.kind == kFc1 || mt.kind == kFc2) {
              const int4 c = __ldcg(P.rctab + mt.rc);
              mt.e = c.x;
              mt.row0 = c.y;
              mt.nrows = c.z;
            }
          }
        }
        // wait until the unit's activation rows are written
        if (mt.kind == kFc2 && !wait_count(ctrl, W, fFc1 + mt.rc, ctrl + cFc1 + kLine * mt.rc, 1, NB1, kErrFc1)) mt.kind = -1;
        if (mt.kind == kSh2 && !wait_count(ctrl, W, fSh1, ctrl + cSh1, kQ, Us1, kErrSh1)) mt.kind = -1;
      }
      // the unit to every lane of the producer warp
      int *mi = reinterpret_cast<int *>(&mt);
#pragma unroll
      for (int f = 0; f < int(sizeof(Meta) / 4); ++f) mi[f] = __shfl_sync(0xffffffffu, mi[f], 0);
      RC = __shfl_sync(0xffffffffu, RC, 0);
      if (mt.kind < 0) break;
      if (mt.kind == kFc1 && lane < mt.nrows) tok = __ldcg(P.perm + mt.row0 + lane) / k;   // its row's token
      const int nst = mt.kind == kEnd ? 1 : mt.nst;
      for (int s = 0; s < nst; ++s, ++it) {
        const int slot = it % kStages;
        int okw = 1;
        if (lane == 0) okw = mbar_wait(&empty[slot], ((it / kStages) & 1) ^ 1, ctrl);
        if (!__shfl_sync(0xffffffffu, okw, 0)) {
          ok = false;
          break;
        }
        Meta ms = mt;
        ms.s = s;
        unsigned char *sl = ring + slot * kSlot;
        if (mt.kind == kEnd) {   // no data: tells the consumers to stop
          if (lane == 0) {
            meta[slot] = ms;
            mbar_arrive(&full[slot]);
          }
          ++it;
          ok = false;
          break;
        }
        if (mt.kind == kFc1 || mt.kind == kFc2) {
          const int c0 = (mt.kind == kFc1 ? 0 : mt.split * P.CH2) + 2 * s;
          const int cend = mt.kind == kFc1 ? d / 128 : (mt.split + 1) * P.CH2;
          ms.nchunk = min(2, cend - c0);
          ms.kbase = c0 * 128;
          const int N = mt.kind == kFc1 ? F1 : d;
          const int chA = mt.kind == kFc1 && swiglu ? mt.cb * 64 : mt.cb * 128;
          const int chB = mt.kind == kFc1 && swiglu ? F + mt.cb * 64 : chA + 64;
          if (lane == 0) {
            meta[slot] = ms;
            mbar_expect_tx(&full[slot], kWB + (GROUPED ? 512 : 0) + mt.nrows * ms.nchunk * 256);
          }
          __syncwarp();
          if (lane < 2) {   // lanes 0-1: the two weight boxes (64 channels x both chunks each)
            tma_2d(sl + lane * 8192, mt.kind == kFc1 ? &M.w1 : &M.w2, c0 * 16, mt.e * N + (lane ? chB : chA),
                   &full[slot]);
          } else if (GROUPED && lane < 4) {   // lanes 2-3: the scale boxes (64 channels x 2 chunk rows)
            tma_2d(sl + kWB + kXB + (lane - 2) * 256, mt.kind == kFc1 ? &M.s1 : &M.s2, lane == 3 ? chB : chA,
                   mt.e * (mt.kind == kFc1 ? G1 : G2) + c0, &full[slot]);
          }
          // activation rows: lane r < nrows copies row r
          if (lane < mt.nrows) {
            const uint16_t *src = mt.kind == kFc1 ? P.x + int64_t(tok) * d : P.h + int64_t(mt.row0 + lane) * F;
            bulk_1d(sl + kWB + lane * kX4, src + c0 * 128, ms.nchunk * 256, &full[slot]);
          }
        } else {   // 16-bit shared expert: a 64-wide slice
          const int j = (mt.kind == kSh1 ? 0 : mt.split * P.CH3) + s;
          ms.kbase = j * 64;
          if (lane == 0) {
            meta[slot] = ms;
            mbar_expect_tx(&full[slot], kWB + T * 128);
          }
          __syncwarp();
          const CUtensorMap *map = mt.kind == kSh1 ? &M.sgu : &M.sd;
          const int rowA = mt.kind == kSh1 ? mt.cb * 64 : mt.cb * 128;
          const int rowB = mt.kind == kSh1 ? P.Fs + mt.cb * 64 : rowA + 64;
          if (lane < 2) tma_2d(sl + lane * 8192, map, j * 64, lane ? rowB : rowA, &full[slot]);
          const uint16_t *base = mt.kind == kSh1 ? P.x : P.hs;
          const int xs = mt.kind == kSh1 ? d : P.Fs;
          if (lane < T) bulk_1d(sl + kWB + lane * kX16, base + int64_t(lane) * xs + j * 64, 128, &full[slot]);
        }
      }
    }
    // drain: every issued copy has landed before the block may leave
    if (lane == 0) {
      const uint32_t first = it >= kStages ? it - kStages : 0;
      for (uint32_t j = first; j < it; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1, ctrl);
    }
  } else {
    // ---------------------------------------------------------- consumers
    float acc[NTS][4];
    uint32_t it = 0;
    for (;;) {
      const int slot = it % kStages;
      if (!mbar_wait(&full[slot], (it / kStages) & 1, ctrl)) break;
      const Meta mt = meta[slot];
      if (mt.kind == kEnd) break;
      const unsigned char *sl = ring + slot * kSlot;
      if (mt.s == 0) {
#pragma unroll
        for (int n = 0; n < NTS; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
      }
      if (mt.kind == kFc1 || mt.kind == kFc2) stage_int4<AT, GROUPED>(sl, mt, mt.kind == kFc1 && swiglu, warp, lane, acc[0]);
      else stage_w16<AT, NTS>(sl, mt.kind == kSh1 && swiglu, warp, lane, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++it;
      if (mt.s != mt.nst - 1) continue;
      // ---- last stage of the unit: epilogue, then the unit's completion is published
      if (mt.kind == kFc1) {
        const int64_t sbase = int64_t(mt.e) * F1;
        int cA, cB;
        if (swiglu) {
          cA = mt.cb * 64 + 8 * warp + row_perm(g);
          cB = F + cA;
        } else {
          cA = mt.cb * 128 + 16 * warp + row_perm(g);
          cB = cA + 8;
        }
        const float sA = GROUPED ? 1.f : h2f<AT>(P.s1[sbase + cA]), sB = GROUPED ? 1.f : h2f<AT>(P.s1[sbase + cB]);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = 2 * t4 + q;
          if (row < mt.nrows) {
            uint16_t *hr = P.h + int64_t(mt.row0 + row) * F;
            const float v0 = acc[0][q] * sA, v1 = acc[0][2 + q] * sB;
            if (swiglu) {
              hr[cA] = f2h<AT>(act_silu(v0) * v1);
            } else {
              hr[cA] = f2h<AT>(act_apply(v0, P.act));
              hr[cB] = f2h<AT>(act_apply(v1, P.act));
            }
          }
        }
      } else if (mt.kind == kFc2) {
        const int cA = mt.cb * 128 + 16 * warp + row_perm(g), cB = cA + 8;
        const float sA = GROUPED ? 1.f : h2f<AT>(P.s2[int64_t(mt.e) * d + cA]);
        const float sB = GROUPED ? 1.f : h2f<AT>(P.s2[int64_t(mt.e) * d + cB]);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = 2 * t4 + q;
          if (row < mt.nrows) {
            float *yr = P.ypart + (int64_t(mt.split) * R + mt.row0 + row) * d;
            yr[cA] = acc[0][q] * sA;
            yr[cB] = acc[0][2 + q] * sB;
          }
        }
      } else if (mt.kind == kSh1) {
        const int hc = mt.cb * 64 + 8 * warp + g;
#pragma unroll
        for (int n = 0; n < NTS; ++n)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int row = n * 8 + 2 * t4 + q;
            if (row < T) P.hs[int64_t(row) * P.Fs + hc] = f2h<AT>(act_silu(acc[n][q]) * acc[n][2 + q]);
          }
      } else {   // kSh2
        const int cA = mt.cb * 128 + 16 * warp + g, cB = cA + 8;
#pragma unroll
        for (int n = 0; n < NTS; ++n)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int row = n * 8 + 2 * t4 + q;
            if (row < T) {
              float *yr = P.yspart + (int64_t(mt.split) * T + row) * d;
              yr[cA] = acc[n][q];
              yr[cB] = acc[n][2 + q];
            }
          }
      }
      fence_acq_rel();
      consumers_sync();
      if (threadIdx.x == 0) {
        int *cnt = mt.kind == kFc1 ? ctrl + cFc1 + kLine * mt.rc
                 : mt.kind == kFc2 ? ctrl + cFc2 + kLine * qb
                 : mt.kind == kSh1 ? ctrl + cSh1 + kLine * qb
                                   : ctrl + cSh2 + kLine * qb;
        atom_add_acq_rel(cnt, 1);
      }
    }
    // ---------------------------------------------------------- combine (token x 256 columns per warp)
    const int NCB = (d + kCombCols - 1) / kCombCols;
    for (int u = blockIdx.x * kCW + warp; u < T * NCB; u += gridDim.x * kCW) {
      if (RC < 0) {   // every FC2 unit done (and every shared FC2 unit)
        int ok = 1, rc = 0;
        if (lane == 0) {
          ok = wait_count(ctrl, W, fReady, ctrl + cReady, 1, 1, kErrRoute);
          if (ok) rc = __ldcg(ctrl + cRC);
          if (ok) ok = wait_count(ctrl, W, fFc2, ctrl + cFc2, kQ, rc * NB2 * P.S2, kErrFc2);
          if (ok && Us2 > 0) ok = wait_count(ctrl, W, fSh2, ctrl + cSh2, kQ, Us2, kErrFc2);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        RC = __shfl_sync(0xffffffffu, rc, 0);
        if (!ok) break;
        fence_acq_rel();
      }
      const int t = u / NCB, cb = u % NCB;
      const int c = cb * kCombCols + lane * 8;
      if (c < d) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = 0.f;
        for (int j = 0; j < k; ++j) {   // entries in j order, split slices in split order
          const int p = __ldcg(P.inv + t * k + j);
          const float gw = __ldcg(P.gate + t * k + j);
          float y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = 0.f;
#pragma unroll 4
          for (int s = 0; s < P.S2; ++s) {
            const float4 *src = reinterpret_cast<const float4 *>(P.ypart + (int64_t(s) * R + p) * d + c);
            const float4 q0 = __ldcg(src), q1 = __ldcg(src + 1);
            y[0] += q0.x; y[1] += q0.y; y[2] += q0.z; y[3] += q0.w;
            y[4] += q1.x; y[5] += q1.y; y[6] += q1.z; y[7] += q1.w;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] += gw * y[i];
        }
        for (int s = 0; s < (Us2 > 0 ? P.S3 : 0); ++s) {
          const float4 *src = reinterpret_cast<const float4 *>(P.yspart + (int64_t(s) * T + t) * d + c);
          const float4 q0 = __ldcg(src), q1 = __ldcg(src + 1);
          a[0] += q0.x; a[1] += q0.y; a[2] += q0.z; a[3] += q0.w;
          a[4] += q1.x; a[5] += q1.y; a[6] += q1.z; a[7] += q1.w;
        }
        uint4 o;
        o.x = uint32_t(f2h<AT>(a[0])) | (uint32_t(f2h<AT>(a[1])) << 16);
        o.y = uint32_t(f2h<AT>(a[2])) | (uint32_t(f2h<AT>(a[3])) << 16);
        o.z = uint32_t(f2h<AT>(a[4])) | (uint32_t(f2h<AT>(a[5])) << 16);
        o.w = uint32_t(f2h<AT>(a[6])) | (uint32_t(f2h<AT>(a[7])) << 16);
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(P.out) + int64_t(t) * d + c) = o;
      }
    }
  }
  // leave: one count per block; the last block resets the control words for the next launch
  fence_acq_rel();
  __syncthreads();
  if (threadIdx.x == 0) s_flag = atom_add_acq_rel(ctrl + cExit, 1) == int(gridDim.x) - 1;
  __syncthreads();
  if (s_flag && warp == 0) {
    for (int i = lane; i < cFc1; i += 32) ctrl[i] = 0;
    for (int rc = lane; rc < P.rcmax; rc += 32) ctrl[cFc1 + kLine * rc] = 0;
    fence_acq_rel();
  }
}

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

// 4-bit codes (rows of K/8 words): 32-word (two chunks) x 64-row boxes, 128-byte swizzle.
int map_int4(EncodeTiledFn enc, CUtensorMap *m, const void *w, int64_t rows, int64_t K) {
  const cuuint64_t dims[2] = {cuuint64_t(K / 8), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(K / 2)};
  const cuuint32_t box[2] = {32u, 64u};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(w), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : set_error(MOE_ERR_CUDA, "decode layer: 4-bit tensor map encode failed (%d)", int(r));
}
// group scales (E * G rows of N 16-bit values): 64-channel x 2-row boxes, no swizzle.
int map_scales(EncodeTiledFn enc, CUtensorMap *m, const void *s, int64_t rows, int64_t N) {
  const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(N) * 2};
  const cuuint32_t box[2] = {64u, 2u};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(s), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : set_error(MOE_ERR_CUDA, "decode layer: scale tensor map encode failed (%d)", int(r));
}
// 16-bit rows of K elements: 64 x 64 boxes with the 128-byte swizzle.
int map_w16(EncodeTiledFn enc, CUtensorMap *m, const void *w, int64_t rows, int64_t K, bool bf) {
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {64u, 64u};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                         const_cast<void *>(w), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : set_error(MOE_ERR_CUDA, "decode layer: 16-bit tensor map encode failed (%d)", int(r));
}

}  // namespace

// ---------------------------------------------------------------- host side

// Whether one launch can run this layer, and how it is cut.  `units` is the number of units
// the later stages are cut to at least (the block count), where the shape allows.
DecodePlan plan_decode(const moe_layer_desc *ds, int64_t T, int64_t units) {
  DecodePlan p{};
  const int64_t R = T * ds->k;
  p.ok = T >= 1 && T <= 32 && ds->bits == 4 && ds->E <= 256 && R <= 256 && ds->d % 128 == 0 && ds->F % 128 == 0 &&
         (ds->Fs == 0 || ds->Fs % 128 == 0) && (ds->d / kCW) % 8 == 0 &&
         (ds->router_dtype == MOE_F32 || ds->router_dtype == ds->dtype);
  if (!p.ok) return p;
  p.nts = T <= 8 ? 1 : (T <= 16 ? 2 : 4);
  p.NCR = 1;
  p.rcmax = int(std::min<int64_t>(ds->E, R) + cdiv(R, 8));
  // routed FC2: K splits of at least 4 chunks each, enough units for every block (routing
  // estimated uniform)
  const double er = double(ds->E);
  const double active = std::max(1.0, er * (1.0 - std::pow(1.0 - 1.0 / er, double(R))));
  const double rc_est = std::max(active, double(R) / 8.0);
  const int nck2 = int(ds->F / 128);
  p.S2 = 1;
  for (int s = 1; s <= nck2; ++s) {
    if (nck2 % s || (nck2 / s < 4 && s > 1)) continue;
    p.S2 = s;
    if (rc_est * double(ds->d / 128) * s >= double(units)) break;
  }
  p.CH2 = nck2 / p.S2;
  p.S3 = 1;
  p.CH3 = 1;
  if (ds->Fs > 0) {
    const int nsl = int(ds->Fs / 64);   // 64-wide slices
    p.CH3 = nsl;
    for (int s = 1; s <= nsl; ++s) {
      if (nsl % s || (nsl / s < 8 && s > 1)) continue;
      p.S3 = s;
      if (double(ds->d / 128) * s >= double(units)) break;
    }
    p.CH3 = nsl / p.S3;
  }
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t at = o;
    o += align256(b);
    return at;
  };
  p.o_rpart = take(0);
  p.o_ypart = take(size_t(p.S2) * R * ds->d * 4);
  p.o_hs = take(size_t(T) * ds->Fs * 2);
  p.o_yspart = take(ds->Fs > 0 ? size_t(p.S3) * T * ds->d * 4 : 0);
  p.o_rctab = take(size_t(p.rcmax) * 16);
  p.o_ctrl = take(size_t(cFc1 + kLine * p.rcmax) * 4);
  p.bytes = o;
  return p;
}

int decode_warps() { return num_sms(); }

// Enqueue the one-launch decode layer.  `fused` points at the plan's region of the workspace;
// ids..h are the regular layer buffers.  zero_ctrl: clear the control words first (they are
// left zero by every launch that completes; a first launch on a workspace needs the clear).
int launch_decode_layer(const moe_layer_desc *ds, const moe_layer_weights *w, const void *x, int64_t T, void *out,
                        int32_t *ids, float *gate, int32_t *offs, int32_t *perm, int32_t *inv, void *h, char *fused,
                        const DecodePlan &pl, bool zero_ctrl, cudaStream_t st) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int64_t d = ds->d, F = ds->F, E = ds->E, Fs = ds->Fs;
  const int64_t F1 = ds->act == MOE_ACT_SWIGLU ? 2 * F : F;
  const bool bf = ds->dtype == MOE_BF16;
  Maps M{};
  MOE_TRY(map_int4(enc, &M.w1, w->w1, E * F1, d));
  MOE_TRY(map_int4(enc, &M.w2, w->w2, E * d, F));
  if (ds->group != 0) {
    MOE_TRY(map_scales(enc, &M.s1, static_cast<const char *>(w->w1) + moe_packed_scale_offset(E, d, F1, 4), E * (d / 128), F1));
    MOE_TRY(map_scales(enc, &M.s2, static_cast<const char *>(w->w2) + moe_packed_scale_offset(E, F, d, 4), E * (F / 128), d));
  }
  if (Fs > 0) {
    MOE_TRY(map_w16(enc, &M.sgu, w->ws_gate_up, 2 * Fs, d, bf));
    MOE_TRY(map_w16(enc, &M.sd, w->ws_down, d, Fs, bf));
  }
  DLP P{};
  P.x = static_cast<const uint16_t *>(x);
  P.wr = w->w_router;
  P.bias = w->router_bias;
  P.s1 = reinterpret_cast<const uint16_t *>(static_cast<const char *>(w->w1) + moe_packed_scale_offset(E, d, F1, 4));
  P.s2 = reinterpret_cast<const uint16_t *>(static_cast<const char *>(w->w2) + moe_packed_scale_offset(E, F, d, 4));
  P.out = out;
  P.ids = ids;
  P.gate = gate;
  P.offsets = offs;
  P.perm = perm;
  P.inv = inv;
  P.h = static_cast<uint16_t *>(h);
  P.ypart = reinterpret_cast<float *>(fused + pl.o_ypart);
  P.hs = reinterpret_cast<uint16_t *>(fused + pl.o_hs);
  P.yspart = reinterpret_cast<float *>(fused + pl.o_yspart);
  P.rctab = reinterpret_cast<int4 *>(fused + pl.o_rctab);
  P.ctrl = reinterpret_cast<int32_t *>(fused + pl.o_ctrl);
  P.T = int(T);
  P.d = int(d);
  P.F = int(F);
  P.E = int(E);
  P.k = ds->k;
  P.Fs = int(Fs);
  P.act = ds->act;
  P.group = ds->group;
  P.renorm = ds->renormalize;
  P.router_f32 = ds->router_dtype == MOE_F32 ? 1 : 0;
  P.S2 = pl.S2;
  P.CH2 = pl.CH2;
  P.S3 = pl.S3;
  P.CH3 = pl.CH3;
  P.rcmax = pl.rcmax;
  if (zero_ctrl && cudaMemsetAsync(P.ctrl, 0, size_t(cFc1 + kLine * pl.rcmax) * 4, st) != cudaSuccess)
    return check_launch("decode layer: clear control words");
  using KFn = void (*)(Maps, DLP);
  KFn fn = nullptr;
  const bool grouped = ds->group != 0;
#define MOE_DL(TT, GG, NN) \
  if ((std::is_same<TT, __nv_bfloat16>::value == bf) && grouped == GG && pl.nts == NN) fn = decode_layer_kernel<TT, GG, NN>;
  MOE_DL(__half, false, 1) MOE_DL(__half, false, 2) MOE_DL(__half, false, 4)
  MOE_DL(__half, true, 1) MOE_DL(__half, true, 2) MOE_DL(__half, true, 4)
  MOE_DL(__nv_bfloat16, false, 1) MOE_DL(__nv_bfloat16, false, 2) MOE_DL(__nv_bfloat16, false, 4)
  MOE_DL(__nv_bfloat16, true, 1) MOE_DL(__nv_bfloat16, true, 2) MOE_DL(__nv_bfloat16, true, 4)
#undef MOE_DL
  if (fn == nullptr) return set_error(MOE_ERR_UNSUPPORTED, "decode layer: no kernel instance");
  const size_t smem = 1024 + size_t(kRingBytes) + kStages * sizeof(Meta) + 2 * kStages * 8 +
                      size_t(2 * (fFc1 + pl.rcmax)) * 4;
  // the shared-memory opt-in is a per-device attribute of each instance: set it every time
  // (cheap) rather than caching it per instance and device
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return check_launch("decode layer: shared-memory attribute");
  fn<<<num_sms(), kThr, smem, st>>>(M, P);
  return check_launch("decode layer");
}

}  // namespace moe
