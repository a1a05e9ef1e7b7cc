// The whole MoE layer of a decode step in one kernel launch.
//
// "Specter" summary page, technical novelty and method step (5): the draft model runs every
// expert sub-computation of a step in a single fused launch, tokens grouped per expert so that
// the per-token GEMVs over fine-grained expert matrices become small GEMMs, then scattered back.
// "Who Says Elephants Can't Run", section 3 workflow: gating, sort by expert id, grouped GEMM
// with dequantization fused (optimized I2F, interleaved INT4 word), un-permute with
// expert_scale; Figure 1: experts without rows load no weights.
//
// One persistent launch runs router + top-k, the counting sort, FC1 (+ activation), FC2, the
// 16-bit shared expert (its two GEMMs) and the combine for T <= 32 tokens.  The work is cut into
// units kept in one global sequence whose order respects the dependencies:
//
//   router (token, 128-row slice of d) -> shared FC1 (8 hidden channels) -> routed FC1 (row
//   chunk, 16 or 32 hidden channels) -> routed FC2 (row chunk, K split, 32 output channels) ->
//   shared FC2 (K split, 16 output channels) -> combine (token, 256 columns)
//
// Every warp takes the next unit from a global counter (an atomic add, fetched one unit ahead),
// so warps that finish early move on to the next kind of work.  A unit waits, before touching
// its inputs, until the units it reads from are done: routed FC1 on the routing tables, a
// routed FC2 unit on the FC1 units of its row chunk, shared FC2 on every shared FC1 unit, the
// combine on every FC2 unit.  A unit only ever waits on units earlier in the sequence, and a
// unit is only taken by a warp that is running, so the waits cannot form a cycle whatever the
// number of resident blocks.  Completion is published with a release fence and an atomic count;
// waiters read the count with acquire loads and read the producers' data through L2 (.cg).
//
// The router's partial logits of a token are summed (in slice order) by the warp that finishes
// the token's last slice; the warp that finishes the last token sorts all rows by expert id
// (stable counting sort by one warp, R = T*k <= 256), cuts every expert's rows into chunks of
// at most 8 and publishes the chunk table.  The last warp to leave resets the control words,
// so the next launch on the same workspace starts from zero.
//
// Every wait is bounded (about a second); on expiry the warp records a code in this file's
// device error word, raises an abort flag that makes every other wait give up, and the launch
// returns with incomplete outputs (moe_device_error reports it).
//
// The expert GEMMs stream the weights through a per-warp ring of cp.async chunk slots in
// shared memory (copies of whole weight rows, the activation pieces lane by lane) and use them
// as the m16n8k16 A operand with the routed rows as B, as the decode weight-stream kernel does.
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

constexpr int kW = 8;                    // warps per block
constexpr int kThr = kW * 32;
constexpr int kRing = 26 * 1024;         // shared-memory ring of one warp (bytes)
constexpr int kRouteRows = 128;          // rows of d per router unit
constexpr int kCombCols = 256;           // columns per combine unit
constexpr long long kTimeout = 2000000000LL;   // ~1 s of clock64 at 2 GHz

// control words (int32) in the workspace.  Words that warps wait on, and the hot atomic
// counters, sit on cache lines of their own (32 words apart).
// The unit sequence is dealt over kQ queues (queue q holds units q, q + kQ, q + 2 kQ, ...; warp w
// of a block takes from queue w % kQ), and the completion counts that many warps bump are kept
// kQ-fold (a waiter sums them), so no single word takes every warp's atomics.
constexpr int kQ = 8;
constexpr int kLine = 32;   // words per cache line
enum : int {
  cGrab = 0,                  // + kLine q: next position in queue q
  cRouteTok = kQ * kLine,     // tokens whose top-k is written
  cReady = cRouteTok + kLine, // routing tables published
  cRC = cReady + 1,           // row chunks
  cAbort = cReady + 2,        // a wait expired: every other wait gives up
  cExit = cReady + kLine,     // blocks that have left
  cTok = cExit + kLine,       // + t: router slices done of token t (t < 32)
  cFc2 = cTok + kLine,        // + kLine q: routed FC2 units done (queue q's share)
  cSh1 = cFc2 + kQ * kLine,   // + kLine q: shared FC1 units done
  cSh2 = cSh1 + kQ * kLine,   // + kLine q: shared FC2 units done
  cFc1 = cSh2 + kQ * kLine,   // + kLine rc: FC1 units done of row chunk rc
};
constexpr int kFc1Stride = kLine;
// waited-on flags, as indices of the per-block wait table: 0 ready, 1 shared FC1, 2 routed FC2,
// 3 shared FC2, 4 + rc the FC1 count of row chunk rc
enum : int { fReady = 0, fSh1 = 1, fFc2 = 2, fSh2 = 3, fFc1 = 4 };
enum : int { kErrRoute = 11, kErrFc1 = 12, kErrSh1 = 13, kErrFc2 = 14 };

struct DLP {
  const uint16_t *x;          // (T, d) activations
  const void *wr;             // (d, E) router weights, fp32 or 16-bit
  const float *bias;          // (E) or nullptr
  const uint4 *w1;            // FC1 codes (E, F1, d/8 words)
  const uint16_t *s1;         // FC1 scales (E, G1, F1)
  const uint4 *w2;            // FC2 codes (E, d, F/8 words)
  const uint16_t *s2;         // FC2 scales (E, G2, d)
  const uint4 *wsgu;          // shared gate|up 16-bit rows (2Fs, d) or nullptr
  const uint4 *wsd;           // shared down 16-bit rows (d, Fs)
  void *out;                  // (T, d)
  int32_t *ids;               // (T, k)
  float *gate;                // (T, k)
  int32_t *offsets;           // (E + 1)
  int32_t *perm, *inv;        // (R)
  float *rpart;               // (T, NCR, E) partial logits
  uint16_t *h;                // (R, F) FC1 output, expert-sorted rows
  float *ypart;               // (S2, R, d) FC2 partial sums
  uint16_t *hs;               // (T, Fs) shared FC1 output
  float *yspart;              // (S3, T, d) shared FC2 partial sums
  int4 *rctab;                // row chunks: (expert, first row, rows, 0)
  int32_t *ctrl;              // control words
  int T, d, F, E, k, Fs;
  int act, group, renorm, router_f32;
  int NCR;                    // router units per token
  int S2, CH2;                // FC2 K splits, 128-wide chunks per split
  int S3, CH3;                // shared FC2 K splits, chunks per split
  int rcmax;                  // row-chunk table capacity
};

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
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
// publish: everything any lane of this warp wrote before is visible to whoever reads the count
// with acquire semantics (each lane's release fence, then one acq_rel add by lane 0; the old
// value tells the last arriver, whose acquire half makes the others' data visible to it)
__device__ __forceinline__ int publish_add(int *p, int v, int lane) {
  fence_acq_rel();
  __syncwarp();
  int old = 0;
  if (lane == 0) old = atom_add_acq_rel(p, v);
  old = __shfl_sync(0xffffffffu, old, 0);
  fence_acq_rel();   // the other lanes of a last arriver read what the others published
  return old;
}

// Per-block wait table in shared memory: for each waited-on flag the largest value any warp of
// the block has seen, and whether a warp is polling it.  One warp per block polls a flag in
// global memory (with a growing pause); the others watch the table, so a flag is read by at most
// one warp per block instead of by every waiting warp.
struct WaitTab {
  int *seen;
  int *poll;
};

// Sum of a count kept in `n` parts kLine words apart (relaxed loads, all in flight together).
__device__ __forceinline__ int ld_sum(const int *p, int n) {
  int v[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) v[q] = q < n ? ld_relaxed(p + q * kLine) : 0;
  int s = 0;
#pragma unroll
  for (int q = 0; q < kQ; ++q) s += v[q];
  return s;
}

// Bounded wait (warp-uniform) until the count at p (n parts) reaches target.  False if it
// expired or another warp gave up.
__device__ __forceinline__ bool wait_geq(const DLP &P, const WaitTab &W, int fi, const int *p, int n, int target,
                                         int code, int lane) {
  int ok = 1;
  if (lane == 0) {
    volatile int *seen = W.seen + fi;
    if (*seen < target) {
      const long long t0 = clock64();
      unsigned pause = 64;
      for (;;) {
        if (atomicCAS(W.poll + fi, 0, 1) == 0) {   // this warp polls for the block
          const int v = ld_sum(p, n);
          atomicMax(W.seen + fi, v);
          atomicExch(W.poll + fi, 0);
          if (v >= target) break;
          if (ld_relaxed(P.ctrl + cAbort)) {
            ok = 0;
            break;
          }
          __nanosleep(pause);
          pause = pause < 512 ? pause * 2 : 512;
        } else {
          __nanosleep(64);
        }
        if (*seen >= target) break;
        if (clock64() - t0 > kTimeout) {
          atomicExch(&g_decode_error, code);
          st_release(P.ctrl + cAbort, 1);
          ok = 0;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {   // every lane: the count is seen reached; acquire what its producers published
    (void)ld_sum(p, n);
    fence_acq_rel();
  }
  return ok != 0;
}

__device__ __forceinline__ float ldcg_f(const float *p) { return __ldcg(p); }
__device__ __forceinline__ int ldcg_i(const int *p) { return __ldcg(p); }

template <typename T> __device__ __forceinline__ float h2f(uint16_t b) {
  if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half(b));
  else return __bfloat162float(__ushort_as_bfloat16(b));
}
template <typename T> __device__ __forceinline__ uint16_t f2h(float v) {
  if constexpr (std::is_same<T, __half>::value) return __half_as_ushort(__float2half_rn(v));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16_cg(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp16_w(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- weight-stream engine

// Slot of the ring: weight rows (16 * MT channels, 16 * BITS bytes each per 128-wide chunk,
// padded for 16-bit rows so a quarter-warp's reads of two rows fall on different banks), the
// activation pieces lane by lane (NT n-tiles), the chunk's scale rows (grouped weights).
template <int BITS, int NT, int MT> struct SL {
  static constexpr int kVec = BITS / 4;
  static constexpr int kRows = 16 * MT;
  static constexpr int kRowBytes = 16 * BITS;
  static constexpr int kRowStride = kRowBytes + (BITS == 4 ? 0 : 16);
  static constexpr int kPiecesPerRow = kRowBytes / 16;
  static constexpr int kRowsPerCopy = 32 / kPiecesPerRow;
  static constexpr int kWPieces = kRows * kRowBytes / 16 / 32;
  static constexpr int kXOff = kRows * kRowStride;
  static constexpr int kSOff = kXOff + NT * 4 * 512;
  static constexpr int kScaleLanes = MT * 2;
  static constexpr int kSlot = (kSOff + kScaleLanes * 16 + 127) / 128 * 128;
  static constexpr int kDepth = kRing / kSlot;
  static_assert(kDepth >= 2, "ring too small for this slot");
};

// Channel of row r (0..15) of m-tile m in channel group grp: SwiGLU groups hold 8 gate channels
// and the 8 matching up channels per m-tile (the D fragment of a lane then holds a pair).
template <int MT>
__device__ __forceinline__ int chan_of(int grp, int m, int r, bool swiglu, int Fh) {
  if (swiglu) return r < 8 ? (grp * MT + m) * 8 + r : Fh + (grp * MT + m) * 8 + (r - 8);
  return (grp * MT + m) * 16 + r;
}

struct Job {
  const uint4 *w;             // expert's weight rows (uint4 units)
  int64_t row_vec;            // uint4 per channel row
  const uint16_t *s;          // expert's scales (E-offset applied) or nullptr
  int N;                      // channels of the weight matrix (scale row stride)
  int grp;                    // channel group
  bool swiglu;
  int Fh;                     // SwiGLU: offset of the up channels
  int c0, nch;                // 128-wide chunks [c0, c0 + nch)
};

// acc[m][n][.] = sum over the job's chunks of A(channels) . B(rows), for the lane's fragment;
// grouped weights get each chunk's scale on the chunk's fp32 sum.  xrow[n]: this lane's
// activation row of n-tile n (row g), or nullptr when the row is beyond the chunk (its output
// column is never stored, so the slot's stale bytes there do no harm).
template <typename T, int BITS, int NT, int MT, bool GROUPED>
__device__ __forceinline__ void stream_job(const Job &J, const uint16_t *const (&xrow)[NT], unsigned char *ring,
                                           int lane, float (&acc)[MT][NT][4]) {
  using C = SL<BITS, NT, MT>;
  constexpr int kDepth = C::kDepth;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t wring = smem_u32(ring);
  const int wrow = lane / C::kPiecesPerRow, wpart = lane % C::kPiecesPerRow;
  int64_t woff[C::kWPieces];
#pragma unroll
  for (int v = 0; v < C::kWPieces; ++v) {
    const int r = v * C::kRowsPerCopy + wrow;
    woff[v] = int64_t(chan_of<MT>(J.grp, r / 16, r % 16, J.swiglu, J.Fh)) * J.row_vec + wpart;
  }
  const uint16_t *ssrc = nullptr;
  if (GROUPED && lane < C::kScaleLanes) ssrc = J.s + chan_of<MT>(J.grp, lane >> 1, 8 * (lane & 1), J.swiglu, J.Fh);
  auto issue = [&](int step, int slot) {
    const int c = J.c0 + step;
    const uint32_t sb = wring + slot * C::kSlot;
#pragma unroll
    for (int v = 0; v < C::kWPieces; ++v) {
      const int r = v * C::kRowsPerCopy + wrow;
      cp16_w(sb + r * C::kRowStride + wpart * 16, J.w + woff[v] + int64_t(c) * BITS);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
      if (xrow[n] != nullptr)
#pragma unroll
        for (int v = 0; v < 4; ++v) cp16_cg(sb + C::kXOff + (n * 4 + v) * 512 + lane * 16, xrow[n] + c * 128 + 32 * t + 8 * v);
    if (GROUPED && lane < C::kScaleLanes) cp16_cg(sb + C::kSOff + lane * 16, ssrc + int64_t(c) * J.N);
  };
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][n][i] = 0.f;
#pragma unroll
  for (int d = 0; d < kDepth - 1; ++d) {
    if (d < J.nch) issue(d, d);
    cp_commit();
  }
  const uint32_t wlane = g * C::kRowStride + t * C::kVec * 16;
  int slot = 0, fill = kDepth - 1;
  for (int j = 0; j < J.nch; ++j) {
    cp_wait<kDepth - 2>();
    __syncwarp();
    if (j + kDepth - 1 < J.nch) issue(j + kDepth - 1, fill);
    cp_commit();
    fill = fill + 1 == kDepth ? 0 : fill + 1;
    const unsigned char *sb = ring + slot * C::kSlot;
    slot = slot + 1 == kDepth ? 0 : slot + 1;
    uint4 xv[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int v = 0; v < 4; ++v) xv[n][v] = *reinterpret_cast<const uint4 *>(sb + C::kXOff + (n * 4 + v) * 512 + lane * 16);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float cs[2] = {1.f, 1.f};
      if constexpr (GROUPED) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          cs[hh] = h2f<T>(*reinterpret_cast<const uint16_t *>(sb + C::kSOff + (m * 2 + hh) * 16 + 2 * g));
      }
      uint4 wv[2][C::kVec];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int v = 0; v < C::kVec; ++v)
          wv[hh][v] = *reinterpret_cast<const uint4 *>(sb + (m * 16 + 8 * hh) * C::kRowStride + wlane + v * 16);
      float tmp[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) tmp[n][i] = 0.f;
      constexpr int kWords = 4 * C::kVec;
      constexpr int kStepsPerWord = 8 / kWords;   // INT4: 2; 16-bit: 0 (two words per step)
#pragma unroll
      for (int wi = 0; wi < kWords; ++wi) {
        const uint32_t wa = (&wv[0][0].x)[wi], wb = (&wv[1][0].x)[wi];
        if constexpr (BITS == 4) {
          uint32_t ha[4], hb[4];
          i2f_int4(wa, ha, T());
          i2f_int4(wb, hb, T());
#pragma unroll
          for (int kk = 0; kk < kStepsPerWord; ++kk) {
            const uint32_t a[4] = {ha[2 * kk], hb[2 * kk], ha[2 * kk + 1], hb[2 * kk + 1]};
            const int st = wi * kStepsPerWord + kk;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const uint4 &xq = xv[n][st >> 1];
              const uint32_t x0 = (st & 1) ? xq.z : xq.x, x1 = (st & 1) ? xq.w : xq.y;
              if constexpr (GROUPED) mma16816(tmp[n], a, x0, x1, T());
              else mma16816(acc[m][n], a, x0, x1, T());
            }
          }
        } else {   // 16-bit weights: this word and the next one form a step
          if (wi % 2 == 0) {
            const uint32_t a[4] = {wa, wb, (&wv[0][0].x)[wi + 1], (&wv[1][0].x)[wi + 1]};
            const int st = wi / 2;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const uint4 &xq = xv[n][st >> 1];
              const uint32_t x0 = (st & 1) ? xq.z : xq.x, x1 = (st & 1) ? xq.w : xq.y;
              mma16816(acc[m][n], a, x0, x1, T());
            }
          }
        }
      }
      if constexpr (GROUPED) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          acc[m][n][0] = fmaf(tmp[n][0], cs[0], acc[m][n][0]);
          acc[m][n][1] = fmaf(tmp[n][1], cs[0], acc[m][n][1]);
          acc[m][n][2] = fmaf(tmp[n][2], cs[1], acc[m][n][2]);
          acc[m][n][3] = fmaf(tmp[n][3], cs[1], acc[m][n][3]);
        }
      }
    }
  }
  cp_wait<0>();
  __syncwarp();   // the ring is free for the next job
}

// ---------------------------------------------------------------- router and sort

// One router unit: partial logits of token t over rows [m0, m0 + rows) of d.  The slice of the
// router weights (rows x E, contiguous in memory) and of x are copied into the warp's scratch
// with every 16-byte piece in flight at once, then lane l sums experts l, l + 32, ... from shared
// memory.
template <typename T>
__device__ void router_slice(const DLP &P, int t, int c, int lane, unsigned char *scratch) {
  const int rows = P.d / P.NCR, m0 = c * rows;
  const int wb = P.router_f32 ? 4 : 2;
  const int wbytes = rows * P.E * wb;   // a multiple of 16 (rows is a multiple of 8)
  const unsigned char *wsrc = static_cast<const unsigned char *>(P.wr) + int64_t(m0) * P.E * wb;
  const uint32_t sw = smem_u32(scratch), sx = sw + uint32_t(wbytes);
  for (int i = lane * 16; i < wbytes; i += 32 * 16) cp16_cg(sw + i, wsrc + i);
  const unsigned char *xsrc = reinterpret_cast<const unsigned char *>(P.x + int64_t(t) * P.d + m0);
  for (int i = lane * 16; i < rows * 2; i += 32 * 16) cp16_cg(sx + i, xsrc + i);
  cp_commit();
  cp_wait<0>();
  __syncwarp();
  const uint16_t *xs = reinterpret_cast<const uint16_t *>(scratch + wbytes);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (P.router_f32) {
    const float *ws = reinterpret_cast<const float *>(scratch);
#pragma unroll 4
    for (int m = 0; m < rows; ++m) {
      const float xm = h2f<T>(xs[m]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (e < P.E) acc[i] = fmaf(xm, ws[m * P.E + e], acc[i]);
      }
    }
  } else {
    const uint16_t *ws = reinterpret_cast<const uint16_t *>(scratch);
#pragma unroll 4
    for (int m = 0; m < rows; ++m) {
      const float xm = h2f<T>(xs[m]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (e < P.E) acc[i] = fmaf(xm, h2f<T>(ws[m * P.E + e]), acc[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e < P.E) P.rpart[(int64_t(t) * P.NCR + c) * P.E + e] = acc[i];
  }
  __syncwarp();   // the scratch is free again
}

// Stable counting sort of the R = T*k rows by expert id (one warp), expert offsets, the
// inverse permutation and the row-chunk table (chunks of at most 8 rows per expert).
__device__ void sort_rows(const DLP &P, int lane, int *sc) {
  int *cnt = sc, *off = sc + 256, *run = sc + 512, *rcs = sc + 768;
  const int E = P.E, R = P.T * P.k;
  for (int e = lane; e < 256; e += 32) {
    cnt[e] = 0;
    run[e] = 0;
  }
  int ide[8];   // R <= 256: every id loaded once, all loads in flight together
#pragma unroll
  for (int b = 0; b < 8; ++b) ide[b] = b * 32 + lane < R ? ldcg_i(P.ids + b * 32 + lane) : -1;
  __syncwarp();
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const int e = ide[b];
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(same) - 1) cnt[e] += __popc(same);
    __syncwarp();
  }
  // exclusive scans of the counts and of the chunk counts; lane owns experts 8 lane .. 8 lane + 7
  int c8[8], r8[8], sc_rows = 0, sc_rc = 0;
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
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const int f = b * 32 + lane;
    const int e = ide[b];
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = off[e] + run[e] + __popc(same & ((1u << lane) - 1u));
      P.perm[pos] = f;
      P.inv[f] = pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(same) - 1) run[e] += __popc(same);
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    if (e < E)
      for (int q = 0; q < r8[i]; ++q)
        P.rctab[rcs[e] + q] = make_int4(e, off[e] + 8 * q, min(8, c8[i] - 8 * q), 0);
  }
  if (lane == 0) P.ctrl[cRC] = total_rc;
}

// ---------------------------------------------------------------- the kernel

template <typename AT, bool GROUPED, int NTS>
__global__ void __launch_bounds__(kThr, 1) decode_layer_kernel(const DLP P) {
  extern __shared__ __align__(128) unsigned char dl_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WaitTab W;
  W.seen = reinterpret_cast<int *>(dl_smem + kW * kRing);
  W.poll = W.seen + fFc1 + P.rcmax;
  for (int i = threadIdx.x; i < 2 * (fFc1 + P.rcmax); i += kThr) W.seen[i] = 0;
  __syncthreads();
  const int g = lane >> 2, t4 = lane & 3;
  unsigned char *ring = dl_smem + warp * kRing;
  int *scratch = reinterpret_cast<int *>(ring);   // router / sort scratch (between jobs)
  int *ctrl = P.ctrl;
  const int T = P.T, d = P.d, F = P.F, E = P.E, k = P.k, R = T * k;
  const bool swiglu = P.act == MOE_ACT_SWIGLU;
  const int F1 = swiglu ? 2 * F : F;
  const int G1 = P.group == 0 ? 1 : d / 128, G2 = P.group == 0 ? 1 : F / 128;
  // units of each kind (routed ones depend on the row-chunk count RC, known after routing)
  const int Ur = T * P.NCR;
  const int Us1 = P.Fs > 0 ? P.Fs / 8 : 0;
  const int NG1 = swiglu ? F / 16 : F / 32;     // FC1 channel groups (two m-tiles each)
  const int NG2 = d / 32;                       // FC2 channel groups
  const int Us2 = P.Fs > 0 ? (d / 16) * P.S3 : 0;
  const int NCB = (d + kCombCols - 1) / kCombCols;
  const int Uc = T * NCB;
  int RC = -1;

  const int qw = warp % kQ;   // this warp's queue
  auto grab = [&]() -> int {
    int i = 0;
    if (lane == 0) i = atomicAdd(ctrl + cGrab + kLine * qw, 1);
    return qw + kQ * i;   // lane 0's value; broadcast by the caller when needed
  };
  int pending = grab();
  for (;;) {
    int u = __shfl_sync(0xffffffffu, pending, 0);
    pending = grab();   // the next unit, fetched while this one runs
    // ---------------------------------------------------------- router
    if (u < Ur) {
      const int t = u / P.NCR, c = u % P.NCR;
      router_slice<AT>(P, t, c, lane, ring);
      if (publish_add(ctrl + cTok + t, 1, lane) != P.NCR - 1) continue;
      // last slice of token t: logits in slice order (+ bias), top-k, softmax
      float *lg = reinterpret_cast<float *>(scratch);
      for (int e = lane; e < E; e += 32) {   // slices summed in order, eight loads in flight
        float v = 0.f;
        for (int c0 = 0; c0 < P.NCR; c0 += 8) {
          float q[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) q[u] = c0 + u < P.NCR ? ldcg_f(P.rpart + (int64_t(t) * P.NCR + c0 + u) * E + e) : 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) v += q[u];
        }
        lg[e] = v + (P.bias ? P.bias[e] : 0.f);
      }
      __syncwarp();
      topk_softmax_warp(lg, E, k, P.renorm, P.ids + t * k, P.gate + t * k);
      if (publish_add(ctrl + cRouteTok, 1, lane) != T - 1) continue;
      // last token: sort the rows by expert and publish the tables
      sort_rows(P, lane, scratch);
      fence_acq_rel();
      __syncwarp();
      if (lane == 0) st_release(ctrl + cReady, 1);
      continue;
    }
    u -= Ur;
    // ---------------------------------------------------------- shared FC1 (x only)
    if (u < Us1) {
      const uint16_t *xrow[NTS];
#pragma unroll
      for (int n = 0; n < NTS; ++n) xrow[n] = n * 8 + g < T ? P.x + int64_t(n * 8 + g) * d : nullptr;
      Job J{P.wsgu, d / 8, nullptr, 2 * P.Fs, u, true, P.Fs, 0, d / 128};
      float acc[1][NTS][4];
      stream_job<AT, 16, NTS, 1, false>(J, xrow, ring, lane, acc);
      const int hch = u * 8 + g;
#pragma unroll
      for (int n = 0; n < NTS; ++n)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = n * 8 + 2 * t4 + q;
          if (row < T) P.hs[int64_t(row) * P.Fs + hch] = f2h<AT>(act_silu(acc[0][n][q]) * acc[0][n][2 + q]);
        }
      publish_add(ctrl + cSh1 + kLine * qw, 1, lane);
      continue;
    }
    u -= Us1;
    // everything below reads the routing tables
    if (RC < 0) {
      if (!wait_geq(P, W, fReady, ctrl + cReady, 1, 1, kErrRoute, lane)) break;
      RC = ldcg_i(ctrl + cRC);
    }
    const int Uf1 = RC * NG1, Uf2 = RC * NG2 * P.S2;
    // ---------------------------------------------------------- routed FC1 (+ activation)
    if (u < Uf1) {
      const int rc = u / NG1, grp = u % NG1;
      const int4 ch = __ldcg(P.rctab + rc);   // (expert, first row, rows)
      const int e = ch.x, row0 = ch.y, nrows = ch.z;
      const uint16_t *xrow[1];
      xrow[0] = nullptr;
      if (g < nrows) xrow[0] = P.x + int64_t(ldcg_i(P.perm + row0 + g) / k) * d;
      Job J{P.w1 + int64_t(e) * F1 * (d / 32), d / 32, P.s1 + int64_t(e) * G1 * F1, F1, grp, swiglu, F, 0, d / 128};
      float acc[2][1][4];
      stream_job<AT, 4, 1, 2, GROUPED>(J, xrow, ring, lane, acc);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int c0 = chan_of<2>(grp, m, g, swiglu, F), c1 = chan_of<2>(grp, m, g + 8, swiglu, F);
        float sc0 = 1.f, sc1 = 1.f;
        if (!GROUPED) {
          sc0 = h2f<AT>(P.s1[int64_t(e) * F1 + c0]);
          sc1 = h2f<AT>(P.s1[int64_t(e) * F1 + c1]);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = 2 * t4 + q;
          if (row < nrows) {
            uint16_t *hr = P.h + int64_t(row0 + row) * F;
            const float v0 = acc[m][0][q] * sc0, v1 = acc[m][0][2 + q] * sc1;
            if (swiglu) {
              hr[(grp * 2 + m) * 8 + g] = f2h<AT>(act_silu(v0) * v1);
            } else {
              hr[c0] = f2h<AT>(act_apply(v0, P.act));
              hr[c1] = f2h<AT>(act_apply(v1, P.act));
            }
          }
        }
      }
      publish_add(ctrl + cFc1 + kFc1Stride * rc, 1, lane);
      continue;
    }
    u -= Uf1;
    // ---------------------------------------------------------- routed FC2 (fp32 split partials)
    if (u < Uf2) {
      const int rc = u / (NG2 * P.S2), rem = u % (NG2 * P.S2);
      const int s2 = rem / NG2, grp = rem % NG2;
      if (!wait_geq(P, W, fFc1 + rc, ctrl + cFc1 + kFc1Stride * rc, 1, NG1, kErrFc1, lane)) break;
      const int4 ch = __ldcg(P.rctab + rc);
      const int e = ch.x, row0 = ch.y, nrows = ch.z;
      const uint16_t *xrow[1];
      xrow[0] = g < nrows ? P.h + int64_t(row0 + g) * F : nullptr;
      Job J{P.w2 + int64_t(e) * d * (F / 32), F / 32, P.s2 + int64_t(e) * G2 * d, d, grp, false, 0, s2 * P.CH2, P.CH2};
      float acc[2][1][4];
      stream_job<AT, 4, 1, 2, GROUPED>(J, xrow, ring, lane, acc);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int c0 = (grp * 2 + m) * 16 + g, c1 = c0 + 8;
        float sc0 = 1.f, sc1 = 1.f;
        if (!GROUPED) {
          sc0 = h2f<AT>(P.s2[int64_t(e) * d + c0]);
          sc1 = h2f<AT>(P.s2[int64_t(e) * d + c1]);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = 2 * t4 + q;
          if (row < nrows) {
            float *yr = P.ypart + (int64_t(s2) * R + row0 + row) * d;
            yr[c0] = acc[m][0][q] * sc0;
            yr[c1] = acc[m][0][2 + q] * sc1;
          }
        }
      }
      publish_add(ctrl + cFc2 + kLine * qw, 1, lane);
      continue;
    }
    u -= Uf2;
    // ---------------------------------------------------------- shared FC2 (fp32 split partials)
    if (u < Us2) {
      const int s3 = u / (d / 16), grp = u % (d / 16);
      if (!wait_geq(P, W, fSh1, ctrl + cSh1, kQ, Us1, kErrSh1, lane)) break;
      const uint16_t *xrow[NTS];
#pragma unroll
      for (int n = 0; n < NTS; ++n) xrow[n] = n * 8 + g < T ? P.hs + int64_t(n * 8 + g) * P.Fs : nullptr;
      Job J{P.wsd, P.Fs / 8, nullptr, d, grp, false, 0, s3 * P.CH3, P.CH3};
      float acc[1][NTS][4];
      stream_job<AT, 16, NTS, 1, false>(J, xrow, ring, lane, acc);
      const int c0 = grp * 16 + g, c1 = c0 + 8;
#pragma unroll
      for (int n = 0; n < NTS; ++n)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = n * 8 + 2 * t4 + q;
          if (row < T) {
            float *yr = P.yspart + (int64_t(s3) * T + row) * d;
            yr[c0] = acc[0][n][q];
            yr[c1] = acc[0][n][2 + q];
          }
        }
      publish_add(ctrl + cSh2 + kLine * qw, 1, lane);
      continue;
    }
    u -= Us2;
    // ---------------------------------------------------------- combine
    if (u < Uc) {
      if (!wait_geq(P, W, fFc2, ctrl + cFc2, kQ, Uf2, kErrFc2, lane)) break;
      if (Us2 > 0 && !wait_geq(P, W, fSh2, ctrl + cSh2, kQ, Us2, kErrFc2, lane)) break;
      const int t = u / NCB, cb = u % NCB;
      const int c = cb * kCombCols + lane * 8;
      if (c < d) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = 0.f;
        for (int j = 0; j < k; ++j) {   // entries in j order, split slices in split order
          const int p = ldcg_i(P.inv + t * k + j);
          const float gw = ldcg_f(P.gate + t * k + j);
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
      continue;
    }
    break;   // past the last unit
  }
  // leave: one count per block; the last block's warp 0 resets the control words for the next
  // launch
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (threadIdx.x == 0) s_last = atomicAdd(ctrl + cExit, 1) == int(gridDim.x) - 1;
  __syncthreads();
  const int last = s_last && warp == 0;
  if (last) {
    __threadfence();
    for (int i = lane; i < cFc1; i += 32) ctrl[i] = 0;
    for (int rc = lane; rc < P.rcmax; rc += 32) ctrl[cFc1 + kFc1Stride * rc] = 0;
    __threadfence();
  }
}

}  // namespace

// ---------------------------------------------------------------- host side

// Whether one launch can run this layer, and how it is cut.  `warps` is the number of warps
// the launch has (units of the later stages are cut to at least that many where the shape
// allows).
DecodePlan plan_decode(const moe_layer_desc *ds, int64_t T, int64_t warps) {
  DecodePlan p{};
  const int64_t R = T * ds->k;
  p.ok = T >= 1 && T <= 32 && ds->bits == 4 && ds->E <= 256 && R <= 256 && ds->d % 128 == 0 && ds->F % 128 == 0 &&
         (ds->Fs == 0 || ds->Fs % 128 == 0) && ds->d >= kRouteRows && (ds->router_dtype == MOE_F32 || ds->router_dtype == ds->dtype);
  if (!p.ok) return p;
  p.nts = T <= 8 ? 1 : (T <= 16 ? 2 : 4);
  // router slice: rows x E weights and rows of x in the warp's scratch (rows a power of two,
  // at least 8 so that every slice is whole 16-byte pieces)
  const int64_t wb = ds->router_dtype == MOE_F32 ? 4 : 2;
  int64_t rows = kRouteRows;
  while (rows > 8 && rows * (ds->E * wb + 2) > kRing) rows /= 2;
  p.NCR = int(ds->d / rows);
  // row chunks: at most one ragged chunk per active expert plus R / 8 full ones
  p.rcmax = int(std::min<int64_t>(ds->E, R) + cdiv(R, 8));
  // routed FC2: split K so that the units outnumber the warps (routing estimated uniform)
  const double er = double(ds->E);
  const double active = std::max(1.0, er * (1.0 - std::pow(1.0 - 1.0 / er, double(R))));
  const double rc_est = std::max(active, double(R) / 8.0);
  const int nck2 = int(ds->F / 128);
  p.S2 = 1;
  for (int s = 1; s <= nck2; ++s) {   // units of at least 4 chunks (fewer only if K is that short)
    if (nck2 % s || (nck2 / s < 4 && s > 1)) continue;
    p.S2 = s;
    if (rc_est * double(ds->d / 32) * s >= double(warps)) break;
  }
  p.CH2 = nck2 / p.S2;
  p.S3 = 1;
  p.CH3 = 1;
  if (ds->Fs > 0) {
    const int nck3 = int(ds->Fs / 128);
    for (int s = 1; s <= nck3; ++s) {
      if (nck3 % s || (nck3 / s < 4 && s > 1)) continue;
      p.S3 = s;
      if (double(ds->d / 16) * s >= double(warps)) break;
    }
    p.CH3 = nck3 / p.S3;
  }
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t at = o;
    o += align256(b);
    return at;
  };
  p.o_rpart = take(size_t(T) * p.NCR * ds->E * 4);
  p.o_ypart = take(size_t(p.S2) * R * ds->d * 4);
  p.o_hs = take(size_t(T) * ds->Fs * 2);
  p.o_yspart = take(ds->Fs > 0 ? size_t(p.S3) * T * ds->d * 4 : 0);
  p.o_rctab = take(size_t(p.rcmax) * 16);
  p.o_ctrl = take(size_t(cFc1 + kFc1Stride * p.rcmax) * 4);
  p.bytes = o;
  return p;
}

int decode_warps() { return num_sms() * kW; }

// Enqueue the one-launch decode layer.  `fused` points at the plan's region of the workspace;
// ids..h are the regular layer buffers.  zero_ctrl: clear the control words first (they are
// left zero by every launch that completes; a first launch on a workspace needs the clear).
int launch_decode_layer(const moe_layer_desc *ds, const moe_layer_weights *w, const void *x, int64_t T, void *out,
                        int32_t *ids, float *gate, int32_t *offs, int32_t *perm, int32_t *inv, void *h, char *fused,
                        const DecodePlan &pl, bool zero_ctrl, cudaStream_t st) {
  DLP P{};
  P.x = static_cast<const uint16_t *>(x);
  P.wr = w->w_router;
  P.bias = w->router_bias;
  const int64_t d = ds->d, F = ds->F, E = ds->E;
  const int64_t F1 = ds->act == MOE_ACT_SWIGLU ? 2 * F : F;
  P.w1 = static_cast<const uint4 *>(w->w1);
  P.s1 = reinterpret_cast<const uint16_t *>(static_cast<const char *>(w->w1) + moe_packed_scale_offset(E, d, F1, 4));
  P.w2 = static_cast<const uint4 *>(w->w2);
  P.s2 = reinterpret_cast<const uint16_t *>(static_cast<const char *>(w->w2) + moe_packed_scale_offset(E, F, d, 4));
  P.wsgu = static_cast<const uint4 *>(w->ws_gate_up);
  P.wsd = static_cast<const uint4 *>(w->ws_down);
  P.out = out;
  P.ids = ids;
  P.gate = gate;
  P.offsets = offs;
  P.perm = perm;
  P.inv = inv;
  P.h = static_cast<uint16_t *>(h);
  P.rpart = reinterpret_cast<float *>(fused + pl.o_rpart);
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
  P.Fs = int(ds->Fs);
  P.act = ds->act;
  P.group = ds->group;
  P.renorm = ds->renormalize;
  P.router_f32 = ds->router_dtype == MOE_F32 ? 1 : 0;
  P.NCR = pl.NCR;
  P.S2 = pl.S2;
  P.CH2 = pl.CH2;
  P.S3 = pl.S3;
  P.CH3 = pl.CH3;
  P.rcmax = pl.rcmax;
  if (zero_ctrl && cudaMemsetAsync(P.ctrl, 0, size_t(cFc1 + kFc1Stride * pl.rcmax) * 4, st) != cudaSuccess)
    return check_launch("decode layer: clear control words");
  using KFn = void (*)(DLP);
  KFn fn = nullptr;
  const bool bf = ds->dtype == MOE_BF16, grouped = ds->group != 0;
#define MOE_DL(TT, GG, NN) \
  if ((std::is_same<TT, __nv_bfloat16>::value == bf) && grouped == GG && pl.nts == NN) fn = decode_layer_kernel<TT, GG, NN>;
  MOE_DL(__half, false, 1) MOE_DL(__half, false, 2) MOE_DL(__half, false, 4)
  MOE_DL(__half, true, 1) MOE_DL(__half, true, 2) MOE_DL(__half, true, 4)
  MOE_DL(__nv_bfloat16, false, 1) MOE_DL(__nv_bfloat16, false, 2) MOE_DL(__nv_bfloat16, false, 4)
  MOE_DL(__nv_bfloat16, true, 1) MOE_DL(__nv_bfloat16, true, 2) MOE_DL(__nv_bfloat16, true, 4)
#undef MOE_DL
  if (fn == nullptr) return set_error(MOE_ERR_UNSUPPORTED, "decode layer: no kernel instance");
  const size_t smem = size_t(kW) * kRing + size_t(2 * (fFc1 + pl.rcmax)) * 4;
  // the shared-memory opt-in is a per-device attribute of each instance: set it every time
  // (cheap) rather than caching it per instance and device
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return check_launch("decode layer: shared-memory attribute");
  fn<<<num_sms(), kThr, smem, st>>>(P);
  return check_launch("decode layer");
}

}  // namespace moe
