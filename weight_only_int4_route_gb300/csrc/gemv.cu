// Grouped GEMM for decode-sized batches (a few routed rows per expert): a weight stream.
//
// "Who Says Elephants Can't Run", section 3: grouped GEMM over every expert in one launch with
// the dequantization fused (optimized I2F, interleaved INT4 word); Figure 1: experts without rows
// load nothing.  "Specter", method step 5 and technical novelty: the rows of one expert are
// gathered so the per-token GEMVs over fine-grained expert matrices become one small GEMM.
//
// With at most a few rows per expert the layer reads each weight once and does ~2 FLOPs per row
// with it, so the kernel is a stream over the weights at HBM speed.  Mapping of the warp MMA
// m16n8k16: the weights fill M (16 output channels per m-tile: for SwiGLU 8 gate channels and
// the 8 matching up channels, so the D fragment of one thread holds a gate/up pair), the routed
// rows fill N (8 per n-tile).  A lane (g = lane/4, t = lane%4) takes the 32 consecutive reduction
// indices [32t, 32t+32) of each 128-wide chunk for channels g and g+8 -- 16 bytes each for INT4 --
// and MMA step s (0..7) of the chunk takes reduction indices 32t + 4s + {0,1,2,3} from lane t (the
// MMA's K order is free as long as both operands agree), so its A registers are exactly the lane's
// dequantized pairs and its B registers 8 bytes of the activation row.
//
// Work unit = (expert row chunk, channel group of MT m-tiles, K split).  Every warp walks its own
// sequence of units with no block-level synchronization.  The warp streams the unit's weight,
// activation and scale bytes with cp.async into its own ring of kDepth chunk slots in shared
// memory and reads them back right before the MMAs; the ring holds the bytes in flight without
// holding registers.  Weight rows are copied warp-wide (consecutive lanes take consecutive
// 16-byte pieces of a row, so every request fills whole sectors) and read by other lanes, so a
// step waits for the lane's own copy group and then for the whole warp (__syncwarp).  K splits
// write fp32 partial sums that are summed later in split order.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

MOE_DEFINE_CHECK_WORD(gemv)

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxE = 256;

// Shared memory of one chunk slot of a warp: weights row by row (row = one of the unit's 16 * MT
// channels, 16 * BITS bytes of it per chunk, padded when that keeps the lanes' reads apart), the
// activation pieces lane by lane, and the unit's scale rows for the chunk.
template <int BITS, int NT, int MT> struct GV {
  static constexpr int kVec = BITS / 4;                      // 16-byte pieces per channel per lane
  static constexpr int kRows = 16 * MT;                      // weight rows per unit
  static constexpr int kRowBytes = 16 * BITS;                // bytes of one row per chunk
  static constexpr int kRowStride = kRowBytes + (BITS == 4 ? 0 : 16);
  // A quarter-warp reads the same pieces of two adjacent rows: 64-byte INT4 rows put them on
  // different banks as they are, the 16 bytes of padding do it for 8- and 16-bit rows.  Copies
  // write whole rows, kRowsPerCopy of them per warp-wide copy.
  static constexpr int kWPieces = kRows * kRowBytes / 16 / 32;   // pieces a lane copies per chunk
  static constexpr int kPiecesPerRow = kRowBytes / 16;
  static constexpr int kRowsPerCopy = 32 / kPiecesPerRow;          // rows one warp-wide copy covers
  static constexpr int kXOff = kRows * kRowStride;
  static constexpr int kSOff = kXOff + NT * 4 * 512;
  static constexpr int kScaleLanes = MT * 2;                 // 16-byte scale pieces per chunk
  static constexpr int kSlotBytes = (kSOff + kScaleLanes * 16 + 127) / 128 * 128;
  // ring depth: the one that fits the most warps per SM (228 KB of shared memory, 1 KB of it
  // reserved per block), then the deeper one
  static constexpr int kStatic = (2 * (kMaxE + 1) + 32) * 4 + 1024;
  static constexpr int blocks(int d) { return 233472 / (kWarps * d * kSlotBytes + kStatic); }
  static constexpr int score(int d) { return blocks(d) * 16 + d; }
  static constexpr int kDepth = score(4) > score(3) ? 4 : 3;
  static constexpr int kWarpBytes = kDepth * kSlotBytes;
  static constexpr int kSmem = kWarps * kWarpBytes;
};

struct GvParams {
  const uint16_t *a;
  const uint4 *w;
  const uint16_t *scales;
  const int32_t *offsets;
  void *out;
  float *partial;
  int R, E, K, N;
  int group, act, out_dtype;
  int swiglu, partial_mode;
  int S, CH;   // K splits, 128-wide chunks per split
  int NG;      // channel groups (16 * MT channels each)
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// weights: read once, cached in L2 only, with the neighbouring 128 bytes fetched along
__device__ __forceinline__ void cp_w16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
// activations and scales: shared by the warps of a block, cached in L1; zero-filled when
// src_bytes == 0
__device__ __forceinline__ void cp_x16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// Shared-memory reads are plain loads: the compiler keeps them after the cp.async wait and the
// warp barrier (both order memory) but may start them early among the MMAs.
__device__ __forceinline__ uint4 lds16(const unsigned char *a) { return *reinterpret_cast<const uint4 *>(a); }
__device__ __forceinline__ uint32_t lds_u16(const unsigned char *a) {
  return *reinterpret_cast<const uint16_t *>(a);
}

__device__ __forceinline__ void st_dt(void *o, int dt, int64_t i, float v) {
  if (dt == MOE_F32) static_cast<float *>(o)[i] = v;
  else if (dt == MOE_F16) static_cast<__half *>(o)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16 *>(o)[i] = __float2bfloat16_rn(v);
}

template <typename T> __device__ __forceinline__ float u16_to_f32(uint32_t b) {
  if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half(uint16_t(b)));
  else return __bfloat162float(__ushort_as_bfloat16(uint16_t(b)));
}

struct Unit {
  int e, row0, nrows, grp, s;
};

// A warp's units are u = wid, wid + wstride, wid + 2 wstride, ...; unit u is, from the fastest
// digit, (channel group, K split, row chunk) -- consecutive warps of a block share the row chunk
// and K split, so they read the same activation slice -- and row chunk rc belongs to the expert
// whose chunk range holds it.  The cursor keeps u's digits and steps them by wstride's digits,
// so no division runs per unit; the expert of a row chunk is found by binary search from the
// previous one (row chunks only grow along the sequence).
struct Cursor {
  int grp, s, rc, e;
};
struct Stride {
  int grp, s, rc;
};

__device__ __forceinline__ int expert_of(int rc, int lo, int E, const int *s_rcstart) {
  int hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_rcstart[mid] <= rc) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ void cursor_step(Cursor &c, const Stride &d, const GvParams &p, const int *s_rcstart) {
  c.grp += d.grp;
  int carry = c.grp >= p.NG;
  if (carry) c.grp -= p.NG;
  c.s += d.s + carry;
  carry = c.s >= p.S;
  if (carry) c.s -= p.S;
  c.rc += d.rc + carry;
  c.e = expert_of(c.rc, c.e, p.E, s_rcstart);
}
template <int NT>
__device__ __forceinline__ Unit unit_of(const Cursor &c, const int *s_rcstart, const int *s_off) {
  Unit x;
  x.e = c.e;
  x.grp = c.grp;
  x.s = c.s;
  x.row0 = s_off[c.e] + (c.rc - s_rcstart[c.e]) * (8 * NT);
  x.nrows = min(8 * NT, s_off[c.e + 1] - x.row0);
  return x;
}

// GROUPED: one scale per 128-wide reduction chunk (applied to the chunk's fp32 sum); otherwise
// per-channel scales (applied at the end) or none (16-bit weights).
template <typename T, int BITS, int NT, int MT, bool GROUPED>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GvParams p) {
  pdl_enter();   // see launch_pdl
  using C = GV<BITS, NT, MT>;
  constexpr int kVec = C::kVec, kDepth = C::kDepth;
  extern __shared__ __align__(128) unsigned char gv_ring[];
  __shared__ int s_rcstart[kMaxE + 1];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int scratch[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int E = p.E;

  // row chunks per expert and their exclusive prefix (each thread takes two consecutive experts)
  int cnt[2] = {0, 0};
  // checked build: unusable offsets leave the kernel without units (nothing is read or written)
  const bool off_ok = p.offsets == nullptr || offsets_usable(p.offsets, E, p.R, [] { check_fail(kCheckOffsets); });
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int e = 2 * tid + q;
    if (e < E && off_ok) {
      const int o0 = p.offsets ? p.offsets[e] : 0;
      const int o1 = p.offsets ? p.offsets[e + 1] : p.R;
      cnt[q] = (o1 - o0 + 8 * NT - 1) / (8 * NT);
      s_off[e] = o0;
      if (e == E - 1) s_off[E] = o1;
    }
  }
  int start = 0;
  const int total_rc = block_exclusive_scan(cnt[0] + cnt[1], &start, scratch);
  if (2 * tid < E) s_rcstart[2 * tid] = start;
  if (2 * tid + 1 < E) s_rcstart[2 * tid + 1] = start + cnt[0];
  __syncthreads();

  const int U = total_rc * p.NG * p.S;
  const int wid = blockIdx.x * kWarps + warp;
  const int wstride = gridDim.x * kWarps;
  const int nunits = wid < U ? (U - wid + wstride - 1) / wstride : 0;   // units of this warp
  const int nsteps = nunits * p.CH;
  if (nsteps == 0) return;
  const int64_t w_row_vec = int64_t(p.K) * BITS / 128;   // 16-byte pieces per channel row
  const int G = p.group == 0 ? 1 : p.K / p.group;
  constexpr bool grouped = GROUPED;
  constexpr bool per_channel = !GROUPED && BITS != 16;
  const int F = p.N >> 1;
  const uint32_t wring = smem_u32(gv_ring) + warp * C::kWarpBytes;
  const unsigned char *rring = gv_ring + warp * C::kWarpBytes;   // the same ring, for reads
  // this lane's weight reads: row g (+ 8 h + 16 m), pieces from t * kVec
  const uint32_t wlane = g * C::kRowStride + t * kVec * 16;

  // output channel of m-tile m, A row r (0..15), channel group grp
  auto channel = [&](int grp, int m, int r) -> int {
    if (p.swiglu) return r < 8 ? (grp * MT + m) * 8 + r : F + (grp * MT + m) * 8 + (r - 8);
    return (grp * MT + m) * 16 + r;
  };

  // ---- copy side.  Copy v of a step moves C::kRowsPerCopy whole weight rows (consecutive lanes
  // take consecutive 16-byte pieces of a row, so every request fills whole sectors); lane i takes
  // piece i % kPiecesPerRow of row v * kRowsPerCopy + i / kPiecesPerRow.  Each lane also copies its own
  // activation pieces (row g of each n-tile, reduction indices [32t, 32t+32)), and lanes below
  // kScaleLanes one 16-byte piece of the scale rows.
  const int wrow = lane / C::kPiecesPerRow;   // row of copy 0; copy v adds v * kRowsPerCopy
  const int wpart = lane % C::kPiecesPerRow;
  Stride dstep;
  Cursor icur, ccur;   // issue side and compute side
  {
    dstep.grp = wstride % p.NG;
    dstep.s = (wstride / p.NG) % p.S;
    dstep.rc = wstride / (p.NG * p.S);
    icur.grp = wid % p.NG;
    icur.s = (wid / p.NG) % p.S;
    icur.rc = wid / (p.NG * p.S);
    icur.e = expert_of(icur.rc, 0, E, s_rcstart);
    ccur = icur;
  }
  int iu = 0, ic = 0;
  const uint4 *wbase = nullptr;   // the unit's expert and K range; rows at woff[v] pieces from it
  int woff[C::kWPieces];
  const uint4 *ssrc = nullptr;
  const uint4 *xsrc[NT];
  int xbytes[NT];
  auto load_unit = [&]() {
    const Unit x = unit_of<NT>(icur, s_rcstart, s_off);
    const int kc0 = x.s * p.CH;
    wbase = p.w + int64_t(x.e) * p.N * w_row_vec + int64_t(kc0) * BITS + wpart;
#pragma unroll
    for (int v = 0; v < C::kWPieces; ++v) {
      const int r = v * C::kRowsPerCopy + wrow;
      woff[v] = channel(x.grp, r / 16, r % 16) * int(w_row_vec);
    }
    if (grouped && lane < C::kScaleLanes) {   // piece q: the 8 channels of A rows 8 (q % 2) .. of m-tile q / 2
      const int c0 = channel(x.grp, lane >> 1, 8 * (lane & 1));
      ssrc = reinterpret_cast<const uint4 *>(p.scales + (int64_t(x.e) * G + kc0) * p.N + c0);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int row = n * 8 + g;
      const bool ok = row < x.nrows;
      xsrc[n] = reinterpret_cast<const uint4 *>(p.a + int64_t(x.row0 + (ok ? row : 0)) * p.K + kc0 * 128 + 32 * t);
      xbytes[n] = ok ? 16 : 0;
    }
  };
  auto issue = [&](int slot) {
    const uint32_t sb = wring + slot * C::kSlotBytes;
#pragma unroll
    for (int v = 0; v < C::kWPieces; ++v) {
      const int r = v * C::kRowsPerCopy + wrow;
      cp_w16(sb + r * C::kRowStride + wpart * 16, wbase + (woff[v] + ic * BITS));
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int v = 0; v < 4; ++v)
        cp_x16(sb + C::kXOff + (n * 4 + v) * 512 + lane * 16, xsrc[n] + ic * 16 + v, xbytes[n]);
    if (grouped && lane < C::kScaleLanes)
      cp_x16(sb + C::kSOff + lane * 16, reinterpret_cast<const uint16_t *>(ssrc) + int64_t(ic) * p.N, 16);
    if (++ic == p.CH) {
      ic = 0;
      if (++iu < nunits) {
        cursor_step(icur, dstep, p, s_rcstart);
        load_unit();
      }
    }
  };

  load_unit();
#pragma unroll
  for (int d = 0; d < kDepth - 1; ++d) {
    if (d < nsteps) issue(d);
    cp_commit();
  }

  float acc[MT][NT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][n][i] = 0.f;

  int cu = 0, cc = 0, slot = 0, fill = kDepth - 1;
  for (int j = 0; j < nsteps; ++j) {
    cp_wait<kDepth - 2>();   // this lane's copies of step j have landed
    __syncwarp();            // ... and every lane's; every lane is done reading the slot of step j-1
    if (j + kDepth - 1 < nsteps) issue(fill);   // step j + kDepth - 1 into the slot of step j - 1
    cp_commit();
    fill = fill + 1 == kDepth ? 0 : fill + 1;

    const unsigned char *sb = rring + slot * C::kSlotBytes;
    slot = slot + 1 == kDepth ? 0 : slot + 1;
    uint4 xv[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int v = 0; v < 4; ++v) xv[n][v] = lds16(sb + C::kXOff + (n * 4 + v) * 512 + lane * 16);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float cs[2] = {1.f, 1.f};
      if constexpr (grouped) {
#pragma unroll
        for (int h = 0; h < 2; ++h) cs[h] = u16_to_f32<T>(lds_u16(sb + C::kSOff + (m * 2 + h) * 16 + 2 * g));
      }
      uint4 wv[2][kVec];   // channel g (h = 0) and g + 8 (h = 1): reduction indices [32t, 32t+32)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int v = 0; v < kVec; ++v)
          wv[h][v] = lds16(sb + (m * 16 + 8 * h) * C::kRowStride + wlane + v * 16);
      float tmp[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) tmp[n][i] = 0.f;
      // each 32-bit word of the lane's weights holds the pairs of 2 (INT4) or 1 (INT8) MMA steps;
      // it is converted once and feeds those steps
      constexpr int kWords = 4 * kVec;
      constexpr int kStepsPerWord = 8 / kWords;
#pragma unroll
      for (int wi = 0; wi < kWords; ++wi) {
        const uint32_t wa = (&wv[0][0].x)[wi], wb = (&wv[1][0].x)[wi];
        uint32_t ha[2 * kStepsPerWord > 0 ? 2 * kStepsPerWord : 1], hb[2 * kStepsPerWord > 0 ? 2 * kStepsPerWord : 1];
        if constexpr (BITS == 4) {
          uint32_t qa[4], qb[4];
          i2f_int4(wa, qa, T());
          i2f_int4(wb, qb, T());
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            ha[q] = qa[q];
            hb[q] = qb[q];
          }
        } else if constexpr (BITS == 8) {
          i2f_int8(wa, ha, T());
          i2f_int8(wb, hb, T());
        }
#pragma unroll
        for (int k = 0; k < (BITS == 16 ? 1 : kStepsPerWord); ++k) {
          uint32_t a[4];
          if constexpr (BITS == 16) {   // two words per step: this word and the next one
            if (wi % 2) continue;
            a[0] = wa;
            a[1] = wb;
            a[2] = (&wv[0][0].x)[wi + 1];
            a[3] = (&wv[1][0].x)[wi + 1];
          } else {
            a[0] = ha[2 * k];
            a[1] = hb[2 * k];
            a[2] = ha[2 * k + 1];
            a[3] = hb[2 * k + 1];
          }
          const int st = BITS == 16 ? wi / 2 : wi * kStepsPerWord + k;   // MMA step 0..7
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const uint4 &xq = xv[n][st >> 1];
            const uint32_t x0 = (st & 1) ? xq.z : xq.x;
            const uint32_t x1 = (st & 1) ? xq.w : xq.y;
            if constexpr (grouped) mma16816(tmp[n], a, x0, x1, T());
            else mma16816(acc[m][n], a, x0, x1, T());
          }
        }
      }
      if constexpr (grouped) {   // group-128 scale on the chunk's fp32 sum: s * sum(x q) (channel g | g+8)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          acc[m][n][0] = fmaf(tmp[n][0], cs[0], acc[m][n][0]);
          acc[m][n][1] = fmaf(tmp[n][1], cs[0], acc[m][n][1]);
          acc[m][n][2] = fmaf(tmp[n][2], cs[1], acc[m][n][2]);
          acc[m][n][3] = fmaf(tmp[n][3], cs[1], acc[m][n][3]);
        }
      }
    }

    if (++cc == p.CH) {   // unit finished: write its outputs
      cc = 0;
      const Unit x = unit_of<NT>(ccur, s_rcstart, s_off);
      if (++cu < nunits) cursor_step(ccur, dstep, p, s_rcstart);
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int row = n * 8 + 2 * t + q;
            if (row < x.nrows) {
              const int64_t grow = x.row0 + row;
              float v0 = acc[m][n][q], v1 = acc[m][n][2 + q];   // channel g, channel g + 8
              const int ch0 = channel(x.grp, m, g), ch1 = channel(x.grp, m, g + 8);
              if constexpr (per_channel) {
                v0 *= u16_to_f32<T>(p.scales[int64_t(x.e) * p.N + ch0]);
                v1 *= u16_to_f32<T>(p.scales[int64_t(x.e) * p.N + ch1]);
              }
              if (p.partial_mode) {
                float *pp = p.partial + (int64_t(x.s) * p.R + grow) * p.N;
                pp[ch0] = v0;
                pp[ch1] = v1;
              } else if (p.swiglu) {
                st_dt(p.out, p.out_dtype, grow * F + ch0, act_silu(v0) * v1);
              } else {
                st_dt(p.out, p.out_dtype, grow * p.N + ch0, act_apply(v0, p.act));
                st_dt(p.out, p.out_dtype, grow * p.N + ch1, act_apply(v1, p.act));
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[m][n][i] = 0.f;
        }
    }
  }
  cp_wait<0>();
}

using KernelFn = void (*)(GvParams);

template <typename T, int BITS, int NT, int MT, bool G> KernelFn kernel_of() { return gemv_kernel<T, BITS, NT, MT, G>; }

template <int BITS, int NT, int MT> constexpr int smem_of() { return GV<BITS, NT, MT>::kSmem; }

struct Inst {
  KernelFn fn;
  int smem;
};

// Instances: 4- and 8-bit weights take two m-tiles per unit (N is a multiple of 64, so the
// channel count always splits that way), 16-bit weights one.
template <typename T> Inst pick_t(int bits, int nt, int mt, bool grouped) {
#define MOE_GV(B, N_, M_, G_)                                            \
  if (bits == B && nt == N_ && mt == M_ && grouped == G_)                \
    return Inst{kernel_of<T, B, N_, M_, G_>(), smem_of<B, N_, M_>()};
  MOE_GV(4, 1, 2, true) MOE_GV(4, 2, 2, true) MOE_GV(4, 1, 2, false) MOE_GV(4, 2, 2, false)
  MOE_GV(4, 1, 4, true) MOE_GV(4, 2, 4, true) MOE_GV(4, 1, 4, false) MOE_GV(4, 2, 4, false)
  MOE_GV(8, 1, 2, true) MOE_GV(8, 2, 2, true) MOE_GV(8, 1, 2, false) MOE_GV(8, 2, 2, false)
  MOE_GV(16, 1, 1, false) MOE_GV(16, 2, 1, false)
#undef MOE_GV
  return Inst{nullptr, 0};
}
Inst pick(bool bf, int bits, int nt, int mt, bool grouped) {
  return bf ? pick_t<__nv_bfloat16>(bits, nt, mt, grouped) : pick_t<__half>(bits, nt, mt, grouped);
}

// Resident blocks per SM of one instance (the dynamic shared memory opt-in, a per-device
// attribute of the kernel, is set on the way); computed once per instance and device.
int blocks_per_sm(bool bf, int bits, int nt, int mt, bool grouped) {
  static std::mutex mu;
  static int cache[64][2][3][2][4][2] = {};
  if (nt < 1 || nt > 2 || mt < 1 || mt > 4) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();   // the launch then reports the problem
    return 1;
  }
  const int bi = bits == 4 ? 0 : (bits == 8 ? 1 : 2);
  std::lock_guard<std::mutex> lock(mu);
  int &c = cache[dev][bf ? 1 : 0][bi][nt - 1][mt - 1][grouped ? 1 : 0];
  if (c == 0) {
    const Inst in = pick(bf, bits, nt, mt, grouped);
    int nb = 0;
    if (in.fn == nullptr ||
        cudaFuncSetAttribute(in.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, in.smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, in.fn, kThreads, in.smem) != cudaSuccess)
      nb = 0;
    if (nb < 1) {
      cudaGetLastError();   // the launch then reports the problem
      return 1;
    }
    c = nb;
  }
  return c;
}

}  // namespace

bool gemv_shape_ok(int64_t K, int64_t N, int bits, int act) {
  const int64_t m16 = act == MOE_ACT_SWIGLU ? (N / 2) / 8 : N / 16;   // 16-channel m-tiles
  // one expert's rows are addressed by 32-bit offsets in 16-byte pieces
  return K % 128 == 0 && (act == MOE_ACT_SWIGLU ? (N / 2) % 8 == 0 : N % 16 == 0) &&
         (bits == 16 || m16 % 2 == 0) && N * (K * bits / 128) < (int64_t(1) << 31);
}

// Plan for the decode kernel.  The routing is not known on the host, so the number of row
// chunks is estimated (experts drawn uniformly); the split S (a divisor of K/128) minimizes the
// bytes the busiest warp streams, counting the fp32 partial slices a split writes and re-reads.
GemmPlan plan_gemv(int64_t R, int64_t E, int64_t K, int64_t N, int bits, int act, bool want_partial) {
  const double er = double(std::max<int64_t>(E, 1));
  const double active = std::max(1.0, er * (1.0 - std::pow(1.0 - 1.0 / er, double(std::max<int64_t>(R, 1)))));
  const double avg = double(std::max<int64_t>(R, 1)) / active;
  const int nt = avg <= 8.0 ? 1 : 2;
  const int64_t m16 = act == MOE_ACT_SWIGLU ? (N / 2) / 8 : N / 16;   // 16-channel m-tiles
  const int64_t nck = K / 128;
  // row chunks: one ragged tail per active expert on average, never more than the rows allow
  const double rc = std::min(std::ceil(active + 0.5 * double(R) / (8.0 * nt)),
                             active - 1.0 + std::ceil(double(R) / (8.0 * nt)));
  const size_t kPartialCap = size_t(256) << 20;
  // For one m16 tile count per unit (mt): the K split with the least per-warp byte load (units
  // dealt round-robin over the resident warps); *steps = the 128-wide chunks a warp streams.
  auto plan_for = [&](int mt, double *steps) {
    GemmPlan pl{};
    pl.kind = kKindGemv;
    pl.nt = nt;
    pl.mt = mt;
    pl.ng = int(m16 / mt);
    const int wps = blocks_per_sm(false, bits, nt, mt, bits != 16) * kWarps;
    const int64_t warps = int64_t(num_sms()) * wps;
    const double step_bytes = double(mt) * 16 * 128 * bits / 8;   // weight bytes per warp per chunk
    double best = 0, best_per = 1;
    int64_t S = 1;
    for (int64_t s = 1; s <= nck; ++s) {
      if (nck % s) continue;
      if (s > 1 && size_t(s) * size_t(R) * size_t(N) * 4 > kPartialCap) break;
      const double units = rc * double(pl.ng) * double(s);
      const double per = std::ceil(units / double(warps));
      double cost = per * double(nck / s) * step_bytes;
      if (want_partial || s > 1) cost += 2.0 * double(s) * double(R) * double(N) * 4 / double(warps);
      if (s == 1 || cost < best * 0.98) {
        best = cost;
        best_per = per;
        S = s;
      }
    }
    pl.splits = int(S);
    pl.ks = int(nck / S) * 128;
    pl.ch = int(nck / S);
    pl.partial = want_partial || S > 1;
    *steps = best_per * double(pl.ch);
    return pl;
  };
  double st2 = 0, st4 = 0;
  if (bits == 16) return plan_for(1, &st2);   // 16-bit weights: one m-tile keeps the ring small
  const GemmPlan p2 = plan_for(2, &st2);
  if (bits != 4 || m16 % 4 != 0) return p2;
  // 4 m16 tiles per unit carry twice the weight bytes per ring slot for the same activation slice
  // (half the warps per SM, each with twice the bytes in flight): measured on GB300 4-8 % faster
  // where each warp streams a long run of chunks (Phi-shaped decode GEMMs), up to 17 % slower
  // where it streams a few (Qwen-shaped T = 8 FC1, 16 chunks), so it takes the long runs
  const GemmPlan p4 = plan_for(4, &st4);
  return st4 >= 32 ? p4 : p2;
}

int launch_gemv(const GemmArgs &g, const GemmPlan &pl, cudaStream_t st) {
  if (g.R == 0) return MOE_OK;
  if (g.E > kMaxE) return set_error(MOE_ERR_UNSUPPORTED, "decode GEMM takes at most %d experts", kMaxE);
  const bool bf = g.a_dtype == MOE_BF16;
  const bool grouped = g.bits != 16 && g.group != 0;
  const Inst in = pick(bf, g.bits, pl.nt, pl.mt, grouped);
  if (in.fn == nullptr) return set_error(MOE_ERR_UNSUPPORTED, "no decode GEMM instance for this shape");
  GvParams gp{};
  gp.a = static_cast<const uint16_t *>(g.a);
  gp.w = static_cast<const uint4 *>(g.w);
  gp.scales = static_cast<const uint16_t *>(g.scales);
  gp.offsets = g.offsets;
  gp.out = g.out;
  gp.partial = g.partial;
  gp.R = int(g.R);
  gp.E = g.E;
  gp.K = g.K;
  gp.N = g.N;
  gp.group = g.group;
  gp.act = g.act;
  gp.out_dtype = g.out_dtype;
  gp.swiglu = g.act == MOE_ACT_SWIGLU ? 1 : 0;
  gp.partial_mode = pl.partial ? 1 : 0;
  gp.S = pl.splits;
  gp.CH = pl.ch;
  gp.NG = pl.ng;
  // the kernel counts units in 32-bit integers: bound the largest count the routing can give
  const int64_t rc_max = std::min<int64_t>(g.E, g.R) + cdiv(g.R, 8 * pl.nt);
  const int64_t units_max = rc_max * pl.ng * pl.splits;
  if (units_max * pl.ch >= (int64_t(1) << 31))
    return set_error(MOE_ERR_UNSUPPORTED, "decode GEMM: %lld work units exceed the 32-bit range",
                     static_cast<long long>(units_max));
  const int64_t resident = int64_t(num_sms()) * blocks_per_sm(bf, g.bits, pl.nt, pl.mt, grouped);
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(resident, cdiv(units_max, kWarps))));
  // a plain launch: placed early, its blocks (all of the SMs' shared memory) would wait there and
  // keep a concurrent branch (the shared expert's stream) off the SMs
  in.fn<<<grid, kThreads, in.smem, st>>>(gp);
  return check_launch("grouped_gemv");
}

}  // namespace moe
