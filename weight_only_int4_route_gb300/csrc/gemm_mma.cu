// Grouped GEMM over experts with the weight dequantization fused into the mainloop, on the
// warp-level tensor-core MMA (m16n8k16, fp32 accumulate).  This is the path for experts with
// few routed rows (decode / speculative-verify batches): it streams the packed weights from
// HBM exactly once per row tile, converts them in registers and never stages them in shared
// memory.
//
// "Who Says Elephants Can't Run", section 3: grouped GEMM computing every expert's
// sub-matrix in one launch (Figure 1), dequantization fused into the GEMM (section 4 table),
// optimized I2F with the interleaved INT4 word; "Specter", method step 5: tokens grouped by
// expert turn per-token GEMVs into per-expert GEMMs.  Figure 1's batch pruning: experts
// with no routed rows own no tile and load no weights.
//
// Mapping.  The weights are the MMA's B operand (n8 = 8 output channels per warp), the
// routed rows are the A operand (m16 row tiles).  A lane (g = lane/4, t = lane%4) owns
// channel g of its warp and the 32 consecutive reduction indices [32t, 32t+32) of every
// 128-wide chunk, i.e. one 16-byte load of INT4 words (two for INT8, four for 16-bit).  The
// MMA's reduction order is free as long as A and B agree, so MMA step s (0..7) of a chunk
// takes reduction indices 32t + 4s + {0,1,2,3} from lane t: the B pair registers are then
// exactly the dequantized pairs (2s, 2s+1) of the lane's own words.  A is staged in shared
// memory in that permuted order (8-byte piece (s, t) at position 4s + t, rows padded to 288
// bytes) so each A fragment is one conflict-free 8-byte load per row.
//
// Work item = (expert row tile, 64-channel block, K split).  A persistent grid walks the
// items; the per-expert tile table is rebuilt by every CTA from the device offsets, so no
// host synchronization is needed.  With several K splits the fp32 partial sums go to a
// workspace and are reduced later (by launch_reduce_act or the combine kernel).
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

MOE_DEFINE_CHECK_WORD(gemm_mma)

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kNB = 64;         // channels per CTA
constexpr int kKC = 128;        // reduction chunk
constexpr int kRowBytes = kKC * 2 + 32;
constexpr int kMaxE = 256;
constexpr int kEpStride = kNB + 8;  // fp32 epilogue tile row stride
constexpr int kTcMinRows = 17;      // rows per active expert from which the tcgen05 path is used
constexpr int kTcMinRows16 = 17;    // the same for 16-bit weights (measured: 17-63 rows of the
                                    // Qwen-shaped shared expert take 42 us there, 63-80 us here)
constexpr int kGemvMaxRows = 16;    // rows per active expert up to which the decode stream kernel is used

template <int BITS> struct WT {
  static constexpr int kVec = BITS == 4 ? 1 : (BITS == 8 ? 2 : 4);  // uint4 per lane per chunk
  static constexpr int kPre = BITS == 4 ? 4 : (BITS == 8 ? 2 : 1);  // chunks prefetched ahead
};

struct KParams {
  const uint16_t *a;
  const uint4 *w;
  const uint16_t *scales;
  const int32_t *offsets;
  void *out;
  float *partial;
  int R, E, K, N;
  int group, act, out_dtype;
  int partial_mode, swiglu_fused;
  int S, KS, ncb;
};

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <typename T, int BITS>
__device__ __forceinline__ void dequant_chunk(const uint4 (&w)[WT<BITS>::kVec], uint32_t (&pr)[16]) {
  if constexpr (BITS == 4) {
    const uint32_t words[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h[4];
      i2f_int4(words[i], h, T());
#pragma unroll
      for (int q = 0; q < 4; ++q) pr[4 * i + q] = h[q];
    }
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const uint32_t words[4] = {w[v].x, w[v].y, w[v].z, w[v].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t h[2];
        i2f_int8(words[i], h, T());
        pr[8 * v + 2 * i] = h[0];
        pr[8 * v + 2 * i + 1] = h[1];
      }
    }
  } else {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      pr[4 * v + 0] = w[v].x;
      pr[4 * v + 1] = w[v].y;
      pr[4 * v + 2] = w[v].z;
      pr[4 * v + 3] = w[v].w;
    }
  }
}

template <typename OT> __device__ __forceinline__ void store_out(void *out, int64_t idx, float v) {
  static_cast<OT *>(out)[idx] = from_f32<OT>(v);
}
__device__ __forceinline__ void store_any(void *out, int dt, int64_t idx, float v) {
  if (dt == MOE_F32) store_out<float>(out, idx, v);
  else if (dt == MOE_F16) store_out<__half>(out, idx, v);
  else store_out<__nv_bfloat16>(out, idx, v);
}

template <typename T>
__device__ __forceinline__ float ld_scale(const uint16_t *s, int64_t idx) {
  const uint16_t b = s[idx];
  if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half(b));
  else return __bfloat162float(__ushort_as_bfloat16(b));
}

template <typename T, int BITS, int MB>
__global__ void __launch_bounds__(kThreads) gemm_mma_kernel(const KParams p) {
  pdl_enter();   // see launch_pdl
  constexpr int MT = 16 * MB;
  constexpr int kVec = WT<BITS>::kVec;
  constexpr int kPre = WT<BITS>::kPre;
  static_assert(MT * kEpStride * 4 <= 2 * MT * kRowBytes, "epilogue tile must fit the A buffers");
  __shared__ __align__(16) uint8_t smem[2 * MT * kRowBytes];
  __shared__ int s_tstart[kMaxE + 1];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int scratch[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int E = p.E;

  // ---- per-expert row-tile table (prefix over experts of ceil(rows / MT)) ----
  int cnt = 0;
  // checked build: unusable offsets leave the kernel without tiles (nothing is read or written)
  const bool off_ok = p.offsets == nullptr || offsets_usable(p.offsets, E, p.R, [] { check_fail(kCheckOffsets); });
  if (tid < E && off_ok) {
    const int o0 = p.offsets ? p.offsets[tid] : 0;
    const int o1 = p.offsets ? p.offsets[tid + 1] : p.R;
    cnt = (o1 - o0 + MT - 1) / MT;
    s_off[tid] = o0;
    if (tid == E - 1) s_off[E] = o1;
  }
  int start = 0;
  const int total_tiles = block_exclusive_scan(cnt, &start, scratch);
  if (tid < E) s_tstart[tid] = start;
  __syncthreads();

  const int64_t items = int64_t(total_tiles) * p.ncb * p.S;
  const int64_t w_row_vec = int64_t(p.K) * BITS / 128;  // uint4 per channel row
  const bool per_channel = p.group == 0 && BITS != 16;
  const int G = p.group == 0 ? 1 : p.K / p.group;

  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int s = int(item % p.S);
    const int64_t rest = item / p.S;
    const int cb = int(rest % p.ncb);
    const int tile = int(rest / p.ncb);
    int lo = 0, hi = E - 1;  // last expert whose first tile is <= tile (skips empty experts)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tstart[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    const int row0 = s_off[e] + (tile - s_tstart[e]) * MT;
    const int nrows = min(MT, s_off[e + 1] - row0);
    const int k0 = s * p.KS;
    const int k1 = min(p.K, k0 + p.KS);
    const int nch = (k1 - k0) / kKC;

    int ch;
    if (p.swiglu_fused) {
      const int F = p.N >> 1;
      ch = warp < kWarps / 2 ? cb * (kNB / 2) + warp * 8 + g : F + cb * (kNB / 2) + (warp - kWarps / 2) * 8 + g;
    } else {
      ch = cb * kNB + warp * 8 + g;
    }
    const uint4 *wrow = p.w + (int64_t(e) * p.N + ch) * w_row_vec + int64_t(k0) * BITS / 128 + kVec * t;
    const uint16_t *srow = p.scales + int64_t(e) * G * p.N + ch;

    auto load_chunk = [&](int c, uint4 (&dst)[kVec], uint32_t &sc) {
#pragma unroll
      for (int v = 0; v < kVec; ++v) dst[v] = ld_stream(wrow + int64_t(c) * (kKC * BITS / 128) + v);
      if (BITS != 16 && p.group != 0) {
        const uint16_t b = srow[int64_t((k0 + c * kKC) / p.group) * p.N];
        sc = uint32_t(b) | (uint32_t(b) << 16);
      }
    };
    auto stage_a = [&](int c, int buf) {
      uint8_t *dst = smem + buf * (MT * kRowBytes);
      for (int i = tid; i < MT * 32; i += kThreads) {
        const int r = i >> 5, j8 = i & 31;
        const int q = 4 * (j8 & 7) + (j8 >> 3);
        const bool ok = r < nrows;
        const uint16_t *src = p.a + int64_t(row0 + (ok ? r : 0)) * p.K + k0 + c * kKC + 4 * j8;
        cp_async8(dst + r * kRowBytes + 8 * q, src, ok ? 8 : 0);
      }
    };

    float acc[MB][4];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mb][j] = 0.f;

    uint4 ring[kPre][kVec];
    uint32_t sring[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      sring[i] = 0;
      if (i < nch) load_chunk(i, ring[i], sring[i]);
    }
    stage_a(0, 0);
    cp_async_commit();

    for (int c0 = 0; c0 < nch; c0 += kPre) {
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        const int c = c0 + i;
        if (c < nch) {
          uint4 cur[kVec];
#pragma unroll
          for (int v = 0; v < kVec; ++v) cur[v] = ring[i][v];
          const uint32_t csc = sring[i];
          if (c + kPre < nch) load_chunk(c + kPre, ring[i], sring[i]);
          if (c + 1 < nch) stage_a(c + 1, (c + 1) & 1);
          cp_async_commit();
          cp_async_wait<1>();
          __syncthreads();

          uint32_t pr[16];
          dequant_chunk<T, BITS>(cur, pr);
          if (BITS != 16 && p.group != 0) {
#pragma unroll
            for (int q = 0; q < 16; ++q) pr[q] = scale_pair(pr[q], csc, T());
          }
          const uint8_t *abuf = smem + (c & 1) * (MT * kRowBytes);
#pragma unroll
          for (int st = 0; st < 8; ++st) {
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              const uint2 lo2 = *reinterpret_cast<const uint2 *>(abuf + (mb * 16 + g) * kRowBytes + 8 * (4 * st + t));
              const uint2 hi2 = *reinterpret_cast<const uint2 *>(abuf + (mb * 16 + g + 8) * kRowBytes + 8 * (4 * st + t));
              const uint32_t a[4] = {lo2.x, hi2.x, lo2.y, hi2.y};
              mma16816(acc[mb], a, pr[2 * st], pr[2 * st + 1], T());
            }
          }
          __syncthreads();
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- epilogue through shared memory ----
    float *ep = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const int col = warp * 8 + 2 * t;
      *reinterpret_cast<float2 *>(&ep[(mb * 16 + g) * kEpStride + col]) = make_float2(acc[mb][0], acc[mb][1]);
      *reinterpret_cast<float2 *>(&ep[(mb * 16 + g + 8) * kEpStride + col]) = make_float2(acc[mb][2], acc[mb][3]);
    }
    __syncthreads();
    const uint16_t *sc_e = p.scales + int64_t(e) * G * p.N;
    if (p.partial_mode) {
      for (int i = tid; i < nrows * kNB; i += kThreads) {
        const int r = i / kNB, cc = i % kNB;
        const int n = cb * kNB + cc;
        float v = ep[r * kEpStride + cc];
        if (per_channel) v *= ld_scale<T>(sc_e, n);
        p.partial[(int64_t(s) * p.R + row0 + r) * p.N + n] = v;
      }
    } else if (p.swiglu_fused) {
      const int F = p.N >> 1;
      for (int i = tid; i < nrows * (kNB / 2); i += kThreads) {
        const int r = i / (kNB / 2), cc = i % (kNB / 2);
        const int n = cb * (kNB / 2) + cc;
        float gt = ep[r * kEpStride + cc];
        float up = ep[r * kEpStride + kNB / 2 + cc];
        if (per_channel) {
          gt *= ld_scale<T>(sc_e, n);
          up *= ld_scale<T>(sc_e, F + n);
        }
        store_any(p.out, p.out_dtype, int64_t(row0 + r) * F + n, act_silu(gt) * up);
      }
    } else {
      for (int i = tid; i < nrows * kNB; i += kThreads) {
        const int r = i / kNB, cc = i % kNB;
        const int n = cb * kNB + cc;
        float v = ep[r * kEpStride + cc];
        if (per_channel) v *= ld_scale<T>(sc_e, n);
        store_any(p.out, p.out_dtype, int64_t(row0 + r) * p.N + n, act_apply(v, p.act));
      }
    }
    __syncthreads();
  }
}

template <typename T, int BITS, int MB>
int launch_one(const KParams &kp, int64_t items_upper, cudaStream_t st) {
  static int occ[64] = {0};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (occ[dev] == 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, gemm_mma_kernel<T, BITS, MB>, kThreads, 0) != cudaSuccess || b < 1)
      b = 1;
    occ[dev] = b;
  }
  const int64_t cap = int64_t(num_sms()) * occ[dev];
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items_upper, cap)));
  launch_pdl(gemm_mma_kernel<T, BITS, MB>, dim3(grid), dim3(kThreads), 0, st, kp);
  return check_launch("grouped_gemm");
}

template <typename T, int BITS>
int launch_mb(const KParams &kp, int mb, int64_t items_upper, cudaStream_t st) {
  if (mb == 1) return launch_one<T, BITS, 1>(kp, items_upper, st);
  if (mb == 2) return launch_one<T, BITS, 2>(kp, items_upper, st);
  return launch_one<T, BITS, 4>(kp, items_upper, st);
}

// Row-tile estimate used for grid sizing and the split-K choice.
int64_t est_tiles(int64_t R, int64_t E, int mt) { return std::min<int64_t>(E, R) + cdiv(R, mt); }

}  // namespace

GemmPlan plan_gemm(int64_t R, int64_t E, int64_t K, int64_t N, int bits, int act, bool want_partial) {
  GemmPlan pl{};
  const int64_t active = std::max<int64_t>(1, std::min<int64_t>(E, R));
  const int64_t avg = cdiv(std::max<int64_t>(R, 1), active);
  if (avg <= kGemvMaxRows && gemv_shape_ok(K, N, bits, act)) return plan_gemv(R, E, K, N, bits, act, want_partial);
  pl.kind = kKindMma;
  pl.mb = avg <= 16 ? 1 : (avg <= 32 ? 2 : 4);
  const int64_t nck = K / kKC;
  const bool swiglu = act == MOE_ACT_SWIGLU;
  const int64_t ncb_fused = swiglu ? (N / 2) / (kNB / 2) : N / kNB;
  const int64_t tiles = est_tiles(R, E, 16 * pl.mb);
  int64_t S = 1;
  const int64_t target = 2 * int64_t(num_sms());
  // the tcgen05 kernel takes these whole, without split-K (group is not known here: group 128 is
  // the only grouped size the API accepts, and the kernel takes it)
  const bool tc_rows = avg >= (bits == 16 ? kTcMinRows16 : kTcMinRows) && tc_shape_ok(E, K, N, bits, 0, act);
  while (!tc_rows && S * 2 <= std::max<int64_t>(1, nck / 2) && tiles * ncb_fused * S < target) S *= 2;
  const int64_t cps = cdiv(nck, S);
  pl.ks = int(cps * kKC);
  pl.splits = int(cdiv(nck, cps));
  pl.partial = want_partial || pl.splits > 1;
  pl.ncb = int(pl.partial ? N / kNB : ncb_fused);
  pl.tc = pl.splits == 1 && tc_rows;
  if (pl.tc) pl.kind = kKindTc;
  return pl;
}

int launch_gemm(const GemmArgs &g, const GemmPlan &pl, cudaStream_t st) {
  if (pl.kind == kKindGemv) return launch_gemv(g, pl, st);
  if (pl.tc && tc_supported(g) && (!pl.partial || g.act == MOE_ACT_NONE)) {
    GemmArgs t = g;
    if (pl.partial) {  // single split: the fp32 "partial" slice is the output itself
      t.out = g.partial;
      t.out_dtype = MOE_F32;
    }
    return launch_gemm_tc(t, st);
  }
  return launch_gemm_mma(g, pl, st);
}

int launch_gemm_mma(const GemmArgs &g, const GemmPlan &pl, cudaStream_t st) {
  KParams kp{};
  kp.a = static_cast<const uint16_t *>(g.a);
  kp.w = static_cast<const uint4 *>(g.w);
  kp.scales = static_cast<const uint16_t *>(g.scales);
  kp.offsets = g.offsets;
  kp.out = g.out;
  kp.partial = g.partial;
  kp.R = int(g.R);
  kp.E = g.E;
  kp.K = g.K;
  kp.N = g.N;
  kp.group = g.group;
  kp.act = g.act;
  kp.out_dtype = g.out_dtype;
  kp.partial_mode = pl.partial ? 1 : 0;
  kp.swiglu_fused = (!pl.partial && g.act == MOE_ACT_SWIGLU) ? 1 : 0;
  kp.S = pl.splits;
  kp.KS = pl.ks;
  kp.ncb = pl.ncb;
  if (g.R == 0) return MOE_OK;
  const int64_t items_upper = est_tiles(g.R, g.E, 16 * pl.mb) * pl.ncb * pl.splits;
  const bool bf = g.a_dtype == MOE_BF16;
  if (g.bits == 4) return bf ? launch_mb<__nv_bfloat16, 4>(kp, pl.mb, items_upper, st) : launch_mb<__half, 4>(kp, pl.mb, items_upper, st);
  if (g.bits == 8) return bf ? launch_mb<__nv_bfloat16, 8>(kp, pl.mb, items_upper, st) : launch_mb<__half, 8>(kp, pl.mb, items_upper, st);
  return bf ? launch_mb<__nv_bfloat16, 16>(kp, pl.mb, items_upper, st) : launch_mb<__half, 16>(kp, pl.mb, items_upper, st);
}

}  // namespace moe
