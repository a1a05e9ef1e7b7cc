// Router: logits = x . Wr (+ bias), top-k (descending, ties -> lower id), softmax gates.
//
// "Specter: Fast MoE Inference via Quantization-Enabled Multi-Step Speculative Offloading",
// background on MoE: each token's hidden state is scored by the router and only the top-k
// experts are activated; background on GPTQ INT4: the router stays in 16-bit.
// "Who Says Elephants Can't Run", section 3 model table: top-1 (Switch) gating.
//
// 16-bit router weights use the warp tensor-core MMA with fp32 accumulation, split over K so
// that a decode step (a few tokens) spreads the d x E weight read over many CTAs; partial
// logits are summed in split order by the top-k kernel (deterministic).  fp32 router weights
// (small routers) use fp32 FMAs in one kernel.  The top-k and softmax run one warp per token
// over the E logits kept in shared memory.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTok = 16;     // tokens per CTA
constexpr int kMaxE = 256;
constexpr int kThreads = 128;

// fp32 router weights: fp32 FMA logits (small routers).  CTA = kTok tokens, kF32Threads
// threads; the (token, expert) pairs are spread over the threads (expert fastest, so a warp reads
// consecutive weights).  The reduction runs over chunks of at most kXW columns of x and kWChunk
// router weights (so few experts give long chunks), staged in shared memory.  With d % 8 == 0
// the staging loads are 16-byte vectors, every one of a chunk issued before any is stored, and
// the next chunk's loads are issued before the current chunk is multiplied (register double
// buffer), so a lone CTA (a decode step) waits on memory about once per launch rather than once
// per chunk; other d take the same route with scalar loads.  A thread owns NP (token, expert)
// pairs (NP = ceil(kTok * E / kF32Threads), rounded up to a power of two) and steps through the
// chunk's reduction index once, advancing all NP sums together.  The top-k and softmax run one
// warp per token (two tokens per warp).
constexpr int kF32Threads = 256;
constexpr int kWChunk = 2048;
constexpr int kXW = 256;
constexpr int kWV = kWChunk / 4 / kF32Threads;           // float4 weight pieces per thread per chunk
constexpr int kXV = kTok * kXW / 8 / kF32Threads;        // 16-byte activation pieces per thread per chunk
constexpr int kSU = 8;                                   // scalar path: loads in flight per thread

template <typename T, int NP, bool VEC>
__global__ void __launch_bounds__(kF32Threads, 1) route_f32_kernel(const T *__restrict__ x,
                                                                 const float *__restrict__ wr,
                                                                 const float *__restrict__ bias,
                                                                 int T_, int d, int E, int k,
                                                                 int renorm, int32_t *__restrict__ ids,
                                                                 float *__restrict__ gates) {
  pdl_enter();   // see launch_pdl
  __shared__ __align__(16) float ws[kWChunk];
  __shared__ float xs[kTok][kXW + 1];   // +1: the rows of one warp's tokens fall in different banks
  __shared__ float lg[kTok][kMaxE + 1];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int tok0 = blockIdx.x * kTok;
  // columns per chunk: as many as fit kWChunk weights, at most kXW, a multiple of 8
  const int rows = min(kXW, (kWChunk / E) & ~7);
  const int npairs = kTok * E;
  float acc[NP];
  int xo[NP], eo[NP];   // the pair's x row offset and expert; pairs past npairs compute a dummy
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    acc[i] = 0.f;
    const int pidx = min(tid + i * kF32Threads, npairs - 1), r = pidx / E;
    xo[i] = r * (kXW + 1);
    eo[i] = pidx - r * E;
  }
  const float *xf = &xs[0][0];
  auto multiply = [&](int kc) {
#pragma unroll 4
    for (int c = 0; c < kc; ++c) {
#pragma unroll
      for (int i = 0; i < NP; ++i) acc[i] = fmaf(xf[xo[i] + c], ws[c * E + eo[i]], acc[i]);
    }
  };
  if constexpr (VEC) {
    // piece q of a chunk: weights q < nw / 4 (float4), activations: row q / (kc / 8), 8 columns
    float4 wv[kWV];
    uint4 xv[kXV];
    auto load = [&](int k0) {
      const int kc = min(rows, d - k0), nw4 = kc * E / 4, nx8 = kTok * (kc / 8);
      const float4 *wsrc = reinterpret_cast<const float4 *>(wr + int64_t(k0) * E);
#pragma unroll
      for (int u = 0; u < kWV; ++u) {
        const int q = tid + u * kF32Threads;
        if (q < nw4) wv[u] = __ldg(wsrc + q);
      }
#pragma unroll
      for (int u = 0; u < kXV; ++u) {
        const int q = tid + u * kF32Threads, r = q / (kc / 8), c8 = q - r * (kc / 8);
        xv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (q < nx8 && tok0 + r < T_)
          xv[u] = __ldg(reinterpret_cast<const uint4 *>(x + int64_t(tok0 + r) * d + k0) + c8);
      }
    };
    auto store = [&](int k0) {
      const int kc = min(rows, d - k0), nw4 = kc * E / 4, nx8 = kTok * (kc / 8);
#pragma unroll
      for (int u = 0; u < kWV; ++u) {
        const int q = tid + u * kF32Threads;
        if (q < nw4) reinterpret_cast<float4 *>(ws)[q] = wv[u];
      }
#pragma unroll
      for (int u = 0; u < kXV; ++u) {
        const int q = tid + u * kF32Threads, r = q / (kc / 8), c8 = q - r * (kc / 8);
        if (q < nx8) {
          const T *h = reinterpret_cast<const T *>(&xv[u]);
#pragma unroll
          for (int j = 0; j < 8; ++j) xs[r][8 * c8 + j] = to_f32(h[j]);
        }
      }
    };
    load(0);
    for (int k0 = 0; k0 < d; k0 += rows) {
      store(k0);
      __syncthreads();
      if (k0 + rows < d) load(k0 + rows);   // next chunk in flight while this one is multiplied
      multiply(min(rows, d - k0));
      __syncthreads();
    }
  } else {
    for (int k0 = 0; k0 < d; k0 += rows) {
      const int kc = min(rows, d - k0);
      const int nw = kc * E, nx = kTok * kc;
      const float *wsrc = wr + int64_t(k0) * E;
      for (int b = tid; b < nw; b += kF32Threads * kSU) {
        float v[kSU];
#pragma unroll
        for (int u = 0; u < kSU; ++u) {
          const int i = b + u * kF32Threads;
          v[u] = i < nw ? __ldg(wsrc + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kSU; ++u) {
          const int i = b + u * kF32Threads;
          if (i < nw) ws[i] = v[u];
        }
      }
      for (int b = tid; b < nx; b += kF32Threads * kSU) {
        float v[kSU];
#pragma unroll
        for (int u = 0; u < kSU; ++u) {
          const int i = b + u * kF32Threads, r = i / kc, c = i - r * kc;
          v[u] = (i < nx && tok0 + r < T_) ? to_f32(x[int64_t(tok0 + r) * d + k0 + c]) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kSU; ++u) {
          const int i = b + u * kF32Threads, r = i / kc;
          if (i < nx) xs[r][i - r * kc] = v[u];
        }
      }
      __syncthreads();
      multiply(kc);
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int pidx = tid + i * kF32Threads;
    if (pidx < npairs) {
      const int r = pidx / E, e = pidx - r * E;
      lg[r][e] = acc[i] + (bias ? bias[e] : 0.f);
    }
  }
  __syncthreads();
  for (int r = warp; r < kTok; r += kF32Threads / 32) {
    const int tok = tok0 + r;
    if (tok < T_) topk_softmax_warp(lg[r], E, k, renorm, ids + int64_t(tok) * k, gates + int64_t(tok) * k);
  }
}


// NP = the smallest power of two >= need_np (need_np <= kTok * kMaxE / kF32Threads = 16)
template <typename T, bool VEC>
void launch_route_f32_v(int need_np, unsigned grid, cudaStream_t st, const T *x, const float *wr, const float *bias,
                        int T_, int d, int E, int k, int renorm, int32_t *ids, float *gates) {
  auto go = [&](auto kern) {
    launch_pdl(kern, dim3(grid), dim3(kF32Threads), 0, st, x, wr, bias, T_, d, E, k, renorm, ids, gates);
  };
  if (need_np <= 1) go(route_f32_kernel<T, 1, VEC>);
  else if (need_np <= 2) go(route_f32_kernel<T, 2, VEC>);
  else if (need_np <= 4) go(route_f32_kernel<T, 4, VEC>);
  else if (need_np <= 8) go(route_f32_kernel<T, 8, VEC>);
  else go(route_f32_kernel<T, 16, VEC>);
}
template <typename T>
void launch_route_f32(unsigned grid, cudaStream_t st, const T *x, const float *wr, const float *bias, int T_, int d,
                      int E, int k, int renorm, int32_t *ids, float *gates) {
  const int need_np = int(cdiv(int64_t(kTok) * E, kF32Threads));
  if (d % 8 == 0) launch_route_f32_v<T, true>(need_np, grid, st, x, wr, bias, T_, d, E, k, renorm, ids, gates);
  else launch_route_f32_v<T, false>(need_np, grid, st, x, wr, bias, T_, d, E, k, renorm, ids, gates);
}
static_assert(kTok * kMaxE / kF32Threads <= 16, "route_f32_kernel instances cover every E");
static_assert(kWChunk % (4 * kF32Threads) == 0 && (kTok * kXW) % (8 * kF32Threads) == 0, "staging pieces");

// ---- split-K router: partial logits per (K split, token, expert), then a fixed-order reduce ----
// CTA = 64 tokens (4 warps x m16) x one K range; the router weights are staged row-major with
// plain coalesced loads and turned into MMA B pairs by transposing ldmatrix reads; each chunk's
// global loads are issued while the previous chunk is multiplied.  Decode batches (a handful of
// tokens) spread the d x E weight read over many CTAs this way.
constexpr int kPTok = 64;
constexpr int kPKC = 64;
// experts per pass (kPEG): 32 when E <= 32 (half the accumulators), else 64

template <typename T, int kPEG>
__global__ void __launch_bounds__(kThreads) route_partial_kernel(const T *__restrict__ x, const T *__restrict__ wr,
                                                                 int T_, int d, int E, int KS,
                                                                 float *__restrict__ part) {
  pdl_enter();   // see launch_pdl
  __shared__ __align__(16) uint16_t xs[kPTok][kPKC + 8];
  __shared__ __align__(16) uint16_t ws[kPKC][kPEG + 8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tok0 = blockIdx.x * kPTok;
  const int s = blockIdx.y;
  const int k_begin = s * KS, k_end = min(d, k_begin + KS);
  const uint16_t *xg = reinterpret_cast<const uint16_t *>(x);
  const uint16_t *wg = reinterpret_cast<const uint16_t *>(wr);
  for (int g0 = 0; g0 < E; g0 += kPEG) {
    const int EG = min(kPEG, E - g0);
    const int ntiles = (EG + 7) >> 3;
    float acc[kPEG / 8][4];
#pragma unroll
    for (int i = 0; i < kPEG / 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    // chunk loads go to registers first: the next chunk's loads are in flight while the
    // current one is multiplied
    constexpr int kXPer = kPTok * (kPKC / 8) / kThreads;   // 16-byte pieces of x per thread
    constexpr int kWPer = kPKC * kPEG / 2 / kThreads;       // 32-bit words of Wr per thread
    uint4 xr[kXPer];
    uint32_t wr2[kWPer];
    const bool even_e = (E & 1) == 0;
    auto load_chunk = [&](int k0) {
      const int kc = min(kPKC, k_end - k0);
#pragma unroll
      for (int j = 0; j < kXPer; ++j) {
        const int i = tid + j * kThreads;
        const int r = i / (kPKC / 8), c8 = (i % (kPKC / 8)) * 8;
        xr[j] = (tok0 + r < T_ && c8 < kc) ? *reinterpret_cast<const uint4 *>(xg + int64_t(tok0 + r) * d + k0 + c8)
                                           : make_uint4(0, 0, 0, 0);
      }
      if (even_e) {
#pragma unroll
        for (int j = 0; j < kWPer; ++j) {
          const int i = tid + j * kThreads;
          const int kk = i / (kPEG / 2), ew = i % (kPEG / 2);
          wr2[j] = (kk < kc && 2 * ew < EG) ? *reinterpret_cast<const uint32_t *>(wg + int64_t(k0 + kk) * E + g0 + 2 * ew)
                                            : 0u;
        }
      } else {   // odd E: 16-bit reads, packed into the same words
#pragma unroll
        for (int j = 0; j < kWPer; ++j) {
          const int i = tid + j * kThreads;
          const int kk = i / (kPEG / 2), ew = i % (kPEG / 2);
          const uint32_t lo = (kk < kc && 2 * ew < EG) ? wg[int64_t(k0 + kk) * E + g0 + 2 * ew] : 0u;
          const uint32_t hi = (kk < kc && 2 * ew + 1 < EG) ? wg[int64_t(k0 + kk) * E + g0 + 2 * ew + 1] : 0u;
          wr2[j] = lo | (hi << 16);
        }
      }
    };
    if (k_begin < k_end) load_chunk(k_begin);
    for (int k0 = k_begin; k0 < k_end; k0 += kPKC) {
#pragma unroll
      for (int j = 0; j < kXPer; ++j) {
        const int i = tid + j * kThreads;
        *reinterpret_cast<uint4 *>(&xs[i / (kPKC / 8)][(i % (kPKC / 8)) * 8]) = xr[j];
      }
#pragma unroll
      for (int j = 0; j < kWPer; ++j) {
        const int i = tid + j * kThreads;
        *reinterpret_cast<uint32_t *>(&ws[i / (kPEG / 2)][2 * (i % (kPEG / 2))]) = wr2[j];
      }
      __syncthreads();
      if (k0 + kPKC < k_end) load_chunk(k0 + kPKC);
#pragma unroll
      for (int ks = 0; ks < kPKC / 16; ++ks) {
        const int c = ks * 16 + 2 * t;
        uint32_t a[4];
        a[0] = *reinterpret_cast<const uint32_t *>(&xs[warp * 16 + g][c]);
        a[1] = *reinterpret_cast<const uint32_t *>(&xs[warp * 16 + g + 8][c]);
        a[2] = *reinterpret_cast<const uint32_t *>(&xs[warp * 16 + g][c + 8]);
        a[3] = *reinterpret_cast<const uint32_t *>(&xs[warp * 16 + g + 8][c + 8]);
        // B pairs of two n8 tiles from the row-major (k, e) block: one transposing ldmatrix;
        // lanes 0-7 / 8-15 / 16-23 / 24-31 address rows k0..7 / k8..15 of experts e0.. / e0+8..
#pragma unroll
        for (int np = 0; np < kPEG / 16; ++np) {
          if (2 * np < ntiles) {
            const int krow = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ecol = np * 16 + (lane >> 4) * 8;
            const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(&ws[krow][ecol]));
            uint32_t b[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
                         : "r"(addr));
            mma16816(acc[2 * np], a, b[0], b[1], T());
            if (2 * np + 1 < ntiles) mma16816(acc[2 * np + 1], a, b[2], b[3], T());
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int nt = 0; nt < kPEG / 8; ++nt) {
      if (nt < ntiles) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int e = nt * 8 + 2 * t + h;
          const int r0 = tok0 + warp * 16 + g;
          if (e < EG) {
            if (r0 < T_) part[(int64_t(s) * T_ + r0) * E + g0 + e] = acc[nt][h];
            if (r0 + 8 < T_) part[(int64_t(s) * T_ + r0 + 8) * E + g0 + e] = acc[nt][2 + h];
          }
        }
      }
    }
  }
}

// One warp per token: logits = sum over K splits in split order (+ bias), then top-k / softmax.
__global__ void __launch_bounds__(kThreads) route_reduce_topk_kernel(const float *__restrict__ part, int S, int T_,
                                                                     int E, const float *__restrict__ bias, int k,
                                                                     int renorm, int32_t *__restrict__ ids,
                                                                     float *__restrict__ gates) {
  pdl_enter();   // see launch_pdl
  __shared__ float lg[kThreads / 32][kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tok = blockIdx.x * (kThreads / 32) + warp;
  if (tok >= T_) return;
  const int64_t sstride = int64_t(T_) * E;
  for (int e = lane; e < E; e += 32) {
    const float *pe = part + int64_t(tok) * E + e;
    float v = 0.f;
    for (int s = 0; s < S; s += 8) {   // up to eight loads in flight, summed in split order
      float q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) q[u] = s + u < S ? pe[(s + u) * sstride] : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (s + u < S) v += q[u];
    }
    lg[warp][e] = v + (bias ? bias[e] : 0.f);
  }
  __syncwarp();
  topk_softmax_warp(lg[warp], E, k, renorm, ids + int64_t(tok) * k, gates + int64_t(tok) * k);
}

// Few tokens, many K splits (decode): one CTA per token; warp w sums the slices s = w, w+8, ...
// for every expert, warp 0 adds the 8 partial sums in warp order (+ bias), then top-k.  The order
// is fixed (deterministic), different from the one-warp kernel's.
__global__ void __launch_bounds__(kThreads * 2) route_reduce_small_kernel(const float *__restrict__ part, int S,
                                                                        int T_, int E, const float *__restrict__ bias,
                                                                        int k, int renorm, int32_t *__restrict__ ids,
                                                                        float *__restrict__ gates) {
  pdl_enter();   // see launch_pdl
  constexpr int kW = kThreads * 2 / 32;
  __shared__ float red[kW][kMaxE];
  __shared__ float lg[kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tok = blockIdx.x;
  const int64_t sstride = int64_t(T_) * E;
  for (int e = lane; e < E; e += 32) {
    float v = 0.f;
    for (int s = warp; s < S; s += kW) v += part[s * sstride + int64_t(tok) * E + e];
    red[warp][e] = v;
  }
  __syncthreads();
  if (warp == 0) {
    for (int e = lane; e < E; e += 32) {
      float v = 0.f;
      for (int w = 0; w < kW; ++w) v += red[w][e];
      lg[e] = v + (bias ? bias[e] : 0.f);
    }
    __syncwarp();
    topk_softmax_warp(lg, E, k, renorm, ids + int64_t(tok) * k, gates + int64_t(tok) * k);
  }
}

int route_splits(int64_t T, int64_t d) {
  const int64_t ntt = cdiv(T, kPTok);
  const int64_t nkc = cdiv(d, kPKC);
  int64_t S = cdiv(2 * int64_t(num_sms()), ntt);
  if (S > nkc) S = nkc;
  if (S < 1) S = 1;
  const int64_t ks = cdiv(nkc, S) * kPKC;
  return int(cdiv(d, ks));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_topk_workspace_size(int64_t T, int64_t d, int64_t E) {
  if (T <= 0 || d < 8 || E < 1) return 0;
  return align256(size_t(route_splits(T, d)) * size_t(T) * size_t(E) * 4);
}

extern "C" int moe_route_topk(const void *x, int x_dtype, const void *w_router, int wr_dtype,
                              const float *bias, int64_t T, int64_t d, int64_t E, int k,
                              int renormalize, int32_t *ids, float *gate_w, void *workspace,
                              size_t workspace_bytes, moe_stream_t stream) {
  MOE_REQUIRE(is16(x_dtype), "x_dtype must be MOE_F16 or MOE_BF16");
  MOE_REQUIRE(wr_dtype == MOE_F32 || wr_dtype == x_dtype, "router weights must be fp32 or the x dtype");
  MOE_REQUIRE(T >= 0 && d >= 8 && d % 8 == 0, "need T >= 0 and d %% 8 == 0 (d=%lld)", (long long)d);
  MOE_REQUIRE(E >= 1 && E <= kMaxE && k >= 1 && k <= E, "need 1 <= k <= E <= 256 (E=%lld k=%d)",
              (long long)E, k);
  MOE_REQUIRE(T < (int64_t(1) << 31) && d < (int64_t(1) << 31), "T and d must fit in int32");
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && w_router && ids && gate_w, "null pointer argument");
  MOE_REQUIRE(aligned16(x) && aligned16(w_router) && aligned16(ids) && aligned16(gate_w) &&
                  (bias == nullptr || aligned16(bias)),
              "pointers must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const unsigned grid = unsigned(cdiv(T, kTok));
  if (wr_dtype == MOE_F32) {
    if (x_dtype == MOE_F16)
      launch_route_f32<__half>(grid, st, static_cast<const __half *>(x), static_cast<const float *>(w_router), bias,
                               int(T), int(d), int(E), k, renormalize, ids, gate_w);
    else
      launch_route_f32<__nv_bfloat16>(grid, st, static_cast<const __nv_bfloat16 *>(x),
                                      static_cast<const float *>(w_router), bias, int(T), int(d), int(E), k,
                                      renormalize, ids, gate_w);
  } else {
    const size_t need = moe_route_topk_workspace_size(T, d, E);
    MOE_REQUIRE(workspace && aligned16(workspace), "workspace must be non-null and 16-byte aligned");
    if (workspace_bytes < need)
      return set_error(MOE_ERR_WORKSPACE, "router workspace %zu < %zu bytes", workspace_bytes, need);
    const int S = route_splits(T, d);
    const int KS = int(cdiv(cdiv(d, kPKC), S) * kPKC);
    float *part = static_cast<float *>(workspace);
    const dim3 pgrid(unsigned(cdiv(T, kPTok)), unsigned(S));
    const bool narrow = E <= 32;
    if (x_dtype == MOE_F16) {
      const __half *xh = static_cast<const __half *>(x), *wh = static_cast<const __half *>(w_router);
      if (narrow) launch_pdl(route_partial_kernel<__half, 32>, dim3(pgrid), dim3(kThreads), 0, st, xh, wh, int(T), int(d), int(E), KS, part);
      else launch_pdl(route_partial_kernel<__half, 64>, dim3(pgrid), dim3(kThreads), 0, st, xh, wh, int(T), int(d), int(E), KS, part);
    } else {
      const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x), *wb = static_cast<const __nv_bfloat16 *>(w_router);
      if (narrow) launch_pdl(route_partial_kernel<__nv_bfloat16, 32>, dim3(pgrid), dim3(kThreads), 0, st, xb, wb, int(T), int(d), int(E), KS, part);
      else launch_pdl(route_partial_kernel<__nv_bfloat16, 64>, dim3(pgrid), dim3(kThreads), 0, st, xb, wb, int(T), int(d), int(E), KS, part);
    }
    MOE_TRY(check_launch("route_partial"));
    if (S >= 8 && T <= int64_t(num_sms()) * 2)
      launch_pdl(route_reduce_small_kernel, dim3(unsigned(T)), dim3(kThreads * 2), 0, st, part, S, int(T), int(E), bias, k, renormalize,
                                                                       ids, gate_w);
    else
      launch_pdl(route_reduce_topk_kernel, dim3(unsigned(cdiv(T, kThreads / 32))), dim3(kThreads), 0, st, part, S, int(T), int(E), bias, k,
                                                                                   renormalize, ids, gate_w);
  }
  return check_launch("route_topk");
}
