// Router: logits = x . Wr (+ bias), top-k (descending, ties -> lower id), softmax gates.
//
// "Specter: Fast MoE Inference via Quantization-Enabled Multi-Step Speculative Offloading",
// background on MoE: each token's hidden state is scored by the router and only the top-k
// experts are activated; background on GPTQ INT4: the router stays in 16-bit.
// "Who Says Elephants Can't Run", section 3 model table: top-1 (Switch) gating.
//
// One CTA handles 16 tokens.  16-bit router weights use the warp tensor-core MMA with fp32
// accumulation (a 16 x E x d product per CTA); fp32 router weights use fp32 FMAs.  The top-k
// and softmax run one warp per token over the E logits kept in shared memory.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTok = 16;     // tokens per CTA
constexpr int kKC = 64;      // reduction chunk staged in shared memory
constexpr int kMaxE = 256;
constexpr int kThreads = 128;

// Top-k + softmax for one token (one warp).  logits: E floats in shared memory.
__device__ void topk_softmax_warp(const float *logits, int E, int k, int renorm, int32_t *ids,
                                  float *gates) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = kMaxE / 32;
  float v[kPer];
  bool taken[kPer];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? logits[e] : -INFINITY;
    taken[i] = e >= E;
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < E) sum += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  float gsum = 0.f;
  float my_gate = 0.f;  // lane j keeps gate j
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i == bi) taken[i] = true;
    const float g = expf(bv - mx) / sum;
    gsum += g;
    if (lane == j) {
      my_gate = g;
      my_id = bi;
    }
  }
  if (lane < k) {
    ids[lane] = my_id;
    gates[lane] = renorm ? my_gate / gsum : my_gate;
  }
}

// 16-bit router weights: tensor-core logits.
template <typename T>
__global__ void __launch_bounds__(kThreads) route_mma_kernel(const T *__restrict__ x,
                                                              const T *__restrict__ wr,
                                                              const float *__restrict__ bias,
                                                              int T_, int d, int E, int k,
                                                              int renorm, int32_t *__restrict__ ids,
                                                              float *__restrict__ gates) {
  // The logits tile reuses the weight-chunk storage once the reduction is finished.
  constexpr int kWsBytes = kMaxE * (kKC + 8) * 2;
  static_assert(kWsBytes >= kTok * (kMaxE + 1) * 4, "logit tile must fit the weight chunk");
  __shared__ __align__(16) uint16_t xs[kTok][kKC + 8];
  __shared__ __align__(16) unsigned char raw[kWsBytes];
  auto ws = reinterpret_cast<uint16_t(*)[kKC + 8]>(raw);  // transposed chunk: ws[e][kk]
  auto lg = reinterpret_cast<float(*)[kMaxE + 1]>(raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tok0 = blockIdx.x * kTok;
  const int Ep = (E + 7) & ~7;
  const int ntiles = Ep / 8;
  float acc[kMaxE / 8 / 4][4];
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const uint16_t *xg = reinterpret_cast<const uint16_t *>(x);
  const uint16_t *wg = reinterpret_cast<const uint16_t *>(wr);
  for (int k0 = 0; k0 < d; k0 += kKC) {
    const int kc = min(kKC, d - k0);
    for (int i = tid; i < kTok * (kKC / 8); i += kThreads) {  // 16-byte pieces of x
      const int r = i / (kKC / 8), c8 = (i % (kKC / 8)) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (tok0 + r < T_ && c8 < kc) v = *reinterpret_cast<const uint4 *>(xg + int64_t(tok0 + r) * d + k0 + c8);
      *reinterpret_cast<uint4 *>(&xs[r][c8]) = v;
    }
    for (int i = tid; i < kKC * Ep; i += kThreads) {
      const int kk = i / Ep, e = i % Ep;
      ws[e][kk] = (kk < kc && e < E) ? wg[int64_t(k0 + kk) * E + e] : uint16_t(0);
    }
    __syncthreads();
#pragma unroll
    for (int ks = 0; ks < kKC / 16; ++ks) {
      uint32_t a[4];
      const int c = ks * 16 + 2 * t;
      a[0] = *reinterpret_cast<const uint32_t *>(&xs[g][c]);
      a[1] = *reinterpret_cast<const uint32_t *>(&xs[g + 8][c]);
      a[2] = *reinterpret_cast<const uint32_t *>(&xs[g][c + 8]);
      a[3] = *reinterpret_cast<const uint32_t *>(&xs[g + 8][c + 8]);
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) {
        const int nt = warp + 4 * i;
        if (nt < ntiles) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&ws[nt * 8 + g][c]);
          const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&ws[nt * 8 + g][c + 8]);
          mma16816(acc[i], a, b0, b1, T());
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int nt = warp + 4 * i;
    if (nt < ntiles) {
      const int e0 = nt * 8 + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h;
        if (e < E) {
          const float b = bias ? bias[e] : 0.f;
          lg[g][e] = acc[i][h] + b;
          lg[g + 8][e] = acc[i][2 + h] + b;
        }
      }
    }
  }
  __syncthreads();
  for (int r = warp; r < kTok; r += kThreads / 32) {
    const int tok = tok0 + r;
    if (tok < T_) topk_softmax_warp(lg[r], E, k, renorm, ids + int64_t(tok) * k, gates + int64_t(tok) * k);
  }
}

// fp32 router weights: fp32 FMA logits (small routers).
template <typename T>
__global__ void __launch_bounds__(kThreads) route_f32_kernel(const T *__restrict__ x,
                                                              const float *__restrict__ wr,
                                                              const float *__restrict__ bias,
                                                              int T_, int d, int E, int k,
                                                              int renorm, int32_t *__restrict__ ids,
                                                              float *__restrict__ gates) {
  __shared__ float xs[kTok][kKC];
  __shared__ float lg[kTok][kMaxE + 1];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int tok0 = blockIdx.x * kTok;
  constexpr int kPairs = kTok * kMaxE / kThreads;
  float acc[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < d; k0 += kKC) {
    const int kc = min(kKC, d - k0);
    for (int i = tid; i < kTok * kKC; i += kThreads) {
      const int r = i / kKC, c = i % kKC;
      xs[r][c] = (tok0 + r < T_ && c < kc) ? to_f32(x[int64_t(tok0 + r) * d + k0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const int pidx = tid + i * kThreads;
      const int r = pidx / kMaxE, e = pidx % kMaxE;
      if (e < E) {
        float s = acc[i];
        for (int c = 0; c < kc; ++c) s = fmaf(xs[r][c], wr[int64_t(k0 + c) * E + e], s);
        acc[i] = s;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const int pidx = tid + i * kThreads;
    const int r = pidx / kMaxE, e = pidx % kMaxE;
    if (e < E) lg[r][e] = acc[i] + (bias ? bias[e] : 0.f);
  }
  __syncthreads();
  for (int r = warp; r < kTok; r += kThreads / 32) {
    const int tok = tok0 + r;
    if (tok < T_) topk_softmax_warp(lg[r], E, k, renorm, ids + int64_t(tok) * k, gates + int64_t(tok) * k);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route_topk(const void *x, int x_dtype, const void *w_router, int wr_dtype,
                              const float *bias, int64_t T, int64_t d, int64_t E, int k,
                              int renormalize, int32_t *ids, float *gate_w, moe_stream_t stream) {
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
      route_f32_kernel<__half><<<grid, kThreads, 0, st>>>(static_cast<const __half *>(x),
          static_cast<const float *>(w_router), bias, int(T), int(d), int(E), k, renormalize, ids, gate_w);
    else
      route_f32_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16 *>(x),
          static_cast<const float *>(w_router), bias, int(T), int(d), int(E), k, renormalize, ids, gate_w);
  } else if (x_dtype == MOE_F16) {
    route_mma_kernel<__half><<<grid, kThreads, 0, st>>>(static_cast<const __half *>(x),
        static_cast<const __half *>(w_router), bias, int(T), int(d), int(E), k, renormalize, ids, gate_w);
  } else {
    route_mma_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16 *>(x),
        static_cast<const __nv_bfloat16 *>(w_router), bias, int(T), int(d), int(E), k, renormalize, ids, gate_w);
  }
  return check_launch("route_topk");
}
