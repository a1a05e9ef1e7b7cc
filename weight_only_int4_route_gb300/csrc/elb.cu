// Expert lookahead buffer (ELB): per-layer expert counts over draft steps, and the top-M experts
// of every layer at a chunk boundary.
//
// "Specter" (paper summary page), method step (2): while the draft advances, the analyzer keeps
// on the GPU, per layer j and expert e, ELB_cnt[j, e] = number of draft steps whose routed set
// in layer j contains e; step (3): at each boundary the planner snapshots the buffer and takes
// each layer's top-M experts as the next prefetch batch.
//
// Counts are integers, so every order of accumulation gives the same result.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kThreads = 256;

// One CTA per layer: a shared-memory histogram of the layer's S x k ids (an expert once per
// step; ids outside [0, E) skipped), then added to the layer's counts.
__global__ void __launch_bounds__(kThreads) elb_accumulate_kernel(const int32_t *__restrict__ ids, int S, int k,
                                                                  int E, int32_t *__restrict__ counts) {
  __shared__ int hist[kMaxE];
  const int layer = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const int32_t *lid = ids + int64_t(layer) * S * k;
  for (int i = threadIdx.x; i < S; i += kThreads) {
    const int32_t *row = lid + int64_t(i) * k;
    for (int a = 0; a < k; ++a) {
      const int e = row[a];
      if (e < 0 || e >= E) continue;
      bool seen = false;
      for (int b = 0; b < a; ++b) seen |= row[b] == e;
      if (!seen) atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) counts[int64_t(layer) * E + e] += hist[e];
}

// One CTA per layer: expert e's place in the order (count descending, id ascending) is the
// number of experts before it; places below M are written.
__global__ void __launch_bounds__(kThreads) elb_topm_kernel(const int32_t *__restrict__ counts, int E, int M,
                                                            int32_t *__restrict__ experts, int32_t *__restrict__ vals) {
  __shared__ int c[kMaxE];
  const int layer = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += kThreads) c[e] = counts[int64_t(layer) * E + e];
  __syncthreads();
  const int m = M < E ? M : E;
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int place = 0;
    for (int f = 0; f < E; ++f) place += (c[f] > c[e]) || (c[f] == c[e] && f < e);
    if (place < m) {
      experts[int64_t(layer) * m + place] = e;
      vals[int64_t(layer) * m + place] = c[e];
    }
  }
}

// Both in one launch (one CTA per layer): add the window's histogram to the counts, then select
// the layer's top-M from the updated counts.
__global__ void __launch_bounds__(kThreads) elb_step_kernel(const int32_t *__restrict__ ids, int S, int k, int E,
                                                            int32_t *__restrict__ counts, int M,
                                                            int32_t *__restrict__ experts, int32_t *__restrict__ vals) {
  __shared__ int hist[kMaxE];
  const int layer = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const int32_t *lid = ids + int64_t(layer) * S * k;
  for (int i = threadIdx.x; i < S; i += kThreads) {
    const int32_t *row = lid + int64_t(i) * k;
    for (int a = 0; a < k; ++a) {
      const int e = row[a];
      if (e < 0 || e >= E) continue;
      bool seen = false;
      for (int b = 0; b < a; ++b) seen |= row[b] == e;
      if (!seen) atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    const int c = counts[int64_t(layer) * E + e] + hist[e];
    counts[int64_t(layer) * E + e] = c;
    hist[e] = c;   // each thread rewrites only its own entries
  }
  __syncthreads();
  const int m = M < E ? M : E;
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int place = 0;
    for (int f = 0; f < E; ++f) place += (hist[f] > hist[e]) || (hist[f] == hist[e] && f < e);
    if (place < m) {
      experts[int64_t(layer) * m + place] = e;
      vals[int64_t(layer) * m + place] = hist[e];
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_elb_step(const int32_t *ids, int64_t L, int64_t S, int k, int64_t E, int32_t *counts, int M,
                            int32_t *experts, int32_t *vals, moe_stream_t stream) {
  MOE_REQUIRE(L >= 0 && L <= 65535 && S >= 0 && k >= 1 && k <= 64 && M >= 1, "need 0 <= L <= 65535, S >= 0, 1 <= k <= 64, M >= 1");
  MOE_REQUIRE(E >= 1 && E <= kMaxE && S * k < (int64_t(1) << 31), "need 1 <= E <= 256 and S*k in int32");
  if (L == 0) return MOE_OK;
  MOE_REQUIRE(counts && experts && vals && (ids || S == 0), "null pointer argument");
  elb_step_kernel<<<unsigned(L), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ids, int(S), k, int(E), counts,
                                                                                        M, experts, vals);
  return check_launch("elb_step");
}

extern "C" int moe_elb_accumulate(const int32_t *ids, int64_t L, int64_t S, int k, int64_t E, int32_t *counts,
                                  moe_stream_t stream) {
  MOE_REQUIRE(L >= 0 && S >= 0 && k >= 1 && k <= 64, "need L, S >= 0 and 1 <= k <= 64");
  MOE_REQUIRE(E >= 1 && E <= kMaxE, "need 1 <= E <= 256");
  MOE_REQUIRE(L <= 65535 && S * k < (int64_t(1) << 31), "L <= 65535 and S*k must fit in int32");
  if (L == 0 || S == 0) return MOE_OK;
  MOE_REQUIRE(ids && counts, "null pointer argument");
  elb_accumulate_kernel<<<unsigned(L), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ids, int(S), k, int(E),
                                                                                              counts);
  return check_launch("elb_accumulate");
}

extern "C" int moe_elb_topm(const int32_t *counts, int64_t L, int64_t E, int M, int32_t *experts, int32_t *vals,
                            moe_stream_t stream) {
  MOE_REQUIRE(L >= 0 && L <= 65535 && E >= 1 && E <= kMaxE && M >= 1, "need 0 <= L <= 65535, 1 <= E <= 256, M >= 1");
  if (L == 0) return MOE_OK;
  MOE_REQUIRE(counts && experts && vals, "null pointer argument");
  elb_topm_kernel<<<unsigned(L), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(counts, int(E), M, experts, vals);
  return check_launch("elb_topm");
}
