// Token routing by expert: stable counting sort of flat rows f = t*k + j by expert id, then
// gather of the activation rows into expert-contiguous order.
//
// "Who Says Elephants Can't Run", section 3 workflow: the row index is appended to the
// gating output, the tuples are sorted with expert_idx as the key and the activation matrix
// is permuted by the result.  The page uses a library radix sort; with at most 256 keys a
// three-pass counting sort gives the same (stable) order:
//   1. per 256-row tile, count rows per expert;
//   2. the tile counts become expert offsets and per-(tile, expert) bases (one CTA, or each
//      scatter CTA for its own tile when the count table is small);
//   3. per tile, each row's rank among equal keys in the tile (warp match + per-warp
//      counts, so the order is stable in f) gives its position p; perm, inv_perm and the
//      gathered row xp[p] = x[f / k] are written.  kSub CTAs share a tile: each recomputes
//      the tile's positions (cheap) and copies its own slice of the rows, so the row copy --
//      the bulk of the bytes -- runs on many SMs.
#include <type_traits>

#include "moe_internal.cuh"

namespace moe {

MOE_DEFINE_CHECK_WORD(permute)

namespace {

constexpr int kTile = 256;
constexpr int kMaxE = 256;
constexpr int kSub = 32;  // CTAs per tile in the scatter (each copies kTile / kSub rows: one per warp)
constexpr int kFusedScanMax = 16384;   // tile-count entries up to which the scatter does the scan

__global__ void __launch_bounds__(kTile) count_kernel(const int32_t *__restrict__ ids, int64_t R,
                                                      int E, int32_t *__restrict__ tile_counts) {
  pdl_enter();   // see launch_pdl
  __shared__ int cnt[kMaxE];
  for (int e = threadIdx.x; e < E; e += kTile) cnt[e] = 0;
  __syncthreads();
  const int64_t f = int64_t(blockIdx.x) * kTile + threadIdx.x;
  if (f < R) {
    const int e = ids[f];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // out-of-range ids are dropped
    else if (MOE_CHECKED) check_fail(kCheckExpertId);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTile) tile_counts[int64_t(blockIdx.x) * E + e] = cnt[e];
}

// One CTA of kMaxE threads; thread e walks the tiles of expert e (loads batched so they are
// in flight together), then the expert totals are scanned and the bases written once.
__global__ void __launch_bounds__(kMaxE) scan_kernel(const int32_t *__restrict__ tile_counts,
                                                     int ntiles, int E, int32_t *__restrict__ tile_base,
                                                     int32_t *__restrict__ offsets) {
  pdl_enter();   // see launch_pdl
  __shared__ int scratch[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    int t = 0;
    for (; t + 8 <= ntiles; t += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = tile_counts[int64_t(t + u) * E + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) total += c[u];
    }
    for (; t < ntiles; ++t) total += tile_counts[int64_t(t) * E + e];
  }
  int start = 0;
  const int all = block_exclusive_scan(e < E ? total : 0, &start, scratch);
  if (e < E) {
    offsets[e] = start;
    int run = start;
    int t = 0;
    for (; t + 8 <= ntiles; t += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = tile_counts[int64_t(t + u) * E + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        tile_base[int64_t(t + u) * E + e] = run;
        run += c[u];
      }
    }
    for (; t < ntiles; ++t) {
      tile_base[int64_t(t) * E + e] = run;
      run += tile_counts[int64_t(t) * E + e];
    }
  }
  if (e == 0) offsets[E] = all;
}

// Copy one row: the lane's pieces are all loaded before any is stored (the loads of a row are
// in flight together).
template <int VEC_BYTES>
__device__ __forceinline__ void copy_row(const uint8_t *src, uint8_t *dst, int64_t row_bytes, int lane) {
  using V = typename std::conditional<VEC_BYTES == 16, uint4, uint2>::type;
  constexpr int kBatch = 4;
  for (int64_t c0 = int64_t(lane) * VEC_BYTES; c0 < row_bytes; c0 += int64_t(kBatch) * 32 * VEC_BYTES) {
    V v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t c = c0 + int64_t(b) * 32 * VEC_BYTES;
      if (c < row_bytes) v[b] = *reinterpret_cast<const V *>(src + c);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t c = c0 + int64_t(b) * 32 * VEC_BYTES;
      if (c < row_bytes) *reinterpret_cast<V *>(dst + c) = v[b];
    }
  }
}

// tile_base == nullptr: the CTA derives its tile's bases from all tile counts itself (expert
// totals and the counts of earlier tiles, summed with shared-memory integer atomics, so the
// result does not depend on their order) and CTA 0 writes the expert offsets; used when the
// count table is small, which saves the scan launch.
template <int VEC_BYTES>
__global__ void __launch_bounds__(kTile) scatter_kernel(const int32_t *__restrict__ ids,
                                                        const int32_t *__restrict__ tile_counts,
                                                        const int32_t *__restrict__ tile_base,
                                                        int ntiles, const uint8_t *__restrict__ x, int64_t R,
                                                        int E, int k, int64_t row_bytes,
                                                        int32_t *__restrict__ offsets,
                                                        int32_t *__restrict__ perm,
                                                        int32_t *__restrict__ inv_perm,
                                                        uint8_t *__restrict__ xp) {
  pdl_enter();   // see launch_pdl
  __shared__ int wcount[kTile / 32][kMaxE];
  __shared__ int dest[kTile];
  __shared__ int tot[kMaxE], pre[kMaxE];
  __shared__ int scratch[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tile = blockIdx.x / kSub, sub = blockIdx.x % kSub;
  for (int i = threadIdx.x; i < (kTile / 32) * E; i += kTile) wcount[i / E][i % E] = 0;
  if (tile_base == nullptr)
    for (int e = threadIdx.x; e < E; e += kTile) tot[e] = pre[e] = 0;
  __syncthreads();
  if (tile_base == nullptr) {
    for (int i = threadIdx.x; i < ntiles * E; i += kTile) {
      const int t = i / E, e = i % E;
      const int c = tile_counts[i];
      if (c) {
        atomicAdd(&tot[e], c);
        if (t < tile) atomicAdd(&pre[e], c);
      }
    }
    __syncthreads();
    int start = 0;
    const int v = threadIdx.x < E ? tot[threadIdx.x] : 0;   // E <= kMaxE == kTile
    const int all = block_exclusive_scan(v, &start, scratch);
    if (threadIdx.x < E) {
      pre[threadIdx.x] += start;   // base of (this tile, expert)
      if (blockIdx.x == 0) offsets[threadIdx.x] = start;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) offsets[E] = all;
  }
  const int64_t f = int64_t(tile) * kTile + threadIdx.x;
  int e = f < R ? ids[f] : -1;
  if (e < 0 || e >= E) e = -1;
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank_in_warp == 0) wcount[warp][e] = __popc(same);
  __syncthreads();
  dest[threadIdx.x] = -1;
  if (e >= 0) {
    int p = (tile_base ? tile_base[int64_t(tile) * E + e] : pre[e]) + rank_in_warp;
    for (int w = 0; w < warp; ++w) p += wcount[w][e];
    if (sub == 0) {
      perm[p] = int32_t(f);
      inv_perm[f] = p;
    }
    dest[threadIdx.x] = p;
  } else if (sub == 0 && f < R) {
    inv_perm[f] = -1;   // dropped row: no position
  }
  __syncthreads();
  // gather this CTA's slice of the tile's rows: one warp per row
  const int64_t base = int64_t(tile) * kTile;
  const int nrows = int(R - base < kTile ? R - base : kTile);
  const int r_end = min(nrows, (sub + 1) * (kTile / kSub));
  for (int r = sub * (kTile / kSub) + warp; r < r_end; r += kTile / 32) {
    if (dest[r] < 0) continue;  // row with an out-of-range id has no position
    copy_row<VEC_BYTES>(x + ((base + r) / k) * row_bytes, xp + int64_t(dest[r]) * row_bytes, row_bytes, lane);
  }
}

// Whole permute in one CTA for small batches (R <= 1024 rows, decode steps): per-warp counts,
// prefix over warps and experts, stable ranks from warp matches, then the row gather; one
// launch instead of three.
constexpr int kSmall = 1024;

template <int VEC_BYTES>
__global__ void __launch_bounds__(kSmall) permute_small_kernel(const int32_t *__restrict__ ids,
                                                               const uint8_t *__restrict__ x, int R, int E, int k,
                                                               int64_t row_bytes, int32_t *__restrict__ offsets,
                                                               int32_t *__restrict__ perm,
                                                               int32_t *__restrict__ inv_perm,
                                                               uint8_t *__restrict__ xp) {
  pdl_enter();   // see launch_pdl
  __shared__ int wcount[kSmall / 32][kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int dest[kSmall];
  __shared__ int scratch[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < (kSmall / 32) * E; i += kSmall) wcount[i / E][i % E] = 0;
  __syncthreads();
  int e = tid < R ? ids[tid] : -1;
  if (tid < R && (e < 0 || e >= E)) {
    e = -1;
    inv_perm[tid] = -1;   // dropped row: no position
    if (MOE_CHECKED) check_fail(kCheckExpertId);
  }
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank_in_warp == 0) wcount[warp][e] = __popc(same);
  __syncthreads();
  int total = 0;
  if (tid < E)
    for (int w = 0; w < kSmall / 32; ++w) {
      const int c = wcount[w][tid];
      wcount[w][tid] = total;
      total += c;
    }
  int start = 0;
  const int all = block_exclusive_scan(tid < E ? total : 0, &start, scratch);
  if (tid < E) {
    s_off[tid] = start;
    offsets[tid] = start;
  }
  if (tid == 0) offsets[E] = all;
  __syncthreads();
  dest[tid] = -1;
  if (e >= 0) {
    const int p = s_off[e] + wcount[warp][e] + rank_in_warp;
    perm[p] = tid;
    inv_perm[tid] = p;
    dest[tid] = p;
  }
  __syncthreads();
  for (int r = warp; r < R; r += kSmall / 32) {
    if (dest[r] < 0) continue;
    const uint8_t *src = x + int64_t(r / k) * row_bytes;
    uint8_t *dst = xp + int64_t(dest[r]) * row_bytes;
    copy_row<VEC_BYTES>(src, dst, row_bytes, lane);
  }
}

}  // namespace

int permute_launches(int64_t R, int64_t E) {
  if (R <= kSmall) return 1;
  return cdiv(R, kTile) * E <= kFusedScanMax ? 2 : 3;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int64_t T, int64_t E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  const int64_t ntiles = cdiv(T * k, kTile);
  return 2 * align256(size_t(ntiles) * size_t(E) * 4);
}

extern "C" int moe_permute(const int32_t *ids, const void *x, int x_dtype, int64_t T, int64_t d,
                           int64_t E, int k, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                           void *xp, void *workspace, size_t workspace_bytes, moe_stream_t stream) {
  MOE_REQUIRE(is16(x_dtype), "x_dtype must be MOE_F16 or MOE_BF16");
  MOE_REQUIRE(T >= 0 && d >= 4 && d % 4 == 0, "need T >= 0 and d %% 4 == 0");
  MOE_REQUIRE(E >= 1 && E <= kMaxE && k >= 1 && k <= E, "need 1 <= k <= E <= 256");
  MOE_REQUIRE(T * k < (int64_t(1) << 31), "T*k must fit in int32");
  MOE_REQUIRE(offsets && aligned16(offsets), "offsets must be non-null and 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t R = T * k;
  if (R == 0) {
    if (cudaMemsetAsync(offsets, 0, size_t(E + 1) * 4, st) != cudaSuccess) return check_launch("permute memset");
    return MOE_OK;
  }
  MOE_REQUIRE(ids && x && perm && inv_perm && xp, "null pointer argument");
  MOE_REQUIRE(aligned16(ids) && aligned16(x) && aligned16(perm) && aligned16(inv_perm) && aligned16(xp),
              "pointers must be 16-byte aligned");
  const size_t need = moe_permute_workspace_size(T, E, k);
  MOE_REQUIRE(workspace && aligned16(workspace), "workspace must be non-null and 16-byte aligned");
  if (workspace_bytes < need)
    return set_error(MOE_ERR_WORKSPACE, "permute workspace %zu < %zu bytes", workspace_bytes, need);
  const int64_t row_bytes = d * 2;
  if (R <= kSmall) {
    if (row_bytes % 16 == 0)
      launch_pdl(permute_small_kernel<16>, dim3(1), dim3(kSmall), 0, st, ids, static_cast<const uint8_t *>(x), int(R), int(E), k, row_bytes,
                                                     offsets, perm, inv_perm, static_cast<uint8_t *>(xp));
    else
      launch_pdl(permute_small_kernel<8>, dim3(1), dim3(kSmall), 0, st, ids, static_cast<const uint8_t *>(x), int(R), int(E), k, row_bytes,
                                                    offsets, perm, inv_perm, static_cast<uint8_t *>(xp));
    return check_launch("permute_small");
  }
  const int ntiles = int(cdiv(R, kTile));
  int32_t *tile_counts = static_cast<int32_t *>(workspace);
  int32_t *tile_base = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                                   align256(size_t(ntiles) * size_t(E) * 4));
  launch_pdl(count_kernel, dim3(ntiles), dim3(kTile), 0, st, ids, R, int(E), tile_counts);
  const bool fused = int64_t(ntiles) * E <= kFusedScanMax;
  if (!fused) launch_pdl(scan_kernel, dim3(1), dim3(kMaxE), 0, st, tile_counts, ntiles, int(E), tile_base, offsets);
  const int32_t *tb = fused ? nullptr : tile_base;
  const uint8_t *xb = static_cast<const uint8_t *>(x);
  uint8_t *xpb = static_cast<uint8_t *>(xp);
  if (row_bytes % 16 == 0)
    launch_pdl(scatter_kernel<16>, dim3(ntiles * kSub), dim3(kTile), 0, st, ids, tile_counts, tb, ntiles, xb, R, int(E), k, row_bytes,
                                                        offsets, perm, inv_perm, xpb);
  else
    launch_pdl(scatter_kernel<8>, dim3(ntiles * kSub), dim3(kTile), 0, st, ids, tile_counts, tb, ntiles, xb, R, int(E), k, row_bytes,
                                                       offsets, perm, inv_perm, xpb);
  return check_launch("permute");
}
