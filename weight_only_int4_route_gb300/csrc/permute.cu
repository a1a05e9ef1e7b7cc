// Token routing by expert: stable counting sort of flat rows f = t*k + j by expert id, then
// gather of the activation rows into expert-contiguous order.
//
// "Who Says Elephants Can't Run", section 3 workflow: the row index is appended to the
// gating output, the tuples are sorted with expert_idx as the key and the activation matrix
// is permuted by the result.  The page uses a library radix sort; with at most 256 keys a
// three-pass counting sort gives the same (stable) order:
//   1. per 256-row tile, count rows per expert;
//   2. one CTA turns the tile counts into expert offsets and per-(tile, expert) bases;
//   3. per tile, each row's rank among equal keys in the tile (warp match + per-warp
//      counts, so the order is stable in f) gives its position p; perm, inv_perm and the
//      gathered row xp[p] = x[f / k] are written.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTile = 256;
constexpr int kMaxE = 256;

__global__ void __launch_bounds__(kTile) count_kernel(const int32_t *__restrict__ ids, int64_t R,
                                                      int E, int32_t *__restrict__ tile_counts) {
  __shared__ int cnt[kMaxE];
  for (int e = threadIdx.x; e < E; e += kTile) cnt[e] = 0;
  __syncthreads();
  const int64_t f = int64_t(blockIdx.x) * kTile + threadIdx.x;
  if (f < R) {
    const int e = ids[f];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // out-of-range ids are dropped
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTile) tile_counts[int64_t(blockIdx.x) * E + e] = cnt[e];
}

// One CTA of kMaxE threads; thread e walks the tiles of expert e.
__global__ void __launch_bounds__(kMaxE) scan_kernel(const int32_t *__restrict__ tile_counts,
                                                     int ntiles, int E, int32_t *__restrict__ tile_base,
                                                     int32_t *__restrict__ offsets) {
  __shared__ int scratch[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E)
    for (int t = 0; t < ntiles; ++t) {
      tile_base[int64_t(t) * E + e] = total;
      total += tile_counts[int64_t(t) * E + e];
    }
  int start = 0;
  const int all = block_exclusive_scan(e < E ? total : 0, &start, scratch);
  if (e < E) {
    offsets[e] = start;
    for (int t = 0; t < ntiles; ++t) tile_base[int64_t(t) * E + e] += start;
  }
  if (e == 0) offsets[E] = all;
}

template <int VEC_BYTES>
__global__ void __launch_bounds__(kTile) scatter_kernel(const int32_t *__restrict__ ids,
                                                        const int32_t *__restrict__ tile_base,
                                                        const uint8_t *__restrict__ x, int64_t R,
                                                        int E, int k, int64_t row_bytes,
                                                        int32_t *__restrict__ perm,
                                                        int32_t *__restrict__ inv_perm,
                                                        uint8_t *__restrict__ xp) {
  __shared__ int wcount[kTile / 32][kMaxE];
  __shared__ int dest[kTile];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kTile / 32) * E; i += kTile) wcount[i / E][i % E] = 0;
  __syncthreads();
  const int64_t f = int64_t(blockIdx.x) * kTile + threadIdx.x;
  int e = f < R ? ids[f] : -1;
  if (e >= E) e = -1;
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank_in_warp == 0) wcount[warp][e] = __popc(same);
  __syncthreads();
  dest[threadIdx.x] = -1;
  if (e >= 0) {
    int p = tile_base[int64_t(blockIdx.x) * E + e] + rank_in_warp;
    for (int w = 0; w < warp; ++w) p += wcount[w][e];
    perm[p] = int32_t(f);
    inv_perm[f] = p;
    dest[threadIdx.x] = p;
  }
  __syncthreads();
  // gather rows: one warp per row, VEC_BYTES per lane per step
  const int64_t base = int64_t(blockIdx.x) * kTile;
  const int nrows = int(R - base < kTile ? R - base : kTile);
  for (int r = warp; r < nrows; r += kTile / 32) {
    if (dest[r] < 0) continue;  // row with an out-of-range id has no position
    const int64_t src_row = (base + r) / k;
    const uint8_t *src = x + src_row * row_bytes;
    uint8_t *dst = xp + int64_t(dest[r]) * row_bytes;
    for (int64_t c = int64_t(lane) * VEC_BYTES; c < row_bytes; c += 32 * VEC_BYTES) {
      if constexpr (VEC_BYTES == 16)
        *reinterpret_cast<uint4 *>(dst + c) = *reinterpret_cast<const uint4 *>(src + c);
      else
        *reinterpret_cast<uint2 *>(dst + c) = *reinterpret_cast<const uint2 *>(src + c);
    }
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
  __shared__ int wcount[kSmall / 32][kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int dest[kSmall];
  __shared__ int scratch[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < (kSmall / 32) * E; i += kSmall) wcount[i / E][i % E] = 0;
  __syncthreads();
  int e = tid < R ? ids[tid] : -1;
  if (e >= E) e = -1;
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
    for (int64_t c = int64_t(lane) * VEC_BYTES; c < row_bytes; c += 32 * VEC_BYTES) {
      if constexpr (VEC_BYTES == 16)
        *reinterpret_cast<uint4 *>(dst + c) = *reinterpret_cast<const uint4 *>(src + c);
      else
        *reinterpret_cast<uint2 *>(dst + c) = *reinterpret_cast<const uint2 *>(src + c);
    }
  }
}

}  // namespace
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
      permute_small_kernel<16><<<1, kSmall, 0, st>>>(ids, static_cast<const uint8_t *>(x), int(R), int(E), k, row_bytes,
                                                     offsets, perm, inv_perm, static_cast<uint8_t *>(xp));
    else
      permute_small_kernel<8><<<1, kSmall, 0, st>>>(ids, static_cast<const uint8_t *>(x), int(R), int(E), k, row_bytes,
                                                    offsets, perm, inv_perm, static_cast<uint8_t *>(xp));
    return check_launch("permute_small");
  }
  const int ntiles = int(cdiv(R, kTile));
  int32_t *tile_counts = static_cast<int32_t *>(workspace);
  int32_t *tile_base = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                                   align256(size_t(ntiles) * size_t(E) * 4));
  count_kernel<<<ntiles, kTile, 0, st>>>(ids, R, int(E), tile_counts);
  scan_kernel<<<1, kMaxE, 0, st>>>(tile_counts, ntiles, int(E), tile_base, offsets);
  if (row_bytes % 16 == 0)
    scatter_kernel<16><<<ntiles, kTile, 0, st>>>(ids, tile_base, static_cast<const uint8_t *>(x), R,
                                                 int(E), k, row_bytes, perm, inv_perm, static_cast<uint8_t *>(xp));
  else
    scatter_kernel<8><<<ntiles, kTile, 0, st>>>(ids, tile_base, static_cast<const uint8_t *>(x), R,
                                                int(E), k, row_bytes, perm, inv_perm, static_cast<uint8_t *>(xp));
  return check_launch("permute");
}
