// Weight packing and the Algorithm 1 dequant export.
//
// Storage ("Who Says Elephants Can't Run", section 3: expert quantization, Algorithm 1;
// optimized I2F, 8-bit and 4-bit dequantization): codes are kept offset-binary so that a
// kernel can OR them straight into the mantissa of a 16-bit magic number, and INT4 words
// use the interleaved nibble order [e0,e2,e4,e6,e1,e3,e5,e7] over 8 consecutive
// reduction-dim elements of one output channel.  Words are stored output-channel-major,
// (E, N, K/8), so each channel's reduction run is contiguous (K-major operand).
#include <type_traits>

#include "moe_internal.cuh"

namespace moe {
namespace {

// nibble slot of element i of an 8-element run: even i -> i/2, odd i -> 4 + i/2
__device__ __forceinline__ int int4_slot(int i) { return (i & 1) ? 4 + (i >> 1) : (i >> 1); }

__global__ void pack_int4_kernel(const int8_t *__restrict__ codes, uint32_t *__restrict__ words,
                                 int64_t E, int64_t K, int64_t N) {
  const int64_t J = K / 8;
  const int64_t total = E * J * N;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = idx % N, j = (idx / N) % J, e = idx / (N * J);
    const int8_t *src = codes + (e * K + 8 * j) * N + n;
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t u = uint32_t(int32_t(src[i * N]) + 8) & 0xFu;
      w |= u << (4 * int4_slot(i));
    }
    words[(e * N + n) * J + j] = w;
  }
}

__global__ void pack_int8_kernel(const int8_t *__restrict__ codes, uint32_t *__restrict__ words,
                                 int64_t E, int64_t K, int64_t N) {
  const int64_t J = K / 4;
  const int64_t total = E * J * N;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = idx % N, j = (idx / N) % J, e = idx / (N * J);
    const int8_t *src = codes + (e * K + 4 * j) * N + n;
    uint32_t w = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) w |= (uint32_t(int32_t(src[b * N]) + 128) & 0xFFu) << (8 * b);
    words[(e * N + n) * J + j] = w;
  }
}

// (E, K, N) -> (E, N, K) transpose of 16-bit values through a 32x32 shared tile.
__global__ void transpose16_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                   int64_t K, int64_t N) {
  __shared__ uint16_t tile[32][33];
  const int64_t e = blockIdx.z;
  const int64_t k0 = int64_t(blockIdx.y) * 32, n0 = int64_t(blockIdx.x) * 32;
  const uint16_t *s = src + e * K * N;
  uint16_t *d = dst + e * K * N;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t k = k0 + r, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[r][threadIdx.x] = s[k * N + n];
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t n = n0 + r, k = k0 + threadIdx.x;
    if (k < K && n < N) d[n * K + k] = tile[threadIdx.x][r];
  }
}

template <typename ST> __device__ __forceinline__ uint32_t bcast_pair(ST s) {
  typename Vec2<ST>::type v;
  v.x = s;
  v.y = s;
  return h2_as_u32(v);
}

template <typename OT> __device__ __forceinline__ OT cvt_from_pair(uint32_t h, int hi, __half) {
  const __half2 v = u32_as_h2(h);
  return from_f32<OT>(__half2float(hi ? __high2half(v) : __low2half(v)));
}
template <typename OT> __device__ __forceinline__ OT cvt_from_pair(uint32_t h, int hi, __nv_bfloat16) {
  const __nv_bfloat162 v = u32_as_b2(h);
  return from_f32<OT>(__bfloat162float(hi ? __high2bfloat16(v) : __low2bfloat16(v)));
}

// Algorithm 1 from the packed buffer.  When the output type is the scale type the value is
// produced by the mainloop's own routine (I2F, then RN(q*s) in that type); otherwise q*s is
// formed exactly in fp32 and rounded once to the output type.
template <typename ST, typename OT, int BITS>
__global__ void dequant_kernel(const uint32_t *__restrict__ words, const ST *__restrict__ scales,
                               OT *__restrict__ out, int64_t E, int64_t K, int64_t N, int group) {
  constexpr int PER = BITS == 4 ? 8 : 4;
  const int64_t J = K / PER;
  const int64_t G = group == 0 ? 1 : K / group;
  const int64_t total = E * J * N;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = idx % N, j = (idx / N) % J, e = idx / (N * J);
    const uint32_t w = words[(e * N + n) * J + j];
    const int64_t k0 = j * PER;
    const ST s = scales[(e * G + (group == 0 ? 0 : k0 / group)) * N + n];
    uint32_t h[PER / 2];
    if constexpr (BITS == 4) {
      uint32_t t[4];
      i2f_int4(w, t, ST());
#pragma unroll
      for (int p = 0; p < 4; ++p) h[p] = t[p];
    } else {
      uint32_t t[2];
      i2f_int8(w, t, ST());
      h[0] = t[0];
      h[1] = t[1];
    }
#pragma unroll
    for (int p = 0; p < PER / 2; ++p) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        OT v;
        if constexpr (sizeof(OT) == 2 && std::is_same<OT, ST>::value) {
          const uint32_t prod = scale_pair(h[p], bcast_pair(s), ST());
          v = cvt_from_pair<OT>(prod, hi, ST());
        } else {
          const float q = to_f32(cvt_from_pair<ST>(h[p], hi, ST()));
          v = from_f32<OT>(q * to_f32(s));  // exact product in fp32, one rounding
        }
        out[(e * K + k0 + 2 * p + hi) * N + n] = v;
      }
    }
  }
}

__global__ void untranspose16_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                     int64_t K, int64_t N) {
  // src (E, N, K) -> dst (E, K, N)
  __shared__ uint16_t tile[32][33];
  const int64_t e = blockIdx.z;
  const int64_t n0 = int64_t(blockIdx.y) * 32, k0 = int64_t(blockIdx.x) * 32;
  const uint16_t *s = src + e * K * N;
  uint16_t *d = dst + e * K * N;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t n = n0 + r, k = k0 + threadIdx.x;
    if (k < K && n < N) tile[r][threadIdx.x] = s[n * K + k];
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t k = k0 + r, n = n0 + threadIdx.x;
    if (k < K && n < N) d[k * N + n] = tile[threadIdx.x][r];
  }
}

int grid_for(int64_t total, int threads) {
  const int64_t want = cdiv(total, threads);
  const int64_t cap = int64_t(num_sms()) * 16;
  return int(want < cap ? (want > 0 ? want : 1) : cap);
}

int check_pack_args(int64_t E, int64_t K, int64_t N, int bits, int group) {
  MOE_REQUIRE(E >= 1 && K >= 1 && N >= 1, "E, K, N must be positive (E=%lld K=%lld N=%lld)",
              (long long)E, (long long)K, (long long)N);
  MOE_REQUIRE(bits == 4 || bits == 8 || bits == 16, "bits must be 4, 8 or 16 (got %d)", bits);
  MOE_REQUIRE(group == 0 || group == 128, "group must be 0 or 128 (got %d)", group);
  MOE_REQUIRE(bits != 16 || group == 0, "16-bit weights take no scales (group must be 0)");
  MOE_REQUIRE(bits != 4 || K % 8 == 0, "INT4 needs K %% 8 == 0 (K=%lld)", (long long)K);
  MOE_REQUIRE(bits != 8 || K % 4 == 0, "INT8 needs K %% 4 == 0 (K=%lld)", (long long)K);
  MOE_REQUIRE(group != 128 || K % 128 == 0, "group 128 needs K %% 128 == 0 (K=%lld)", (long long)K);
  MOE_REQUIRE(N % 8 == 0, "N %% 8 == 0 required (N=%lld)", (long long)N);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_packed_scale_offset(int64_t E, int64_t K, int64_t N, int bits) {
  if (E < 1 || K < 1 || N < 1 || (bits != 4 && bits != 8 && bits != 16)) return 0;
  return align256(packed_code_bytes(E, K, N, bits));
}

extern "C" size_t moe_packed_size(int64_t E, int64_t K, int64_t N, int bits, int group) {
  if (check_pack_args(E, K, N, bits, group) != MOE_OK) return 0;
  size_t bytes = align256(packed_code_bytes(E, K, N, bits));
  if (bits != 16) bytes += align256(size_t(E) * size_t(scale_groups(K, group)) * size_t(N) * 2);
  return bytes;
}

extern "C" int moe_pack_weights(const void *codes, const void *scales, int w_dtype, int64_t E,
                                int64_t K, int64_t N, int bits, int group, void *packed,
                                size_t packed_bytes, moe_stream_t stream) {
  MOE_TRY(check_pack_args(E, K, N, bits, group));
  MOE_REQUIRE(is16(w_dtype), "w_dtype must be MOE_F16 or MOE_BF16");
  MOE_REQUIRE(codes && packed, "codes and packed must be non-null");
  MOE_REQUIRE(aligned16(codes) && aligned16(packed), "codes and packed must be 16-byte aligned");
  MOE_REQUIRE(bits == 16 ? scales == nullptr : scales != nullptr,
              bits == 16 ? "16-bit weights take no scales" : "scales must be non-null");
  MOE_REQUIRE(packed_bytes >= moe_packed_size(E, K, N, bits, group),
              "packed buffer too small (%zu < %zu)", packed_bytes, moe_packed_size(E, K, N, bits, group));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int threads = 256;
  if (bits == 4) {
    pack_int4_kernel<<<grid_for(E * (K / 8) * N, threads), threads, 0, st>>>(
        static_cast<const int8_t *>(codes), static_cast<uint32_t *>(packed), E, K, N);
  } else if (bits == 8) {
    pack_int8_kernel<<<grid_for(E * (K / 4) * N, threads), threads, 0, st>>>(
        static_cast<const int8_t *>(codes), static_cast<uint32_t *>(packed), E, K, N);
  } else {
    MOE_SUPPORT(E <= 65535, "16-bit packing supports E <= 65535");
    dim3 grid(unsigned(cdiv(N, 32)), unsigned(cdiv(K, 32)), unsigned(E));
    transpose16_kernel<<<grid, dim3(32, 8), 0, st>>>(static_cast<const uint16_t *>(codes),
                                                     static_cast<uint16_t *>(packed), K, N);
  }
  MOE_TRY(check_launch("pack"));
  if (bits != 16) {
    MOE_REQUIRE(aligned16(scales), "scales must be 16-byte aligned");
    const size_t sbytes = size_t(E) * size_t(scale_groups(K, group)) * size_t(N) * 2;
    char *dst = static_cast<char *>(packed) + moe_packed_scale_offset(E, K, N, bits);
    if (cudaMemcpyAsync(dst, scales, sbytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return check_launch("pack scales copy");
  }
  return MOE_OK;
}

extern "C" int moe_dequant(const void *packed, int w_dtype, int64_t E, int64_t K, int64_t N,
                           int bits, int group, int out_dtype, void *w_out, moe_stream_t stream) {
  MOE_TRY(check_pack_args(E, K, N, bits, group));
  MOE_REQUIRE(is16(w_dtype), "w_dtype must be MOE_F16 or MOE_BF16");
  MOE_REQUIRE(out_dtype == MOE_F16 || out_dtype == MOE_BF16 || out_dtype == MOE_F32, "bad out_dtype");
  MOE_REQUIRE(packed && w_out && aligned16(packed) && aligned16(w_out),
              "packed and w_out must be non-null and 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int threads = 256;
  if (bits == 16) {
    MOE_SUPPORT(E <= 65535, "16-bit dequant supports E <= 65535");
    MOE_SUPPORT(out_dtype == w_dtype, "16-bit weights dequantize to their own type only");
    dim3 grid(unsigned(cdiv(K, 32)), unsigned(cdiv(N, 32)), unsigned(E));
    untranspose16_kernel<<<grid, dim3(32, 8), 0, st>>>(static_cast<const uint16_t *>(packed),
                                                       static_cast<uint16_t *>(w_out), K, N);
    return check_launch("dequant16");
  }
  const uint32_t *words = static_cast<const uint32_t *>(packed);
  const void *sc = static_cast<const char *>(packed) + moe_packed_scale_offset(E, K, N, bits);
  const int64_t total = E * (K / (bits == 4 ? 8 : 4)) * N;
  const int grid = grid_for(total, threads);
#define MOE_DQ(ST, OT, B)                                                                    \
  dequant_kernel<ST, OT, B><<<grid, threads, 0, st>>>(words, static_cast<const ST *>(sc),    \
                                                      static_cast<OT *>(w_out), E, K, N, group)
#define MOE_DQ_OUT(ST, B)                                              \
  do {                                                                 \
    if (out_dtype == MOE_F16) MOE_DQ(ST, __half, B);                    \
    else if (out_dtype == MOE_BF16) MOE_DQ(ST, __nv_bfloat16, B);       \
    else MOE_DQ(ST, float, B);                                          \
  } while (0)
  if (w_dtype == MOE_F16) {
    if (bits == 4) MOE_DQ_OUT(__half, 4); else MOE_DQ_OUT(__half, 8);
  } else {
    if (bits == 4) MOE_DQ_OUT(__nv_bfloat16, 4); else MOE_DQ_OUT(__nv_bfloat16, 8);
  }
#undef MOE_DQ_OUT
#undef MOE_DQ
  return check_launch("dequant");
}
