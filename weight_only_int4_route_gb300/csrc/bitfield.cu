// Lossless BF16 bit-field codec for expert weights: split a BF16 tensor into its exponent bytes
// and its sign|mantissa bytes, and merge the two back.
//
// "ZipMoE" (paper summary page), method details: the exponent bits of each BF16 expert tensor
// are low-entropy and are compressed on the host (E-chunks); the sign and mantissa bits are
// near random and stored byte-aligned (SM-chunks); after the host decompresses the exponent
// bytes, a device kernel merges both parts back into the original BF16 tensor, bit for bit.
//
// BF16: bit 15 sign, bits 14..7 exponent, bits 6..0 mantissa.  SM byte: sign in bit 7,
// mantissa in bits 6..0.  Both kernels stream 16 elements per thread (16-byte loads and stores
// of each plane) and handle the last n % 16 elements one by one.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kVecElems = 16;

__device__ __forceinline__ uint32_t merge2(uint32_t e2, uint32_t s2) {
  // e2, s2: two bytes each in the low bytes of the 16-bit lanes
  return ((s2 & 0x00800080u) << 8) | (e2 << 7) | (s2 & 0x007F007Fu);
}

__global__ void recombine_kernel(const uint8_t *__restrict__ exp, const uint8_t *__restrict__ sm, int64_t n,
                                 uint16_t *__restrict__ out) {
  const int64_t nvec = n / kVecElems;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < nvec; v += stride) {
    const uint4 e = reinterpret_cast<const uint4 *>(exp)[v];
    const uint4 s = reinterpret_cast<const uint4 *>(sm)[v];
    const uint32_t ew[4] = {e.x, e.y, e.z, e.w}, sw[4] = {s.x, s.y, s.z, s.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // bytes 0,1 and 2,3 of each word -> two 16-bit lanes
      o[2 * i] = merge2(__byte_perm(ew[i], 0u, 0x4140), __byte_perm(sw[i], 0u, 0x4140));
      o[2 * i + 1] = merge2(__byte_perm(ew[i], 0u, 0x4342), __byte_perm(sw[i], 0u, 0x4342));
    }
    uint4 *dst = reinterpret_cast<uint4 *>(out) + 2 * v;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  for (int64_t i = nvec * kVecElems + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += stride) {
    const uint32_t e = exp[i], s = sm[i];
    out[i] = uint16_t(((s & 0x80u) << 8) | (e << 7) | (s & 0x7Fu));
  }
}

__global__ void split_kernel(const uint16_t *__restrict__ in, int64_t n, uint8_t *__restrict__ exp,
                             uint8_t *__restrict__ sm) {
  const int64_t nvec = n / kVecElems;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < nvec; v += stride) {
    const uint4 a = reinterpret_cast<const uint4 *>(in)[2 * v], b = reinterpret_cast<const uint4 *>(in)[2 * v + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t eo[4], so[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // words 2i, 2i+1 hold elements 4i .. 4i+3
      const uint32_t e01 = (w[2 * i] >> 7) & 0x00FF00FFu, e23 = (w[2 * i + 1] >> 7) & 0x00FF00FFu;
      const uint32_t s01 = ((w[2 * i] >> 8) & 0x00800080u) | (w[2 * i] & 0x007F007Fu);
      const uint32_t s23 = ((w[2 * i + 1] >> 8) & 0x00800080u) | (w[2 * i + 1] & 0x007F007Fu);
      eo[i] = __byte_perm(e01, e23, 0x6420);   // low bytes of the four 16-bit lanes
      so[i] = __byte_perm(s01, s23, 0x6420);
    }
    reinterpret_cast<uint4 *>(exp)[v] = make_uint4(eo[0], eo[1], eo[2], eo[3]);
    reinterpret_cast<uint4 *>(sm)[v] = make_uint4(so[0], so[1], so[2], so[3]);
  }
  for (int64_t i = nvec * kVecElems + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += stride) {
    const uint32_t b = in[i];
    exp[i] = uint8_t((b >> 7) & 0xFFu);
    sm[i] = uint8_t(((b >> 8) & 0x80u) | (b & 0x7Fu));
  }
}

unsigned codec_grid(int64_t n) {
  const int64_t want = cdiv(std::max<int64_t>(n / kVecElems, 1), 256);
  const int64_t cap = int64_t(num_sms()) * 8;
  return unsigned(want < cap ? want : cap);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_bf16_recombine(const uint8_t *exp, const uint8_t *sm, int64_t n, uint16_t *out,
                                  moe_stream_t stream) {
  MOE_REQUIRE(n >= 0, "n must be >= 0");
  if (n == 0) return MOE_OK;
  MOE_REQUIRE(exp && sm && out, "null pointer argument");
  MOE_REQUIRE(aligned16(exp) && aligned16(sm) && aligned16(out), "pointers must be 16-byte aligned");
  recombine_kernel<<<codec_grid(n), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(exp, sm, n, out);
  return check_launch("bf16_recombine");
}

extern "C" int moe_bf16_split(const uint16_t *in, int64_t n, uint8_t *exp, uint8_t *sm, moe_stream_t stream) {
  MOE_REQUIRE(n >= 0, "n must be >= 0");
  if (n == 0) return MOE_OK;
  MOE_REQUIRE(in && exp && sm, "null pointer argument");
  MOE_REQUIRE(aligned16(in) && aligned16(exp) && aligned16(sm), "pointers must be 16-byte aligned");
  split_kernel<<<codec_grid(n), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(in, n, exp, sm);
  return check_launch("bf16_split");
}
