// Internal helpers shared by the libmoe translation units (device and host).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

// Checked build (compiled with -DMOE_CHECKED=1 into a separate library): kernels bounds-check
// the indices they read from device memory -- expert ids, expert row offsets, permutation
// entries -- skip the access when one is out of range and record the kind of violation in a
// device check word (moe_check_status reads it).  The plain build checks nothing beyond what
// its documented behaviour needs.
#ifndef MOE_CHECKED
#define MOE_CHECKED 0
#endif

namespace moe {

// Bits of the device check word.
enum : int { kCheckExpertId = 1, kCheckOffsets = 2, kCheckPerm = 4 };

// One check word per translation unit (device variables are not shared across separately
// compiled files); check_word_take_<tu> ORs the word into *out and clears it.
#define MOE_DEFINE_CHECK_WORD(tu)                                                               \
  namespace {                                                                                   \
  __device__ int g_check_word = 0;                                                              \
  __device__ __forceinline__ void check_fail(int bit) { atomicOr(&g_check_word, bit); }         \
  }                                                                                             \
  int check_word_take_##tu(int *out) {                                                          \
    int v = 0;                                                                                  \
    if (cudaMemcpyFromSymbol(&v, g_check_word, sizeof(int)) != cudaSuccess)                     \
      return check_launch("check word read");                                                   \
    if (v != 0) {                                                                               \
      const int zero = 0;                                                                       \
      if (cudaMemcpyToSymbol(g_check_word, &zero, sizeof(int)) != cudaSuccess)                  \
        return check_launch("check word reset");                                                \
    }                                                                                           \
    *out |= v;                                                                                  \
    return MOE_OK;                                                                              \
  }
int check_word_take_permute(int *out);
int check_word_take_combine(int *out);
int check_word_take_gemm_tc(int *out);
int check_word_take_gemv(int *out);
int check_word_take_gemm_mma(int *out);

// ---------------------------------------------------------------- host side

int set_error(int code, const char *fmt, ...);
int check_launch(const char *what);  // MOE_OK or MOE_ERR_CUDA with the runtime's message
int num_sms();                       // SM count of the current device (cached)

// Programmatic dependent launch.  The kernels of the layer chain are launched with programmatic
// stream serialization: a kernel may be placed on the SMs while its predecessor in the stream is
// still running, and its first act (pdl_enter) is to let its own successor be launched likewise
// and then wait until the predecessor has completed and its memory is visible -- before any
// global memory is read or written, so the stream order of every access is as without it.  A
// kernel launched without the attribute passes the wait at once.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool is16(int dt) { return dt == MOE_F16 || dt == MOE_BF16; }
inline size_t dtype_size(int dt) { return dt == MOE_F32 ? 4 : 2; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

#define MOE_REQUIRE(cond, ...)                                        \
  do {                                                                \
    if (!(cond)) return ::moe::set_error(MOE_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define MOE_SUPPORT(cond, ...)                                        \
  do {                                                                \
    if (!(cond)) return ::moe::set_error(MOE_ERR_UNSUPPORTED, __VA_ARGS__); \
  } while (0)
#define MOE_TRY(expr)            \
  do {                           \
    int _st = (expr);            \
    if (_st != MOE_OK) return _st; \
  } while (0)

// Packed-weight geometry (see include/moe.h).
inline size_t packed_code_bytes(int64_t E, int64_t K, int64_t N, int bits) {
  return size_t(E) * size_t(N) * size_t(K) * size_t(bits) / 8;
}
inline int64_t scale_groups(int64_t K, int group) { return group == 0 ? 1 : K / group; }

// Which grouped-GEMM kernel runs and how it is split (shared by size queries and launches).
enum : int { kKindMma = 0, kKindTc = 1, kKindGemv = 2 };
struct GemmPlan {
  int kind;    // kKindMma (warp MMA, mid-size batches), kKindTc (tcgen05), kKindGemv (decode stream)
  int nt;      // decode kernel: n8 tiles of routed rows per unit
  int ch;      // decode kernel: 128-wide chunks per K split
  int ng;      // decode kernel: channel groups of mt m16 tiles
  int mt;      // decode kernel: m16 tiles (16 channels each) per unit
  int mb;      // m16 tiles per CTA tile (rows per tile = 16 * mb)
  int splits;  // split-K factor
  int ks;      // K per split (multiple of 128)
  int ncb;     // channel blocks
  bool partial;  // fp32 partial slices instead of the fused epilogue
  bool tc;       // rows per active expert large enough for the tcgen05 path
};
GemmPlan plan_gemm(int64_t R, int64_t E, int64_t K, int64_t N, int bits, int act, bool want_partial);
bool gemv_shape_ok(int64_t K, int64_t N, int bits, int act);
GemmPlan plan_gemv(int64_t R, int64_t E, int64_t K, int64_t N, int bits, int act, bool want_partial);

struct GemmArgs {
  const void *a;
  const void *w;       // code / 16-bit weight region of the packed buffer
  const void *scales;  // scale region or nullptr
  const int32_t *offsets;
  void *out;
  float *partial;
  int64_t R;
  int E, K, N;
  int group;
  int act;
  int out_dtype;
  int a_dtype;
  int bits;
  // tcgen05 kernel only, top-1 un-permute fused into the epilogue: permuted row p is written to
  // output row row_dest[p], times row_gate[row_dest[p]] (nullptr: row p, no factor)
  const int32_t *row_dest;
  const float *row_gate;
};
// Enqueue the grouped GEMM described by `g` with plan `pl`.  When pl.partial, the fp32
// accumulators (times per-channel scales) go to g.partial (splits, R, N).  Dispatches to the
// tcgen05 kernel when the plan and the shapes allow it, else to the warp-MMA kernel.
int launch_gemm(const GemmArgs &g, const GemmPlan &pl, cudaStream_t st);
int launch_gemm_mma(const GemmArgs &g, const GemmPlan &pl, cudaStream_t st);
int launch_gemv(const GemmArgs &g, const GemmPlan &pl, cudaStream_t st);
bool tc_supported(const GemmArgs &g);
// Shapes the tcgen05 kernel takes (the launch also needs an offsets array).
bool tc_shape_ok(int64_t E, int64_t K, int64_t N, int bits, int group, int act);
int launch_gemm_tc(const GemmArgs &g, cudaStream_t st);
// CTA pairs for the quantized tcgen05 GEMM (moe_set_gemm_pairs): returns the previous setting
int set_gemm_pairs(int on);
int read_device_error(cudaStream_t st, int *out);
int decode_error_take(int *out);   // device error word of the one-launch decode layer

// One-launch decode layer (decode_layer.cu): whether it takes a layer of T tokens, how the work
// is cut, and the layout of its own region of the layer workspace.
struct DecodePlan {
  bool ok;
  int NCR, S2, CH2, S3, CH3, rcmax, nts;
  size_t o_rpart, o_ypart, o_hs, o_yspart, o_rctab, o_ctrl, bytes;   // offsets inside the region
};
DecodePlan plan_decode(const moe_layer_desc *ds, int64_t T, int64_t warps);
int decode_warps();
int launch_decode_layer(const moe_layer_desc *ds, const moe_layer_weights *w, const void *x, int64_t T, void *out,
                        int32_t *ids, float *gate, int32_t *offs, int32_t *perm, int32_t *inv, void *h, char *fused,
                        const DecodePlan &pl, bool zero_ctrl, cudaStream_t st);
// Kernel launches of one moe_permute call for R rows over E experts.
int permute_launches(int64_t R, int64_t E);
// out[r, c] = act(sum_s part[s, r, c]) (SWIGLU pairs column c with c + N/2).
int launch_reduce_act(const float *part, int splits, int64_t R, int N, int act, void *out,
                      int out_dtype, cudaStream_t st);
// Combine with split slices: out[t] = sum_j g[t,j] * sum_s y[s, inv[t*k+j]] + sum_s sh[s, t].
int launch_combine(const void *y, int y_dtype, int ysplits, const int32_t *inv_perm,
                   const float *gate, const void *sh, int sh_dtype, int shsplits, int64_t T,
                   int64_t d, int k, void *out, int out_dtype, cudaStream_t st);

// ---------------------------------------------------------------- device side

template <typename T> struct Vec2;
template <> struct Vec2<__half> { using type = __half2; };
template <> struct Vec2<__nv_bfloat16> { using type = __nv_bfloat162; };

__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }
__device__ __forceinline__ uint32_t h2_as_u32(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ __nv_bfloat162 u32_as_b2(uint32_t v) {
  return *reinterpret_cast<__nv_bfloat162 *>(&v);
}

// ---- magic-number integer-to-float ("optimized I2F", FT-MoE review section 3) ----------
// An fp16 with exponent field 1024 keeps an integer 0 <= u < 1024 exactly in its mantissa:
// OR-ing u into 0x6400 gives 1024 + u.  bf16 keeps only 7 mantissa bits, so 128.0 (0x4300)
// is the magic there and u must stay below 128.

// INT4 word -> four 16-bit pairs (e0,e1) (e2,e3) (e4,e5) (e6,e7) holding q = u - 8.
// Pair p lives in bits 4p and 16 + 4p (nibble slots p and p + 4 of the interleaved word).
//
// The steps are written as single PTX instructions (one lop3 per masked OR, one shr per
// shift): this conversion is the integer-ALU bound part of a weight stream, and the plain C++
// form of the same expressions was measured to compile to about four more integer instructions
// per word.
__device__ __forceinline__ void i2f_int4(uint32_t w, uint32_t (&h)[4], __half) {
  uint32_t w8, t[4];
  asm("shr.b32 %0, %1, 8;\n" : "=r"(w8) : "r"(w));
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;\n" : "=r"(t[0]) : "r"(w));    // 1024 + u
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;\n" : "=r"(t[1]) : "r"(w));    // 1024 + 16 u
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;\n" : "=r"(t[2]) : "r"(w8));
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;\n" : "=r"(t[3]) : "r"(w8));
  // lower nibble: (1024 + u) - 1032; upper nibble kept in place: (1024 + 16 u) / 16 - 72
  const uint32_t bias = 0x64086408u, sixteenth = 0x2C002C00u, bias16 = 0xD480D480u;   // 1032, 1/16, -72
  asm("sub.f16x2 %0, %1, %2;\n" : "=r"(h[0]) : "r"(t[0]), "r"(bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(h[1]) : "r"(t[1]), "r"(sixteenth), "r"(bias16));
  asm("sub.f16x2 %0, %1, %2;\n" : "=r"(h[2]) : "r"(t[2]), "r"(bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(h[3]) : "r"(t[3]), "r"(sixteenth), "r"(bias16));
}

__device__ __forceinline__ void i2f_int4(uint32_t w, uint32_t (&h)[4], __nv_bfloat16) {
  uint32_t t[4];
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;\n" : "=r"(t[0]) : "r"(w));    // 128 + u
  asm("{\n .reg .b32 s;\n shr.b32 s, %1, 4;\n lop3.b32 %0, s, 0x000F000F, 0x43004300, 0xEA;\n}\n"
      : "=r"(t[1]) : "r"(w));
  asm("{\n .reg .b32 s;\n shr.b32 s, %1, 8;\n lop3.b32 %0, s, 0x000F000F, 0x43004300, 0xEA;\n}\n"
      : "=r"(t[2]) : "r"(w));
  asm("{\n .reg .b32 s;\n shr.b32 s, %1, 12;\n lop3.b32 %0, s, 0x000F000F, 0x43004300, 0xEA;\n}\n"
      : "=r"(t[3]) : "r"(w));
#pragma unroll
  for (int p = 0; p < 4; ++p) asm("sub.bf16x2 %0, %1, %2;\n" : "=r"(h[p]) : "r"(t[p]), "r"(0x43084308u));   // - 136
}

// INT8 word (byte b = element b, u = q + 128) -> two pairs (e0,e1) (e2,e3).
__device__ __forceinline__ void i2f_int8(uint32_t w, uint32_t (&h)[2], __half) {
  const uint32_t t0 = __byte_perm(w, 0x64646464u, 0x5140);  // [u0, 0x64, u1, 0x64] = 1024 + u
  const uint32_t t1 = __byte_perm(w, 0x64646464u, 0x5342);
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152 = 1024 + 128
  h[0] = h2_as_u32(__hsub2(u32_as_h2(t0), bias));
  h[1] = h2_as_u32(__hsub2(u32_as_h2(t1), bias));
}

// bf16 cannot hold a byte in its mantissa; go through the fp32 magic 2^23 (exact for
// |q| <= 128, which also fits bf16's 8 significant bits).
__device__ __forceinline__ float i2f_int8_byte_f32(uint32_t w, int b) {
  const uint32_t sel = 0x7540u | uint32_t(b);                 // [u_b, 0, 0, 0x4B]
  return __uint_as_float(__byte_perm(w, 0x4B000000u, sel)) - 8388736.0f;  // 2^23 + 128
}
__device__ __forceinline__ void i2f_int8(uint32_t w, uint32_t (&h)[2], __nv_bfloat16) {
  h[0] = h2_as_u32(__floats2bfloat162_rn(i2f_int8_byte_f32(w, 0), i2f_int8_byte_f32(w, 1)));
  h[1] = h2_as_u32(__floats2bfloat162_rn(i2f_int8_byte_f32(w, 2), i2f_int8_byte_f32(w, 3)));
}

// Multiply a pair by a broadcast scale: RN(q * s), one rounding of the exact product.
__device__ __forceinline__ uint32_t scale_pair(uint32_t h, uint32_t s2, __half) {
  return h2_as_u32(__hmul2(u32_as_h2(h), u32_as_h2(s2)));
}
__device__ __forceinline__ uint32_t scale_pair(uint32_t h, uint32_t s2, __nv_bfloat16) {
  return h2_as_u32(__hmul2(u32_as_b2(h), u32_as_b2(s2)));
}

// ---- activations ----------------------------------------------------------------------
__device__ __forceinline__ float act_relu(float x) { return fmaxf(x, 0.0f); }
// GELU(x) = 0.5 x (1 + erf(x / sqrt 2)).  erf from Abramowitz & Stegun, Handbook of Mathematical
// Functions, formula 7.1.26 (Hastings' approximation): for z >= 0,
//   erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),   t = 1 / (1 + p z),
// with the book's coefficients and |error| <= 1.5e-7; by odd symmetry
//   x >= 0: GELU = x - q,   x < 0: GELU = q,   q = 0.5 x (a1 t + ... + a5 t^5) exp(-x^2 / 2).
// The reciprocal and the exponential are the hardware approximations (rcp.approx, ex2.approx),
// adding ~1e-7; no branch, so a warp holding both signs runs one path.  Measured against a
// float64 erf it stays within 1e-6 * max(1, |x|) (GPU test), far below the 16-bit rounding of
// every output it feeds.
__device__ __forceinline__ float act_gelu(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  float t, e;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(t) : "f"(fmaf(0.3275911f, z, 1.0f)));
  float P = fmaf(1.061405429f, t, -1.453152027f);
  P = fmaf(P, t, 1.421413741f);
  P = fmaf(P, t, -0.284496736f);
  P = fmaf(P, t, 0.254829592f);
  P *= t;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(e) : "f"(-(z * z) * 1.4426950408889634f));
  const float q = 0.5f * x * P * e;
  return x >= 0.f ? x - q : q;
}
// Two GELUs with the same operations in the same order as act_gelu (so the same bits), the
// fp32 arithmetic done by the paired .f32x2 instructions (two lanes of fp32 per instruction);
// the reciprocal and the exponential stay per element.
__device__ __forceinline__ void act_gelu2(float &x0, float &x1) {
  float r0, r1;
  asm("{\n"
      " .reg .b64 x, z, d, t, P, a, e, q, h, c;\n"
      " .reg .f32 z0, z1, d0, d1, t0, t1, a0, a1, e0, e1, r0, r1, q0, q1;\n"
      " .reg .pred p0, p1;\n"
      " mov.b64 x, {%2, %3};\n"
      " mul.f32 z0, %2, 0f3F3504F3;\n"           // |x| / sqrt 2 (abs folded below)
      " abs.f32 z0, z0;\n"
      " mul.f32 z1, %3, 0f3F3504F3;\n"
      " abs.f32 z1, z1;\n"
      " mov.b64 z, {z0, z1};\n"
      " mov.b64 c, {0f3EA7BA05, 0f3EA7BA05};\n"   // p = 0.3275911
      " mov.b64 h, {0f3F800000, 0f3F800000};\n"
      " fma.rn.f32x2 d, c, z, h;\n"
      " mov.b64 {d0, d1}, d;\n"
      " rcp.approx.ftz.f32 t0, d0;\n"
      " rcp.approx.ftz.f32 t1, d1;\n"
      " mov.b64 t, {t0, t1};\n"
      " mov.b64 c, {0f3F87DC22, 0f3F87DC22};\n"   // a5 = 1.061405429
      " mov.b64 h, {0fBFBA00E3, 0fBFBA00E3};\n"   // a4 = -1.453152027
      " fma.rn.f32x2 P, c, t, h;\n"
      " mov.b64 h, {0f3FB5F0E3, 0f3FB5F0E3};\n"   // a3 = 1.421413741
      " fma.rn.f32x2 P, P, t, h;\n"
      " mov.b64 h, {0fBE91A98E, 0fBE91A98E};\n"   // a2 = -0.284496736
      " fma.rn.f32x2 P, P, t, h;\n"
      " mov.b64 h, {0f3E827906, 0f3E827906};\n"   // a1 = 0.254829592
      " fma.rn.f32x2 P, P, t, h;\n"
      " mul.rn.f32x2 P, P, t;\n"
      " mul.rn.f32x2 a, z, z;\n"
      " mov.b64 c, {0fBFB8AA3B, 0fBFB8AA3B};\n"   // -log2(e)
      " mul.rn.f32x2 a, a, c;\n"
      " mov.b64 {a0, a1}, a;\n"
      " ex2.approx.ftz.f32 e0, a0;\n"
      " ex2.approx.ftz.f32 e1, a1;\n"
      " mov.b64 e, {e0, e1};\n"
      " mov.b64 c, {0f3F000000, 0f3F000000};\n"   // 0.5
      " mul.rn.f32x2 q, c, x;\n"
      " mul.rn.f32x2 q, q, P;\n"
      " mul.rn.f32x2 q, q, e;\n"
      " sub.rn.f32x2 d, x, q;\n"
      " mov.b64 {d0, d1}, d;\n"
      " mov.b64 {q0, q1}, q;\n"
      " setp.ge.f32 p0, %2, 0f00000000;\n"
      " setp.ge.f32 p1, %3, 0f00000000;\n"
      " selp.f32 %0, d0, q0, p0;\n"
      " selp.f32 %1, d1, q1, p1;\n"
      "}\n"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1));
  x0 = r0;
  x1 = r1;
}
// SiLU(x) = x / (1 + exp(-x)) with the hardware exponential and reciprocal approximations
// (relative error a few 1e-7, far below the 16-bit rounding of every output it feeds); for very
// negative x the exponential overflows to +inf and the result is -0, the limit.
__device__ __forceinline__ float act_silu(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(1.0f + e));
  return x * r;
}
// Two SiLUs, the same operations in the same order as act_silu, fp32 arithmetic paired.
__device__ __forceinline__ void act_silu2(float &x0, float &x1) {
  float r0, r1;
  asm("{\n"
      " .reg .b64 x, c, a, d, r;\n"
      " .reg .f32 a0, a1, e0, e1, d0, d1, q0, q1;\n"
      " mov.b64 x, {%2, %3};\n"
      " mov.b64 c, {0fBFB8AA3B, 0fBFB8AA3B};\n"   // -log2(e)
      " mul.rn.f32x2 a, x, c;\n"
      " mov.b64 {a0, a1}, a;\n"
      " ex2.approx.ftz.f32 e0, a0;\n"
      " ex2.approx.ftz.f32 e1, a1;\n"
      " mov.b64 d, {e0, e1};\n"
      " mov.b64 c, {0f3F800000, 0f3F800000};\n"
      " add.rn.f32x2 d, c, d;\n"
      " mov.b64 {d0, d1}, d;\n"
      " rcp.approx.ftz.f32 q0, d0;\n"
      " rcp.approx.ftz.f32 q1, d1;\n"
      " mov.b64 r, {q0, q1};\n"
      " mul.rn.f32x2 r, x, r;\n"
      " mov.b64 {%0, %1}, r;\n"
      "}\n"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1));
  x0 = r0;
  x1 = r1;
}
__device__ __forceinline__ float act_apply(float x, int act) {
  return act == MOE_ACT_RELU ? act_relu(x) : (act == MOE_ACT_GELU ? act_gelu(x) : x);
}

// Checked build: whether the expert row offsets are usable (0 <= off[e] <= off[e+1] <= R for
// every e < E).  Every thread of the block must call it (it contains a barrier); a thread
// whose expert entry is bad calls fail().  In the plain build it is true without a look.
template <typename Fail>
__device__ __forceinline__ bool offsets_usable(const int32_t *off, int E, int64_t R, Fail fail) {
#if MOE_CHECKED
  int bad = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int o0 = off[e], o1 = off[e + 1];
    bad |= (o0 < 0 || o1 < o0 || int64_t(o1) > R) ? 1 : 0;
  }
  if (bad) fail();
  return __syncthreads_or(bad) == 0;
#else
  (void)off; (void)E; (void)R; (void)fail;
  return true;
#endif
}

// Top-k + softmax for one token (one warp), E <= 256 logits in shared memory: the k largest
// logits in descending order (equal logits: lower expert id first), gate = softmax over all E
// logits taken at the chosen ids (divided by the k gates' sum when renorm != 0).  Lane j < k
// writes ids[j] and gates[j].
__device__ __forceinline__ void topk_softmax_warp(const float *logits, int E, int k, int renorm, int32_t *ids,
                                  float *gates) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = 256 / 32;   // E <= 256
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

__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// ---- warp-level tensor-core MMA (m16n8k16, fp32 accumulate) ---------------------------
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, __half) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, __nv_bfloat16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---- cp.async (8-byte, zero-fill when src_bytes == 0) ----------------------------------
__device__ __forceinline__ void cp_async8(void *smem, const void *gmem, int src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Exclusive prefix sum over blockDim.x (<= 1024, multiple of 32) ints; returns the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *out, int *scratch /*32 ints*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int base = warp > 0 ? scratch[warp - 1] : 0;
  *out = base + x - v;
  const int total = scratch[nw - 1];
  __syncthreads();
  return total;
}

}  // namespace moe
