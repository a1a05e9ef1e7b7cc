// Split-K reduction with the FC1 activation, and the un-permute / combine step.
//
// "Who Says Elephants Can't Run", section 3 workflow: the rows are restored to their
// original order and multiplied by expert_scale; "Specter", method step 5: results are
// scattered back to their positions.  out[t] = sum_j gate[t, j] * y[inv_perm[t*k + j]]
// (+ shared expert), summed in fp32 in j order and rounded once.
#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float ld_any(const void *p, int dt, int64_t i) {
  if (dt == MOE_F32) return static_cast<const float *>(p)[i];
  if (dt == MOE_F16) return __half2float(static_cast<const __half *>(p)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
}
__device__ __forceinline__ void st_any(void *p, int dt, int64_t i, float v) {
  if (dt == MOE_F32) static_cast<float *>(p)[i] = v;
  else if (dt == MOE_F16) static_cast<__half *>(p)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

// out[r, c] = act(sum_s part[s, r, c]); SWIGLU: silu(sum part[.., c]) * sum part[.., c + N/2].
__global__ void reduce_act_kernel(const float *__restrict__ part, int splits, int64_t R, int N,
                                  int act, void *__restrict__ out, int out_dtype) {
  const int Nout = act == MOE_ACT_SWIGLU ? N / 2 : N;
  const int64_t total = R * Nout;
  const int64_t slice = R * int64_t(N);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / Nout;
    const int c = int(i % Nout);
    float v = 0.f;
    const float *pv = part + r * N + c;
    int s = 0;
    for (; s + 4 <= splits; s += 4) {
      const float q0 = pv[s * slice], q1 = pv[(s + 1) * slice], q2 = pv[(s + 2) * slice], q3 = pv[(s + 3) * slice];
      v += q0; v += q1; v += q2; v += q3;
    }
    for (; s < splits; ++s) v += pv[s * slice];
    if (act == MOE_ACT_SWIGLU) {
      float u = 0.f;
      const float *pu = pv + Nout;
      s = 0;
      for (; s + 4 <= splits; s += 4) {
        const float q0 = pu[s * slice], q1 = pu[(s + 1) * slice], q2 = pu[(s + 2) * slice], q3 = pu[(s + 3) * slice];
        u += q0; u += q1; u += q2; u += q3;
      }
      for (; s < splits; ++s) u += pu[s * slice];
      v = act_silu(v) * u;
    } else {
      v = act_apply(v, act);
    }
    st_any(out, out_dtype, i, v);
  }
}

// One thread per (token, 4 columns); y has `ysplits` slices of (R, d), sh `shsplits` of (T, d).
__global__ void combine_kernel(const void *__restrict__ y, int y_dtype, int ysplits,
                               const int32_t *__restrict__ inv_perm, const float *__restrict__ gate,
                               const void *__restrict__ sh, int sh_dtype, int shsplits, int64_t T,
                               int64_t d, int k, void *__restrict__ out, int out_dtype) {
  const int64_t R = T * k;
  const int64_t d4 = d / 4;
  const int64_t total = T * d4;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t tok = i / d4;
    const int64_t c = (i % d4) * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int64_t p = inv_perm[tok * k + j];
      if (p < 0 || p >= R) continue;  // malformed permutation: contributes nothing
      const float gw = gate[tok * k + j];
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (y_dtype == MOE_F32) {
        const float *yf = static_cast<const float *>(y) + p * d + c;
        int s = 0;
        for (; s + 4 <= ysplits; s += 4) {   // four independent loads in flight, summed in split order
          float4 q[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) q[u] = *reinterpret_cast<const float4 *>(yf + (s + u) * R * d);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            v[0] += q[u].x; v[1] += q[u].y; v[2] += q[u].z; v[3] += q[u].w;
          }
        }
        for (; s < ysplits; ++s) {
          const float4 q = *reinterpret_cast<const float4 *>(yf + s * R * d);
          v[0] += q.x; v[1] += q.y; v[2] += q.z; v[3] += q.w;
        }
      } else {
        for (int s = 0; s < ysplits; ++s) {
          const int64_t base = s * R * d + p * d + c;
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] += ld_any(y, y_dtype, base + q);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] += gw * v[q];
    }
    if (sh) {
      if (sh_dtype == MOE_F32) {
        const float *sf = static_cast<const float *>(sh) + tok * d + c;
        int s = 0;
        for (; s + 4 <= shsplits; s += 4) {
          float4 q[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) q[u] = *reinterpret_cast<const float4 *>(sf + (s + u) * T * d);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[0] += q[u].x; acc[1] += q[u].y; acc[2] += q[u].z; acc[3] += q[u].w;
          }
        }
        for (; s < shsplits; ++s) {
          const float4 q = *reinterpret_cast<const float4 *>(sf + s * T * d);
          acc[0] += q.x; acc[1] += q.y; acc[2] += q.z; acc[3] += q.w;
        }
      } else {
        for (int s = 0; s < shsplits; ++s) {
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[q] += ld_any(sh, sh_dtype, s * T * d + tok * d + c + q);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) st_any(out, out_dtype, tok * d + c + q, acc[q]);
  }
}

int grid_1d(int64_t total, int threads) {
  const int64_t want = cdiv(total, threads);
  const int64_t cap = int64_t(num_sms()) * 8;
  return int(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

int launch_reduce_act(const float *part, int splits, int64_t R, int N, int act, void *out,
                      int out_dtype, cudaStream_t st) {
  const int Nout = act == MOE_ACT_SWIGLU ? N / 2 : N;
  if (R == 0) return MOE_OK;
  reduce_act_kernel<<<grid_1d(R * Nout, 256), 256, 0, st>>>(part, splits, R, N, act, out, out_dtype);
  return check_launch("reduce_act");
}

int launch_combine(const void *y, int y_dtype, int ysplits, const int32_t *inv_perm,
                   const float *gate, const void *sh, int sh_dtype, int shsplits, int64_t T,
                   int64_t d, int k, void *out, int out_dtype, cudaStream_t st) {
  if (T == 0) return MOE_OK;
  combine_kernel<<<grid_1d(T * (d / 4), 256), 256, 0, st>>>(y, y_dtype, ysplits, inv_perm, gate, sh,
                                                           sh_dtype, shsplits, T, d, k, out, out_dtype);
  return check_launch("combine");
}

}  // namespace moe

using namespace moe;

extern "C" int moe_unpermute_combine(const void *yp, int yp_dtype, const int32_t *inv_perm,
                                     const float *gate_w, const void *shared, int shared_dtype,
                                     int64_t T, int64_t d, int k, void *out, int out_dtype,
                                     moe_stream_t stream) {
  auto okdt = [](int dt) { return dt == MOE_F16 || dt == MOE_BF16 || dt == MOE_F32; };
  MOE_REQUIRE(okdt(yp_dtype) && okdt(out_dtype), "bad dtype");
  MOE_REQUIRE(shared == nullptr || okdt(shared_dtype), "bad shared dtype");
  MOE_REQUIRE(T >= 0 && d >= 4 && d % 4 == 0 && k >= 1, "need T >= 0, d %% 4 == 0, k >= 1");
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(yp && inv_perm && gate_w && out, "null pointer argument");
  MOE_REQUIRE(aligned16(yp) && aligned16(inv_perm) && aligned16(gate_w) && aligned16(out) &&
                  (shared == nullptr || aligned16(shared)),
              "pointers must be 16-byte aligned");
  return launch_combine(yp, yp_dtype, 1, inv_perm, gate_w, shared, shared_dtype, 1, T, d, k, out,
                        out_dtype, reinterpret_cast<cudaStream_t>(stream));
}
