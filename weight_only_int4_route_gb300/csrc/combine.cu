// Split-K reduction with the FC1 activation, and the un-permute / combine step.
//
// "Who Says Elephants Can't Run", section 3 workflow: the rows are restored to their
// original order and multiplied by expert_scale; "Specter", method step 5: results are
// scattered back to their positions.  out[t] = sum_j gate[t, j] * y[inv_perm[t*k + j]]
// (+ shared expert), summed in fp32 in j order and rounded once.
#include "moe_internal.cuh"

namespace moe {

MOE_DEFINE_CHECK_WORD(combine)

namespace {

__device__ __forceinline__ void st_any(void *p, int dt, int64_t i, float v) {
  if (dt == MOE_F32) static_cast<float *>(p)[i] = v;
  else if (dt == MOE_F16) static_cast<__half *>(p)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

// out[r, c] = act(sum_s part[s, r, c]); SWIGLU: silu(sum part[.., c]) * sum part[.., c + N/2].
__global__ void reduce_act_kernel(const float *__restrict__ part, int splits, int64_t R, int N,
                                  int act, void *__restrict__ out, int out_dtype) {
  pdl_enter();   // see launch_pdl
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

// Work item = (TPW consecutive tokens, column group of 128 * CPT columns), one per warp; y has
// `ysplits` slices of (R, d), sh `shsplits` of (T, d).  Lane l reads one (token, entry) row
// position and gate (32 at a time) and broadcasts them; lane l covers columns 4l .. 4l+3 of each
// 128 of the group, so a position read feeds CPT independent row loads.  Many tokens: TPW = 2,
// CPT = 4 (bytes in flight per position read); a few tokens: 1 x 1 (parallelism across columns).
// Every sum runs in entry order, split slices in split order.
constexpr int kCombineWarps = 8;

__device__ __forceinline__ float4 ld4(const void *p, int dt, int64_t i) {
  if (dt == MOE_F32) return *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
  const uint2 v = *reinterpret_cast<const uint2 *>(static_cast<const char *>(p) + i * 2);
  if (dt == MOE_F16) {
    const float2 a = __half22float2(u32_as_h2(v.x)), b = __half22float2(u32_as_h2(v.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  const float2 a = __bfloat1622float2(u32_as_b2(v.x)), b = __bfloat1622float2(u32_as_b2(v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void add4(float (&a)[4], const float4 &q) {
  a[0] += q.x; a[1] += q.y; a[2] += q.z; a[3] += q.w;
}
// acc += sum over s < splits of src[(s * rows + row) * d + c], in split order
__device__ __forceinline__ void split_sum(const void *src, int dt, int splits, int64_t rows, int64_t row, int64_t d,
                                          int64_t c, float (&acc)[4]) {
  int s = 0;
  for (; s + 8 <= splits; s += 8) {
    float4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = ld4(src, dt, ((s + u) * rows + row) * d + c);
#pragma unroll
    for (int u = 0; u < 8; ++u) add4(acc, q[u]);
  }
  for (; s < splits; ++s) add4(acc, ld4(src, dt, (s * rows + row) * d + c));
}

template <int CPT, int TPW>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(
    const void *__restrict__ y, int y_dtype, int ysplits, const int32_t *__restrict__ inv_perm,
    const float *__restrict__ gate, const void *__restrict__ sh, int sh_dtype, int shsplits, int64_t T,
    int64_t d, int k, void *__restrict__ out, int out_dtype) {
  pdl_enter();   // see launch_pdl
  const int lane = threadIdx.x & 31;
  const int64_t R = T * k;
  const int64_t ngroups = (d + 128 * CPT - 1) / (128 * CPT);
  const int64_t nblk = (T + TPW - 1) / TPW;
  for (int64_t task = int64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5); task < nblk * ngroups;
       task += int64_t(gridDim.x) * kCombineWarps) {   // warp-uniform
    const int64_t tok0 = (task / ngroups) * TPW;
    const int64_t cbase = (task % ngroups) * 128 * CPT + int64_t(lane) * 4;
    float acc[TPW][CPT][4];
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
      for (int u = 0; u < CPT; ++u)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][u][q] = 0.f;
    // entries of the TPW tokens, flattened (token i, entry j) -> i * k + j, 32 per round
    const int nent = TPW * k;
    for (int jb = 0; jb < nent; jb += 32) {
      int pl = -1;
      float gl = 0.f;
      {
        const int l = jb + lane;
        const int64_t tok = tok0 + l / k;
        if (l < nent && tok < T) {
          pl = inv_perm[tok * k + l % k];
          gl = gate[tok * k + l % k];
          if (pl < 0 || pl >= R) {   // dropped row (or a malformed permutation): contributes nothing
            if (MOE_CHECKED) check_fail(kCheckPerm);
            pl = -1;
          }
        }
      }
      const int nj = nent - jb < 32 ? nent - jb : 32;
      if (ysplits == 1 && TPW * k <= 32) {   // one slice: every row load of the round in flight together
        float4 q[TPW][CPT];
        float gw[TPW];
#pragma unroll
        for (int i = 0; i < TPW; ++i) gw[i] = 0.f;
        for (int j = 0; j < k; ++j) {
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            const int p = __shfl_sync(0xffffffffu, pl, i * k + j);
            gw[i] = __shfl_sync(0xffffffffu, gl, i * k + j);
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
              const int64_t c = cbase + u * 128;
              q[i][u] = (p >= 0 && c < d) ? ld4(y, y_dtype, int64_t(p) * d + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
              acc[i][u][0] += gw[i] * q[i][u].x;
              acc[i][u][1] += gw[i] * q[i][u].y;
              acc[i][u][2] += gw[i] * q[i][u].z;
              acc[i][u][3] += gw[i] * q[i][u].w;
            }
        }
      } else {
        for (int jj = 0; jj < nj; ++jj) {
          const int p = __shfl_sync(0xffffffffu, pl, jj);
          const float gw = __shfl_sync(0xffffffffu, gl, jj);
          if (p < 0) continue;
          const int i = (jb + jj) / k;   // token of this entry within the block
#pragma unroll
          for (int ii = 0; ii < TPW; ++ii) {
            if (ii != i) continue;
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
              const int64_t c = cbase + u * 128;
              if (c >= d) continue;
              float v[4] = {0.f, 0.f, 0.f, 0.f};
              split_sum(y, y_dtype, ysplits, R, p, d, c, v);
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[ii][u][q] += gw * v[q];
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      const int64_t tok = tok0 + i;
      if (tok >= T) continue;
#pragma unroll
      for (int u = 0; u < CPT; ++u) {
        const int64_t c = cbase + u * 128;
        if (c >= d) continue;
        if (sh) split_sum(sh, sh_dtype, shsplits, T, tok, d, c, acc[i][u]);
        if (out_dtype == MOE_F32) {
          *reinterpret_cast<float4 *>(static_cast<float *>(out) + tok * d + c) =
              make_float4(acc[i][u][0], acc[i][u][1], acc[i][u][2], acc[i][u][3]);
        } else {   // four 16-bit values in one 8-byte store
          uint2 v;
          if (out_dtype == MOE_F16) {
            v.x = h2_as_u32(__floats2half2_rn(acc[i][u][0], acc[i][u][1]));
            v.y = h2_as_u32(__floats2half2_rn(acc[i][u][2], acc[i][u][3]));
          } else {
            v.x = h2_as_u32(__floats2bfloat162_rn(acc[i][u][0], acc[i][u][1]));
            v.y = h2_as_u32(__floats2bfloat162_rn(acc[i][u][2], acc[i][u][3]));
          }
          *reinterpret_cast<uint2 *>(static_cast<char *>(out) + (tok * d + c) * 2) = v;
        }
      }
    }
  }
}

// Few output groups and many split slices (decode steps): summing the slices one after another
// in each thread is a chain of dependent memory round trips.  Instead a CTA owns one (row,
// 128-column group); its 8 warps each sum an interleaved subset of the (entry, slice) terms
// (lane l: columns 4l .. 4l+3) and warp 0 adds the 8 partial sums in warp order.  The order is
// fixed, so results are deterministic (it is a different order from the one-thread kernels).
constexpr int kSmallWarps = 8;

// out[r, c] = act(sum_s part[s, r, c]) (SWIGLU pairs c with c + N/2); Nout % 4 == 0.
__global__ void __launch_bounds__(kSmallWarps * 32) reduce_act_small_kernel(const float *__restrict__ part, int splits,
                                                                           int64_t R, int N, int act,
                                                                           void *__restrict__ out, int out_dtype) {
  pdl_enter();   // see launch_pdl
  __shared__ float4 red[2][kSmallWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool swiglu = act == MOE_ACT_SWIGLU;
  const int Nout = swiglu ? N / 2 : N;
  const int ngroups = (Nout + 127) / 128;
  const int64_t r = blockIdx.x / ngroups;
  const int c = (blockIdx.x % ngroups) * 128 + lane * 4;
  const bool in = c < Nout;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f), u = v;
  if (in) {
    const int64_t slice = R * int64_t(N);
    const float *pv = part + r * N + c;
    for (int s = warp; s < splits; s += kSmallWarps) {
      const float4 q = *reinterpret_cast<const float4 *>(pv + s * slice);
      v.x += q.x; v.y += q.y; v.z += q.z; v.w += q.w;
      if (swiglu) {
        const float4 w = *reinterpret_cast<const float4 *>(pv + s * slice + Nout);
        u.x += w.x; u.y += w.y; u.z += w.z; u.w += w.w;
      }
    }
  }
  red[0][warp][lane] = v;
  red[1][warp][lane] = u;
  __syncthreads();
  if (warp == 0 && in) {
    float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
    for (int w = 0; w < kSmallWarps; ++w) {
      const float4 x = red[0][w][lane], y = red[1][w][lane];
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
      b[0] += y.x; b[1] += y.y; b[2] += y.z; b[3] += y.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float o = swiglu ? act_silu(a[q]) * b[q] : act_apply(a[q], act);
      st_any(out, out_dtype, r * Nout + c + q, o);
    }
  }
}

// out[t] = sum_j gate[t, j] * sum_s y[s, inv[t*k + j]] + sum_s sh[s, t] for one (token,
// 128-column group) per CTA; k <= 32 (lane j holds entry j).  Term q < k*ysplits is entry
// q / ysplits, slice q % ysplits; the rest are shared-expert slices.
__global__ void __launch_bounds__(kSmallWarps * 32) combine_small_kernel(
    const void *__restrict__ y, int y_dtype, int ysplits, const int32_t *__restrict__ inv_perm,
    const float *__restrict__ gate, const void *__restrict__ sh, int sh_dtype, int shsplits, int64_t T,
    int64_t d, int k, void *__restrict__ out, int out_dtype) {
  pdl_enter();   // see launch_pdl
  __shared__ float4 red[kSmallWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t R = T * k;
  const int64_t ngroups = (d + 127) / 128;
  const int64_t tok = blockIdx.x / ngroups;
  const int64_t c = (blockIdx.x % ngroups) * 128 + lane * 4;
  const bool in = c < d;
  int pl = -1;
  float gl = 0.f;
  if (lane < k) {
    pl = inv_perm[tok * k + lane];
    gl = gate[tok * k + lane];
    if (pl < 0 || pl >= R) {   // dropped row (or a malformed permutation): contributes nothing
      if (MOE_CHECKED) check_fail(kCheckPerm);
      pl = -1;
    }
  }
  const int ny = k * ysplits;
  const int nterms = ny + (sh ? shsplits : 0);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q = warp; q < nterms; q += kSmallWarps) {   // warp-uniform
    if (q < ny) {
      const int j = q / ysplits, s = q - j * ysplits;
      const int p = __shfl_sync(0xffffffffu, pl, j);
      const float g = __shfl_sync(0xffffffffu, gl, j);
      if (p >= 0 && in) {
        const float4 v = ld4(y, y_dtype, (int64_t(s) * R + p) * d + c);
        acc.x += g * v.x; acc.y += g * v.y; acc.z += g * v.z; acc.w += g * v.w;
      }
    } else if (in) {
      const float4 v = ld4(sh, sh_dtype, (int64_t(q - ny) * T + tok) * d + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
  }
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && in) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    for (int w = 0; w < kSmallWarps; ++w) {
      const float4 x = red[w][lane];
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
    }
    if (out_dtype == MOE_F32) {
      *reinterpret_cast<float4 *>(static_cast<float *>(out) + tok * d + c) = make_float4(a[0], a[1], a[2], a[3]);
    } else {
      uint2 v;
      if (out_dtype == MOE_F16) {
        v.x = h2_as_u32(__floats2half2_rn(a[0], a[1]));
        v.y = h2_as_u32(__floats2half2_rn(a[2], a[3]));
      } else {
        v.x = h2_as_u32(__floats2bfloat162_rn(a[0], a[1]));
        v.y = h2_as_u32(__floats2bfloat162_rn(a[2], a[3]));
      }
      *reinterpret_cast<uint2 *>(static_cast<char *>(out) + (tok * d + c) * 2) = v;
    }
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
  const int64_t groups = R * cdiv(Nout, 128);
  if (splits >= 4 && Nout % 4 == 0 && groups <= int64_t(num_sms()) * 4)   // few outputs, many slices
    launch_pdl(reduce_act_small_kernel, dim3(unsigned(groups)), dim3(kSmallWarps * 32), 0, st, part, splits, R, N, act, out, out_dtype);
  else
    launch_pdl(reduce_act_kernel, dim3(grid_1d(R * Nout, 256)), dim3(256), 0, st, part, splits, R, N, act, out, out_dtype);
  return check_launch("reduce_act");
}

int launch_combine(const void *y, int y_dtype, int ysplits, const int32_t *inv_perm,
                   const float *gate, const void *sh, int sh_dtype, int shsplits, int64_t T,
                   int64_t d, int k, void *out, int out_dtype, cudaStream_t st) {
  if (T == 0) return MOE_OK;
  const int64_t ngroups = T * cdiv(d, 128);
  if (k <= 32 && k * ysplits + (sh ? shsplits : 0) >= 8 && ngroups <= int64_t(num_sms()) * 4) {
    launch_pdl(combine_small_kernel, dim3(unsigned(ngroups)), dim3(kSmallWarps * 32), 0, st, y, y_dtype, ysplits, inv_perm, gate, sh,
                                                                         sh_dtype, shsplits, T, d, k, out, out_dtype);
    return check_launch("combine");
  }
  // two tokens x four 128-column strides per warp when that still leaves 16 work items per SM,
  // else one token x one stride (parallelism across columns for a few tokens)
  const int64_t g1 = T * cdiv(d, 128);
  const bool wide = g1 / 8 >= int64_t(num_sms()) * 16;
  const int64_t tasks = wide ? cdiv(T, 2) * cdiv(d, 512) : g1;
  const int64_t want = cdiv(tasks, kCombineWarps);
  const int64_t cap = int64_t(num_sms()) * 8;
  const unsigned grid = unsigned(want < cap ? want : cap);
  if (wide)
    launch_pdl(combine_kernel<4, 2>, dim3(grid), dim3(kCombineWarps * 32), 0, st, y, y_dtype, ysplits, inv_perm, gate, sh, sh_dtype,
                                                              shsplits, T, d, k, out, out_dtype);
  else
    launch_pdl(combine_kernel<1, 1>, dim3(grid), dim3(kCombineWarps * 32), 0, st, y, y_dtype, ysplits, inv_perm, gate, sh, sh_dtype,
                                                              shsplits, T, d, k, out, out_dtype);
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
