// Public entry points that chain kernels (grouped GEMM, shared expert, whole layer), the
// error reporting and the small host helpers.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "moe_internal.cuh"

namespace moe {

namespace {
thread_local char g_err[512] = "no error";
}

int set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

int check_gemm_args(int bits, const void *a, int a_dtype, const void *packed_w, int64_t E, int64_t K,
                    int64_t N, int group, const int32_t *offsets, int64_t R, int act, const void *out,
                    int out_dtype) {
  MOE_REQUIRE(is16(a_dtype), "a_dtype must be MOE_F16 or MOE_BF16");
  MOE_REQUIRE(out_dtype == MOE_F16 || out_dtype == MOE_BF16 || out_dtype == MOE_F32, "bad out_dtype");
  MOE_REQUIRE(act >= MOE_ACT_NONE && act <= MOE_ACT_SWIGLU, "bad act %d", act);
  MOE_REQUIRE(E >= 1 && E <= 256, "need 1 <= E <= 256 (E=%lld)", (long long)E);
  MOE_REQUIRE(group == 0 || group == 128, "group must be 0 or 128");
  MOE_REQUIRE(bits != 16 || group == 0, "16-bit weights take no group");
  MOE_REQUIRE(R >= 0 && R < (int64_t(1) << 31), "R out of range");
  MOE_REQUIRE(K >= 128 && K % 128 == 0 && K < (int64_t(1) << 30), "K must be a positive multiple of 128 (K=%lld)", (long long)K);
  if (act == MOE_ACT_SWIGLU)
    MOE_SUPPORT(N % 64 == 0 && N >= 64, "SWIGLU needs N %% 64 == 0 (N=%lld)", (long long)N);
  else
    MOE_SUPPORT(N % 64 == 0 && N >= 64, "N must be a multiple of 64 (N=%lld)", (long long)N);
  MOE_REQUIRE(N < (int64_t(1) << 30), "N too large");
  MOE_REQUIRE(offsets != nullptr || E == 1, "offsets may be NULL only when E == 1");
  if (R == 0) return MOE_OK;
  MOE_REQUIRE(a && packed_w && out, "null pointer argument");
  MOE_REQUIRE(aligned16(a) && aligned16(packed_w) && aligned16(out) && (offsets == nullptr || aligned16(offsets)),
              "pointers must be 16-byte aligned");
  return MOE_OK;
}

size_t gemm_ws_bytes(const GemmPlan &pl, int64_t R, int64_t N) {
  return pl.partial ? align256(size_t(pl.splits) * size_t(R) * size_t(N) * 4) : 0;
}

int grouped_gemm(int bits, const void *a, int a_dtype, const void *packed_w, int64_t E, int64_t K,
                 int64_t N, int group, const int32_t *offsets, int64_t R, int act, void *out,
                 int out_dtype, void *workspace, size_t workspace_bytes, cudaStream_t st) {
  MOE_TRY(check_gemm_args(bits, a, a_dtype, packed_w, E, K, N, group, offsets, R, act, out, out_dtype));
  if (R == 0) return MOE_OK;
  const GemmPlan pl = plan_gemm(R, E, K, N, bits, act, false);
  const size_t need = gemm_ws_bytes(pl, R, N);
  if (need) {
    MOE_REQUIRE(workspace && aligned16(workspace), "workspace must be non-null and 16-byte aligned");
    if (workspace_bytes < need)
      return set_error(MOE_ERR_WORKSPACE, "grouped GEMM workspace %zu < %zu bytes", workspace_bytes, need);
  }
  GemmArgs g{};
  g.a = a;
  g.w = packed_w;
  g.scales = bits == 16 ? nullptr
                        : static_cast<const char *>(packed_w) + moe_packed_scale_offset(E, K, N, bits);
  g.offsets = offsets;
  g.out = out;
  g.partial = static_cast<float *>(workspace);
  g.R = R;
  g.E = int(E);
  g.K = int(K);
  g.N = int(N);
  g.group = group;
  g.act = act;
  g.out_dtype = out_dtype;
  g.a_dtype = a_dtype;
  g.bits = bits;
  MOE_TRY(launch_gemm(g, pl, st));
  if (pl.partial) MOE_TRY(launch_reduce_act(g.partial, pl.splits, R, int(N), act, out, out_dtype, st));
  return MOE_OK;
}

// ---- layer workspace layout -------------------------------------------------------------
struct LayerPlan {
  int64_t T, R;
  GemmPlan fc1, fc2, sh1, sh2;
  bool fused_combine;   // top-1, no shared expert, FC2 on tcgen05: FC2 writes the layer output
  DecodePlan dec;       // the one-launch decode layer (dec.ok: it takes this T)
  size_t o_ids, o_gate, o_off, o_perm, o_inv, o_rws, o_pws, o_xp, o_p1, o_h, o_y, o_hs, o_ps1, o_ys, o_dec, total;
};

// How a decode step runs (moe_set_decode_mode): 0 automatic, 1 always the chain of kernels,
// 2 one launch whenever the layer allows it.
std::atomic<int> g_decode_mode{0};
// Automatic choice: one launch when the step streams at most this many weight bytes.  Measured
// on GB300: a small layer (1 MB of expert weights, T = 16) takes 29 us as one launch and 42 us as
// the chain (launch and dependency latency dominate), while from the Qwen-shaped T = 1 step
// (88 MB) up the chain's many-warp weight-stream kernels stream faster than the one-launch
// kernel's one block per SM (51 vs 48 us; Phi-shaped T = 16: 231 vs 168 us).
constexpr double kDecodeLaunchMaxBytes = 16e6;

int check_desc(const moe_layer_desc *d) {
  MOE_REQUIRE(d != nullptr, "desc is NULL");
  MOE_REQUIRE(is16(d->dtype), "desc.dtype must be MOE_F16 or MOE_BF16");
  MOE_REQUIRE(d->router_dtype == MOE_F32 || d->router_dtype == d->dtype, "desc.router_dtype must be F32 or dtype");
  MOE_REQUIRE(d->bits == 4 || d->bits == 8, "desc.bits must be 4 or 8");
  MOE_REQUIRE(d->group == 0 || d->group == 128, "desc.group must be 0 or 128");
  MOE_REQUIRE(d->act >= MOE_ACT_RELU && d->act <= MOE_ACT_SWIGLU, "desc.act must be RELU, GELU or SWIGLU");
  MOE_REQUIRE(d->E >= 1 && d->E <= 256 && d->k >= 1 && d->k <= d->E, "need 1 <= k <= E <= 256");
  MOE_REQUIRE(d->d >= 128 && d->d % 128 == 0, "d must be a multiple of 128 (d=%lld)", (long long)d->d);
  MOE_REQUIRE(d->F >= 128 && d->F % 128 == 0, "F must be a multiple of 128 (F=%lld)", (long long)d->F);
  MOE_REQUIRE(d->Fs >= 0 && (d->Fs == 0 || d->Fs % 128 == 0), "Fs must be 0 or a multiple of 128");
  return MOE_OK;
}

LayerPlan plan_layer(const moe_layer_desc *d, int64_t T, bool for_size = false) {
  LayerPlan p{};
  p.T = T;
  p.R = T * d->k;
  const int64_t F1 = d->act == MOE_ACT_SWIGLU ? 2 * d->F : d->F;
  p.fc1 = plan_gemm(p.R, d->E, d->d, F1, d->bits, d->act, false);
  p.fc2 = plan_gemm(p.R, d->E, d->F, d->d, d->bits, MOE_ACT_NONE, true);
  // one routed row per token and nothing else to add: the un-permute and gate of the combine
  // step go into FC2's epilogue (the tcgen05 kernel's), the same arithmetic with one rounding
  p.fused_combine = d->k == 1 && d->Fs == 0 && p.fc2.kind == kKindTc && p.fc2.splits == 1 &&
                    tc_shape_ok(d->E, d->F, d->d, d->bits, d->group, MOE_ACT_NONE);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  p.o_ids = take(size_t(p.R) * 4);
  p.o_gate = take(size_t(p.R) * 4);
  p.o_off = take(size_t(d->E + 1) * 4);
  p.o_perm = take(size_t(p.R) * 4);
  p.o_inv = take(size_t(p.R) * 4);
  p.o_rws = take(moe_route_topk_workspace_size(T, d->d, d->E));
  p.o_pws = take(moe_permute_workspace_size(T, d->E, d->k));
  p.o_xp = take(size_t(p.R) * d->d * 2);
  p.o_p1 = take(p.fc1.partial ? size_t(p.fc1.splits) * p.R * F1 * 4 : 0);
  p.o_h = take(size_t(p.R) * d->F * 2);
  p.o_y = take(size_t(p.fc2.splits) * p.R * d->d * 4);
  if (d->Fs > 0) {
    p.sh1 = plan_gemm(T, 1, d->d, 2 * d->Fs, 16, MOE_ACT_SWIGLU, false);
    p.sh2 = plan_gemm(T, 1, d->Fs, d->d, 16, MOE_ACT_NONE, true);
    p.o_hs = take(size_t(T) * d->Fs * 2);
    p.o_ps1 = take(p.sh1.partial ? size_t(p.sh1.splits) * T * 2 * d->Fs * 4 : 0);
    p.o_ys = take(size_t(p.sh2.splits) * T * d->d * 4);
  }
  // the one-launch decode layer's own region, last in the workspace.  For a size query it is the
  // largest any T' <= min(T, 32) needs (moe_layer_workspace_size then takes the largest total
  // over every T' <= T).
  p.dec = plan_decode(d, std::min<int64_t>(T, 32), decode_warps());
  if (p.dec.ok) {
    size_t bytes = p.dec.bytes;
    if (for_size)
      for (int64_t t = 1; t < std::min<int64_t>(T, 32); ++t) bytes = std::max(bytes, plan_decode(d, t, decode_warps()).bytes);
    p.o_dec = take(bytes);
    if (T > 32) p.dec.ok = false;
  }
  p.total = o;
  return p;
}

// Expert and shared-expert weight bytes a step of T tokens streams (experts drawn uniformly).
double decode_bytes(const moe_layer_desc *d, int64_t T) {
  const double er = double(d->E), R = double(T * d->k);
  const double active = std::min(er, std::max(1.0, er * (1.0 - std::pow(1.0 - 1.0 / er, R))));
  const double F1 = d->act == MOE_ACT_SWIGLU ? 2.0 * d->F : double(d->F);
  const double per_expert = (double(d->d) * F1 + double(d->F) * d->d) * d->bits / 8.0;
  return active * per_expert + 3.0 * d->d * d->Fs * 2.0;
}

bool use_decode_launch(const moe_layer_desc *d, const LayerPlan &p) {
  if (!p.dec.ok) return false;
  const int mode = g_decode_mode.load(std::memory_order_relaxed);
  if (mode == 1) return false;
  return mode == 2 || decode_bytes(d, p.T) <= kDecodeLaunchMaxBytes;
}

// The shared expert reads only x, so it runs on a second stream beside the routed chain
// (router, sort, two grouped GEMMs) and joins back before the combine: its 16-bit weight stream
// overlaps the chain's short, latency-bound kernels.  One stream and two events per thread and
// device, made on first use and kept for the life of the process (a graph capture records the
// fork and the join as graph edges).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

int side_stream(SideStream **out) {
  thread_local SideStream tl[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("side stream: cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(MOE_ERR_UNSUPPORTED, "side stream: device index %d >= 64", dev);
  SideStream &sd = tl[dev];
  if (sd.s == nullptr) {
    cudaStream_t s = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
      if (j) cudaEventDestroy(j);
      if (f) cudaEventDestroy(f);
      if (s) cudaStreamDestroy(s);
      return check_launch("side stream: create");
    }
    sd.s = s;
    sd.fork = f;
    sd.join = j;
  }
  *out = &sd;
  return MOE_OK;
}

GemmArgs make_args(int bits, const void *a, int dt, const void *w, int64_t E, int64_t K, int64_t N,
                   int group, const int32_t *offsets, int64_t R, int act, void *out, int out_dtype,
                   float *partial) {
  GemmArgs g{};
  g.a = a;
  g.w = w;
  g.scales = bits == 16 ? nullptr : static_cast<const char *>(w) + moe_packed_scale_offset(E, K, N, bits);
  g.offsets = offsets;
  g.out = out;
  g.partial = partial;
  g.R = R;
  g.E = int(E);
  g.K = int(K);
  g.N = int(N);
  g.group = group;
  g.act = act;
  g.out_dtype = out_dtype;
  g.a_dtype = dt;
  g.bits = bits;
  return g;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" const char *moe_last_error_string(void) { return g_err; }

extern "C" int moe_device_error(moe_stream_t stream, int32_t *host_code) {
  MOE_REQUIRE(host_code != nullptr, "host_code is NULL");
  int v = 0;
  MOE_TRY(read_device_error(reinterpret_cast<cudaStream_t>(stream), &v));
  MOE_TRY(decode_error_take(&v));
  *host_code = v;
  return MOE_OK;
}
extern "C" int moe_version(void) { return 1; }

extern "C" int moe_checked_build(void) { return MOE_CHECKED; }

extern "C" int moe_set_decode_mode(int mode) {
  MOE_REQUIRE(mode >= 0 && mode <= 2, "decode mode must be 0 (automatic), 1 (kernel chain) or 2 (one launch)");
  return g_decode_mode.exchange(mode);
}

extern "C" int moe_set_gemm_pairs(int on) {
  MOE_REQUIRE(on == 0 || on == 1, "on must be 0 or 1");
  return set_gemm_pairs(on);
}

extern "C" int moe_check_status(moe_stream_t stream, int32_t *host_flags) {
  MOE_REQUIRE(host_flags != nullptr, "host_flags is NULL");
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return check_launch("check status: stream synchronize");
  int v = 0;
  MOE_TRY(check_word_take_permute(&v));
  MOE_TRY(check_word_take_combine(&v));
  MOE_TRY(check_word_take_gemm_tc(&v));
  MOE_TRY(check_word_take_gemv(&v));
  MOE_TRY(check_word_take_gemm_mma(&v));
  *host_flags = v;
  if (v != 0)
    return set_error(MOE_ERR_DEVICE_CHECK, "device bounds check failed (flags 0x%x:%s%s%s)", v,
                     (v & kCheckExpertId) ? " expert id out of range" : "",
                     (v & kCheckOffsets) ? " expert offsets unusable" : "",
                     (v & kCheckPerm) ? " permutation entry out of range" : "");
  return MOE_OK;
}

extern "C" int moe_gemm_path(int64_t R, int64_t E, int64_t K, int64_t N, int bits, int group, int act) {
  if (R <= 0 || E < 1 || K < 128 || N < 64) return 0;
  const GemmPlan pl = plan_gemm(R, E, K, N, bits, act, false);
  static const int32_t dummy = 0;
  const GemmArgs g = make_args(bits, nullptr, MOE_F16, nullptr, E, K, N, group, &dummy, R, act, nullptr,
                               MOE_F16, nullptr);
  if (pl.kind == kKindGemv) return 2;
  return (pl.tc && tc_supported(g)) ? 1 : 0;
}

extern "C" size_t moe_grouped_gemm_workspace_size(int64_t R, int64_t E, int64_t K, int64_t N, int bits,
                                                  int act) {
  if (R <= 0 || E < 1 || K < 128 || N < 64) return 0;
  return gemm_ws_bytes(plan_gemm(R, E, K, N, bits, act, false), R, N);
}

extern "C" int moe_grouped_gemm_w4a16(const void *a, int a_dtype, const void *packed_w, int64_t E,
                                      int64_t K, int64_t N, int group, const int32_t *offsets, int64_t R,
                                      int act, void *out, int out_dtype, void *workspace,
                                      size_t workspace_bytes, moe_stream_t stream) {
  return grouped_gemm(4, a, a_dtype, packed_w, E, K, N, group, offsets, R, act, out, out_dtype, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_grouped_gemm_w8a16(const void *a, int a_dtype, const void *packed_w, int64_t E,
                                      int64_t K, int64_t N, int group, const int32_t *offsets, int64_t R,
                                      int act, void *out, int out_dtype, void *workspace,
                                      size_t workspace_bytes, moe_stream_t stream) {
  return grouped_gemm(8, a, a_dtype, packed_w, E, K, N, group, offsets, R, act, out, out_dtype, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_grouped_gemm_w16a16(const void *a, int a_dtype, const void *packed_w, int64_t E,
                                       int64_t K, int64_t N, const int32_t *offsets, int64_t R, int act,
                                       void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                                       moe_stream_t stream) {
  return grouped_gemm(16, a, a_dtype, packed_w, E, K, N, 0, offsets, R, act, out, out_dtype, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t moe_shared_expert_workspace_size(int64_t T, int64_t d, int64_t Fs) {
  if (T <= 0 || d < 128 || Fs < 128) return 0;
  const GemmPlan p1 = plan_gemm(T, 1, d, 2 * Fs, 16, MOE_ACT_SWIGLU, false);
  const GemmPlan p2 = plan_gemm(T, 1, Fs, d, 16, MOE_ACT_NONE, true);
  return align256(size_t(T) * Fs * 2) + gemm_ws_bytes(p1, T, 2 * Fs) + gemm_ws_bytes(p2, T, d);
}

extern "C" int moe_shared_expert(const void *x, int x_dtype, const void *w_gate_up_packed,
                                 const void *w_down_packed, int64_t T, int64_t d, int64_t Fs, void *out,
                                 int out_dtype, void *workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  MOE_REQUIRE(out_dtype == MOE_F32 || out_dtype == x_dtype, "out_dtype must be F32 or the x dtype");
  MOE_TRY(check_gemm_args(16, x, x_dtype, w_gate_up_packed, 1, d, 2 * Fs, 0, nullptr, T, MOE_ACT_SWIGLU, out, out_dtype));
  MOE_TRY(check_gemm_args(16, x, x_dtype, w_down_packed, 1, Fs, d, 0, nullptr, T, MOE_ACT_NONE, out, out_dtype));
  if (T == 0) return MOE_OK;
  const size_t need = moe_shared_expert_workspace_size(T, d, Fs);
  MOE_REQUIRE(workspace && aligned16(workspace), "workspace must be non-null and 16-byte aligned");
  if (workspace_bytes < need)
    return set_error(MOE_ERR_WORKSPACE, "shared-expert workspace %zu < %zu bytes", workspace_bytes, need);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const GemmPlan p1 = plan_gemm(T, 1, d, 2 * Fs, 16, MOE_ACT_SWIGLU, false);
  const GemmPlan p2 = plan_gemm(T, 1, Fs, d, 16, MOE_ACT_NONE, true);
  char *ws = static_cast<char *>(workspace);
  void *hs = ws;
  float *pa = reinterpret_cast<float *>(ws + align256(size_t(T) * Fs * 2));
  float *pb = reinterpret_cast<float *>(reinterpret_cast<char *>(pa) + gemm_ws_bytes(p1, T, 2 * Fs));
  MOE_TRY(launch_gemm(make_args(16, x, x_dtype, w_gate_up_packed, 1, d, 2 * Fs, 0, nullptr, T,
                                    MOE_ACT_SWIGLU, hs, x_dtype, pa), p1, st));
  if (p1.partial) MOE_TRY(launch_reduce_act(pa, p1.splits, T, int(2 * Fs), MOE_ACT_SWIGLU, hs, x_dtype, st));
  MOE_TRY(launch_gemm(make_args(16, hs, x_dtype, w_down_packed, 1, Fs, d, 0, nullptr, T,
                                    MOE_ACT_NONE, nullptr, MOE_F32, pb), p2, st));
  return launch_reduce_act(pb, p2.splits, T, int(d), MOE_ACT_NONE, out, out_dtype, st);
}

extern "C" size_t moe_layer_workspace_size(const moe_layer_desc *desc, int64_t T) {
  if (check_desc(desc) != MOE_OK || T < 0) return 0;
  // A smaller batch can need more than a larger one (its split-K GEMM plans write partial sums
  // in more slices), so the size is the largest requirement over every T' <= T: a workspace of
  // this size serves every call with at most T tokens.  A plan costs a few microseconds.  Split
  // plans exist only while the rows give fewer tiles than two waves of CTAs (under 64 rows per
  // CTA of 2 x 256 SMs, 32768 rows) or at most 16 rows per expert (4096 rows): from 65536 tokens
  // on every plan is unsplit and every region grows with T, so the scan stops there.
  size_t best = plan_layer(desc, T, true).total;
  const int64_t scan = std::min<int64_t>(T - 1, 65536);
  for (int64_t t = 1; t <= scan; ++t) best = std::max(best, plan_layer(desc, t, true).total);
  return best;
}

extern "C" int moe_layer_routing_view(const moe_layer_desc *desc, int64_t T, void *workspace,
                                      moe_layer_routing *view) {
  MOE_TRY(check_desc(desc));
  MOE_REQUIRE(T >= 0 && workspace && view, "bad arguments");
  const LayerPlan p = plan_layer(desc, T);
  char *ws = static_cast<char *>(workspace);
  view->ids = reinterpret_cast<int32_t *>(ws + p.o_ids);
  view->gate_w = reinterpret_cast<float *>(ws + p.o_gate);
  view->offsets = reinterpret_cast<int32_t *>(ws + p.o_off);
  view->perm = reinterpret_cast<int32_t *>(ws + p.o_perm);
  view->inv_perm = reinterpret_cast<int32_t *>(ws + p.o_inv);
  return MOE_OK;
}

extern "C" int moe_layer_launch_count(const moe_layer_desc *desc, int64_t T) {
  if (check_desc(desc) != MOE_OK || T <= 0) return 0;
  const LayerPlan p = plan_layer(desc, T);
  if (use_decode_launch(desc, p)) return 1;
  int n = (desc->router_dtype == MOE_F32 ? 1 : 2) /*route*/ + permute_launches(p.R, desc->E) /*permute*/ + 1 /*fc1*/ + (p.fc1.partial ? 1 : 0) + 1 /*fc2*/ + (p.fused_combine ? 0 : 1) /*combine*/;
  if (desc->Fs > 0) n += 2 + (p.sh1.partial ? 1 : 0);
  return n;
}

extern "C" int moe_layer_forward(const moe_layer_desc *desc, const moe_layer_weights *w, const void *x,
                                 int64_t T, void *out, void *workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  return moe_layer_forward_profiled(desc, w, x, T, out, workspace, workspace_bytes, stream, nullptr);
}

extern "C" int moe_layer_forward_profiled(const moe_layer_desc *desc, const moe_layer_weights *w,
                                          const void *x, int64_t T, void *out, void *workspace,
                                          size_t workspace_bytes, moe_stream_t stream,
                                          void *const *stage_events) {
  MOE_TRY(check_desc(desc));
  MOE_REQUIRE(w != nullptr, "weights struct is NULL");
  MOE_REQUIRE(T >= 0 && T * desc->k < (int64_t(1) << 31), "T out of range");
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && out && w->w_router && w->w1 && w->w2, "null pointer argument");
  MOE_REQUIRE(desc->Fs == 0 || (w->ws_gate_up && w->ws_down), "shared-expert weights missing");
  const LayerPlan p = plan_layer(desc, T);
  MOE_REQUIRE(workspace && aligned16(workspace), "workspace must be non-null and 16-byte aligned");
  if (workspace_bytes < p.total)
    return set_error(MOE_ERR_WORKSPACE, "layer workspace %zu < %zu bytes", workspace_bytes, p.total);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  int32_t *ids = reinterpret_cast<int32_t *>(ws + p.o_ids);
  float *gate = reinterpret_cast<float *>(ws + p.o_gate);
  int32_t *offs = reinterpret_cast<int32_t *>(ws + p.o_off);
  int32_t *perm = reinterpret_cast<int32_t *>(ws + p.o_perm);
  int32_t *inv = reinterpret_cast<int32_t *>(ws + p.o_inv);
  void *xp = ws + p.o_xp;
  float *p1 = reinterpret_cast<float *>(ws + p.o_p1);
  void *h = ws + p.o_h;
  float *y = reinterpret_cast<float *>(ws + p.o_y);
  const int dt = desc->dtype;
  const int64_t d = desc->d, F = desc->F, E = desc->E;
  const int k = desc->k;
  const int64_t F1 = desc->act == MOE_ACT_SWIGLU ? 2 * F : F;
  if (!stage_events && use_decode_launch(desc, p)) {
    // one launch for the whole layer; its control words are cleared first, except inside a
    // stream capture, where the launch relies on them being zero (every completed launch leaves
    // them so; moe_layer_graph_create runs one call before it captures)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return check_launch("layer: capture status");
    return launch_decode_layer(desc, w, x, T, out, ids, gate, offs, perm, inv, h, ws + p.o_dec, p.dec,
                               cs == cudaStreamCaptureStatusNone, st);
  }

  auto mark = [&](int stage) -> int {
    if (!stage_events) return MOE_OK;
    if (cudaEventRecord(static_cast<cudaEvent_t>(stage_events[stage]), st) != cudaSuccess)
      return check_launch("stage event");
    return MOE_OK;
  };
  // shared expert beside the routed chain (serial when stage events are recorded, so that every
  // stage boundary stays a point in one stream)
  SideStream *side = nullptr;
  if (desc->Fs > 0 && !stage_events) {
    MOE_TRY(side_stream(&side));
    if (cudaEventRecord(side->fork, st) != cudaSuccess) return check_launch("shared expert: fork");
  }
  auto shared_expert = [&](cudaStream_t s) -> int {
    void *hs = ws + p.o_hs;
    float *ps1 = reinterpret_cast<float *>(ws + p.o_ps1);
    float *ys = reinterpret_cast<float *>(ws + p.o_ys);
    MOE_TRY(launch_gemm(make_args(16, x, dt, w->ws_gate_up, 1, d, 2 * desc->Fs, 0, nullptr, T,
                                  MOE_ACT_SWIGLU, hs, dt, ps1), p.sh1, s));
    if (p.sh1.partial) MOE_TRY(launch_reduce_act(ps1, p.sh1.splits, T, int(2 * desc->Fs), MOE_ACT_SWIGLU, hs, dt, s));
    return launch_gemm(make_args(16, hs, dt, w->ws_down, 1, desc->Fs, d, 0, nullptr, T, MOE_ACT_NONE, nullptr,
                                 MOE_F32, ys), p.sh2, s);
  };
  MOE_TRY(mark(MOE_STAGE_START));
  MOE_TRY(moe_route_topk(x, dt, w->w_router, desc->router_dtype, w->router_bias, T, d, E, k,
                         desc->renormalize, ids, gate, ws + p.o_rws, moe_route_topk_workspace_size(T, d, E),
                         stream));
  if (side) {   // enqueued after the router, so the router's blocks are placed first
    if (cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess) return check_launch("shared expert: wait");
    MOE_TRY(shared_expert(side->s));
    if (cudaEventRecord(side->join, side->s) != cudaSuccess) return check_launch("shared expert: join");
  }
  MOE_TRY(mark(MOE_STAGE_ROUTED));
  MOE_TRY(moe_permute(ids, x, dt, T, d, E, k, offs, perm, inv, xp, ws + p.o_pws,
                      moe_permute_workspace_size(T, E, k), stream));
  MOE_TRY(mark(MOE_STAGE_PERMUTED));
  MOE_TRY(launch_gemm(make_args(desc->bits, xp, dt, w->w1, E, d, F1, desc->group, offs, p.R, desc->act,
                                    h, dt, p1), p.fc1, st));
  if (p.fc1.partial) MOE_TRY(launch_reduce_act(p1, p.fc1.splits, p.R, int(F1), desc->act, h, dt, st));
  MOE_TRY(mark(MOE_STAGE_FC1));
  if (p.fused_combine) {
    GemmArgs g2 = make_args(desc->bits, h, dt, w->w2, E, F, d, desc->group, offs, p.R, MOE_ACT_NONE, out, dt,
                            nullptr);
    g2.row_dest = perm;   // k == 1: perm[p] is the token of permuted row p
    g2.row_gate = gate;
    MOE_TRY(launch_gemm_tc(g2, st));
    MOE_TRY(mark(MOE_STAGE_FC2));
    MOE_TRY(mark(MOE_STAGE_SHARED));
    return mark(MOE_STAGE_DONE);
  }
  MOE_TRY(launch_gemm(make_args(desc->bits, h, dt, w->w2, E, F, d, desc->group, offs, p.R, MOE_ACT_NONE,
                                    nullptr, MOE_F32, y), p.fc2, st));
  MOE_TRY(mark(MOE_STAGE_FC2));
  const void *sh = nullptr;
  int shs = 0;
  if (desc->Fs > 0) {
    if (side) {
      if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return check_launch("shared expert: join wait");
    } else {
      MOE_TRY(shared_expert(st));
    }
    sh = ws + p.o_ys;
    shs = p.sh2.splits;
  }
  MOE_TRY(mark(MOE_STAGE_SHARED));
  MOE_TRY(launch_combine(y, MOE_F32, p.fc2.splits, inv, gate, sh, MOE_F32, shs, T, d, k, out, dt, st));
  return mark(MOE_STAGE_DONE);
}

// ---------------------------------------------------------------- CUDA graph of the chain

struct moe_layer_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" int moe_layer_graph_create(const moe_layer_desc *desc, const moe_layer_weights *w, const void *x,
                                      int64_t T, void *out, void *workspace, size_t workspace_bytes,
                                      moe_stream_t stream, moe_layer_graph *graph) {
  MOE_REQUIRE(graph != nullptr, "graph handle pointer is NULL");
  *graph = nullptr;
  MOE_REQUIRE(T > 0, "a graph needs T > 0");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_REQUIRE(st != nullptr, "capture needs a created stream (not the legacy default stream)");
  // eager run: validates the arguments and fills the per-kernel caches before capture
  MOE_TRY(moe_layer_forward(desc, w, x, T, out, workspace, workspace_bytes, stream));
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return check_launch("layer graph: begin capture");
  const int rc = moe_layer_forward(desc, w, x, T, out, workspace, workspace_bytes, stream);
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(st, &g);
  if (rc != MOE_OK || ec != cudaSuccess || g == nullptr) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != MOE_OK ? rc : set_error(MOE_ERR_CUDA, "layer graph: capture failed: %s", cudaGetErrorString(ec));
  }
  cudaGraphExec_t ex = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&ex, g, 0);
  if (ei != cudaSuccess) {
    cudaGraphDestroy(g);
    return set_error(MOE_ERR_CUDA, "layer graph: instantiate failed: %s", cudaGetErrorString(ei));
  }
  auto *h = new moe_layer_graph_s;
  h->graph = g;
  h->exec = ex;
  *graph = h;
  return MOE_OK;
}

extern "C" int moe_layer_graph_launch(moe_layer_graph graph, moe_stream_t stream) {
  MOE_REQUIRE(graph != nullptr && graph->exec != nullptr, "graph is NULL");
  if (cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return check_launch("layer graph launch");
  return MOE_OK;
}

extern "C" int moe_layer_graph_destroy(moe_layer_graph graph) {
  if (graph == nullptr) return MOE_OK;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
  return MOE_OK;
}
