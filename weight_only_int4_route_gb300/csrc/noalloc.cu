// Grouped W4A16 GEMM that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory when they run this GEMM: a serving runtime that
// carves all device memory into fixed pools at start-up and forbids later allocation, a host
// framework that owns the device allocator and hands plug-ins only their input and output
// buffers, or code that must not call cudaMalloc while a stream is being captured into a CUDA
// graph.  For them the split-K partial sums, the only scratch memory this GEMM uses, live in
// one fixed array that is part of the library itself.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds it
// until the process exits.  In host code its name is only a host-side stand-in: the device
// address is obtained once per device with cudaGetSymbolAddress, with that device current,
// and passed to the kernels.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};

// Device address of the scratch array on the current device (looked up on first use).
int static_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("static scratch: cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(MOE_ERR_UNSUPPORTED, "static scratch: device index %d >= 64", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(MOE_ERR_CUDA, "static scratch: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_grouped_gemm_w4a16_static(const void *a, int a_dtype, const void *packed_w, int64_t E,
                                             int64_t K, int64_t N, int group, const int32_t *offsets,
                                             int64_t R, int act, void *out, int out_dtype,
                                             moe_stream_t stream) {
  const size_t need = moe_grouped_gemm_workspace_size(R, E, K, N, 4, act);
  if (need > kStaticScratchBytes)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "this GEMM needs %zu bytes of scratch; the library's built-in buffer holds %zu "
                     "(use moe_grouped_gemm_w4a16 with a workspace instead)",
                     need, kStaticScratchBytes);
  void *scratch = nullptr;
  if (need > 0) MOE_TRY(static_scratch(&scratch));
  return moe_grouped_gemm_w4a16(a, a_dtype, packed_w, E, K, N, group, offsets, R, act, out, out_dtype, scratch,
                                need > 0 ? kStaticScratchBytes : 0, stream);
}
