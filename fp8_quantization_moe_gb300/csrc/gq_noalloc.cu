// gq_noalloc.cu -- gq_fp8_colwise_noalloc: the colwise call for callers that
// cannot allocate device memory where they quantize.
//
// Such a caller may run inside another runtime that owns every byte of the
// device heap and exposes no way to borrow a workspace, or on a hot path
// where cudaMalloc / cudaFree are off limits because they can synchronize
// the whole device.  This entry point therefore needs no workspace argument:
// its scratch (the work-claiming counters and the per-(group, column) amax
// words) is one fixed array in this library's device memory.  The array
// exists on every GPU that loads the library and stays there until the
// process exits.
//
// Nothing here allocates.  The first call on each device looks up the
// array's device address with cudaGetSymbolAddress, with that device
// current; a host-side name of a __device__ array is not a device address,
// so the kernel must never be handed `g_noalloc_scratch` itself.  The actual
// work goes through the same validation and kernel as gq_fp8_colwise, which
// clears the used part of the scratch with cudaMemsetAsync on the caller's
// stream before the kernel runs.
#include <mutex>

#include "gq_internal.h"

namespace {

constexpr size_t kScratchBytes = GQ_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size keeps 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Once per device, with that device current.
void lookup_scratch(int dev) {
  void* p = nullptr;
  g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  g_scratch_addr[dev] = p;
}

}  // namespace

extern "C" gq_status gq_fp8_colwise_noalloc(const void* x, int64_t M, int64_t K,
                                            const int32_t* offs,
                                            int32_t n_groups, void* out,
                                            float* scales,
                                            gq_stream_t stream) {
  const size_t need = gq_workspace_bytes(GQ_KIND_COLWISE, M, K, n_groups);
  if (need > kScratchBytes)
    return gq::fail(GQ_ERR_UNSUPPORTED,
                    "gq_fp8_colwise_noalloc: this call needs %zu bytes of "
                    "scratch but the built-in array holds %zu "
                    "(GQ_NOALLOC_SCRATCH_BYTES); use gq_fp8_colwise with a "
                    "workspace",
                    need, kScratchBytes);
  if (need == 0)  // empty or invalid: gq_fp8_colwise checks and handles it
    return gq_fp8_colwise(x, M, K, offs, n_groups, out, scales, nullptr, 0,
                          stream);
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return gq::fail(GQ_ERR_CUDA, "gq_fp8_colwise_noalloc: cudaGetDevice: %s",
                    cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return gq::fail(GQ_ERR_UNSUPPORTED,
                    "gq_fp8_colwise_noalloc: device ordinal %d out of range", dev);
  std::call_once(g_scratch_once[dev], lookup_scratch, dev);
  if (g_scratch_err[dev] != cudaSuccess || g_scratch_addr[dev] == nullptr)
    return gq::fail(GQ_ERR_CUDA,
                    "gq_fp8_colwise_noalloc: scratch address lookup failed: %s",
                    cudaGetErrorString(g_scratch_err[dev]));
  return gq_fp8_colwise(x, M, K, offs, n_groups, out, scales,
                        g_scratch_addr[dev], kScratchBytes, stream);
}
