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
// so the kernel must never be handed `g_noalloc_scratch` itself.  Only a
// successful lookup is kept: a lookup that failed (for instance one made
// while the stream was being captured) is tried again on the next call.  The actual
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
void* g_scratch_addr[kMaxDevices];  // null until a lookup succeeded
std::mutex g_scratch_mu;

// The array's device address on `dev` (the current device), looked up on
// the first call that succeeds and kept from then on.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();  // leave no stale error for a later launch check
      return e;
    }
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
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
  void* scratch = nullptr;
  const cudaError_t le = scratch_address(dev, &scratch);
  if (le != cudaSuccess)
    return gq::fail(GQ_ERR_CUDA,
                    "gq_fp8_colwise_noalloc: scratch address lookup failed "
                    "(tried again on the next call): %s",
                    cudaGetErrorString(le));
  return gq_fp8_colwise(x, M, K, offs, n_groups, out, scales, scratch,
                        kScratchBytes, stream);
}
