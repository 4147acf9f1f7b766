// gq_api.cu -- the C ABI of libgqfp8 (declared in include/gq_fp8.h):
// argument validation, per-device set-up, TMA descriptor encoding, the
// per-device error word, and dispatch to the two kernels.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {

// Per-device error word; kernels get its device address as a parameter.
__device__ unsigned g_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
gq_status g_dev_status[kMaxDevices];
DebugKnobs g_dbg;
thread_local char g_msg[512] = "";

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
gq_status g_encode_status = GQ_OK;

void load_encode_fn() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  const cudaError_t e = cudaGetDriverEntryPointByVersion(
      "cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    g_encode_status = fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                           cudaGetErrorString(e));
    return;
  }
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}

void setup_device(int dev) {
  DeviceInfo& info = g_dev[dev];
  info.device = dev;
  gq_status& st = g_dev_status[dev];
  int major = 0, minor = 0;
  st = check_cuda(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev),
                  "query compute capability");
  if (st != GQ_OK) return;
  st = check_cuda(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev),
                  "query compute capability");
  if (st != GQ_OK) return;
  if (major != 10 || minor != 3) {
    st = fail(GQ_ERR_UNSUPPORTED,
              "device %d is sm_%d%d; libgqfp8 is built for sm_103a only", dev,
              major, minor);
    return;
  }
  st = check_cuda(cudaDeviceGetAttribute(&info.sm_count,
                                         cudaDevAttrMultiProcessorCount, dev),
                  "query SM count");
  if (st != GQ_OK) return;
  void* addr = nullptr;
  st = check_cuda(cudaGetSymbolAddress(&addr, g_error_word), "error word address");
  if (st != GQ_OK) return;
  info.err_word = static_cast<unsigned*>(addr);
  st = colwise::setup(info);
  if (st != GQ_OK) return;
  st = rowwise::setup(info);
  if (st != GQ_OK) return;
  st = mx::setup(info);
  if (st != GQ_OK) return;
  st = wgrad::setup(info);
  if (st != GQ_OK) return;
  st = rows::setup(info);
}

// Set-up for the current device (once per device per process).
gq_status current_device(const DeviceInfo** out) {
  int dev = -1;
  gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != GQ_OK) return st;
  if (dev < 0 || dev >= kMaxDevices)
    return fail(GQ_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::call_once(g_dev_once[dev], setup_device, dev);
  if (g_dev_status[dev] != GQ_OK) {
    return fail(g_dev_status[dev], "device %d set-up failed earlier", dev);
  }
  *out = &g_dev[dev];
  return GQ_OK;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

constexpr int64_t kMaxExtent = (int64_t(1) << 31) - 4096;

__global__ void fill_scales_kernel(float* s, int64_t n, float v) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    s[i] = v;
}

}  // namespace

gq_status fail(gq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

gq_status check_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return GQ_OK;
  return fail(GQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

gq_status encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype,
                          void* base, uint64_t dim0, uint64_t dim1,
                          uint64_t row_stride_bytes, uint32_t box0,
                          uint32_t box1, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, load_encode_fn);
  if (g_encode == nullptr) return g_encode_status;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llux%llu",
                static_cast<int>(r), static_cast<unsigned long long>(dim0),
                static_cast<unsigned long long>(dim1));
  return GQ_OK;
}

WorkspaceLayout colwise_workspace(int64_t K, int64_t G) {
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  WorkspaceLayout L;
  L.counters = 256;
  L.amax = L.counters + up(static_cast<size_t>(G * ((K + colwise::kW - 1) / colwise::kW)) * 4);
  L.total = L.amax + up(static_cast<size_t>(G * K) * 4);
  return L;
}

gq_status launch_fill_empty_scales(float* scales, int64_t n, uint32_t flags,
                                   cudaStream_t stream) {
  if (n <= 0) return GQ_OK;
  float v = kFp8Max / kEps;  // IEEE fp32 division on the host
  if (flags & GQ_SCALE_POW2) {  // the power of two below: clear the mantissa
    uint32_t b;
    memcpy(&b, &v, sizeof b);
    b &= 0xFF800000u;
    memcpy(&v, &b, sizeof v);
  }
  const int threads = 256;
  const int64_t blocks64 = (n + threads - 1) / threads;
  const int blocks = static_cast<int>(blocks64 < 4096 ? blocks64 : 4096);
  fill_scales_kernel<<<blocks, threads, 0, stream>>>(scales, n, v);
  return check_cuda(cudaGetLastError(), "fill empty-group scales");
}

}  // namespace gq

using namespace gq;

namespace {

// the calls that take a workspace
constexpr uint32_t kRowwiseFlags = GQ_SCALE_POW2 | GQ_WORKSPACE_ZEROED;
constexpr uint32_t kColwiseFlags = kRowwiseFlags | GQ_TWO_PHASE;

gq_status validate_common(const void* in, const void* out, const int32_t* offs,
                          int32_t n_groups, const float* scales, int64_t rows,
                          int64_t cols, const char* name) {
  if (rows < 0 || cols < 0)
    return fail(GQ_ERR_INVALID_ARG, "%s: negative size (%lld, %lld)", name,
                static_cast<long long>(rows), static_cast<long long>(cols));
  if (n_groups < 1)
    return fail(GQ_ERR_INVALID_ARG, "%s: n_groups must be >= 1 (got %d)", name,
                n_groups);
  if (n_groups > GQ_MAX_GROUPS)
    return fail(GQ_ERR_UNSUPPORTED, "%s: n_groups %d > %d", name, n_groups,
                GQ_MAX_GROUPS);
  if (offs == nullptr) return fail(GQ_ERR_INVALID_ARG, "%s: offs is NULL", name);
  if (!aligned(offs, 4))
    return fail(GQ_ERR_INVALID_ARG, "%s: offs not 4-byte aligned", name);
  if (rows > 0 && cols > 0) {
    if (in == nullptr || out == nullptr)
      return fail(GQ_ERR_INVALID_ARG, "%s: input or output is NULL", name);
    if (!aligned(in, 16) || !aligned(out, 16))
      return fail(GQ_ERR_INVALID_ARG,
                  "%s: input and output must be 16-byte aligned", name);
  }
  if (rows > kMaxExtent || cols > kMaxExtent)
    return fail(GQ_ERR_UNSUPPORTED, "%s: extent >= 2^31", name);
  (void)scales;
  return GQ_OK;
}

gq_status validate_ws(void* ws, size_t ws_bytes, size_t need, const char* name) {
  if (need == 0) return GQ_OK;
  if (ws == nullptr || ws_bytes < need)
    return fail(GQ_ERR_INVALID_ARG, "%s: workspace needs %zu bytes (got %zu%s)",
                name, need, ws_bytes, ws == nullptr ? ", NULL" : "");
  if (!aligned(ws, 256))
    return fail(GQ_ERR_INVALID_ARG, "%s: workspace not 256-byte aligned", name);
  return GQ_OK;
}

}  // namespace

extern "C" {

size_t gq_workspace_bytes(int kind, int64_t rows, int64_t cols,
                          int32_t n_groups) {
  if (rows < 0 || cols < 0 || n_groups < 1 || n_groups > GQ_MAX_GROUPS) return 0;
  if (kind == GQ_KIND_COLWISE) {
    const int64_t M = rows, K = cols;
    if (M == 0 || K == 0) return 0;
    return colwise_workspace(K, n_groups).total;
  }
  if (kind == GQ_KIND_ROWWISE_T) {
    const int64_t N = rows, Mg = cols;
    if (N == 0 || Mg == 0) return 0;
    return rowwise::workspace_bytes(N, Mg, n_groups);
  }
  return 0;
}

gq_status gq_fp8_colwise(const void* x, int64_t M, int64_t K,
                         const int32_t* offs, int32_t n_groups, void* out,
                         float* scales, void* workspace,
                         size_t workspace_bytes, gq_stream_t stream) {
  return gq_fp8_colwise_ex(x, M, K, offs, n_groups, out, scales, 0u, workspace,
                           workspace_bytes, stream);
}

gq_status gq_fp8_colwise_ex(const void* x, int64_t M, int64_t K,
                            const int32_t* offs, int32_t n_groups, void* out,
                            float* scales, uint32_t flags, void* workspace,
                            size_t workspace_bytes, gq_stream_t stream) {
  const char* name = "gq_fp8_colwise";
  if (flags & ~kColwiseFlags)
    return fail(GQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags & ~kColwiseFlags);
  gq_status st = validate_common(x, out, offs, n_groups, scales, M, K, name);
  if (st != GQ_OK) return st;
  if (K % 16 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: K = %lld is not a multiple of 16", name,
                static_cast<long long>(K));
  if (K > 0 && (scales == nullptr || !aligned(scales, 4)))
    return fail(GQ_ERR_INVALID_ARG, "%s: scales NULL or misaligned", name);
  const size_t need = gq_workspace_bytes(GQ_KIND_COLWISE, M, K, n_groups);
  st = validate_ws(workspace, workspace_bytes, need, name);
  if (st != GQ_OK) return st;
  if (K == 0) return GQ_OK;  // nothing to write
  const DeviceInfo* info = nullptr;
  st = current_device(&info);
  if (st != GQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0)
    return launch_fill_empty_scales(scales, static_cast<int64_t>(n_groups) * K, flags, s);
  return colwise::launch(*info, g_dbg, x, static_cast<int32_t>(M),
                         static_cast<int32_t>(K), offs, 0, n_groups, out, scales,
                         flags, workspace, s);
}

gq_status gq_fp8_expert_dim1(const void* w, int64_t E, int64_t K, int64_t N, void* out,
                             float* scales, uint32_t flags, void* workspace,
                             size_t workspace_bytes, gq_stream_t stream) {
  const char* name = "gq_fp8_expert_dim1";
  if (flags & ~kColwiseFlags)
    return fail(GQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags & ~kColwiseFlags);
  if (E < 1 || K < 0 || N < 0)
    return fail(GQ_ERR_INVALID_ARG, "%s: bad sizes (%lld, %lld, %lld)", name,
                static_cast<long long>(E), static_cast<long long>(K),
                static_cast<long long>(N));
  if (E > GQ_MAX_GROUPS)
    return fail(GQ_ERR_UNSUPPORTED, "%s: %lld experts > %d", name,
                static_cast<long long>(E), GQ_MAX_GROUPS);
  if (K > kMaxExtent || (K > 0 && E * K > kMaxExtent))  // E <= 1024: no overflow
    return fail(GQ_ERR_UNSUPPORTED, "%s: E * K >= 2^31", name);
  const int64_t M = E * K;
  if (N > kMaxExtent) return fail(GQ_ERR_UNSUPPORTED, "%s: extent >= 2^31", name);
  if (N % 16 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: N = %lld is not a multiple of 16", name,
                static_cast<long long>(N));
  if (M > 0 && N > 0) {
    if (w == nullptr || out == nullptr)
      return fail(GQ_ERR_INVALID_ARG, "%s: input or output is NULL", name);
    if (!aligned(w, 16) || !aligned(out, 16))
      return fail(GQ_ERR_INVALID_ARG, "%s: input and output must be 16-byte aligned", name);
  }
  if (N > 0 && (scales == nullptr || !aligned(scales, 4)))
    return fail(GQ_ERR_INVALID_ARG, "%s: scales NULL or misaligned", name);
  const size_t need = gq_workspace_bytes(GQ_KIND_COLWISE, M, N, static_cast<int32_t>(E));
  gq_status st = validate_ws(workspace, workspace_bytes, need, name);
  if (st != GQ_OK) return st;
  if (N == 0) return GQ_OK;
  const DeviceInfo* info = nullptr;
  st = current_device(&info);
  if (st != GQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) return launch_fill_empty_scales(scales, E * N, flags, s);
  return colwise::launch(*info, g_dbg, w, static_cast<int32_t>(M), static_cast<int32_t>(N),
                         nullptr, static_cast<int32_t>(K), static_cast<int32_t>(E), out, scales,
                         flags, workspace, s);
}

gq_status gq_fp8_expert_rowwise(const void* w, int64_t E, int64_t N, int64_t K, void* out,
                                float* scales, uint32_t flags, gq_stream_t stream) {
  const char* name = "gq_fp8_expert_rowwise";
  if (flags & ~static_cast<uint32_t>(GQ_SCALE_POW2))
    return fail(GQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name,
                flags & ~static_cast<uint32_t>(GQ_SCALE_POW2));
  if (E < 1 || N < 0 || K < 0)
    return fail(GQ_ERR_INVALID_ARG, "%s: bad sizes (%lld, %lld, %lld)", name,
                static_cast<long long>(E), static_cast<long long>(N),
                static_cast<long long>(K));
  if (E > kMaxExtent || N > kMaxExtent || K > kMaxExtent)
    return fail(GQ_ERR_UNSUPPORTED, "%s: extent >= 2^31", name);
  if (K % 8 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: K = %lld is not a multiple of 8", name,
                static_cast<long long>(K));
  const int64_t rows = E * N;  // both below 2^31: no overflow
  if (rows == 0) return GQ_OK;
  if (scales == nullptr || !aligned(scales, 4))
    return fail(GQ_ERR_INVALID_ARG, "%s: scales NULL or misaligned", name);
  if (K > 0) {
    if (w == nullptr || out == nullptr)
      return fail(GQ_ERR_INVALID_ARG, "%s: input or output is NULL", name);
    if (!aligned(w, 16) || !aligned(out, 16))
      return fail(GQ_ERR_INVALID_ARG, "%s: input and output must be 16-byte aligned", name);
  }
  const DeviceInfo* info = nullptr;
  gq_status st = current_device(&info);
  if (st != GQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_fill_empty_scales(scales, rows, flags, s);
  return rows::launch(*info, w, rows, K, out, scales, (flags & GQ_SCALE_POW2) != 0, s);
}

gq_status gq_fp8_rowwise_t(const void* a, int64_t N, int64_t Mg,
                           const int32_t* offs, int32_t n_groups, void* out_t,
                           float* scales, void* workspace,
                           size_t workspace_bytes, gq_stream_t stream) {
  return gq_fp8_rowwise_t_ex(a, N, Mg, offs, n_groups, out_t, scales, 0u, workspace,
                             workspace_bytes, stream);
}

gq_status gq_fp8_rowwise_t_ex(const void* a, int64_t N, int64_t Mg,
                              const int32_t* offs, int32_t n_groups, void* out_t,
                              float* scales, uint32_t flags, void* workspace,
                              size_t workspace_bytes, gq_stream_t stream) {
  const char* name = "gq_fp8_rowwise_t";
  if (flags & ~kRowwiseFlags)
    return fail(GQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags & ~kRowwiseFlags);
  gq_status st = validate_common(a, out_t, offs, n_groups, scales, N, Mg, name);
  if (st != GQ_OK) return st;
  if (N % 16 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: N = %lld is not a multiple of 16", name,
                static_cast<long long>(N));
  if (Mg % 8 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: Mg = %lld is not a multiple of 8", name,
                static_cast<long long>(Mg));
  if (N > 0 && (scales == nullptr || !aligned(scales, 4)))
    return fail(GQ_ERR_INVALID_ARG, "%s: scales NULL or misaligned", name);
  const size_t need = gq_workspace_bytes(GQ_KIND_ROWWISE_T, N, Mg, n_groups);
  st = validate_ws(workspace, workspace_bytes, need, name);
  if (st != GQ_OK) return st;
  if (N == 0) return GQ_OK;
  const DeviceInfo* info = nullptr;
  st = current_device(&info);
  if (st != GQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (Mg == 0)
    return launch_fill_empty_scales(scales, N * static_cast<int64_t>(n_groups), flags, s);
  return rowwise::launch(*info, g_dbg, a, static_cast<int32_t>(N),
                         static_cast<int32_t>(Mg), offs, n_groups, out_t, scales,
                         flags, workspace, s);
}

gq_status gq_mxfp8_dim0(const void* x, int64_t M, int64_t K, void* out, uint8_t* scales,
                        int mode, gq_stream_t stream) {
  const char* name = "gq_mxfp8_dim0";
  if (mode != GQ_MX_FLOOR && mode != GQ_MX_RCEIL)
    return fail(GQ_ERR_INVALID_ARG, "%s: unknown mode %d", name, mode);
  if (M < 0 || K < 0)
    return fail(GQ_ERR_INVALID_ARG, "%s: negative size (%lld, %lld)", name,
                static_cast<long long>(M), static_cast<long long>(K));
  if (M > kMaxExtent || K > kMaxExtent)
    return fail(GQ_ERR_UNSUPPORTED, "%s: extent >= 2^31", name);
  if (K % 32 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: K = %lld is not a multiple of 32", name,
                static_cast<long long>(K));
  if (M == 0 || K == 0) return GQ_OK;
  if (x == nullptr || out == nullptr || scales == nullptr)
    return fail(GQ_ERR_INVALID_ARG, "%s: NULL pointer", name);
  if (!aligned(x, 16) || !aligned(out, 16))
    return fail(GQ_ERR_INVALID_ARG, "%s: input and output must be 16-byte aligned", name);
  const DeviceInfo* info = nullptr;
  gq_status st = current_device(&info);
  if (st != GQ_OK) return st;
  return mx::launch(*info, x, M, K, out, scales, mode, reinterpret_cast<cudaStream_t>(stream));
}

gq_status gq_grouped_wgrad(const void* qa_t, const float* sa, const void* qx, const float* sx,
                           int64_t T, int64_t N, int64_t K, const int32_t* offs,
                           int32_t n_groups, void* out, gq_stream_t stream) {
  const char* name = "gq_grouped_wgrad";
  if (T < 0 || N < 0 || K < 0)
    return fail(GQ_ERR_INVALID_ARG, "%s: negative size (%lld, %lld, %lld)", name,
                static_cast<long long>(T), static_cast<long long>(N), static_cast<long long>(K));
  if (n_groups < 1 || n_groups > GQ_MAX_GROUPS)
    return fail(GQ_ERR_INVALID_ARG, "%s: n_groups = %d out of range", name, n_groups);
  if (T > kMaxExtent || N > kMaxExtent || K > kMaxExtent)
    return fail(GQ_ERR_UNSUPPORTED, "%s: extent >= 2^31", name);
  if (N % 16 != 0 || K % 16 != 0)
    return fail(GQ_ERR_UNSUPPORTED, "%s: N = %lld and K = %lld must be multiples of 16", name,
                static_cast<long long>(N), static_cast<long long>(K));
  if (N == 0 || K == 0) return GQ_OK;
  if (out == nullptr || sa == nullptr || sx == nullptr || offs == nullptr)
    return fail(GQ_ERR_INVALID_ARG, "%s: NULL pointer", name);
  if (!aligned(out, 16) || !aligned(sa, 4) || !aligned(sx, 4))
    return fail(GQ_ERR_INVALID_ARG, "%s: misaligned output or scales", name);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t out_bytes = static_cast<size_t>(n_groups) * N * K * 2;
  if (T == 0)  // every group is empty
    return check_cuda(cudaMemsetAsync(out, 0, out_bytes, s), "grouped_wgrad: zero output");
  if (qa_t == nullptr || qx == nullptr)
    return fail(GQ_ERR_INVALID_ARG, "%s: NULL operand", name);
  if (!aligned(qa_t, 16) || !aligned(qx, 16))
    return fail(GQ_ERR_INVALID_ARG, "%s: operands must be 16-byte aligned", name);
  const DeviceInfo* info = nullptr;
  gq_status st = current_device(&info);
  if (st != GQ_OK) return st;
  return wgrad::launch(*info, g_dbg, qa_t, sa, qx, sx, static_cast<int32_t>(T),
                       static_cast<int32_t>(N), static_cast<int32_t>(K), offs, n_groups, out, s);
}

gq_status gq_check_device_error(gq_stream_t stream) {
  const DeviceInfo* info = nullptr;
  gq_status st = current_device(&info);
  if (st != GQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = check_cuda(cudaStreamSynchronize(s), "stream synchronize");
  if (st != GQ_OK) return st;
  unsigned word = 0;
  st = check_cuda(cudaMemcpy(&word, info->err_word, sizeof word,
                             cudaMemcpyDeviceToHost),
                  "read error word");
  if (st != GQ_OK) return st;
  if (word != 0) {
    const unsigned zero = 0;
    st = check_cuda(cudaMemcpy(info->err_word, &zero, sizeof zero,
                               cudaMemcpyHostToDevice),
                    "clear error word");
    if (st != GQ_OK) return st;
    return fail(GQ_ERR_TIMEOUT,
                "a bounded wait expired on the GPU (error bits 0x%x: %s%s)", word,
                (word & kErrDepTimeout) ? "dependency " : "",
                (word & kErrMbarTimeout) ? "mbarrier" : "");
  }
  return GQ_OK;
}

const char* gq_status_string(gq_status status) {
  switch (status) {
    case GQ_OK: return "ok";
    case GQ_ERR_INVALID_ARG: return "invalid argument";
    case GQ_ERR_UNSUPPORTED: return "unsupported";
    case GQ_ERR_CUDA: return "CUDA error";
    case GQ_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* gq_last_error(void) { return g_msg; }

int gq_version(void) { return 200; }  // 0.2.0: mxfp8_dim0, grouped_wgrad, GQ_WORKSPACE_ZEROED

gq_status gq_set_lag(int kind, int32_t lag) {
  if (kind != GQ_KIND_COLWISE && kind != GQ_KIND_ROWWISE_T)
    return fail(GQ_ERR_INVALID_ARG, "gq_set_lag: unknown kind %d", kind);
  if (lag < 0) return fail(GQ_ERR_INVALID_ARG, "gq_set_lag: negative lag");
  g_dbg.lag[kind] = lag;
  return GQ_OK;
}

gq_status gq_debug_set(int flags, int64_t wait_timeout_ns) {
  if (wait_timeout_ns < 0)
    return fail(GQ_ERR_INVALID_ARG, "gq_debug_set: negative timeout");
  if (flags & ~3)
    return fail(GQ_ERR_INVALID_ARG, "gq_debug_set: unknown flags 0x%x", flags & ~3);
  g_dbg.skip_arrival = flags & 1;
  g_dbg.no_split = (flags >> 1) & 1;
  g_dbg.timeout_ns = wait_timeout_ns == 0 ? 1000000000ull
                                          : static_cast<uint64_t>(wait_timeout_ns);
  return GQ_OK;
}

}  // extern "C"
