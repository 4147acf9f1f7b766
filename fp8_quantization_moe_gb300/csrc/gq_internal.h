// gq_internal.h -- host-side declarations shared by the translation units of
// libgqfp8 (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gq_fp8.h"

namespace gq {

// Per-device facts and handles, filled once per device.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  unsigned* err_word = nullptr;  // device address of the error word
  int colwise_ctas_per_sm = 0;
  int rowwise_ctas_per_sm = 0;
  int mx_ctas_per_sm = 0;
  int rows_ctas_per_sm = 0;
};

// Launch-time knobs (test hooks).
struct DebugKnobs {
  int skip_arrival = 0;
  int no_split = 0;  // rowwise_t: never split units across blocks
  uint64_t timeout_ns = 1000000000ull;
  int32_t lag[2] = {0, 0};  // per kind; 0 = automatic
};

// Encodes a 2-D tiled tensor map (row-major, dim0 innermost).
gq_status encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype,
                          void* base, uint64_t dim0, uint64_t dim1,
                          uint64_t row_stride_bytes, uint32_t box0,
                          uint32_t box1, CUtensorMapSwizzle swizzle);

// Records a message for gq_last_error() and returns `st`.
gq_status fail(gq_status st, const char* fmt, ...);

// Returns GQ_ERR_CUDA with the runtime's message if `e` is an error.
gq_status check_cuda(cudaError_t e, const char* what);

// Colwise workspace layout: a 256-byte header (work counters), one counter
// per (group, 128-column slab) strip, then the (G, K) amax words.  Offsets
// in bytes; every region starts on a 256-byte boundary.  Every launch
// leaves all of it zero.
struct WorkspaceLayout {
  size_t counters = 0;  // start of the strip counters
  size_t amax = 0;      // start of the amax words
  size_t total = 0;
};
WorkspaceLayout colwise_workspace(int64_t K, int64_t G);

namespace colwise {
constexpr int kW = 128;  // columns per slab
gq_status setup(DeviceInfo& info);
// offs == nullptr: G groups of `uniform` rows each.
gq_status launch(const DeviceInfo& info, const DebugKnobs& dbg, const void* x,
                 int32_t M, int32_t K, const int32_t* offs, int32_t uniform, int32_t G,
                 void* out, float* scales, uint32_t flags, void* ws, cudaStream_t stream);
}  // namespace colwise

namespace rowwise {
constexpr int kTn = 64;  // rows of A per window: one row band
constexpr int kTm = 64;  // token columns per window
constexpr size_t kHeaderBytes = 256;  // unit counter, finished-blocks counter, padded
constexpr int kSplitWords = 68;        // per split unit: kTn amax words, a counter, padding
// Workspace of a call: the header, then kSplitWords words for every
// (row band, group) unit that may be split (groups of 4090 tokens or more).
size_t workspace_bytes(int64_t N, int64_t Mg, int64_t G);
gq_status setup(DeviceInfo& info);
gq_status launch(const DeviceInfo& info, const DebugKnobs& dbg, const void* a,
                 int32_t N, int32_t Mg, const int32_t* offs, int32_t G,
                 void* out_t, float* scales, uint32_t flags, void* ws, cudaStream_t stream);
}  // namespace rowwise

namespace mx {
gq_status setup(DeviceInfo& info);
gq_status launch(const DeviceInfo& info, const void* x, int64_t M, int64_t K, void* out,
                 uint8_t* scales, int mode, cudaStream_t stream);
}  // namespace mx

namespace rows {
gq_status setup(DeviceInfo& info);
gq_status launch(const DeviceInfo& info, const void* w, int64_t rows, int64_t K, void* out,
                 float* scales, bool pow2, cudaStream_t stream);
}  // namespace rows

namespace wgrad {
gq_status setup(DeviceInfo& info);
gq_status launch(const DeviceInfo& info, const DebugKnobs& dbg, const void* qa_t, const float* sa,
                 const void* qx, const float* sx, int32_t T, int32_t N, int32_t K,
                 const int32_t* offs, int32_t G, void* out, cudaStream_t stream);
}  // namespace wgrad

// Writes the scale of an empty group -- 448 / 1e-12 (fp32), or its power
// of two below with GQ_SCALE_POW2 -- into n scales: every group is empty
// when the token extent is 0.
gq_status launch_fill_empty_scales(float* scales, int64_t n, uint32_t flags,
                                   cudaStream_t stream);

}  // namespace gq
