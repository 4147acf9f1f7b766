// gq_rows.cu -- stacked expert weights W (E, N, K) scaled per row: one scale
// per (expert, row), the amax taken over the row's K elements, the output
// in W's layout (the "fp8 rowwise kernels for expert weights" of the
// pytorch/ao #2668 page's PR stack, #2696; the scale and the cast as in the
// per-group kernels: 448 / max(amax, 1e-12) in IEEE fp32, then e4m3 of the
// fp32 product, round-to-nearest-even, saturating).
//
// The E * N rows are independent, so this is a plain stream: one warp per
// row, a persistent grid stepping through the rows.  A row of up to kHold
// 16-byte chunks per lane (4096 elements) is read once into registers --
// all of its loads issued before the first is used -- reduced across the
// warp by shuffles, then scaled, cast and stored from the same registers.
// A longer row takes two passes: the amax pass keeps its lines in L2 and
// the cast pass reads them again from there.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace rows {

constexpr int kThreads = 256;  // 8 warps, one row each at a time
constexpr int kWarps = kThreads / 32;
constexpr int kHold = 16;      // 16-byte chunks per lane held in registers

struct Params {
  const uint4* w;  // 16-byte chunks of W: 8 bf16
  uint2* q;        // 8-byte chunks of the output: 8 e4m3
  float* scales;   // one per row
  int64_t rows;    // E * N
  int32_t chunks;  // K / 8 chunks per row
  bool pow2;       // scales rounded down to powers of two
};

// The largest |x| of a warp's bf16x2 accumulators, as fp32 bits.
__device__ __forceinline__ uint32_t warp_amax_bits(uint32_t acc) {
  uint32_t m = amax_bits_of(acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

__device__ __forceinline__ uint32_t absmax_chunk(uint32_t acc, const uint4& v) {
  return absmax_bf16x2(absmax_bf16x2(acc, v.x), absmax_bf16x2(absmax_bf16x2(v.y, v.z), v.w));
}

__device__ __forceinline__ uint2 cast_chunk(const uint4& v, float s) {
  return make_uint2(quant4(v.x, v.y, s, s, s, s), quant4(v.z, v.w, s, s, s, s));
}

// kInRegs: every row has at most 32 * kHold chunks.
template <bool kInRegs>
__global__ void __launch_bounds__(kThreads) rows_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); r < p.rows;
       r += nwarps) {
    const uint4* src = p.w + r * p.chunks;
    uint2* dst = p.q + r * p.chunks;
    uint32_t acc = 0u;
    if (kInRegs) {
      uint4 v[kHold];
#pragma unroll
      for (int i = 0; i < kHold; ++i) {
        const int c = lane + 32 * i;
        v[i] = c < p.chunks ? __ldcs(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kHold; ++i) acc = absmax_chunk(acc, v[i]);
      const float s = scale_from_amax_bits(warp_amax_bits(acc), p.pow2);
      if (lane == 0) p.scales[r] = s;
#pragma unroll
      for (int i = 0; i < kHold; ++i) {
        const int c = lane + 32 * i;
        if (c < p.chunks) __stcs(dst + c, cast_chunk(v[i], s));
      }
    } else {
      for (int c = lane; c < p.chunks; c += 32) acc = absmax_chunk(acc, __ldg(src + c));
      const float s = scale_from_amax_bits(warp_amax_bits(acc), p.pow2);
      if (lane == 0) p.scales[r] = s;
      for (int c = lane; c < p.chunks; c += 32) __stcs(dst + c, cast_chunk(__ldcs(src + c), s));
    }
  }
}

gq_status setup(DeviceInfo& info) {
  int occ = 0;
  gq_status st = check_cuda(
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rows_kernel<true>, kThreads, 0),
      "expert_rowwise: occupancy");
  if (st != GQ_OK) return st;
  info.rows_ctas_per_sm = occ > 0 ? occ : 1;
  return GQ_OK;
}

gq_status launch(const DeviceInfo& info, const void* w, int64_t rows, int64_t K, void* out,
                 float* scales, bool pow2, cudaStream_t stream) {
  Params p;
  p.w = static_cast<const uint4*>(w);
  p.q = static_cast<uint2*>(out);
  p.scales = scales;
  p.rows = rows;
  p.chunks = static_cast<int32_t>(K / 8);
  p.pow2 = pow2;
  const int64_t per_launch = static_cast<int64_t>(info.sm_count) * info.rows_ctas_per_sm;
  const int64_t need = (rows + kWarps - 1) / kWarps;
  const int grid = static_cast<int>(need < per_launch ? need : per_launch);
  if (p.chunks <= 32 * kHold)
    rows_kernel<true><<<grid, kThreads, 0, stream>>>(p);
  else
    rows_kernel<false><<<grid, kThreads, 0, stream>>>(p);
  return check_cuda(cudaGetLastError(), "expert_rowwise: launch");
}

}  // namespace rows
}  // namespace gq
