// gq_mxfp8.cu -- mxfp8 cast along dim0 on sm_103a.
//
// X (M, K) bf16 row-major, K % 32 == 0.  Every 32 consecutive elements of a
// row form a block that shares one power-of-two scale 2^E, stored as an e8m0
// byte E + 127; elements are e4m3(fp32(x * 2^-E)).  This is the mxfp8 cast
// of the pytorch/ao page "[mxfp8 moe training] fix mxfp8 a2a bench script;
// set mxfp8 a2a scaling type to RCEIL" (Summary: the dim0_mxfp8_floor cast
// benchmark, and the RCEIL scaling type), with the two scaling types:
//   FLOOR: E = floor(log2(amax)) - 8  (8: the exponent of 448, e4m3's largest);
//   RCEIL: E = ceil(log2(fp32(amax / 448))).
// E is clamped to [-127, 127]; a block whose amax is 0 gets E = -127.
//
// The cast is a pure stream -- every block depends on its own 64 bytes
// alone -- so the kernel is plain coalesced loads and stores: lane l of a
// warp takes 16-byte chunk l of each 512-byte stretch (four stretches in
// flight per warp), four consecutive lanes hold one block and join their
// maxima with two shuffles, and each lane writes its 8 e4m3 bytes; the first
// lane of a block writes the scale byte.  Loads and stores are streaming
// (evict-first): nothing is read twice.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace mx {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 512-byte stretches per warp and step

struct Params {
  const uint4* x;     // 16-byte chunks of X
  uint2* q;           // 8-byte chunks of the e4m3 output
  uint8_t* scales;    // (M, K / 32) e8m0 bytes
  int64_t chunks;     // M * K / 8 (a multiple of 4: K % 32 == 0)
  int32_t mode;       // GQ_MX_FLOOR or GQ_MX_RCEIL
};

// floor(log2(a)) of a positive finite fp32 given by its bits (subnormals
// included): the exponent field, or the top set bit of a subnormal's
// significand.
__device__ __forceinline__ int floor_log2_bits(uint32_t b) {
  const int ex = static_cast<int>(b >> 23);
  return ex ? ex - 127 : (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
}

// The block exponent E for an amax given by its fp32 bits (sign clear).
__device__ __forceinline__ int mx_exponent(uint32_t amax_bits, int mode) {
  if (amax_bits == 0u) return -127;
  int E;
  if (mode == GQ_MX_FLOOR) {
    E = floor_log2_bits(amax_bits) - 8;
  } else {
    // v > 0: a bf16 amax is at least 2^-133, and 2^-133 / 448 > 2^-149
    const uint32_t v = __float_as_uint(__fdiv_rn(__uint_as_float(amax_bits), kFp8Max));
    const uint32_t sig = (v >> 23) ? (v & 0x7FFFFFu) : (v & 0x7FFFFFu) & ((v & 0x7FFFFFu) - 1u);
    E = floor_log2_bits(v) + (sig != 0u ? 1 : 0);  // ceil: up unless a power of two
  }
  return min(max(E, -127), 127);
}

// 2^n as fp32 for n in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int n) {
  return __uint_as_float(n >= -126 ? static_cast<uint32_t>(n + 127) << 23 : 0x00400000u);
}

__global__ void __launch_bounds__(kThreads)
    mx_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + (threadIdx.x & ~31)) * kUnroll;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads * kUnroll;
  for (int64_t base = warp0; base < p.chunks; base += stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + 32 * u + lane;
      v[u] = c < p.chunks ? __ldcs(p.x + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + 32 * u + lane;
      uint32_t m = amax_bits_of(absmax_bf16x2(absmax_bf16x2(v[u].x, v[u].y),
                                              absmax_bf16x2(v[u].z, v[u].w)));
      // lanes 4j .. 4j+3 hold one block (base is a multiple of 32)
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const int E = mx_exponent(m, p.mode);
      const float f = pow2f(-E);
      if (c < p.chunks) {
        __stcs(p.q + c, make_uint2(quant4(v[u].x, v[u].y, f, f, f, f),
                                   quant4(v[u].z, v[u].w, f, f, f, f)));
        if ((lane & 3) == 0) p.scales[c >> 2] = static_cast<uint8_t>(E + 127);
      }
    }
  }
}

gq_status setup(DeviceInfo& info) {
  int occ = 0;
  const gq_status st = check_cuda(
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, mx_kernel, kThreads, 0),
      "mxfp8: occupancy");
  if (st != GQ_OK) return st;
  if (occ < 1) return fail(GQ_ERR_UNSUPPORTED, "mxfp8 kernel does not fit an SM");
  info.mx_ctas_per_sm = occ;
  return GQ_OK;
}

gq_status launch(const DeviceInfo& info, const void* x, int64_t M, int64_t K, void* out,
                 uint8_t* scales, int mode, cudaStream_t stream) {
  Params p;
  p.x = static_cast<const uint4*>(x);
  p.q = static_cast<uint2*>(out);
  p.scales = scales;
  p.chunks = M * K / 8;
  p.mode = mode;
  const int64_t want = (p.chunks + static_cast<int64_t>(kThreads) * kUnroll - 1) /
                       (static_cast<int64_t>(kThreads) * kUnroll);
  const int64_t cap = static_cast<int64_t>(info.sm_count) * info.mx_ctas_per_sm;
  const int grid = static_cast<int>(want < cap ? want : cap);
  mx_kernel<<<grid, kThreads, 0, stream>>>(p);
  return check_cuda(cudaGetLastError(), "mxfp8: launch");
}

}  // namespace mx
}  // namespace gq
