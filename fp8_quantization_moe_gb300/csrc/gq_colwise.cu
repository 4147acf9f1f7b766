// gq_colwise.cu -- colwise per-token-group fp8 e4m3 scaling on sm_103a.
//
// X (M, K) bf16 row-major; token groups are row ranges [s_g, e_g); one scale
// per (group, column).  This is the per-token-group scaling "along dim0" of
// pytorch/ao #2668 ("use smaller block sizes for per group scaling kernels
// to improve perf", intro); the page's lesson -- the grid was too small to
// fill the SMs -- is answered here by a persistent grid sized to the SM
// count that claims 16 KB tiles one by one.
//
// Tiles are kR = 64 rows x kW = 128 columns (256-byte row runs), loaded by
// TMA into a kStages-deep shared-memory ring.  A column slab (all M rows of
// kW columns) is one dependency group: phase B of a tile of slab d needs the
// amax of every tile of slab d.  See gq_device.cuh for the schedule.
//
// Per tile, phase A: each consumer thread owns one 16-byte column chunk
// (8 columns) and every 8th row; it folds |x| with max.xorsign.abs.bf16x2,
// the CTA reduces over rows through shared memory, and one atomicMax per
// (group, column) goes to the amax words.  Phase B: the scale of each
// (group, column) is 448 / max(amax, 1e-12) (IEEE division), the product
// x * scale is an fp32 multiply, and cvt.rn.satfinite.e4m3x2 packs pairs;
// 8 output bytes per thread and row leave as one 8-byte store, so a warp
// writes two 128-byte row runs.
#include <cstdio>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace colwise {

constexpr int kStages = 6;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kTileBytes = kW * kR * 2;
constexpr int kChunks = kW / 8;  // 16-byte column chunks per tile row
static_assert(kConsumers == kW, "one consumer thread per column in the reduction");
static_assert(kConsumers == kChunks * (kR / 8), "one 16-byte chunk and every 8th row per thread");

using Hdr = TileHdr<kR>;

struct Smem {
  uint8_t tile[kStages][kTileBytes];  // first member: 1024-byte aligned
  Hdr hdr[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t ends_ready;
  int32_t ends[kMaxGroups];
  uint32_t red[kConsumerWarps][kChunks * 4];
  alignas(16) float sc[2][kW];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

struct Params {
  const int32_t* offs;
  uint8_t* out;
  float* scales;
  uint32_t* ticket;  // one word
  uint32_t* done;    // one word per slab
  uint32_t* amax;    // (G, K) fp32 bit patterns
  unsigned* err;
  int32_t M, K, G;
  Schedule sched;
  uint64_t timeout_ns;
  int32_t skip_arrival;
};

__device__ __forceinline__ void producer(Smem& s, const CUtensorMap* xmap,
                                         const Params& p) {
  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  const uint32_t total = 2u * static_cast<uint32_t>(p.sched.units) *
                         static_cast<uint32_t>(p.sched.groups);
  bool ends_ok = false;
  int st = 0;
  uint32_t ph = 0;
  for (;;) {
    if (!mbar_wait(&s.empty[st], ph ^ 1u, 4 * p.timeout_ns, p.err)) return;
    const uint32_t t = atomicAdd(p.ticket, 1u);
    Hdr& h = s.hdr[st];
    if (t >= total) {
      h.phase = -1;
      mbar_arrive(&s.full[st]);
      return;
    }
    const Ticket k = decode_ticket(t, p.sched);
    const int32_t c0 = k.dg * kW;
    const int32_t r0 = k.unit * kR;
    mbar_expect_tx(&s.full[st], kTileBytes);
    tma_load_2d(s.tile[st], xmap, c0, r0, &s.full[st],
                k.phase == 0 ? pol_a : pol_b);
    if (!ends_ok) {
      if (!mbar_wait(&s.ends_ready, 0u, 4 * p.timeout_ns, p.err)) return;
      ends_ok = true;
    }
    h.phase = k.phase;
    h.dg = k.dg;
    fill_segments(h, s.ends, p.G, r0, min(r0 + kR, p.M),
                  k.unit == p.sched.units - 1);
    mbar_arrive(&s.full[st]);
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
}

// Phase A: fold |x| of the tile into the amax words of each segment.
__device__ __forceinline__ void phase_a(Smem& s, const Hdr& h, uint32_t tile,
                                        const Params& p, int t, int warp,
                                        int lane) {
  const int cc = t & (kChunks - 1);  // column chunk
  const int rl = t / kChunks;        // row lane: rows rl, rl + 8, ...
  const int32_t c0 = h.dg * kW;
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    uint32_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
    if (a == 0 && b == kR) {
#pragma unroll
      for (int i = 0; i < kR / 8; ++i) {
        const int r = rl + 8 * i;
        const uint4 v = lds128(tile + (r * kW + cc * 8) * 2);
        acc0 = absmax_bf16x2(acc0, v.x);
        acc1 = absmax_bf16x2(acc1, v.y);
        acc2 = absmax_bf16x2(acc2, v.z);
        acc3 = absmax_bf16x2(acc3, v.w);
      }
    } else {
#pragma unroll 4
      for (int i = 0; i < kR / 8; ++i) {
        const int r = rl + 8 * i;
        if (r >= a && r < b) {
          const uint4 v = lds128(tile + (r * kW + cc * 8) * 2);
          acc0 = absmax_bf16x2(acc0, v.x);
          acc1 = absmax_bf16x2(acc1, v.y);
          acc2 = absmax_bf16x2(acc2, v.z);
          acc3 = absmax_bf16x2(acc3, v.w);
        }
      }
    }
    // lanes l and l ^ 16 hold the same column chunk
    acc0 = absmax_bf16x2(acc0, __shfl_xor_sync(0xffffffffu, acc0, 16));
    acc1 = absmax_bf16x2(acc1, __shfl_xor_sync(0xffffffffu, acc1, 16));
    acc2 = absmax_bf16x2(acc2, __shfl_xor_sync(0xffffffffu, acc2, 16));
    acc3 = absmax_bf16x2(acc3, __shfl_xor_sync(0xffffffffu, acc3, 16));
    if (lane < 16) {
      uint32_t* r = &s.red[warp][lane * 4];
      r[0] = acc0;
      r[1] = acc1;
      r[2] = acc2;
      r[3] = acc3;
    }
    named_bar(1, kConsumers);
    {
      // thread t -> column t of the slab
      const int word = t >> 1;  // chunk * 4 + word-in-chunk
      const int shift = (t & 1) * 16;
      uint32_t m = 0;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const uint32_t v = (s.red[w][word] >> shift) & 0x7FFFu;
        m = v > m ? v : m;
      }
      const int32_t col = c0 + t;
      if (m != 0u && col < p.K)
        atomicMax(p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + col, m << 16);
    }
    named_bar(1, kConsumers);
  }
  if (t == 0) {
    const bool skip = p.skip_arrival && h.dg == 0 && h.lo == 0;
    __threadfence();
    if (!skip) atomicAdd(p.done + h.dg, 1u);
  }
}

// Phase B: scales, then the scaled cast of every row inside a group.
__device__ __forceinline__ void phase_b(Smem& s, const Hdr& h, uint32_t tile,
                                        const Params& p, int t,
                                        uint32_t& sc_seq) {
  const int cc = t & (kChunks - 1);
  const int rl = t / kChunks;
  const int32_t c0 = h.dg * kW;
  if (t == 0)
    wait_counter(p.done + h.dg, static_cast<uint32_t>(p.sched.units),
                 p.timeout_ns, p.err);
  named_bar(1, kConsumers);
  const int32_t col = c0 + t;
  const bool col_in = col < p.K;
  for (int g = h.own_lo; g < h.own_hi; ++g) {
    if (col_in) {
      const size_t i = static_cast<size_t>(g) * p.K + col;
      p.scales[i] = scale_from_amax_bits(ld_cg_u32(p.amax + i));
    }
  }
  const bool chunk_in = c0 + cc * 8 < p.K;
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    float* scb = s.sc[sc_seq & 1u];
    ++sc_seq;
    scb[t] = col_in ? scale_from_amax_bits(ld_cg_u32(
                          p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + col))
                    : 0.0f;
    named_bar(1, kConsumers);
    const float4 sa = *reinterpret_cast<const float4*>(scb + cc * 8);
    const float4 sb = *reinterpret_cast<const float4*>(scb + cc * 8 + 4);
    uint8_t* obase =
        p.out + static_cast<size_t>(h.lo) * p.K + static_cast<size_t>(c0 + cc * 8);
#pragma unroll 4
    for (int i = 0; i < kR / 8; ++i) {
      const int r = rl + 8 * i;
      if (r >= a && r < b && chunk_in) {
        const uint4 v = lds128(tile + (r * kW + cc * 8) * 2);
        const uint32_t w0 =
            cvt_e4m3x2(__fmul_rn(bf16_lo(v.x), sa.x), __fmul_rn(bf16_hi(v.x), sa.y)) |
            (cvt_e4m3x2(__fmul_rn(bf16_lo(v.y), sa.z), __fmul_rn(bf16_hi(v.y), sa.w))
             << 16);
        const uint32_t w1 =
            cvt_e4m3x2(__fmul_rn(bf16_lo(v.z), sb.x), __fmul_rn(bf16_hi(v.z), sb.y)) |
            (cvt_e4m3x2(__fmul_rn(bf16_lo(v.w), sb.z), __fmul_rn(bf16_hi(v.w), sb.w))
             << 16);
        __stcs(reinterpret_cast<uint2*>(obase + static_cast<size_t>(r) * p.K),
               make_uint2(w0, w1));
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    colwise_kernel(const __grid_constant__ CUtensorMap xmap, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kConsumerWarps);
    }
    mbar_init(&s.ends_ready, 32);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tensormap(&xmap);
      producer(s, &xmap, p);
    }
    return;
  }

  if (warp == 0) {
    build_ends(p.offs, p.G, p.M, s.ends, lane);
    __syncwarp();
    mbar_arrive(&s.ends_ready);
  }

  const int t = threadIdx.x;
  int st = 0;
  uint32_t ph = 0;
  uint32_t sc_seq = 0;
  for (;;) {
    const bool ok = mbar_wait(&s.full[st], ph, 4 * p.timeout_ns, p.err);
    if (named_bar_any(1, kConsumers, !ok)) break;  // all consumers agree
    const Hdr& h = s.hdr[st];
    const int phase = h.phase;
    if (phase < 0) break;
    const uint32_t tile = smem_addr(s.tile[st]);
    if (phase == 0)
      phase_a(s, h, tile, p, t, warp, lane);
    else
      phase_b(s, h, tile, p, t, sc_seq);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
}

gq_status setup(DeviceInfo& info) {
  gq_status st = check_cuda(
      cudaFuncSetAttribute(colwise_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)),
      "colwise: set shared memory size");
  if (st != GQ_OK) return st;
  int occ = 0;
  st = check_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &occ, colwise_kernel, kThreads, kSmemBytes),
                  "colwise: occupancy");
  if (st != GQ_OK) return st;
  if (occ < 1) return fail(GQ_ERR_UNSUPPORTED, "colwise kernel does not fit an SM");
  info.colwise_ctas_per_sm = occ;
  return GQ_OK;
}

gq_status launch(const DeviceInfo& info, const DebugKnobs& dbg, const void* x,
                 int32_t M, int32_t K, const int32_t* offs, int32_t G,
                 void* out, float* scales, void* ws, cudaStream_t stream) {
  CUtensorMap xmap;
  gq_status st = encode_tiled_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(x), static_cast<uint64_t>(K),
                                 static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(K) * 2, kW, kR,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;

  Params p;
  p.sched.units = (M + kR - 1) / kR;
  p.sched.groups = (K + kW - 1) / kW;
  const int64_t total = 2ll * p.sched.units * p.sched.groups;
  const int64_t max_ctas =
      static_cast<int64_t>(info.sm_count) * info.colwise_ctas_per_sm;
  const int grid = static_cast<int>(total < max_ctas ? total : max_ctas);
  int64_t lag = (2ll * grid + p.sched.units - 1) / p.sched.units;
  if (lag < 1) lag = 1;
  if (lag > p.sched.groups) lag = p.sched.groups;
  p.sched.lag = static_cast<int32_t>(lag);

  const WorkspaceLayout L =
      workspace_layout(p.sched.groups, static_cast<int64_t>(G) * K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.offs = offs;
  p.out = static_cast<uint8_t*>(out);
  p.scales = scales;
  p.ticket = reinterpret_cast<uint32_t*>(w);
  p.done = reinterpret_cast<uint32_t*>(w + L.counters);
  p.amax = reinterpret_cast<uint32_t*>(w + L.amax);
  p.err = info.err_word;
  p.M = M;
  p.K = K;
  p.G = G;
  p.timeout_ns = dbg.timeout_ns;
  p.skip_arrival = dbg.skip_arrival;

  st = check_cuda(cudaMemsetAsync(ws, 0, L.total, stream), "colwise: clear workspace");
  if (st != GQ_OK) return st;
  colwise_kernel<<<grid, kThreads, kSmemBytes, stream>>>(xmap, p);
  return check_cuda(cudaGetLastError(), "colwise: launch");
}

}  // namespace colwise
}  // namespace gq
