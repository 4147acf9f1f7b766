// gq_colwise.cu -- colwise per-token-group fp8 e4m3 scaling on sm_103a.
//
// X (M, K) bf16 row-major; token groups are row ranges [s_g, e_g); one scale
// per (group, column).  This is the per-token-group scaling "along dim0" of
// pytorch/ao #2668 ("use smaller block sizes for per group scaling kernels
// to improve perf", intro); the page's lesson -- the grid was too small to
// fill the SMs -- is answered here by a persistent grid of two CTAs per SM.
//
// A stage is kR = 64 rows x kW = 128 columns, loaded by TMA as two 64-column
// halves with the 128-byte swizzle (row r of a half is 128 bytes; its
// 16-byte chunk k sits at slot k ^ (r % 8)).  A super tile is kSub = 4
// stages: 256 rows of one column slab.  A column slab (all M rows of kW
// columns) is one dependency group: phase B of slab d needs the amax of every
// super tile of slab d.  See gq_device.cuh for the schedule.  In phase B the
// producer lanes bring the 128 amax words of each of the super tile's first
// kSegA segments into its context (one 16-byte cp.async per lane).
//
// The eight consumer warps work on each stage independently -- no barrier
// among them:
//   phase A: warp w takes a 16-column strip (half w / 4, chunks 2 (w % 4)
//     and 2 (w % 4) + 1); per segment a lane folds |x| of its chunk over
//     every 16th row of every stage the segment covers, with
//     max.xorsign.abs.bf16x2; a butterfly over the 16 lanes of a chunk
//     finishes the column maxima and 16 lanes issue one atomicMax each;
//   phase B: warp w takes rows 8w .. 8w + 7 of every stage; per segment a
//     lane computes four of the 128 scales (448 / max(amax, 1e-12), IEEE
//     division) and gathers the eight of its chunk by shuffles; products
//     are IEEE fp32 multiplies (mul.rn.f32x2), packed with
//     cvt.rn.satfinite.e4m3x2; each warp store writes two 128-byte output
//     row runs.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace colwise {

constexpr int kStages = 5;
constexpr int kSub = 4;             // stages per super tile
constexpr int kSuper = kSub * kR;   // rows per super tile
constexpr int kCtx = 3;             // super-tile contexts in flight
constexpr int kConsumerWarps = 8;
constexpr int kThreads = kConsumerWarps * 32 + 64;  // + producer + signal warps
constexpr int kSigSlots = 16;
constexpr int kHalfBytes = 64 * kR * 2;  // one swizzled 64-column half
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr int kSegA = 4;  // segments whose amax words ride in the context
static_assert(kW == 128 && kR == 64, "tile shape assumed by the lane maps");
static_assert(kW == 32 * 4, "one 16-byte amax chunk per producer lane");
static_assert(kSub < kStages, "a super tile wraps the stage ring at most once");
static_assert(kSigSlots > kStages, "a warp cannot lap the signal ring");

using Hdr = TileHdr<kSuper>;

struct Ctx {
  Hdr hdr;
  alignas(16) uint32_t amax[kSegA][kW];  // phase B amax words
};

struct Smem {
  uint8_t tile[kStages][kTileBytes];  // first member: 1024-byte aligned
  Ctx ctx[kCtx];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t ctx_empty[kCtx];
  uint64_t ends_ready;
  SigRing<kSigSlots> sig;
  DepFlag dep;
  int32_t ends[kMaxGroups];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

struct Params {
  const int32_t* offs;
  uint8_t* out;
  float* scales;
  uint32_t* done;  // one word per slab
  uint32_t* amax;  // (G, K) fp32 bit patterns
  unsigned* err;
  int32_t M, K, G;
  Schedule sched;  // units = super tiles per slab
  uint64_t timeout_ns;
  int32_t skip_arrival;
};

// Shared-memory offset of chunk `k` (0..15, 8 columns each) of stage row r.
__device__ __forceinline__ uint32_t chunk_off(int r, int k) {
  return static_cast<uint32_t>((k >> 3) * kHalfBytes + r * 128 + (((k ^ r) & 7) << 4));
}

// ------------------------------------------------------------- producer --
__device__ __forceinline__ void producer(Smem& s, const CUtensorMap* xmap,
                                         const Params& p, int lane) {
  build_ends(p.offs, p.G, p.M, s.ends, lane);
  __syncwarp();
  if (lane == 0) mbar_arrive(&s.ends_ready);

  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  const int32_t units = p.sched.units;
  const int32_t blocks = 2 * p.sched.groups;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  int32_t ready_dg = -1;  // slabs <= ready_dg are complete
  int st = 0, ci = 0;
  uint32_t ph = 0, cph = 0;
  for (TicketWalk tw(blockIdx.x, gridDim.x, units);; tw.next(units)) {
    Ctx& c = s.ctx[ci];
    Hdr& h = c.hdr;
    if (!mbar_wait(&s.ctx_empty[ci], cph ^ 1u, wait_ns, p.err)) return;
    bool stop = tw.block >= blocks;
    int32_t phase = 0, dg = 0;
    if (!stop) decode_block(tw.block, p.sched, phase, dg);
    if (!stop && phase == 1 && dg > ready_dg) {
      bool ok = true;
      if (lane == 0) ok = wait_dep_flag(s.dep, dg, 2 * p.timeout_ns, p.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) {
        ld_acquire_cta_s32(&s.dep.ready);  // every lane acquires before reading amax
        ready_dg = dg;
      }
      stop = !ok;
    }
    if (!mbar_wait(&s.empty[st], ph ^ 1u, wait_ns, p.err)) return;
    if (stop) {
      if (lane == 0) {
        h.phase = -1;
        mbar_arrive(&s.full[st]);
      }
      return;
    }
    const int32_t c0 = dg * kW;
    const int32_t r0 = tw.unit * kSuper;
    const int32_t r1 = min(r0 + kSuper, p.M);
    const int nsub = (r1 - r0 + kR - 1) / kR;
    build_header_warp(h, s.ends, p.G, r0, r1, tw.unit == units - 1, lane);
    __syncwarp();
    if (phase == 1) {
      const int n = min(static_cast<int>(h.nseg), kSegA);
      const int32_t col = c0 + 4 * lane;
      for (int j = 0; j < n; ++j)
        cp_async_16(smem_addr(&c.amax[j][4 * lane]),
                    p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + (col < p.K ? col : 0),
                    col < p.K ? 16u : 0u);
      cp_async_mbar_arrive(&s.full[st]);  // the first stage waits for them
    }
    if (lane == 0) {
      h.phase = phase;
      h.dg = dg;
      h.nsub = nsub;
    }
    __syncwarp();
    const bool two = c0 + 64 < p.K;  // the second half holds columns
    const uint64_t pol = phase == 0 ? pol_a : pol_b;
    for (int k = 0; k < nsub; ++k) {
      if (k > 0 && !mbar_wait(&s.empty[st], ph ^ 1u, wait_ns, p.err)) return;
      if (lane == 0) {
        mbar_arrive_expect_tx(&s.full[st], two ? kTileBytes : kHalfBytes);
        tma_load_2d(s.tile[st], xmap, c0, r0 + k * kR, &s.full[st], pol);
        if (two)
          tma_load_2d(s.tile[st] + kHalfBytes, xmap, c0 + 64, r0 + k * kR, &s.full[st], pol);
      }
      if (++st == kStages) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (++ci == kCtx) {
      ci = 0;
      cph ^= 1u;
    }
  }
}

// ------------------------------------------------------------ consumers --
// The stages of one super tile, as seen by one consumer warp: acquired in
// order (full barrier), released in order (empty barrier) as soon as the
// warp is done with them.
struct SubTiles {
  int st0;
  uint32_t ph0;
  int nsub, acq, rel;
  uint64_t wait_ns;
  unsigned* err;
  __device__ __forceinline__ int stage(int k) const {
    return st0 + k < kStages ? st0 + k : st0 + k - kStages;
  }
  __device__ __forceinline__ uint32_t parity(int k) const {
    return st0 + k < kStages ? ph0 : ph0 ^ 1u;
  }
  __device__ __forceinline__ bool acquire(Smem& s, int k) {
    for (; acq <= k; ++acq) {
      const bool ok = mbar_wait(&s.full[stage(acq)], parity(acq), wait_ns, err);
      if (__any_sync(0xffffffffu, !ok)) return false;  // the warp leaves together
    }
    return true;
  }
  __device__ __forceinline__ void release(Smem& s, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[stage(rel)]);
    ++rel;
  }
  __device__ __forceinline__ bool finish(Smem& s, int lane) {
    while (rel < nsub) {
      if (!acquire(s, rel)) return false;
      release(s, lane);
    }
    return true;
  }
};

// Phase A, warp w: column maxima of its 16-column strip per segment, one
// atomicMax per (segment, column); then the super tile goes to the signal
// lane.
__device__ __forceinline__ bool phase_a(Smem& s, const Hdr& h, SubTiles& sub,
                                        const Params& p, int warp, int lane,
                                        uint32_t& sig_seq) {
  const int kc = (warp >> 2) * 8 + (warp & 3) * 2 + (lane & 1);  // chunk 0..15
  const int r0 = lane >> 1;                                       // rows r0 + 16 i
  const uint32_t lane_off = chunk_off(r0, kc);  // + 16 i rows = + 2048 i bytes
  const int32_t col = h.dg * kW + 8 * kc + ((lane >> 1) & 7);    // RED column
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    uint32_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
    for (int k = a / kR; k * kR < b; ++k) {
      if (!sub.acquire(s, k)) return false;
      const uint32_t tile = smem_addr(s.tile[sub.stage(k)]) + lane_off;
      const int ra = a - k * kR, rb = b - k * kR;
#pragma unroll
      for (int i = 0; i < kR / 16; ++i) {
        const int r = r0 + 16 * i;
        if (r >= ra && r < rb) {
          const uint4 v = lds128(tile + i * 16 * 128);
          acc0 = absmax_bf16x2(acc0, v.x);
          acc1 = absmax_bf16x2(acc1, v.y);
          acc2 = absmax_bf16x2(acc2, v.z);
          acc3 = absmax_bf16x2(acc3, v.w);
        }
      }
      if (b >= (k + 1) * kR) sub.release(s, lane);
    }
    // lanes of equal parity hold the same chunk
#pragma unroll
    for (int x = 2; x < 32; x <<= 1) {
      acc0 = absmax_bf16x2(acc0, __shfl_xor_sync(0xffffffffu, acc0, x));
      acc1 = absmax_bf16x2(acc1, __shfl_xor_sync(0xffffffffu, acc1, x));
      acc2 = absmax_bf16x2(acc2, __shfl_xor_sync(0xffffffffu, acc2, x));
      acc3 = absmax_bf16x2(acc3, __shfl_xor_sync(0xffffffffu, acc3, x));
    }
    if (lane < 16) {
      const int cc = lane >> 1;  // column within the chunk
      const uint32_t w = cc < 2 ? acc0 : cc < 4 ? acc1 : cc < 6 ? acc2 : acc3;
      const uint32_t m = ((cc & 1) ? (w >> 16) : w) & 0x7FFFu;
      if (m != 0u && col < p.K)
        atomicMax(p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + col, m << 16);
    }
  }
  if (!sub.finish(s, lane)) return false;
  sig_post(s.sig, (p.skip_arrival && h.dg == 0 && h.lo == 0) ? kSigSkip : h.dg,
           warp * 32 + lane, lane, sig_seq, 4 * p.timeout_ns, p.err);
  return true;
}

// Phase B, warp w: rows 8w .. 8w + 7 of every stage, all 128 columns.
__device__ __forceinline__ bool phase_b(Smem& s, const Ctx& c, SubTiles& sub,
                                        const Params& p, int warp, int lane) {
  const Hdr& h = c.hdr;
  const int32_t c0 = h.dg * kW;
  const int kc = lane & 15;  // chunk: columns 8 kc .. 8 kc + 7
  const bool chunk_in = c0 + 8 * kc < p.K;
  const int32_t c4 = c0 + 4 * lane;  // this lane's four scale columns
  const bool c4_in = c4 < p.K;
  const int rl = 8 * warp + (lane >> 4);  // this lane's rows: rl + 2 i
  uint32_t row_off[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) row_off[i] = chunk_off(rl + 2 * i, kc);
  // owned groups without rows: amax 0
  if (warp == 0) {
    for (int g = h.own_lo; g < h.own_hi; ++g) {
      const int32_t gs = g ? s.ends[g - 1] : 0;
      if (c4_in && s.ends[g] == gs) {
        const float e = scale_from_amax_bits(0u);
        *reinterpret_cast<float4*>(p.scales + static_cast<size_t>(g) * p.K + c4) =
            make_float4(e, e, e, e);
      }
    }
  }
  uint8_t* obase = p.out + static_cast<size_t>(h.lo) * p.K + static_cast<size_t>(c0 + 8 * kc);
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    const int g = h.seg_g[j];
    bool have_sc = false;
    float sc[8];
    for (int k = a / kR; k * kR < b; ++k) {
      if (!sub.acquire(s, k)) return false;
      const int ra = a - k * kR, rb = b - k * kR;
      if (8 * warp + 7 >= ra && 8 * warp < rb) {  // the warp has rows here
        if (!have_sc) {
          have_sc = true;
          uint4 am;
          if (j < kSegA) {
            am = *reinterpret_cast<const uint4*>(&c.amax[j][4 * lane]);
          } else if (c4_in) {
            const uint32_t* src = p.amax + static_cast<size_t>(g) * p.K + c4;
            am = make_uint4(ld_cg_u32(src), ld_cg_u32(src + 1), ld_cg_u32(src + 2),
                            ld_cg_u32(src + 3));
          } else {
            am = make_uint4(0u, 0u, 0u, 0u);
          }
          const float s0 = scale_from_amax_bits(am.x), s1 = scale_from_amax_bits(am.y);
          const float s2 = scale_from_amax_bits(am.z), s3 = scale_from_amax_bits(am.w);
          // the group starts inside the super tile at row a: the warp holding
          // row a writes its scales
          if (k == a / kR && warp == (a % kR) / 8 && c4_in && g >= h.own_lo &&
              g < h.own_hi)
            *reinterpret_cast<float4*>(p.scales + static_cast<size_t>(g) * p.K + c4) =
                make_float4(s0, s1, s2, s3);
          const int l0 = 2 * kc, l1 = 2 * kc + 1;  // lanes holding columns 8kc..
          sc[0] = __shfl_sync(0xffffffffu, s0, l0);
          sc[1] = __shfl_sync(0xffffffffu, s1, l0);
          sc[2] = __shfl_sync(0xffffffffu, s2, l0);
          sc[3] = __shfl_sync(0xffffffffu, s3, l0);
          sc[4] = __shfl_sync(0xffffffffu, s0, l1);
          sc[5] = __shfl_sync(0xffffffffu, s1, l1);
          sc[6] = __shfl_sync(0xffffffffu, s2, l1);
          sc[7] = __shfl_sync(0xffffffffu, s3, l1);
        }
        const uint32_t tile = smem_addr(s.tile[sub.stage(k)]);
        uint8_t* ok_base = obase + static_cast<size_t>(k * kR) * p.K;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rl + 2 * i;
          if (r >= ra && r < rb && chunk_in) {
            const uint2 o = quant8(lds128(tile + row_off[i]), sc);
            __stcs(reinterpret_cast<uint2*>(ok_base + static_cast<size_t>(r) * p.K), o);
          }
        }
      }
      if (b >= (k + 1) * kR) sub.release(s, lane);
    }
  }
  return sub.finish(s, lane);
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
    for (int i = 0; i < kCtx; ++i) mbar_init(&s.ctx_empty[i], kConsumerWarps);
    mbar_init(&s.ends_ready, 1);
    sig_init(s.sig, kConsumerWarps);
    s.dep.ready = -1;
    s.dep.fail = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps + 1) {
    if (lane == 0)
      signal_lane(s.sig, s.dep, p.done, p.sched, static_cast<uint32_t>(p.sched.units),
                  p.timeout_ns, 8 * p.timeout_ns, p.err);
    return;
  }
  if (warp == kConsumerWarps) {
    if (lane == 0) prefetch_tensormap(&xmap);
    producer(s, &xmap, p, lane);
    return;
  }

  mbar_wait(&s.ends_ready, 0u, 4 * p.timeout_ns, p.err);
  SubTiles sub;
  sub.st0 = 0;
  sub.ph0 = 0;
  sub.wait_ns = 4 * p.timeout_ns;
  sub.err = p.err;
  int ci = 0;
  uint32_t sig_seq = 0;
  for (;;) {
    // the super tile's first stage also publishes its context
    const bool ok = mbar_wait(&s.full[sub.st0], sub.ph0, sub.wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;
    const Ctx& c = s.ctx[ci];
    const int phase = c.hdr.phase;
    if (phase < 0) break;
    sub.nsub = c.hdr.nsub;
    sub.acq = 1;
    sub.rel = 0;
    const bool done_ok = phase == 0 ? phase_a(s, c.hdr, sub, p, warp, lane, sig_seq)
                                    : phase_b(s, c, sub, p, warp, lane);
    if (!done_ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.ctx_empty[ci]);
    sub.ph0 = sub.parity(sub.nsub);
    sub.st0 = sub.stage(sub.nsub);
    if (++ci == kCtx) ci = 0;
  }
  sig_post(s.sig, kSigEnd, warp * 32 + lane, lane, sig_seq, 4 * p.timeout_ns, p.err);
}

// ---------------------------------------------------------------- host --
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
                                 static_cast<uint64_t>(K) * 2, 64, kR,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;

  Params p;
  p.sched.units = (M + kSuper - 1) / kSuper;
  p.sched.groups = (K + kW - 1) / kW;
  const int64_t total = 2ll * p.sched.units * p.sched.groups;
  const int64_t max_ctas =
      static_cast<int64_t>(info.sm_count) * info.colwise_ctas_per_sm;
  const int grid = static_cast<int>(total < max_ctas ? total : max_ctas);
  p.sched.lag = schedule_lag(dbg.lag[GQ_KIND_COLWISE], p.sched.units, p.sched.groups,
                             grid, kCtx);

  const WorkspaceLayout L =
      workspace_layout(p.sched.groups, static_cast<int64_t>(G) * K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.offs = offs;
  p.out = static_cast<uint8_t*>(out);
  p.scales = scales;
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
  // cooperative: the static ticket order needs every CTA resident
  void* args[] = {&xmap, &p};
  return check_cuda(
      cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(colwise_kernel),
                                  dim3(grid), dim3(kThreads), args, kSmemBytes,
                                  stream),
      "colwise: launch");
}

}  // namespace colwise
}  // namespace gq
