// gq_colwise.cu -- colwise per-token-group fp8 e4m3 scaling on sm_103a.
//
// X (M, K) bf16 row-major; token groups are row ranges [s_g, e_g); one scale
// per (group, column).  This is the per-token-group scaling "along dim0" of
// pytorch/ao #2668 ("use smaller block sizes for per group scaling kernels
// to improve perf", intro); the page's lesson -- the grid was too small to
// fill the SMs -- is answered here by a persistent grid of two CTAs per SM.
//
// A stage is kRows = 32 rows x kW = 128 columns (8 KB, rows of 256 bytes),
// one TMA box; every shared-memory access below reads whole 256-byte rows,
// so the layout needs no swizzle to be bank-conflict free.  A super tile is
// kSub = 8 stages: 256 rows of one column slab.  A column slab (all M rows of
// kW columns) is one dependency group: phase B of slab d needs the amax of
// every phase-A super tile of slab d.  See gq_device.cuh for the schedule.
//
// A producer warp loads the stages of the CTA's tickets into a shared ring
// of kStages buffers; a consumer warp takes the next loaded stage (a shared
// counter), whichever ticket it belongs to, and does all its work.  Lane l
// owns the 16-byte column chunk l % 16 (8 columns) of rows l / 16,
// l / 16 + 2, ...: a warp load covers two 256-byte rows and a warp store two
// 128-byte output rows.
//   phase A: per group segment, |x| is folded with max.xorsign.abs.bf16x2
//     over the lane's rows, one shuffle joins the two row halves, and every
//     lane folds its four column maxima into the super tile's context with
//     shared-memory atomics; the warp finishing the super tile adds them to
//     the amax words in global memory (one atomicMax per column);
//   phase B: per segment a lane computes four of the 128 scales
//     (448 / max(amax, 1e-12), IEEE division) and gathers the eight of its
//     chunk by shuffles; products are IEEE fp32 multiplies (mul.rn.f32x2),
//     packed with cvt.rn.satfinite.e4m3x2.
// The context warp writes each super tile's context: the header, and in
// phase B -- once the slab is complete -- the 128 amax words of each of its
// first kSegA segments (one 16-byte cp.async per lane).
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace colwise {

constexpr int kRows = 32;             // rows per stage
constexpr int kStages = 12;           // shared ring of stage buffers
constexpr int kConsumerWarps = 4;
constexpr int kSub = 8;               // stages per super tile
constexpr int kSuper = kSub * kRows;  // rows per super tile
constexpr int kCtx = 2;               // super-tile contexts in flight
// warps: consumers 0..3, producer 4, context 5, signal 6
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kContextWarp = kConsumerWarps + 1;
constexpr int kSignalWarp = kConsumerWarps + 2;
constexpr int kThreads = (kConsumerWarps + 3) * 32;
constexpr int kSigSlots = 8;
constexpr int kRowBytes = kW * 2;
constexpr int kStageBytes = kRows * kRowBytes;
constexpr int kSegA = 4;  // segments whose amax words ride in the context
static_assert(kW == 128, "lane maps assume 128-column slabs");
static_assert(kW == 32 * 4, "one 16-byte amax chunk per context-warp lane");
static_assert(kSigSlots > kConsumerWarps, "one outstanding post per warp");
static_assert(kRows % 32 == 0, "rows in batches of 16 per lane");

using Hdr = TileHdr<kSuper>;

struct Ctx {
  Hdr hdr;
  // phase A: the super tile's column maxima of its first kSegA segments
  // (shared atomics); phase B: the amax words of those segments
  alignas(16) uint32_t amax[kSegA][kW];
  uint32_t a_done;  // phase A: stages finished
  int32_t ticket;   // the claimed ticket, -1: no more
};

// What a stage holds: stage k of the CTA's ticket `seq` (context slot
// seq % kCtx); seq = -1: no more stages.
struct StageInfo {
  int32_t seq;
  int32_t k;
};

struct Smem {
  uint8_t tile[kStages][kStageBytes];  // first member: 1024-byte aligned
  Ctx ctx[kCtx];
  StageInfo info[kStages];
  uint64_t full[kStages];     // stage loaded (TMA bytes)
  uint64_t empty[kStages];    // stage consumed
  uint64_t ctx_tkt[kCtx];     // context's ticket claimed
  uint64_t ctx_full[kCtx];    // context written
  uint64_t ctx_empty[kCtx];   // kSub stage arrivals: context free
  uint32_t claim;             // next stage a consumer takes
  SigRing<kSigSlots> sig;
  DepFlag dep;
  int32_t ends[kMaxGroups];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

struct Params {
  const int32_t* offs;  // nullptr: groups of `uniform` rows each
  int32_t uniform;
  uint32_t* ticket;  // ticket counter
  uint8_t* out;
  float* scales;
  uint32_t* done;  // one word per slab: finished phase-A super tiles
  uint32_t* amax;  // (G, K) fp32 bit patterns
  unsigned* err;
  int32_t M, K, G;
  Schedule sched;  // units = super tiles per slab
  uint64_t timeout_ns;
  int32_t skip_arrival;
  bool pow2;  // scales rounded down to powers of two
};

// Shared-memory offset of chunk k (0..15, 8 columns each) of stage row r.
__device__ __forceinline__ uint32_t chunk_off(int r, int k) {
  return static_cast<uint32_t>(r * kRowBytes + k * 16);
}

__device__ __forceinline__ int stages_of(int32_t unit, int32_t M) {
  const int32_t r0 = unit * kSuper;
  return (min(r0 + kSuper, M) - r0 + kRows - 1) / kRows;
}

// ---------------------------------------------------------- context warp --
__device__ __forceinline__ void context_warp(Smem& s, const Params& p, int lane) {
  build_ends(p.offs, p.uniform, p.G, p.M, s.ends, lane);
  __syncwarp();
  const int32_t units = p.sched.units;
  const uint32_t total = 2u * static_cast<uint32_t>(units) * static_cast<uint32_t>(p.sched.groups);
  const uint64_t wait_ns = 4 * p.timeout_ns;
  int32_t ready_dg = -1;  // slabs <= ready_dg are complete
  uint32_t next = lane == 0 ? claim_ticket(p.ticket) : 0u;  // claimed one ahead
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % kCtx;
    Ctx& c = s.ctx[ci];
    Hdr& h = c.hdr;
    if (!mbar_wait(&s.ctx_empty[ci], ((seq / kCtx) & 1) ^ 1u, wait_ns, p.err)) return;
    const uint32_t t = __shfl_sync(0xffffffffu, next, 0);
    if (t >= total) {  // no more tickets: a stop context
      if (lane == 0) {
        c.ticket = -1;
        mbar_arrive(&s.ctx_tkt[ci]);
        mbar_arrive(&s.ctx_full[ci]);
      }
      return;
    }
    if (lane == 0) {
      next = claim_ticket(p.ticket);
      c.ticket = static_cast<int32_t>(t);
      mbar_arrive(&s.ctx_tkt[ci]);  // consumers may start loading
    }
    const int32_t unit = static_cast<int32_t>(t % static_cast<uint32_t>(units));
    int32_t phase, dg;
    decode_block(static_cast<int32_t>(t / static_cast<uint32_t>(units)), p.sched, phase, dg);
    if (phase == 1 && dg > ready_dg) {
      bool ok = true;
      if (lane == 0) ok = wait_dep_flag(s.dep, dg, 2 * p.timeout_ns, p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
      ld_acquire_cta_s32(&s.dep.ready);  // every lane acquires before reading amax
      ready_dg = dg;
    }
    const int32_t c0 = dg * kW;
    const int32_t r0 = unit * kSuper;
    build_header_warp(h, s.ends, p.G, r0, min(r0 + kSuper, p.M), unit == units - 1, lane);
    __syncwarp();
    if (phase == 1) {
      const int n = min(static_cast<int>(h.nseg), kSegA);
      const int32_t col = c0 + 4 * lane;
      for (int j = 0; j < n; ++j)
        cp_async_16(smem_addr(&c.amax[j][4 * lane]),
                    p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + (col < p.K ? col : 0),
                    col < p.K ? 16u : 0u);
      cp_async_mbar_arrive(&s.ctx_full[ci]);  // the context also waits for them
    } else {
#pragma unroll
      for (int j = 0; j < kSegA; ++j)
        sts128(smem_addr(&c.amax[j][4 * lane]), make_uint4(0, 0, 0, 0));
    }
    if (lane == 0) {
      c.a_done = 0;
      h.phase = phase;
      h.dg = dg;
      const int nsub = stages_of(unit, p.M);
      h.nsub = nsub;
      // the context is free after kSub stage arrivals: stand in for the
      // stages a short super tile does not have
      for (int k = nsub; k < kSub; ++k) mbar_arrive(&s.ctx_empty[ci]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.ctx_full[ci]);
  }
}

// ---------------------------------------------------------- producer warp --
// Follows the CTA's tickets as the context warp publishes them and loads
// their stages into the shared ring, in order; each stage is tagged with its
// ticket and place.  After the last ticket, one stop stage per consumer warp.
__device__ __forceinline__ void producer_warp(Smem& s, const CUtensorMap* xmap,
                                              const Params& p, int lane) {
  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  const uint64_t wait_ns = 4 * p.timeout_ns;
  const uint32_t units = static_cast<uint32_t>(p.sched.units);
  uint32_t g = 0;  // stages loaded
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % kCtx;
    if (!mbar_wait(&s.ctx_tkt[ci], (seq / kCtx) & 1, wait_ns, p.err)) return;
    const int32_t t = s.ctx[ci].ticket;
    int nsub = kConsumerWarps, phase = 0, dg = 0, unit = 0;
    if (t >= 0) {
      unit = static_cast<int32_t>(static_cast<uint32_t>(t) % units);
      decode_block(static_cast<int32_t>(static_cast<uint32_t>(t) / units), p.sched, phase, dg);
      nsub = stages_of(unit, p.M);
    }
    for (int k = 0; k < nsub; ++k, ++g) {
      const int st = static_cast<int>(g % kStages);
      if (!mbar_wait(&s.empty[st], ((g / kStages) & 1) ^ 1u, wait_ns, p.err)) return;
      if (lane == 0) {
        s.info[st].seq = t >= 0 ? seq : -1;
        s.info[st].k = k;
        if (t >= 0) {
          mbar_arrive_expect_tx(&s.full[st], kStageBytes);
          tma_load_2d(s.tile[st], xmap, dg * kW, unit * kSuper + k * kRows, &s.full[st],
                      phase == 0 ? pol_a : pol_b);
        } else {
          mbar_arrive(&s.full[st]);
        }
      }
    }
    if (t < 0) return;
  }
}

// ------------------------------------------------------------ consumers --
// Phase A of one stage: column maxima of the stage rows inside each
// segment, folded into the context (first kSegA segments) or straight into
// the global amax words.
__device__ __forceinline__ void stage_a(Ctx& c, int k, uint32_t tile, const Params& p,
                                        int lane) {
  const Hdr& h = c.hdr;
  const int kc = lane & 15;  // column chunk
  const int rl = lane >> 4;  // rows rl + 2 i
  const uint32_t base = tile + chunk_off(rl, kc);  // row rl + 2 i: + 2 i rows
  const int rbase = k * kRows;  // super-tile row of stage row 0
  const int cw = 8 * kc + 4 * rl;  // first of this lane's 4 columns within the slab
  const int32_t col = h.dg * kW + cw;
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int ra = h.seg_lo[j] - rbase, rb = h.seg_hi[j] - rbase;
    if (rb <= 0) continue;
    if (ra >= kRows) break;
    uint32_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
    if (ra <= 0 && rb >= kRows) {
#pragma unroll
      for (int hb = 0; hb < kRows / 32; ++hb) {  // batches of 16 rows: loads first
        uint4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = lds128(base + (hb * 16 + i) * 2 * kRowBytes);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc0 = absmax_bf16x2(acc0, v[i].x);
          acc1 = absmax_bf16x2(acc1, v[i].y);
          acc2 = absmax_bf16x2(acc2, v[i].z);
          acc3 = absmax_bf16x2(acc3, v[i].w);
        }
      }
    } else {
#pragma unroll 1
      for (int i = 0; i < kRows / 2; ++i) {
        const int r = rl + 2 * i;
        if (r >= ra && r < rb) {
          const uint4 v = lds128(base + i * 2 * kRowBytes);
          acc0 = absmax_bf16x2(acc0, v.x);
          acc1 = absmax_bf16x2(acc1, v.y);
          acc2 = absmax_bf16x2(acc2, v.z);
          acc3 = absmax_bf16x2(acc3, v.w);
        }
      }
    }
    // lanes l and l ^ 16 hold the same chunk (even and odd rows)
    acc0 = absmax_bf16x2(acc0, __shfl_xor_sync(0xffffffffu, acc0, 16));
    acc1 = absmax_bf16x2(acc1, __shfl_xor_sync(0xffffffffu, acc1, 16));
    acc2 = absmax_bf16x2(acc2, __shfl_xor_sync(0xffffffffu, acc2, 16));
    acc3 = absmax_bf16x2(acc3, __shfl_xor_sync(0xffffffffu, acc3, 16));
    // lanes < 16 take columns 0..3 of the chunk, the others 4..7
    const uint32_t w0 = rl ? acc2 : acc0, w1 = rl ? acc3 : acc1;
    const uint32_t m[4] = {(w0 & 0x7FFFu) << 16, ((w0 >> 16) & 0x7FFFu) << 16,
                           (w1 & 0x7FFFu) << 16, ((w1 >> 16) & 0x7FFFu) << 16};
    if (j < kSegA) {
      const uint32_t dst = smem_addr(&c.amax[j][cw]);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m[e]) red_max_shared(dst + 4 * e, m[e]);
    } else if (col < p.K) {
      uint32_t* dst = p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + col;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m[e]) atomicMax(dst + e, m[e]);
    }
  }
}

// After a warp's phase-A stage: the warp that finishes the super tile's last
// stage adds the context's maxima to the global amax words and posts the
// super tile to the signal lane.
__device__ __forceinline__ void finish_a(Smem& s, Ctx& c, const Params& p, int lane,
                                         uint64_t wait_ns) {
  const Hdr& h = c.hdr;
  __syncwarp();
  uint32_t prev = 0;
  if (lane == 0) prev = atom_add_acq_rel_cta_shared(smem_addr(&c.a_done), 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev + 1 != static_cast<uint32_t>(h.nsub)) return;
  const int32_t col = h.dg * kW + 4 * lane;
  const int n = min(static_cast<int>(h.nseg), kSegA);
  for (int j = 0; j < n; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(&c.amax[j][4 * lane]);
    if (col < p.K) {
      uint32_t* dst = p.amax + static_cast<size_t>(h.seg_g[j]) * p.K + col;
      if (v.x) atomicMax(dst, v.x);
      if (v.y) atomicMax(dst + 1, v.y);
      if (v.z) atomicMax(dst + 2, v.z);
      if (v.w) atomicMax(dst + 3, v.w);
    }
  }
  const bool skip = p.skip_arrival && h.dg == 0 && h.lo == 0;
  sig_post(s.sig, skip ? kSigSkip : h.dg, lane, wait_ns, p.err);
}

// Phase B of one stage: scales, then the scaled cast of every stage row
// inside a group.
__device__ __forceinline__ void stage_b(Smem& s, const Ctx& c, int k, uint32_t tile,
                                        const Params& p, int lane) {
  const Hdr& h = c.hdr;
  const int kc = lane & 15;  // column chunk
  const int rl = lane >> 4;  // rows rl + 2 i
  const int32_t c0 = h.dg * kW;
  const bool chunk_in = c0 + 8 * kc < p.K;
  const int32_t c4 = c0 + 4 * lane;  // this lane's four scale columns
  const bool c4_in = c4 < p.K;
  const int rbase = k * kRows;
  // owned groups without rows: amax 0 (once per super tile)
  if (k == 0) {
    for (int g = h.own_lo; g < h.own_hi; ++g) {
      const int32_t gs = g ? s.ends[g - 1] : 0;
      if (c4_in && s.ends[g] == gs) {
        const float e = scale_from_amax_bits(0u, p.pow2);
        *reinterpret_cast<float4*>(p.scales + static_cast<size_t>(g) * p.K + c4) =
            make_float4(e, e, e, e);
      }
    }
  }
  const uint32_t base = tile + chunk_off(rl, kc);  // row rl + 2 i: + 2 i rows
  const size_t K2 = 2 * static_cast<size_t>(p.K);
  uint8_t* obase = p.out + static_cast<size_t>(h.lo + rbase + rl) * p.K +
                   static_cast<size_t>(c0 + 8 * kc);
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int ra = h.seg_lo[j] - rbase, rb = h.seg_hi[j] - rbase;
    if (rb <= 0) continue;
    if (ra >= kRows) break;
    const int g = h.seg_g[j];
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
    const float s0 = scale_from_amax_bits(am.x, p.pow2), s1 = scale_from_amax_bits(am.y, p.pow2);
    const float s2 = scale_from_amax_bits(am.z, p.pow2), s3 = scale_from_amax_bits(am.w, p.pow2);
    // the group starts inside the super tile at row seg_lo: the stage
    // holding that row writes its scales
    if (ra >= 0 && c4_in && g >= h.own_lo && g < h.own_hi)
      *reinterpret_cast<float4*>(p.scales + static_cast<size_t>(g) * p.K + c4) =
          make_float4(s0, s1, s2, s3);
    float sc[8];
    const int l0 = 2 * kc, l1 = 2 * kc + 1;  // lanes holding columns 8kc .. 8kc+7
    sc[0] = __shfl_sync(0xffffffffu, s0, l0);
    sc[1] = __shfl_sync(0xffffffffu, s1, l0);
    sc[2] = __shfl_sync(0xffffffffu, s2, l0);
    sc[3] = __shfl_sync(0xffffffffu, s3, l0);
    sc[4] = __shfl_sync(0xffffffffu, s0, l1);
    sc[5] = __shfl_sync(0xffffffffu, s1, l1);
    sc[6] = __shfl_sync(0xffffffffu, s2, l1);
    sc[7] = __shfl_sync(0xffffffffu, s3, l1);
    if (!chunk_in) continue;
    if (ra <= 0 && rb >= kRows) {
      // all of the lane's rows: loads first, then the casts and stores, so
      // that sixteen independent chains hide the latency of each step
      uint4 v[kRows / 2];
#pragma unroll
      for (int i = 0; i < kRows / 2; ++i) v[i] = lds128(base + i * 2 * kRowBytes);
#pragma unroll
      for (int i = 0; i < kRows / 2; ++i)
        __stcs(reinterpret_cast<uint2*>(obase + i * K2), quant8(v[i], sc));
    } else {
#pragma unroll 1
      for (int i = 0; i < kRows / 2; ++i) {
        const int r = rl + 2 * i;
        if (r >= ra && r < rb) {
          const uint2 o = quant8(lds128(base + i * 2 * kRowBytes), sc);
          __stcs(reinterpret_cast<uint2*>(obase + i * K2), o);
        }
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
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < kCtx; ++i) {
      mbar_init(&s.ctx_tkt[i], 1);
      mbar_init(&s.ctx_full[i], 1);
      mbar_init(&s.ctx_empty[i], kSub);
    }
    s.claim = 0;
    sig_init(s.sig);
    dep_init(s.dep);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kSignalWarp) {
    if (lane == 0)
      signal_lane(s.sig, s.dep, p.done, static_cast<uint32_t>(p.sched.units), kConsumerWarps,
                  p.timeout_ns, 8 * p.timeout_ns, p.err);
    return;
  }
  if (warp == kContextWarp) {
    context_warp(s, p, lane);
    return;
  }
  if (warp == kProducerWarp) {
    if (lane == 0) prefetch_tensormap(&xmap);
    producer_warp(s, &xmap, p, lane);
    return;
  }

  // consumer warp: takes the next loaded stage, whichever it is
  const uint64_t wait_ns = 4 * p.timeout_ns;
  for (;;) {
    uint32_t g = 0;
    if (lane == 0) g = atomicAdd(&s.claim, 1u);
    g = __shfl_sync(0xffffffffu, g, 0);
    const int st = static_cast<int>(g % kStages);
    // Stages finish out of order, so the stage kStages before g may still be
    // in flight (its TMA outstanding) when g is claimed; its full barrier
    // would then show the parity g waits for.  Wait for that stage's
    // consumption first: then the full barrier is in g's round.
    bool ok = mbar_wait(&s.empty[st], ((g / kStages) & 1) ^ 1u, wait_ns, p.err);
    if (ok) ok = mbar_wait(&s.full[st], (g / kStages) & 1, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;
    const StageInfo inf = s.info[st];
    if (inf.seq < 0) break;
    const int ci = inf.seq % kCtx;
    ok = mbar_wait(&s.ctx_full[ci], (inf.seq / kCtx) & 1, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;
    Ctx& c = s.ctx[ci];
    const uint32_t tile = pin(smem_addr(s.tile[st]));
    if (c.hdr.phase == 0) {
      stage_a(c, inf.k, tile, p, lane);
      finish_a(s, c, p, lane, wait_ns);
    } else {
      stage_b(s, c, inf.k, tile, p, lane);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&s.empty[st]);
      mbar_arrive(&s.ctx_empty[ci]);
    }
  }
  sig_post(s.sig, kSigEnd, lane, wait_ns, p.err);
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
                 int32_t M, int32_t K, const int32_t* offs, int32_t uniform, int32_t G,
                 void* out, float* scales, uint32_t flags, void* ws, cudaStream_t stream) {
  CUtensorMap xmap;
  gq_status st = encode_tiled_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(x), static_cast<uint64_t>(K),
                                 static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(K) * 2, kW, kRows,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;

  Params p;
  p.sched.units = (M + kSuper - 1) / kSuper;
  p.sched.groups = (K + kW - 1) / kW;
  const int64_t total = 2ll * p.sched.units * p.sched.groups;
  const int64_t max_ctas =
      static_cast<int64_t>(info.sm_count) * info.colwise_ctas_per_sm;
  const int grid = static_cast<int>(total < max_ctas ? total : max_ctas);
  p.sched.lag = schedule_lag(dbg.lag[GQ_KIND_COLWISE], p.sched.units, p.sched.groups, grid);

  const WorkspaceLayout L = colwise_workspace(K, G);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.offs = offs;
  p.uniform = uniform;
  p.ticket = reinterpret_cast<uint32_t*>(w);  // first word of the header
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
  p.pow2 = (flags & GQ_SCALE_POW2) != 0;

  st = check_cuda(cudaMemsetAsync(ws, 0, L.total, stream), "colwise: clear workspace");
  if (st != GQ_OK) return st;
  // cooperative: a claimed ticket may wait for tickets of other CTAs, so
  // every CTA must be resident
  void* args[] = {&xmap, &p};
  return check_cuda(
      cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(colwise_kernel),
                                  dim3(grid), dim3(kThreads), args, kSmemBytes,
                                  stream),
      "colwise: launch");
}

}  // namespace colwise
}  // namespace gq
