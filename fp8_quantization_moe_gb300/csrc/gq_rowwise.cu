// gq_rowwise.cu -- rowwise per-token-group fp8 e4m3 scaling with transposed
// output, on sm_103a.
//
// A (N, Mg) bf16 row-major; token groups are column ranges [s_g, e_g) of A;
// one scale per (row, group); the fp8 result is written as A^T, (Mg, N)
// row-major.  This is the per-group rowwise scaling of the backward
// grad_weight GEMM in pytorch/ao #2863 ("test and bench new faster method for
// per group rowwise scaling", Summary).  That page removes the uncoalesced
// global accesses of its first kernel by computing colwise scales on the
// transpose and transposing back; here both sides stay coalesced in a single
// kernel: tiles come in by TMA with 128-byte rows, the transpose happens in
// shared memory (ldmatrix .trans), and the fp8 result leaves by TMA stores
// of 32-byte row runs of A^T.
//
// A stage is kTn = 128 rows of A x kTm = 64 token columns (16 KB), staged
// with the 128-byte TMA swizzle so that row-wise and column-wise
// shared-memory accesses are bank-conflict free.  A super tile is kSub = 4
// stages: 256 token columns of one row band.  A row band (kTn rows, all Mg
// columns) is one dependency group.  See gq_device.cuh for the schedule.  In
// phase B the producer lanes bring the amax words of the band's 128 rows for
// each of the super tile's first kSegA segments into its context.
//
// The eight consumer warps work on each stage independently:
//   phase A: warp w takes rows 16w .. 16w + 15; per segment, lane l folds
//     |x| of row 16w + l % 16 over columns 32 (l / 16) .. + 31 of every stage
//     the segment covers, with max.xorsign.abs.bf16x2; one shuffle joins the
//     two column halves and 16 lanes issue one atomicMax each, into amax
//     words laid out (G, N) so that the 16 atomics of a warp hit one 64-byte
//     run;
//   phase B: warp w takes the 32 x 32 block of rows 32 (w % 4) .. + 31 and
//     columns 32 (w / 4) .. + 31 of every stage: per segment a lane computes
//     the scale of one row (448 / max(amax, 1e-12), IEEE division) and
//     gathers the eight it needs by shuffles; ldmatrix.x4.trans gives every
//     lane the pairs (n, n+1) of one column m, which are multiplied in fp32
//     (mul.rn.f32x2) and packed with cvt.rn.satfinite.e4m3x2 into bytes of
//     A^T; one shuffle between neighbouring lanes assembles 4-byte runs of an
//     output row; each finished 32 x 32-byte block of A^T leaves by the
//     warp's own TMA store.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace rowwise {

constexpr int kStages = 5;
constexpr int kSub = 4;              // stages per super tile
constexpr int kSuper = kSub * kTm;   // token columns per super tile
constexpr int kCtx = 3;              // super-tile contexts in flight
constexpr int kConsumerWarps = 8;
constexpr int kThreads = kConsumerWarps * 32 + 64;  // + producer + signal warps
constexpr int kSigSlots = 16;
constexpr int kTileBytes = kTn * kTm * 2;  // bf16 in
constexpr int kBlk = 32;                   // phase-B block: 32 rows x 32 columns
constexpr int kOutBytes = kBlk * kBlk;     // e4m3 out per warp and buffer
constexpr int kSegA = 4;  // segments whose amax words ride in the context
static_assert(kTm * 2 == 128 && kTn == 128, "128-byte swizzled rows in");
static_assert(kTn == 32 * 4, "one 16-byte amax chunk per producer lane");
static_assert(kConsumerWarps * kBlk * kBlk == kTn * kTm, "warps tile a stage");
static_assert(kSub < kStages, "a super tile wraps the stage ring at most once");
static_assert(kSigSlots > kStages, "a warp cannot lap the signal ring");

using Hdr = TileHdr<kSuper>;

struct Ctx {
  Hdr hdr;
  alignas(16) uint32_t amax[kSegA][kTn];  // phase B amax words
};

struct Smem {
  uint8_t tile[kStages][kTileBytes];  // 1024-byte aligned (swizzle atom)
  uint8_t outt[kConsumerWarps][2][kOutBytes];
  Ctx ctx[kCtx];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t ctx_empty[kCtx];
  uint64_t ends_ready;
  SigRing<kSigSlots> sig;
  DepFlag dep;
  int32_t ends[kMaxGroups];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Params {
  const int32_t* offs;
  uint8_t* out_t;
  float* scales;
  uint32_t* done;  // one word per row band
  uint32_t* amax;  // (G, N) fp32 bit patterns
  unsigned* err;
  int32_t N, Mg, G;
  Schedule sched;  // units = super tiles per band
  uint64_t timeout_ns;
  int32_t skip_arrival;
};

// Shared-memory offset of 16-byte chunk c (8 token columns) of stage row r
// (128-byte TMA swizzle: the chunk index is xor-ed with r % 8).
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// ------------------------------------------------------------- producer --
__device__ __forceinline__ void producer(Smem& s, const CUtensorMap* amap,
                                         const Params& p, int lane) {
  build_ends(p.offs, p.G, p.Mg, s.ends, lane);
  __syncwarp();
  if (lane == 0) mbar_arrive(&s.ends_ready);

  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  const int32_t units = p.sched.units;
  const int32_t blocks = 2 * p.sched.groups;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  int32_t ready_dg = -1;  // bands <= ready_dg are complete
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
    const int32_t n0 = dg * kTn;
    const int32_t m0 = tw.unit * kSuper;
    const int32_t m1 = min(m0 + kSuper, p.Mg);
    const int nsub = (m1 - m0 + kTm - 1) / kTm;
    build_header_warp(h, s.ends, p.G, m0, m1, tw.unit == units - 1, lane);
    __syncwarp();
    if (phase == 1) {
      const int n = min(static_cast<int>(h.nseg), kSegA);
      const int32_t row = n0 + 4 * lane;
      for (int j = 0; j < n; ++j)
        cp_async_16(smem_addr(&c.amax[j][4 * lane]),
                    p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + (row < p.N ? row : 0),
                    row < p.N ? 16u : 0u);
      cp_async_mbar_arrive(&s.full[st]);  // the first stage waits for them
    }
    if (lane == 0) {
      h.phase = phase;
      h.dg = dg;
      h.nsub = nsub;
    }
    __syncwarp();
    const uint64_t pol = phase == 0 ? pol_a : pol_b;
    for (int k = 0; k < nsub; ++k) {
      if (k > 0 && !mbar_wait(&s.empty[st], ph ^ 1u, wait_ns, p.err)) return;
      if (lane == 0) {
        mbar_arrive_expect_tx(&s.full[st], kTileBytes);
        tma_load_2d(s.tile[st], amap, m0 + k * kTm, n0, &s.full[st], pol);
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
};

// Phase A, warp w: per segment, the |x| maxima of rows 16w .. 16w + 15; then
// the super tile goes to the signal lane.
__device__ __forceinline__ bool phase_a(Smem& s, const Hdr& h, SubTiles& sub,
                                        const Params& p, int warp, int lane,
                                        uint32_t& sig_seq) {
  const int r = 16 * warp + (lane & 15);  // stage row
  const int hc = lane >> 4;               // column half: chunks 4 hc .. 4 hc + 3
  const int32_t n = h.dg * kTn + r;
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    uint32_t acc = 0;
    for (int k = a / kTm; k * kTm < b; ++k) {
      if (!sub.acquire(s, k)) return false;
      const uint32_t tile = smem_addr(s.tile[sub.stage(k)]);
      const int ca = a - k * kTm, cb = b - k * kTm;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int c = 4 * hc + cc;
        const int lo = c * 8, hi = lo + 8;
        if (hi <= ca || lo >= cb) continue;
        const uint4 v = lds128(tile + chunk_off(r, c));
        if (lo >= ca && hi <= cb) {
          acc = absmax_bf16x2(acc, v.x);
          acc = absmax_bf16x2(acc, v.y);
          acc = absmax_bf16x2(acc, v.z);
          acc = absmax_bf16x2(acc, v.w);
        } else {
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int col = lo + e;
            if (col >= ca && col < cb) {
              const uint32_t half = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
              acc = absmax_bf16x2(acc, half);
            }
          }
        }
      }
      if (b >= (k + 1) * kTm) sub.release(s, lane);
    }
    acc = absmax_bf16x2(acc, __shfl_xor_sync(0xffffffffu, acc, 16));
    const uint32_t m = amax_bits_of(acc);
    if (lane < 16 && m != 0u && n < p.N)
      atomicMax(p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + n, m);
  }
  while (sub.rel < sub.nsub) {
    if (!sub.acquire(s, sub.rel)) return false;
    sub.release(s, lane);
  }
  sig_post(s.sig, (p.skip_arrival && h.dg == 0 && h.lo == 0) ? kSigSkip : h.dg,
           warp * 32 + lane, lane, sig_seq, 4 * p.timeout_ns, p.err);
  return true;
}

// Phase B state of one warp: its 32 x 32 block, the output buffer it fills.
struct BlockOut {
  int rq, hc;      // block rows 32 rq .., columns 32 hc .. of every stage
  int open;        // stage (sub-tile) whose block is in obuf, -1 if none
  uint32_t ob;     // which of the warp's two buffers
};

// Stores the warp's block of sub-tile k of A^T: by TMA when every token of
// it is covered by a group, else by plain stores of the covered rows only
// (tokens past the last group end stay untouched).
__device__ __forceinline__ void store_block(Smem& s, const Hdr& h, BlockOut& bo,
                                            int k, const CUtensorMap* omap,
                                            const Params& p, int warp, int lane,
                                            int32_t cover, uint64_t pol_out) {
  uint8_t* obuf = s.outt[warp][bo.ob];
  fence_proxy_async_smem();
  __syncwarp();
  const int width = h.hi - h.lo;  // tokens in the super tile
  const int mlo = k * kTm + kBlk * bo.hc;
  if (mlo >= width) return;
  const int32_t n0 = h.dg * kTn + kBlk * bo.rq;
  if (min(mlo + kBlk, width) <= cover) {
    if (lane == 0) {
      tma_store_2d(omap, obuf, n0, h.lo + mlo, pol_out);
      bulk_commit();
    }
    bo.ob ^= 1u;
  } else if (cover > mlo) {
    const uint32_t obase = smem_addr(obuf);
    const int rows = cover - mlo;
    for (int i = lane; i < 2 * rows; i += 32) {
      const int ml = i >> 1, hb = i & 1;
      const int32_t nn = n0 + 16 * hb;
      if (nn < p.N) {
        const uint4 v = lds128(obase + static_cast<uint32_t>(ml * kBlk + 16 * hb));
        *reinterpret_cast<uint4*>(p.out_t + static_cast<size_t>(h.lo + mlo + ml) * p.N + nn) = v;
      }
    }
  }
}

// Phase B, warp w: scale, cast and transpose its block of every stage.
__device__ __forceinline__ bool phase_b(Smem& s, const Ctx& c, SubTiles& sub,
                                        const CUtensorMap* omap, const Params& p,
                                        int warp, int lane, BlockOut& bo,
                                        uint64_t pol_out) {
  const Hdr& h = c.hdr;
  const int32_t nrow = h.dg * kTn + kBlk * bo.rq + lane;  // row whose scale this lane computes
  const bool row_in = nrow < p.N;
  const int q = lane & 3;
  const bool odd = (lane & 1) != 0;
  const int mcol = lane >> 2;  // column within an 8-column chunk
  const uint32_t lrow_off = static_cast<uint32_t>(kBlk * bo.rq + lane) * 128u;
  const int32_t cover = min(h.hi, p.G > 0 ? s.ends[p.G - 1] : 0) - h.lo;
  // owned groups without columns: amax 0
  if (bo.hc == 0) {
    for (int g = h.own_lo; g < h.own_hi; ++g) {
      const int32_t gs = g ? s.ends[g - 1] : 0;
      if (row_in && s.ends[g] == gs)
        p.scales[static_cast<size_t>(nrow) * p.G + g] = scale_from_amax_bits(0u);
    }
  }
  bo.open = -1;
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    const int g = h.seg_g[j];
    bool have_sc = false;
    float sv[8];
    for (int k = a / kTm; k * kTm < b; ++k) {
      if (!sub.acquire(s, k)) return false;
      const int wlo = k * kTm + kBlk * bo.hc, whi = wlo + kBlk;  // super-tile columns
      if (a < whi && b > wlo) {  // the segment meets the warp's columns here
        if (bo.open != k) {
          bo.open = k;
          if (lane == 0) bulk_wait_read<1>();  // the store that last read the buffer is done
          __syncwarp();
        }
        if (!have_sc) {
          have_sc = true;
          const uint32_t bits =
              j < kSegA ? c.amax[j][kBlk * bo.rq + lane]
                        : (row_in ? ld_cg_u32(p.amax + static_cast<size_t>(g) * p.N + nrow)
                                  : 0u);
          const float sc = scale_from_amax_bits(bits);
          // the group starts inside the super tile at column a: the warps
          // holding column a write its scales
          if (k == a / kTm && bo.hc == (a % kTm) / kBlk && row_in && g >= h.own_lo &&
              g < h.own_hi)
            p.scales[static_cast<size_t>(nrow) * p.G + g] = sc;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sv[2 * i] = __shfl_sync(0xffffffffu, sc, 8 * i + 2 * q);
            sv[2 * i + 1] = __shfl_sync(0xffffffffu, sc, 8 * i + 2 * q + 1);
          }
        }
        const uint32_t lrow = smem_addr(s.tile[sub.stage(k)]) + lrow_off;
        const uint32_t obase = smem_addr(s.outt[warp][bo.ob]);
        const int c_first = (max(a, wlo) - k * kTm) >> 3;
        const int c_last = (min(b, whi) - 1 - k * kTm) >> 3;
        for (int cc = c_first; cc <= c_last; ++cc) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_trans(lrow + ((((cc ^ lane) & 7)) << 4), r0, r1, r2, r3);
          const int m = k * kTm + cc * 8 + mcol;  // super-tile column
          // pair i: rows 8i + 2q (+1) of the block, column m -> 2 bytes of A^T
          const float2 f0 = mul_f32x2(make_float2(bf16_lo(r0), bf16_hi(r0)), make_float2(sv[0], sv[1]));
          const float2 f1 = mul_f32x2(make_float2(bf16_lo(r1), bf16_hi(r1)), make_float2(sv[2], sv[3]));
          const float2 f2 = mul_f32x2(make_float2(bf16_lo(r2), bf16_hi(r2)), make_float2(sv[4], sv[5]));
          const float2 f3 = mul_f32x2(make_float2(bf16_lo(r3), bf16_hi(r3)), make_float2(sv[6], sv[7]));
          const uint32_t p0 = cvt_e4m3x2(f0.x, f0.y), p1 = cvt_e4m3x2(f1.x, f1.y);
          const uint32_t p2 = cvt_e4m3x2(f2.x, f2.y), p3 = cvt_e4m3x2(f3.x, f3.y);
          // even lanes keep pairs 0,1 and take the odd neighbour's; odd lanes
          // keep pairs 2,3 -- each lane ends with two 4-byte runs of row m
          const uint32_t send = odd ? (p0 | (p1 << 16)) : (p2 | (p3 << 16));
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
          if (m >= a && m < b) {
            const int nb = 2 * (q & 2);  // first row of the 4-run
            uint32_t wa, wb;
            int na, nb2;
            if (!odd) {
              wa = p0 | ((recv & 0xFFFFu) << 16);  // rows nb + 0..3
              wb = p1 | ((recv >> 16) << 16);      // rows nb + 8 + 0..3
              na = nb;
              nb2 = nb + 8;
            } else {
              wa = (recv >> 16) | (p3 << 16);      // rows nb + 24 + 0..3
              wb = (recv & 0xFFFFu) | (p2 << 16);  // rows nb + 16 + 0..3
              na = nb + 24;
              nb2 = nb + 16;
            }
            const uint32_t rowb = obase + static_cast<uint32_t>((m - wlo) * kBlk);
            sts32(rowb + na, wa);
            sts32(rowb + nb2, wb);
          }
        }
      }
      if (b >= (k + 1) * kTm) {
        if (bo.open == k) {
          store_block(s, h, bo, k, omap, p, warp, lane, cover, pol_out);
          bo.open = -1;
        }
        sub.release(s, lane);
      }
    }
  }
  while (sub.rel < sub.nsub) {
    if (!sub.acquire(s, sub.rel)) return false;
    if (bo.open == sub.rel) {
      store_block(s, h, bo, sub.rel, omap, p, warp, lane, cover, pol_out);
      bo.open = -1;
    }
    sub.release(s, lane);
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 2)
    rowwise_kernel(const __grid_constant__ CUtensorMap amap,
                   const __grid_constant__ CUtensorMap omap, const Params p) {
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
    if (lane == 0) prefetch_tensormap(&amap);
    producer(s, &amap, p, lane);
    return;
  }

  if (lane == 0) prefetch_tensormap(&omap);
  mbar_wait(&s.ends_ready, 0u, 4 * p.timeout_ns, p.err);
  const uint64_t pol_out = policy_evict_first();
  SubTiles sub;
  sub.st0 = 0;
  sub.ph0 = 0;
  sub.wait_ns = 4 * p.timeout_ns;
  sub.err = p.err;
  BlockOut bo;
  bo.rq = warp & 3;
  bo.hc = warp >> 2;
  bo.open = -1;
  bo.ob = 0;
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
    const bool done_ok = phase == 0
                             ? phase_a(s, c.hdr, sub, p, warp, lane, sig_seq)
                             : phase_b(s, c, sub, &omap, p, warp, lane, bo, pol_out);
    if (!done_ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.ctx_empty[ci]);
    sub.ph0 = sub.parity(sub.nsub);
    sub.st0 = sub.stage(sub.nsub);
    if (++ci == kCtx) ci = 0;
  }
  sig_post(s.sig, kSigEnd, warp * 32 + lane, lane, sig_seq, 4 * p.timeout_ns, p.err);
  if (lane == 0) bulk_wait<0>();  // this warp's TMA stores done before exit
}

// ---------------------------------------------------------------- host --
gq_status setup(DeviceInfo& info) {
  gq_status st = check_cuda(
      cudaFuncSetAttribute(rowwise_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)),
      "rowwise_t: set shared memory size");
  if (st != GQ_OK) return st;
  int occ = 0;
  st = check_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &occ, rowwise_kernel, kThreads, kSmemBytes),
                  "rowwise_t: occupancy");
  if (st != GQ_OK) return st;
  if (occ < 1) return fail(GQ_ERR_UNSUPPORTED, "rowwise_t kernel does not fit an SM");
  info.rowwise_ctas_per_sm = occ;
  return GQ_OK;
}

gq_status launch(const DeviceInfo& info, const DebugKnobs& dbg, const void* a,
                 int32_t N, int32_t Mg, const int32_t* offs, int32_t G,
                 void* out_t, float* scales, void* ws, cudaStream_t stream) {
  CUtensorMap amap, omap;
  gq_status st = encode_tiled_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(a), static_cast<uint64_t>(Mg),
                                 static_cast<uint64_t>(N),
                                 static_cast<uint64_t>(Mg) * 2, kTm, kTn,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;
  st = encode_tiled_2d(&omap, CU_TENSOR_MAP_DATA_TYPE_UINT8, out_t,
                       static_cast<uint64_t>(N), static_cast<uint64_t>(Mg),
                       static_cast<uint64_t>(N), kBlk, kBlk,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;

  Params p;
  p.sched.units = (Mg + kSuper - 1) / kSuper;
  p.sched.groups = (N + kTn - 1) / kTn;
  const int64_t total = 2ll * p.sched.units * p.sched.groups;
  const int64_t max_ctas =
      static_cast<int64_t>(info.sm_count) * info.rowwise_ctas_per_sm;
  const int grid = static_cast<int>(total < max_ctas ? total : max_ctas);
  p.sched.lag = schedule_lag(dbg.lag[GQ_KIND_ROWWISE_T], p.sched.units,
                             p.sched.groups, grid, kCtx);

  const WorkspaceLayout L =
      workspace_layout(p.sched.groups, static_cast<int64_t>(N) * G);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.offs = offs;
  p.out_t = static_cast<uint8_t*>(out_t);
  p.scales = scales;
  p.done = reinterpret_cast<uint32_t*>(w + L.counters);
  p.amax = reinterpret_cast<uint32_t*>(w + L.amax);
  p.err = info.err_word;
  p.N = N;
  p.Mg = Mg;
  p.G = G;
  p.timeout_ns = dbg.timeout_ns;
  p.skip_arrival = dbg.skip_arrival;

  st = check_cuda(cudaMemsetAsync(ws, 0, L.total, stream),
                  "rowwise_t: clear workspace");
  if (st != GQ_OK) return st;
  // cooperative: the static ticket order needs every CTA resident
  void* args[] = {&amap, &omap, &p};
  return check_cuda(
      cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(rowwise_kernel),
                                  dim3(grid), dim3(kThreads), args, kSmemBytes,
                                  stream),
      "rowwise_t: launch");
}

}  // namespace rowwise
}  // namespace gq
