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
// kernel: stages come in by TMA with 128-byte rows, the transpose happens on
// the way from shared memory to registers (ldmatrix .trans) and between
// lanes (shuffles), and every warp store writes whole 32-byte sectors of A^T.
//
// A stage is kTn = 64 rows of A x kTm = 64 token columns (8 KB), staged with
// the 128-byte TMA swizzle so that row-wise and column-wise shared-memory
// accesses are bank-conflict free.  A super tile is kSub = 4 stages: 256
// token columns of one row band.  A row band (kTn rows, all Mg columns) is
// one dependency group.  See gq_device.cuh for the schedule.
//
// A producer warp loads the stages of the CTA's tickets into a shared ring
// of kStages buffers; a consumer warp takes the next loaded stage (a shared
// counter), whichever ticket it belongs to, and does all its work:
//   phase A: lane l takes rows l + 32 i; per group segment it folds |x|
//     of the row's columns inside the segment with max.xorsign.abs.bf16x2
//     into the super tile's context with shared-memory atomics; the warp
//     finishing the super tile adds them to the amax words in global memory,
//     laid out (G, N) so that a warp's atomics hit 128-byte runs;
//   phase B: per segment a lane computes the scales of rows l + 32 i
//     (448 / max(amax, 1e-12), IEEE division) and gathers the eight it needs
//     per 32-row half by shuffles; for each half and 8-column chunk,
//     ldmatrix.x4.trans gives lane l the pairs (n, n+1) of rows 8i + 2(l%4)
//     of column 8c + l/4, which are multiplied in fp32 (mul.rn.f32x2) and
//     packed with cvt.rn.satfinite.e4m3x2; a 4x4 exchange of byte pairs among
//     the four lanes of a column leaves each lane 8 consecutive bytes of a
//     row of A^T, stored with one 8-byte store.
// The context warp writes each super tile's context: the header, and in
// phase B -- once the band is complete -- the amax words of the band's rows
// for each of its first kSegA segments.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace rowwise {

constexpr int kStages = 12;           // shared ring of stage buffers
constexpr int kConsumerWarps = 4;
constexpr int kSub = 4;               // stages per super tile
constexpr int kSuper = kSub * kTm;    // token columns per super tile
constexpr int kCtx = 4;               // super-tile contexts in flight
constexpr int kQ = kTn / 32;          // 32-row parts of a stage
// warps: consumers 0..3, producer 4, context 5, signal 6
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kContextWarp = kConsumerWarps + 1;
constexpr int kSignalWarp = kConsumerWarps + 2;
constexpr int kThreads = (kConsumerWarps + 3) * 32;
constexpr int kSigSlots = 8;
constexpr int kStageBytes = kTn * kTm * 2;
constexpr int kSegA = 4;  // segments whose amax words ride in the context
static_assert(kTm * 2 == 128 && kTn % 32 == 0, "128-byte swizzled rows, 32-row parts");
static_assert(kTn % 4 == 0 && kTn / 4 <= 32, "one 16-byte amax chunk per context-warp lane");
static_assert(kSigSlots > kConsumerWarps, "one outstanding post per warp");

using Hdr = TileHdr<kSuper>;

struct Ctx {
  Hdr hdr;
  // phase A: the super tile's row maxima of its first kSegA segments (shared
  // atomics); phase B: the amax words of those segments
  alignas(16) uint32_t amax[kSegA][kTn];
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
  uint8_t tile[kStages][kStageBytes];  // 1024-byte aligned (swizzle atom)
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

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Params {
  const int32_t* offs;
  uint32_t* ticket;  // ticket counter
  uint8_t* out_t;
  float* scales;
  uint32_t* done;  // one word per row band: finished phase-A super tiles
  uint32_t* amax;  // (G, N) fp32 bit patterns
  unsigned* err;
  int32_t N, Mg, G;
  Schedule sched;  // units = super tiles per band
  uint64_t timeout_ns;
  int32_t skip_arrival;
};

__device__ __forceinline__ int stages_of(int32_t unit, int32_t Mg) {
  const int32_t m0 = unit * kSuper;
  return (min(m0 + kSuper, Mg) - m0 + kTm - 1) / kTm;
}

// ---------------------------------------------------------- context warp --
__device__ __forceinline__ void context_warp(Smem& s, const Params& p, int lane) {
  build_ends(p.offs, p.G, p.Mg, s.ends, lane);
  __syncwarp();
  const int32_t units = p.sched.units;
  const uint32_t total = 2u * static_cast<uint32_t>(units) * static_cast<uint32_t>(p.sched.groups);
  const uint64_t wait_ns = 4 * p.timeout_ns;
  int32_t ready_dg = -1;  // bands <= ready_dg are complete
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
    const int32_t n0 = dg * kTn;
    const int32_t m0 = unit * kSuper;
    build_header_warp(h, s.ends, p.G, m0, min(m0 + kSuper, p.Mg), unit == units - 1, lane);
    __syncwarp();
    if (phase == 1) {
      if (lane < kTn / 4) {
        const int n = min(static_cast<int>(h.nseg), kSegA);
        const int32_t row = n0 + 4 * lane;
        for (int j = 0; j < n; ++j)
          cp_async_16(smem_addr(&c.amax[j][4 * lane]),
                      p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + (row < p.N ? row : 0),
                      row < p.N ? 16u : 0u);
      }
      cp_async_mbar_arrive(&s.ctx_full[ci]);  // the context also waits for them
    } else if (lane < kTn / 4) {
#pragma unroll
      for (int j = 0; j < kSegA; ++j)
        sts128(smem_addr(&c.amax[j][4 * lane]), make_uint4(0, 0, 0, 0));
    }
    if (lane == 0) {
      c.a_done = 0;
      h.phase = phase;
      h.dg = dg;
      const int nsub = stages_of(unit, p.Mg);
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
__device__ __forceinline__ void producer_warp(Smem& s, const CUtensorMap* amap,
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
      nsub = stages_of(unit, p.Mg);
    }
    for (int k = 0; k < nsub; ++k, ++g) {
      const int st = static_cast<int>(g % kStages);
      if (!mbar_wait(&s.empty[st], ((g / kStages) & 1) ^ 1u, wait_ns, p.err)) return;
      if (lane == 0) {
        s.info[st].seq = t >= 0 ? seq : -1;
        s.info[st].k = k;
        if (t >= 0) {
          mbar_arrive_expect_tx(&s.full[st], kStageBytes);
          tma_load_2d(s.tile[st], amap, unit * kSuper + k * kTm, dg * kTn, &s.full[st],
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
// Phase A of one stage: per segment, the |x| maxima of rows l + 32 i,
// folded into the context (first kSegA segments) or straight into the global
// amax words.
__device__ __forceinline__ void stage_a(Ctx& c, int k, uint32_t tile, const Params& p,
                                        int lane) {
  const Hdr& h = c.hdr;
  const uint32_t row0 = tile + static_cast<uint32_t>(lane) * 128u;  // row l
  const int sw = lane & 7;  // swizzle of rows l + 32 i
  const int32_t n = h.dg * kTn + lane;
  const int cbase = k * kTm;  // super-tile column of stage column 0
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int ca = h.seg_lo[j] - cbase, cb = h.seg_hi[j] - cbase;
    if (cb <= 0) continue;
    if (ca >= kTm) break;
    uint32_t acc[kQ];
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) acc[qq] = 0;
    if (ca <= 0 && cb >= kTm) {
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {  // two batches of 4 chunks: loads first
        uint4 v[4][kQ];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int qq = 0; qq < kQ; ++qq)
            v[cc][qq] = lds128(row0 + qq * 32 * 128 + (((hb * 4 + cc) ^ sw) << 4));
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int qq = 0; qq < kQ; ++qq) {
            acc[qq] = absmax_bf16x2(absmax_bf16x2(acc[qq], v[cc][qq].x),
                                    absmax_bf16x2(v[cc][qq].y, v[cc][qq].z));
            acc[qq] = absmax_bf16x2(acc[qq], v[cc][qq].w);
          }
      }
    } else {
#pragma unroll 1
      for (int cc = 0; cc < kTm / 8; ++cc) {
        const int lo = cc * 8, hi = lo + 8;
        if (hi <= ca || lo >= cb) continue;
        const uint32_t o = static_cast<uint32_t>((cc ^ sw) << 4);
#pragma unroll
        for (int qq = 0; qq < kQ; ++qq) {
          const uint4 v = lds128(row0 + qq * 32 * 128 + o);
          const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int col = lo + e;
            if (col >= ca && col < cb) {
              const uint32_t sh = (e & 1) ? 16 : 0;
              acc[qq] = absmax_bf16x2(acc[qq], (a[e >> 1] >> sh) & 0xFFFFu);
            }
          }
        }
      }
    }
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) {
      const uint32_t m = amax_bits_of(acc[qq]);
      if (!m) continue;
      if (j < kSegA)
        red_max_shared(smem_addr(&c.amax[j][lane + 32 * qq]), m);
      else if (n + 32 * qq < p.N)
        atomicMax(p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + n + 32 * qq, m);
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
  const int32_t n = h.dg * kTn + lane;
  const int nj = min(static_cast<int>(h.nseg), kSegA);
  for (int j = 0; j < nj; ++j) {
    uint32_t* dst = p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + n;
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) {
      const uint32_t m = c.amax[j][lane + 32 * qq];
      if (m != 0u && n + 32 * qq < p.N) atomicMax(dst + 32 * qq, m);
    }
  }
  const bool skip = p.skip_arrival && h.dg == 0 && h.lo == 0;
  sig_post(s.sig, skip ? kSigSkip : h.dg, lane, wait_ns, p.err);
}

// Phase B of one stage: scale, cast and transpose; store rows of A^T.
__device__ __forceinline__ void stage_b(Smem& s, const Ctx& c, int k, uint32_t tile,
                                        const Params& p, int lane) {
  const Hdr& h = c.hdr;
  const int32_t n0 = h.dg * kTn;
  const int32_t nl = n0 + lane;  // rows nl + 32 i: the scales this lane computes
  const int q = lane & 3;
  const int mcol = lane >> 2;  // column within an 8-column chunk
  const int cbase = k * kTm;
  // owned groups without columns: amax 0 (once per super tile)
  if (k == 0) {
    for (int g = h.own_lo; g < h.own_hi; ++g) {
      const int32_t gs = g ? s.ends[g - 1] : 0;
      if (s.ends[g] == gs) {
        const float e = scale_from_amax_bits(0u);
#pragma unroll
        for (int qq = 0; qq < kQ; ++qq)
          if (nl + 32 * qq < p.N) p.scales[static_cast<size_t>(nl + 32 * qq) * p.G + g] = e;
      }
    }
  }
  // this lane's stores: bytes n0 + 32 i + 8 q .. + 7 of A^T rows
  uint8_t* obase = p.out_t + static_cast<size_t>(h.lo + cbase + mcol) * p.N + n0 + 8 * q;
  const size_t N8 = 8 * static_cast<size_t>(p.N);
  const uint32_t lrow = tile + static_cast<uint32_t>(lane) * 128u;  // ldmatrix row address base
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int ca = h.seg_lo[j] - cbase, cb = h.seg_hi[j] - cbase;
    if (cb <= 0) continue;
    if (ca >= kTm) break;
    const int g = h.seg_g[j];
    float sq[kQ];
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) {
      const int32_t nr = nl + 32 * qq;
      const uint32_t bits =
          j < kSegA ? c.amax[j][lane + 32 * qq]
                    : (nr < p.N ? ld_cg_u32(p.amax + static_cast<size_t>(g) * p.N + nr) : 0u);
      sq[qq] = scale_from_amax_bits(bits);
    }
    // the group starts inside the super tile at column seg_lo: the stage
    // holding that column writes its scales
    if (ca >= 0 && g >= h.own_lo && g < h.own_hi) {
#pragma unroll
      for (int qq = 0; qq < kQ; ++qq)
        if (nl + 32 * qq < p.N) p.scales[static_cast<size_t>(nl + 32 * qq) * p.G + g] = sq[qq];
    }
    const int c_first = max(ca, 0) >> 3;
    const int c_last = (min(cb, kTm) - 1) >> 3;
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) {
      // scales of rows 32 qq + 8 i + 2q (+1), the rows of matrix i
      float sv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sv[2 * i] = __shfl_sync(0xffffffffu, sq[qq], 8 * i + 2 * q);
        sv[2 * i + 1] = __shfl_sync(0xffffffffu, sq[qq], 8 * i + 2 * q + 1);
      }
      const bool st_ok = n0 + 32 * qq + 8 * q < p.N;
      for (int cc = c_first; cc <= c_last; ++cc) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(lrow + qq * 32 * 128 + ((((cc ^ lane) & 7)) << 4), r0, r1, r2, r3);
        // p01: bytes of rows 2q, 2q+1 (matrix 0) and 8+2q, 9+2q (matrix 1);
        // p23: matrices 2 and 3 -- the pairs V[q][i] of lane q
        const uint32_t p01 = quant4(r0, r1, sv[0], sv[1], sv[2], sv[3]);
        const uint32_t p23 = quant4(r2, r3, sv[4], sv[5], sv[6], sv[7]);
        // 4x4 transpose of pairs among the lanes of one column: lane q ends
        // with V[0][q], V[1][q], V[2][q], V[3][q] = rows 8q .. 8q + 7
        const uint32_t x1 = __shfl_xor_sync(0xffffffffu, (q & 2) ? p01 : p23, 2);
        const uint32_t tlo = (q & 2) ? x1 : p01, thi = (q & 2) ? p23 : x1;
        const uint32_t x2 = __shfl_xor_sync(
            0xffffffffu, __byte_perm(tlo, thi, (q & 1) ? 0x5410 : 0x7632), 1);
        const uint32_t w0 = (q & 1) ? __byte_perm(x2, tlo, 0x7610) : __byte_perm(tlo, x2, 0x5410);
        const uint32_t w1 = (q & 1) ? __byte_perm(x2, thi, 0x7632) : __byte_perm(thi, x2, 0x7610);
        const int m = cc * 8 + mcol;  // stage column
        if (m >= ca && m < cb && st_ok)
          __stcs(reinterpret_cast<uint2*>(obase + cc * N8 + qq * 32), make_uint2(w0, w1));
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    rowwise_kernel(const __grid_constant__ CUtensorMap amap, const Params p) {
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
    if (lane == 0) prefetch_tensormap(&amap);
    producer_warp(s, &amap, p, lane);
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
  CUtensorMap amap;
  gq_status st = encode_tiled_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(a), static_cast<uint64_t>(Mg),
                                 static_cast<uint64_t>(N),
                                 static_cast<uint64_t>(Mg) * 2, kTm, kTn,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
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
  p.ticket = reinterpret_cast<uint32_t*>(w);  // first word of the header
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
  // cooperative: a claimed ticket may wait for tickets of other CTAs, so
  // every CTA must be resident
  void* args[] = {&amap, &p};
  return check_cuda(
      cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(rowwise_kernel),
                                  dim3(grid), dim3(kThreads), args, kSmemBytes,
                                  stream),
      "rowwise_t: launch");
}

}  // namespace rowwise
}  // namespace gq
