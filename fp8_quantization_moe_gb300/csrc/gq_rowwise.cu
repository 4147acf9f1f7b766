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
// kernel: windows come in by TMA with 128-byte rows, the transpose happens on
// the way from shared memory to registers (ldmatrix .trans) and between
// lanes (shuffles), and every warp store writes whole 32-byte sectors of A^T.
//
// Work unit: one (row band, group) pair -- kTn = 64 rows of A by the group's
// token columns.  Every scale of the unit depends on the unit alone, so no
// block ever waits for another: a persistent grid claims units from a global
// counter, group by group.  A unit is read through windows of kTn rows x kTm =
// 64 token columns (8 KB, one TMA box with the 128-byte swizzle, so that
// row-wise and column-wise shared-memory accesses are bank-conflict free);
// window 0 starts at s_g rounded down to 8 tokens (the TMA's 16-byte rule).
// A unit of at most kFit windows (groups up to about 760 tokens) keeps them
// in shared memory between its two passes, and A is read from HBM once; a
// longer unit streams its windows twice through the ring, the second time
// from L2 where it can.
//
// A descriptor warp claims units and publishes each in a small ring of unit
// descriptors -- at most `lag` units in flight, about kBudget windows' worth
// of the average unit, so that short units keep the consumers fed and long
// ones do not pile up in the last claims --; a loader warp follows the descriptors and issues the TMA
// loads of the block's window stream into a ring of kStages windows, kIssue
// windows side by side.  Pass A of a unit folds its amax, pass B scales,
// casts and stores it; a pass covers the unit's windows in order.  Resident
// units are visited with a lag of one unit,
//   A(r0), A(r1), B(r0), A(r2), B(r1), ...,
// so that pass B does not wait for the amax; before a long unit L the
// pending resident unit is finished, and L's two passes follow each other:
//   ..., A(r2), B(r1), B(r2), A(L), B(L), A(r3), ...
// A visits load a window; B visits of a resident unit re-read the window A
// left behind, B visits of a long unit load it again.  Consumer warp w takes
// the visits w, w + W, w + 2W, ... of the stream (W = kConsumerWarps), each
// visit alone:
//   A visit: lane l takes rows l and l + 32 of the window, folds |x| over
//     the window's columns inside the group with max.xorsign.abs.bf16x2 and
//     adds the row maxima to the unit's amax words with shared-memory
//     atomics; the last warp through a unit's pass A (an acquire-release
//     counter says which) turns its amax words into scales (448 / max(amax,
//     1e-12), IEEE division), stores them, and completes the unit's amax
//     barrier;
//   B visit: once that barrier completes, for each 32-row half and 8-column
//     chunk, ldmatrix.x4.trans gives lane l the pairs
//     (n, n+1) of rows 8i + 2(l%4) of column 8c + l/4, which are multiplied
//     in fp32 (mul.rn.f32x2) and packed with cvt.rn.satfinite.e4m3x2; a 4x4
//     exchange of words among the four lanes of a column, over both halves,
//     leaves each lane 16 consecutive bytes of a row of A^T, stored with one
//     16-byte store.
// Every warp walks the same stream and derives each visit's ring slot from
// the descriptors, so a window costs one barrier wait to read and one
// arrival to release.
//
// Progress: the ring is a FIFO, so the loads issued between a resident
// unit's first window and its pass B must fit in it next to that unit's
// windows; in the stream above they are the windows of at most one other
// resident unit (2 kFit <= kStages), and a long unit's windows are released
// as they are visited.  A warp's waits only ever name visits earlier in the
// stream.  Every wait is bounded in time nonetheless.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace rowwise {

constexpr int kStages = 24;  // ring of windows
constexpr int kFit = 12;     // windows a unit may keep resident between passes
constexpr int kUnits = 8;    // unit descriptors (at most in flight)
constexpr int kBudget = 40;  // ring loads the units in flight should come to, about
constexpr int kConsumerWarps = 10;
constexpr int kAhead = 2;  // units a block claims before it needs them
constexpr int kIssue = 8;  // producer lanes issuing window loads side by side
constexpr int kLoaderWarp = kConsumerWarps;
constexpr int kDescWarp = kConsumerWarps + 1;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kQ = kTn / 32;  // 32-row halves of a window
constexpr int kStageBytes = kTn * kTm * 2;
static_assert(kTm * 2 == 128 && kTn == 64, "128-byte swizzled rows, two 32-row halves");
static_assert(2 * kFit <= kStages, "the ring holds two consecutive resident units");
static_assert(kUnits >= 2, "pass B of a resident unit follows pass A of the next");
static_assert(kIssue <= kStages && kIssue <= 32, "a batch of loads takes distinct slots");

struct Unit {
  int32_t n0;   // first row of the band; -1: no more units
  int32_t g;    // group
  int32_t x0;   // token column of window 0 (s_g rounded down to 8)
  int32_t lo;   // group columns relative to x0: [lo, hi)
  int32_t hi;
  int32_t nst;  // windows
  int32_t resident;  // 1: windows stay in the ring for pass B
  int32_t hold;      // test hook: the amax is never reported complete
  uint32_t a_done;   // A visits finished
  alignas(16) uint32_t amax[kTn];  // row maxima, fp32 bit patterns
  alignas(16) float scale[kTn];    // written by the last warp through pass A
};

struct Smem {
  uint8_t tile[kStages][kStageBytes];  // 1024-byte aligned (swizzle atom)
  Unit unit[kUnits];
  uint64_t full[kStages];    // window loaded (TMA bytes)
  uint64_t empty[kStages];   // window released
  uint64_t u_full[kUnits];   // descriptor published
  uint64_t u_amax[kUnits];   // pass A done and scales written
  uint64_t u_free[kUnits];   // every warp's B visits done (W arrivals)
  int32_t ends[kMaxGroups];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "fits one SM's shared memory");

struct Params {
  const int32_t* offs;
  uint32_t* ticket;  // unit counter; ticket[1]: blocks finished
  uint8_t* out_t;
  float* scales;
  unsigned* err;
  int32_t N, Mg, G;
  uint32_t units;  // row bands x groups
  uint32_t bands;  // row bands of kTn rows
  int32_t lag;     // units in flight per block (2 .. kUnits)
  uint64_t timeout_ns;
  int32_t skip_arrival;
  bool pow2;  // scales rounded down to powers of two
};

// ------------------------------------------------- descriptor and loader --
// Loads the nst windows of a pass (token columns x0 + 64 k, rows y ...) into
// the ring: lanes 0 .. kIssue-1 take windows kb + lane side by side, each
// waiting for its own slot.
__device__ __forceinline__ bool load_pass(Smem& s, const CUtensorMap* amap, uint32_t& g, int nst,
                                          int32_t x0, int32_t y, uint64_t pol, int lane,
                                          uint64_t wait_ns, unsigned* err) {
  for (int kb = 0; kb < nst; kb += kIssue) {
    const int k = kb + lane;
    bool ok = true;
    if (lane < kIssue && k < nst) {
      const uint32_t ld = g + k;
      const int st = static_cast<int>(ld % kStages);
      ok = mbar_wait(&s.empty[st], ((ld / kStages) & 1) ^ 1u, wait_ns, err);
      if (ok) {
        mbar_arrive_expect_tx(&s.full[st], kStageBytes);
        tma_load_2d(s.tile[st], amap, x0 + k * kTm, y, &s.full[st], pol);
      }
    }
    if (__any_sync(0xffffffffu, !ok)) return false;
  }
  g += static_cast<uint32_t>(nst);
  return true;
}

// Claims units (kAhead ahead), decodes them and publishes their
// descriptors; empty groups get their scales here and no descriptor.  The
// whole warp builds the group-end table first.
__device__ __forceinline__ void descriptor_warp(Smem& s, const Params& p, int lane) {
  build_ends(p.offs, 0, p.G, p.Mg, s.ends, lane);
  __syncwarp();
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t useq = 0;  // units published
  // lane 0 claims units kAhead ahead, so that a claim's round trip to L2
  // overlaps the units before it
  uint32_t q[kAhead];
#pragma unroll
  for (int a = 0; a < kAhead; ++a) q[a] = lane == 0 ? claim_ticket(p.ticket) : 0u;
  for (;;) {
    const uint32_t u = __shfl_sync(0xffffffffu, q[0], 0);
#pragma unroll
    for (int a = 0; a + 1 < kAhead; ++a) q[a] = q[a + 1];
    if (lane == 0 && u < p.units) q[kAhead - 1] = claim_ticket(p.ticket);
    int32_t grp = 0, n0 = -1, s0 = 0, e0 = 0;
    if (u < p.units) {  // else: publish the stop descriptor
      // group-major: the bands of a group are claimed one after another, so
      // the 64-byte runs that neighbouring bands write into each row of A^T
      // reach L2 close together
      grp = static_cast<int32_t>(u / static_cast<uint32_t>(p.bands));
      n0 = static_cast<int32_t>(u % static_cast<uint32_t>(p.bands)) * kTn;
      s0 = grp ? s.ends[grp - 1] : 0;
      e0 = s.ends[grp];
      if (e0 == s0) {  // empty group: amax 0 for every row
        const float e = scale_from_amax_bits(0u, p.pow2);
#pragma unroll
        for (int qq = 0; qq < kQ; ++qq) {
          const int32_t n = n0 + lane + 32 * qq;
          if (n < p.N) p.scales[static_cast<size_t>(n) * p.G + grp] = e;
        }
        continue;
      }
    }
    const int32_t x0 = s0 & ~7;
    const int nst = n0 >= 0 ? (e0 - x0 + kTm - 1) / kTm : 0;
    const int us = static_cast<int>(useq % kUnits);
    // at most p.lag units in flight: unit useq - lag must be finished (units
    // finish in stream order), which also frees this descriptor
    bool ok = true;
    if (useq >= static_cast<uint32_t>(p.lag)) {
      const uint32_t v = useq - static_cast<uint32_t>(p.lag);
      ok = mbar_wait(&s.u_free[v % kUnits], (v / kUnits) & 1, wait_ns, p.err);
    }
    if (__any_sync(0xffffffffu, !ok)) return;
    Unit& U = s.unit[us];
    if (lane < kTn / 4) sts128(smem_addr(&U.amax[4 * lane]), make_uint4(0, 0, 0, 0));
    if (lane == 0) {
      U.n0 = n0;
      U.g = grp;
      U.x0 = x0;
      U.lo = s0 - x0;
      U.hi = e0 - x0;
      U.nst = nst;
      U.resident = nst <= kFit ? 1 : 0;
      U.hold = p.skip_arrival && u == 0u;
      U.a_done = 0u;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.u_full[us]);
    ++useq;
    if (n0 < 0) return;
  }
}

// Follows the published descriptors and loads the window stream: pass A of
// each unit, and a long unit's pass B at once.
__device__ __forceinline__ void loader_warp(Smem& s, const CUtensorMap* amap, const Params& p,
                                            int lane) {
  if (lane == 0) prefetch_tensormap(amap);
  const uint64_t pol_once = policy_evict_first();  // read once
  const uint64_t pol_again = policy_evict_last();  // a long unit's pass A
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t g = 0;  // loads issued
  for (uint32_t useq = 0;; ++useq) {
    const int us = static_cast<int>(useq % kUnits);
    bool ok = mbar_wait(&s.u_full[us], (useq / kUnits) & 1, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;
    const Unit& U = s.unit[us];
    const int32_t n0 = U.n0, x0 = U.x0;
    const int nst = U.nst;
    const bool resident = U.resident != 0;
    if (n0 < 0) break;
    ok = load_pass(s, amap, g, nst, x0, n0, resident ? pol_once : pol_again, lane, wait_ns, p.err);
    if (ok && !resident) ok = load_pass(s, amap, g, nst, x0, n0, pol_once, lane, wait_ns, p.err);
    if (!ok) break;
  }
  // no load may still be in flight when the block exits
  if (lane == 0)
    for (uint32_t d = g > static_cast<uint32_t>(kStages) ? g - kStages : 0u; d < g; ++d)
      mbar_wait(&s.full[d % kStages], (d / kStages) & 1, wait_ns, p.err);
}

// ------------------------------------------------------------ consumers --
// A visit: the |x| maxima of rows l and l + 32 over the window's columns
// [ca, cb) (the group's), added to the unit's amax words.
__device__ __forceinline__ void fold_a(Unit& U, int ca, int cb, uint32_t tile, int lane) {
  const uint32_t row0 = tile + static_cast<uint32_t>(lane) * 128u;  // row l
  const int sw = lane & 7;  // swizzle of rows l + 32 i
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
    for (int cc = max(ca, 0) >> 3; cc <= (min(cb, kTm) - 1) >> 3; ++cc) {
      const int c0 = cc * 8;
      const uint32_t o = static_cast<uint32_t>((cc ^ sw) << 4);
#pragma unroll
      for (int qq = 0; qq < kQ; ++qq) {
        const uint4 v = lds128(row0 + qq * 32 * 128 + o);
        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int col = c0 + e;
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
    if (m) red_max_shared(smem_addr(&U.amax[lane + 32 * qq]), m);
  }
}

// B visit: scale, cast and transpose the window at token column xw (group
// columns [ca, cb) of it); store rows of A^T.  scale[r] is the scale of row
// n0 + r.  Both 32-row halves go through ldmatrix and the cast first, in
// batches of all eight 8-column chunks, so that eight independent chains
// hide the latency of each step; then, per chunk, a 4x4 exchange of words
// among the four lanes of a column leaves each lane 16 consecutive bytes of
// a row of A^T (rows 16 q .. 16 q + 15 of the band), stored with one 16-byte
// store.  Chunks outside [ca, cb) are computed from the window's other
// columns and not stored.  The window's ring slot (`empty`) is released as
// soon as the casts are in registers.
__device__ __forceinline__ void quant_b(int32_t n0, int32_t xw, int ca, int cb,
                                        const float* scale, uint32_t tile, uint64_t* empty,
                                        const Params& p, int lane) {
  const int q = lane & 3;
  const int mcol = lane >> 2;  // column within an 8-column chunk
  // this lane's stores: bytes n0 + 16 q .. + 15 of A^T rows
  uint8_t* obase = p.out_t + static_cast<size_t>(xw + mcol) * p.N + n0 + 16 * q;
  const size_t N8 = 8 * static_cast<size_t>(p.N);
  const uint32_t lrow = tile + static_cast<uint32_t>(lane) * 128u;  // ldmatrix row address base
  constexpr int kC = kTm / 8;  // chunks
  // w[cc][t]: the cast bytes of rows 16 t + (2q, 2q+1, 8+2q, 9+2q) of
  // column 8 cc + mcol (t = 2 qq: matrices 0, 1 of half qq; t = 2 qq + 1:
  // matrices 2, 3)
  uint32_t w[kC][4];
#pragma unroll
  for (int qq = 0; qq < kQ; ++qq) {
    // scales of rows 32 qq + 8 i + 2q (+1), the rows of matrix i
    float sv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = *reinterpret_cast<const float2*>(scale + 32 * qq + 8 * i + 2 * q);
      sv[2 * i] = v.x;
      sv[2 * i + 1] = v.y;
    }
    uint32_t r[kC][4];
#pragma unroll
    for (int cc = 0; cc < kC; ++cc)
      ldsm_x4_trans(lrow + qq * 32 * 128 + ((((cc ^ lane) & 7)) << 4), r[cc][0], r[cc][1],
                    r[cc][2], r[cc][3]);
#pragma unroll
    for (int cc = 0; cc < kC; ++cc) {
      w[cc][2 * qq] = quant4(r[cc][0], r[cc][1], sv[0], sv[1], sv[2], sv[3]);
      w[cc][2 * qq + 1] = quant4(r[cc][2], r[cc][3], sv[4], sv[5], sv[6], sv[7]);
    }
  }
  // the window is read: its slot goes back to the ring before the exchange
  // and the stores, so that the loader can refill it sooner
  __syncwarp();
  if (lane == 0) mbar_arrive(empty);
  // lane q holds M[q][t] = w[.][t] for the four targets t; lane t needs
  // M[0..3][t].  Step 1 (partner q ^ 2) swaps the two words whose target
  // differs from q in bit 1, step 2 (partner q ^ 1) those differing in bit 0.
  const bool b2 = (q & 2) != 0, b1 = (q & 1) != 0;
  // byte order of the 16 rows: words of lanes (0, 1) give rows 0-3 (low
  // halves) and 8-11 (high halves), lanes (2, 3) rows 4-7 and 12-15
  const uint32_t sel_lo = b1 ? 0x1054u : 0x5410u;
  const uint32_t sel_hi = b1 ? 0x3276u : 0x7632u;
  const bool st_ok = n0 + 16 * q < p.N;
#pragma unroll
  for (int cc = 0; cc < kC; ++cc) {
    const uint32_t own0 = b2 ? w[cc][2] : w[cc][0];  // M[q][t0], t0 = q & 2
    const uint32_t own1 = b2 ? w[cc][3] : w[cc][1];  // M[q][t0 + 1]
    const uint32_t g0 = __shfl_xor_sync(0xffffffffu, b2 ? w[cc][0] : w[cc][2], 2);  // M[q^2][t0]
    const uint32_t g1 = __shfl_xor_sync(0xffffffffu, b2 ? w[cc][1] : w[cc][3], 2);  // M[q^2][t0+1]
    const uint32_t a = b1 ? own1 : own0;  // M[q][q]
    const uint32_t c = b1 ? g1 : g0;      // M[q^2][q]
    const uint32_t bb = __shfl_xor_sync(0xffffffffu, b1 ? own0 : own1, 1);  // M[q^1][q]
    const uint32_t d = __shfl_xor_sync(0xffffffffu, b1 ? g0 : g1, 1);       // M[q^3][q]
    // sources 0..3 are (a, bb, c, d) permuted by q: lanes (0,1) -> (P, Q),
    // lanes (2, 3) -> (R, S), each pair swapped when q is odd (sel_*)
    const uint32_t P = b2 ? c : a, Q = b2 ? d : bb, R = b2 ? a : c, S = b2 ? bb : d;
    const int m = cc * 8 + mcol;  // window column
    if (m >= ca && m < cb && st_ok)
      __stcs(reinterpret_cast<uint4*>(obase + cc * N8),
             make_uint4(__byte_perm(P, Q, sel_lo), __byte_perm(R, S, sel_lo),
                        __byte_perm(P, Q, sel_hi), __byte_perm(R, S, sel_hi)));
  }
}

// What a warp keeps of a unit between its two passes.
struct UnitView {
  uint32_t useq;
  int32_t n0, g, x0, lo, hi, nst;
  bool resident;
  uint32_t first;  // ring load of pass A's window 0
};

// Waits until the ring load `ld` is in place.  The load kStages earlier in
// the same slot may still be outstanding -- visits finish out of order -- so
// its release is waited for first; then the full barrier is in ld's round.
__device__ __forceinline__ bool wait_load(Smem& s, uint32_t ld, uint64_t wait_ns, unsigned* err) {
  const int st = static_cast<int>(ld % kStages);
  bool ok = mbar_wait(&s.empty[st], ((ld / kStages) & 1) ^ 1u, wait_ns, err);
  if (ok) ok = mbar_wait(&s.full[st], (ld / kStages) & 1, wait_ns, err);
  return ok;
}

// Pass A of unit `cu` (its windows are ring loads cu.first ...): this warp's
// visits, and from the warp finishing the last of them the unit's scales.
__device__ __forceinline__ bool pass_a(Smem& s, const UnitView& cu, bool hold, uint32_t& j,
                                       const Params& p, int w, int lane, uint64_t wait_ns) {
  unsigned* err = p.err;
  Unit& U = s.unit[cu.useq % kUnits];
  const int k0 = static_cast<int>((w + kConsumerWarps - j % kConsumerWarps) % kConsumerWarps);
  j += static_cast<uint32_t>(cu.nst);
  if (k0 >= cu.nst) return true;  // no visit of this unit
  for (int k = k0; k < cu.nst; k += kConsumerWarps) {
    const uint32_t ld = cu.first + k;
    const bool ok = wait_load(s, ld, wait_ns, err);
    if (__any_sync(0xffffffffu, !ok)) return false;
    const uint32_t tile = pin(smem_addr(s.tile[ld % kStages]));
    fold_a(U, cu.lo - k * kTm, cu.hi - k * kTm, tile, lane);
    if (!cu.resident) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[ld % kStages]);
    }
  }
  // the warp that finishes the unit's last A visit (an acquire-release
  // counter of visits says which) turns the amax words into its scales, once
  const uint32_t mine = static_cast<uint32_t>((cu.nst - k0 + kConsumerWarps - 1) / kConsumerWarps);
  __syncwarp();
  uint32_t prev = 0;
  if (lane == 0) prev = atom_add_acq_rel_cta_shared(smem_addr(&U.a_done), mine);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev + mine == static_cast<uint32_t>(cu.nst)) {
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) {
      const int r = lane + 32 * qq;
      const float sc = scale_from_amax_bits(U.amax[r], p.pow2);
      U.scale[r] = sc;
      if (cu.n0 + r < p.N) p.scales[static_cast<size_t>(cu.n0 + r) * p.G + cu.g] = sc;
    }
    __syncwarp();
    if (lane == 0 && !hold) mbar_arrive(&s.u_amax[cu.useq % kUnits]);
  }
  return true;
}

// Pass B of unit `pv`, whose windows are ring loads `base` ...: this warp's
// visits, then its arrival on the unit's free barrier.
__device__ __forceinline__ bool pass_b(Smem& s, const UnitView& pv, uint32_t base, uint32_t& j,
                                       const Params& p, int w, int lane, uint64_t wait_ns) {
  const int ps = static_cast<int>(pv.useq % kUnits);
  const int k0 = static_cast<int>((w + kConsumerWarps - j % kConsumerWarps) % kConsumerWarps);
  if (k0 < pv.nst) {
    bool ok = mbar_wait(&s.u_amax[ps], (pv.useq / kUnits) & 1, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) return false;
    for (int k = k0; k < pv.nst; k += kConsumerWarps) {
      const uint32_t ld = base + k;
      // a resident window is still in the round its A visit waited for
      ok = pv.resident ? mbar_wait(&s.full[ld % kStages], (ld / kStages) & 1, wait_ns, p.err)
                       : wait_load(s, ld, wait_ns, p.err);
      if (__any_sync(0xffffffffu, !ok)) return false;
      const uint32_t tile = pin(smem_addr(s.tile[ld % kStages]));
      quant_b(pv.n0, pv.x0 + k * kTm, pv.lo - k * kTm, pv.hi - k * kTm, s.unit[ps].scale, tile,
              &s.empty[ld % kStages], p, lane);
    }
  }
  j += static_cast<uint32_t>(pv.nst);
  __syncwarp();
  if (lane == 0) mbar_arrive(&s.u_free[ps]);
  return true;
}

__device__ __forceinline__ void consumer_warp(Smem& s, const Params& p, int w, int lane) {
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t g = 0;  // ring loads of the stream so far (the producer's count)
  uint32_t j = 0;  // visits of the stream so far
  UnitView pv;     // the resident unit whose pass B is pending
  bool pending = false;
  for (uint32_t useq = 0;; ++useq) {
    const int us = static_cast<int>(useq % kUnits);
    const bool ok = mbar_wait(&s.u_full[us], (useq / kUnits) & 1, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) return;
    const Unit& U = s.unit[us];
    UnitView cu;
    cu.useq = useq;
    cu.n0 = U.n0;
    cu.g = U.g;
    cu.x0 = U.x0;
    cu.lo = U.lo;
    cu.hi = U.hi;
    cu.nst = U.nst;
    cu.resident = U.resident != 0;
    cu.first = g;
    const bool hold = U.hold != 0;
    if (cu.n0 < 0) {  // the stop descriptor
      if (pending) pass_b(s, pv, pv.first, j, p, w, lane, wait_ns);
      return;
    }
    if (cu.resident) {
      g += static_cast<uint32_t>(cu.nst);
      if (!pass_a(s, cu, hold, j, p, w, lane, wait_ns)) return;
      if (pending && !pass_b(s, pv, pv.first, j, p, w, lane, wait_ns)) return;
      pv = cu;
      pending = true;
    } else {
      if (pending && !pass_b(s, pv, pv.first, j, p, w, lane, wait_ns)) return;
      pending = false;
      g += static_cast<uint32_t>(cu.nst);
      if (!pass_a(s, cu, hold, j, p, w, lane, wait_ns)) return;
      const uint32_t base = g;  // the windows come again
      g += static_cast<uint32_t>(cu.nst);
      if (!pass_b(s, cu, base, j, p, w, lane, wait_ns)) return;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
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
    for (int i = 0; i < kUnits; ++i) {
      mbar_init(&s.u_full[i], 1);
      mbar_init(&s.u_amax[i], 1);
      mbar_init(&s.u_free[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDescWarp)
    descriptor_warp(s, p, lane);
  else if (warp == kLoaderWarp)
    loader_warp(s, &amap, p, lane);
  else
    consumer_warp(s, p, warp, lane);

  // The last block to finish returns the counters to zero, so that the next
  // call on this workspace may skip its clear (GQ_WORKSPACE_ZEROED).  Every
  // block gets here, also after a bounded wait expired, and has made its
  // last claim before its arrival is counted.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.ticket + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.ticket, 0u);
      atomicExch(p.ticket + 1, 0u);
    }
  }
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
                 void* out_t, float* scales, uint32_t flags, void* ws, cudaStream_t stream) {
  CUtensorMap amap;
  gq_status st = encode_tiled_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(a), static_cast<uint64_t>(Mg),
                                 static_cast<uint64_t>(N),
                                 static_cast<uint64_t>(Mg) * 2, kTm, kTn,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;

  Params p;
  const int64_t bands = (N + kTn - 1) / kTn;
  const int64_t units = bands * G;
  const int64_t max_ctas = static_cast<int64_t>(info.sm_count) * info.rowwise_ctas_per_sm;
  const int grid = static_cast<int>(units < max_ctas ? units : max_ctas);
  // the unit counter ends below units + (kAhead + 1) * grid
  if (units + (kAhead + 1) * static_cast<int64_t>(grid) >= (int64_t(1) << 32))
    return fail(GQ_ERR_UNSUPPORTED, "rowwise_t: (N / 64) x n_groups too large");
  p.offs = offs;
  p.ticket = static_cast<uint32_t*>(ws);  // first word of the header
  p.out_t = static_cast<uint8_t*>(out_t);
  p.scales = scales;
  p.err = info.err_word;
  p.N = N;
  p.Mg = Mg;
  p.G = G;
  p.units = static_cast<uint32_t>(units);
  p.bands = static_cast<uint32_t>(bands);
  // units in flight: about kBudget ring loads' worth of the average unit (a
  // long unit streams twice), at least two -- more overlap the short units'
  // descriptor and scale waits, fewer keep the last claims of a grid with
  // few units per block balanced
  {
    int64_t win = (Mg / G + kTm - 1) / kTm + 1;
    if (win > kFit) win *= 2;
    int64_t lag = kBudget / win;
    p.lag = static_cast<int32_t>(lag < 2 ? 2 : lag > kUnits ? kUnits : lag);
  }
  p.timeout_ns = dbg.timeout_ns;
  p.skip_arrival = dbg.skip_arrival;
  p.pow2 = (flags & GQ_SCALE_POW2) != 0;

  if (!(flags & GQ_WORKSPACE_ZEROED)) {
    st = check_cuda(cudaMemsetAsync(ws, 0, 8, stream), "rowwise_t: clear the counters");
    if (st != GQ_OK) return st;
  }
  rowwise_kernel<<<grid, kThreads, kSmemBytes, stream>>>(amap, p);
  return check_cuda(cudaGetLastError(), "rowwise_t: launch");
}

}  // namespace rowwise
}  // namespace gq
