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
// from L2 where it can.  Where groups are far longer (calls whose groups
// average kSplitAvg tokens or more take a build that can do this), a unit of
// more than kSplitOver windows -- whose two reads, for every row band at
// once, would pass more data than L2 keeps between them -- is cut into parts
// of at most kFit windows, consecutive tickets that other blocks take: each
// part stays resident, adds its row maxima to the unit's words in the
// workspace with atomicMax and counts itself (release); the descriptor warp
// of each part, one unit later, waits for the count (acquire), takes the
// scales and lets the part's pass B start.  Tickets are then assigned
// (block b takes b, b + grid, ...), not claimed, so that a unit's parts lie
// in two consecutive rounds of the grid, and a block's stream visits A of its
// next unit before B of the current one; so a pass B waits only for passes
// A that no wait precedes -- provided every block of the grid is resident,
// which the blocks establish first (a count of arrivals and one CAS that
// settles the decision for all), falling back to unsplit units otherwise.
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

#include <algorithm>

namespace gq {
namespace rowwise {

constexpr int kStages = 24;  // ring of windows
constexpr int kFit = 12;     // windows a unit may keep resident between passes
// A unit of more windows is split into parts of at most kFit windows that
// several blocks take: read twice through the ring, such units (a group of
// thousands of tokens in every row band) would pass more than L2 holds
// between their two reads.
constexpr int kSplitOver = 64;
constexpr int kSplitAvg = 2048;  // average group (tokens) from which a call may split units
constexpr int kUnits = 8;    // unit descriptors (at most in flight)
constexpr int kBudget = 40;  // ring loads the units in flight should come to, about
constexpr int kConsumerWarps = 14;
constexpr int kAhead = 2;  // units a block claims before it needs them
constexpr int kIssue = 8;  // producer lanes issuing window loads side by side
constexpr uint64_t kResidentWaitNs = 200000;  // for every block of the grid to arrive
constexpr int kLoaderWarp = kConsumerWarps;
constexpr int kDescWarp = kConsumerWarps + 1;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kQ = kTn / 32;  // 32-row halves of a window
constexpr int kStageBytes = kTn * kTm * 2;
static_assert(kTm * 2 == 128 && kTn == 64, "128-byte swizzled rows, two 32-row halves");
static_assert(2 * kFit <= kStages, "the ring holds two consecutive resident units");
static_assert(kUnits >= 2, "pass B of a resident unit follows pass A of the next");
static_assert(kIssue <= kStages && kIssue <= 32, "a batch of loads takes distinct slots");
static_assert(kSplitWords >= kTn + 1 && kSplitWords % 4 == 0, "amax words, counter, 16-byte rows");

struct Unit {
  int32_t n0;   // first row of the band; -1: no more units
  int32_t g;    // group
  int32_t sidx;   // split unit: its row of the split words; -1: not split
  int32_t parts;  // parts of the split unit
  int32_t part;   // this part (0 writes the scales)
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
  // tickets of groups before g (tb[G] = all); split units of groups before
  // g (sb[G] = all); both for the call's decomposition
  int32_t tb[kMaxGroups + 1];
  int32_t sb[kMaxGroups + 1];
  int32_t split_mode;  // some unit is split: tickets are assigned, not claimed
  int32_t clear_all;   // the last block clears the split words (after an error)
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "fits one SM's shared memory");

struct Params {
  const int32_t* offs;
  uint32_t* ticket;  // unit counter; [1] blocks finished; [2] blocks arrived; [3] split decision
  uint32_t* split;   // per split unit: kTn amax words and a counter (kSplitWords)
  int32_t max_split; // split units the workspace has room for
  uint64_t split_words;  // 32-bit words of the split region
  uint8_t* out_t;
  float* scales;
  unsigned* err;
  int32_t N, Mg, G;
  uint32_t units;  // row bands x groups
  uint32_t bands;  // row bands of kTn rows
  int32_t lag;     // units in flight per block (2 .. kUnits)
  uint64_t timeout_ns;
  int32_t skip_arrival;
  int32_t no_split;  // test hook: units are never split
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

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* ptr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(ptr), "r"(v)
               : "memory");
  return old;
}

// Windows of the group columns [s0, e0) (window 0 at s0 rounded down to 8).
__device__ __forceinline__ int32_t windows_of(int32_t s0, int32_t e0) {
  return (e0 - (s0 & ~7) + kTm - 1) / kTm;
}

// Parts each unit of a group is cut into: a unit of more than kSplitOver
// windows into parts of at most kFit, so that every part stays resident.
__device__ __forceinline__ int32_t parts_of(int32_t s0, int32_t e0) {
  const int32_t w = e0 > s0 ? windows_of(s0, e0) : 0;
  return w > kSplitOver ? (w + kFit - 1) / kFit : 1;
}

// Largest g in [0, n) with bands * pre[g] <= u, for a nondecreasing pre
// with pre[0] = 0; a whole warp searches 32 probes at a time.
__device__ __forceinline__ int find_group(const int32_t* pre, int n, uint32_t bands, uint32_t u,
                                          int lane) {
  int lo = 0, span = n;
  while (span > 1) {
    const int step = (span + 31) >> 5;
    const int idx = lo + lane * step;
    const bool le = idx < lo + span &&
                    static_cast<uint64_t>(pre[idx]) * bands <= static_cast<uint64_t>(u);
    const unsigned m = __ballot_sync(0xffffffffu, le);  // a prefix of the lanes, lane 0 set
    const int nlo = lo + (31 - __clz(m)) * step;
    span = min(step, lo + span - nlo);
    lo = nlo;
  }
  return lo;
}

// A split unit's part at the end of its pass A: its row maxima join the
// unit's words in global memory and the part is counted (release: after
// the maxima).
__device__ __forceinline__ void merge_part(uint32_t* w, const uint32_t* amax, bool count, int lane) {
#pragma unroll
  for (int qq = 0; qq < kQ; ++qq) {
    const uint32_t a = amax[lane + 32 * qq];
    if (a) atomicMax(w + lane + 32 * qq, a);
  }
  __syncwarp();
  if (lane == 0 && count) red_release_add(w + kTn, 1u);
}

// The scales of split unit v, once every part's maxima are in its words
// (the counter shows all parts: acquire); the unit's pass B may then start.
// Each part's read is counted too, and the last of them returns the words
// and the counter to zero.
__device__ __forceinline__ bool split_scales(Smem& s, const Params& p, uint32_t v, int lane) {
  Unit& U = s.unit[v % kUnits];
  uint32_t* w = p.split + static_cast<size_t>(U.sidx) * kSplitWords;
  const uint32_t parts = static_cast<uint32_t>(U.parts);
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    const uint32_t c = ld_acquire_u32(w + kTn);
    if (__all_sync(0xffffffffu, c >= parts)) break;
    if (ld_volatile_u32(p.err) != 0u || global_timer_ns() - t0 > p.timeout_ns) {
      if (lane == 0) atomicOr(p.err, kErrDepTimeout);
      return false;
    }
    __nanosleep(64);
  }
#pragma unroll
  for (int qq = 0; qq < kQ; ++qq) {
    const int r = lane + 32 * qq;
    const float sc = scale_from_amax_bits(ld_cg_u32(w + r), p.pow2);
    U.scale[r] = sc;
    if (U.part == 0 && U.n0 + r < p.N) p.scales[static_cast<size_t>(U.n0 + r) * p.G + U.g] = sc;
  }
  __syncwarp();
  if (lane == 0 && !U.hold) mbar_arrive(&s.u_amax[v % kUnits]);
  uint32_t old = 0;
  if (lane == 0) old = atom_add_acq_rel_gpu(w + kTn, 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old + 1u == 2u * parts) {
#pragma unroll
    for (int qq = 0; qq < kQ; ++qq) w[lane + 32 * qq] = 0u;
    __syncwarp();
    if (lane == 0) w[kTn] = 0u;
  }
  return true;
}

// Decodes units and publishes their descriptors; empty groups get their
// scales here and no descriptor.  The whole warp builds the group-end table
// and the call's decomposition first.  Without split units, units are
// claimed from the counter, kAhead ahead; with them, block b takes tickets
// b, b + grid, b + 2 grid, ... (the parts of a split unit are consecutive
// tickets, so they lie in two consecutive rounds of the grid, and every
// block's stream visits A of its next unit before B of the current one: a
// part's pass B waits only for passes A that no wait precedes).  One unit
// behind its publication, a split unit's scales are taken here.
template <bool kSplit>
__device__ __forceinline__ void descriptor_warp(Smem& s, const Params& p, int lane) {
  build_ends(p.offs, 0, p.G, p.Mg, s.ends, lane);
  __syncwarp();
  // parts per unit of each group; prefix sums of parts and of split groups
  // (only if some group is split at all)
  bool any_split = false;
  if (kSplit)
    for (int g = lane; g < p.G; g += 32)
      any_split |= parts_of(g ? s.ends[g - 1] : 0, s.ends[g]) > 1;
  if (!__any_sync(0xffffffffu, any_split)) {
    if (lane == 0) s.split_mode = 0;
    __syncwarp();
  } else {
    int32_t cp = 0, cs = 0, maxp = 1;
    for (int base = 0; base < p.G; base += 32) {
      const int g = base + lane;
      int32_t np = 0, sp = 0;
      if (g < p.G) {
        np = parts_of(g ? s.ends[g - 1] : 0, s.ends[g]);
        sp = np > 1 ? 1 : 0;
      }
      int32_t xp = np, xs = sp;  // inclusive scans
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t yp = __shfl_up_sync(0xffffffffu, xp, o);
        const int32_t ys = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) {
          xp += yp;
          xs += ys;
        }
      }
      if (g < p.G) {
        s.tb[g] = cp + xp - np;
        s.sb[g] = cs + xs - sp;
      }
      cp += __shfl_sync(0xffffffffu, xp, 31);
      cs += __shfl_sync(0xffffffffu, xs, 31);
      maxp = max(maxp, np);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
    // split only where a unit's parts fit one round of the grid, the
    // workspace has the words, and every block of the grid is resident (a
    // part waits for passes A that other blocks run): each block counts
    // its arrival, and the first to see all of them -- or the first to
    // give up waiting -- settles the decision for all (one CAS)
    bool split = !p.no_split && cs > 0 && maxp <= static_cast<int32_t>(gridDim.x) &&
                 static_cast<int64_t>(cs) * p.bands <= p.max_split;
    if (split) {
      uint32_t d = 0;
      if (lane == 0) {
        atomicAdd(p.ticket + 2, 1u);
        const uint64_t t0 = global_timer_ns();
        for (;;) {
          d = ld_acquire_u32(p.ticket + 3);
          if (d != 0u) break;
          if (ld_acquire_u32(p.ticket + 2) >= gridDim.x) {
            atomicCAS(p.ticket + 3, 0u, 1u);
          } else if (global_timer_ns() - t0 > kResidentWaitNs) {
            atomicCAS(p.ticket + 3, 0u, 2u);
          } else {
            __nanosleep(128);
          }
        }
      }
      split = __shfl_sync(0xffffffffu, d, 0) == 1u;
    }
    if (lane == 0) {
      s.tb[p.G] = cp;
      s.sb[p.G] = cs;
      s.split_mode = split ? 1 : 0;
    }
    __syncwarp();
  }
  const bool split_mode = kSplit && s.split_mode != 0;
  const uint32_t total = split_mode ? p.bands * static_cast<uint32_t>(s.tb[p.G]) : p.units;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t useq = 0;  // units published
  bool pend = false;  // unit useq - 1 is split: its scales are due
  // lane 0 claims units kAhead ahead, so that a claim's round trip to L2
  // overlaps the units before it
  uint32_t q[kAhead];
#pragma unroll
  for (int a = 0; a < kAhead; ++a)
    q[a] = split_mode ? blockIdx.x + a * gridDim.x : lane == 0 ? claim_ticket(p.ticket) : 0u;
  for (;;) {
    const uint32_t u = split_mode ? q[0] : __shfl_sync(0xffffffffu, q[0], 0);
#pragma unroll
    for (int a = 0; a + 1 < kAhead; ++a) q[a] = q[a + 1];
    if (split_mode)
      q[kAhead - 1] = q[kAhead - 2] + gridDim.x;
    else if (lane == 0 && u < total)
      q[kAhead - 1] = claim_ticket(p.ticket);
    int32_t grp = 0, n0 = -1, x0 = 0, lo = 0, hi = 0, nst = 0, sidx = -1, np = 1, part = 0;
    if (u < total) {  // else: publish the stop descriptor
      // group-major: the bands of a group are taken one after another, so
      // the 64-byte runs that neighbouring bands write into each row of A^T
      // reach L2 close together; a split unit's parts are consecutive
      uint32_t r = u;
      if (split_mode) {
        grp = find_group(s.tb, p.G, p.bands, u, lane);
        np = s.tb[grp + 1] - s.tb[grp];
        r = u - p.bands * static_cast<uint32_t>(s.tb[grp]);
        n0 = static_cast<int32_t>(r / static_cast<uint32_t>(np)) * kTn;
        part = static_cast<int32_t>(r % static_cast<uint32_t>(np));
      } else {
        grp = static_cast<int32_t>(u / p.bands);
        n0 = static_cast<int32_t>(u % p.bands) * kTn;
      }
      const int32_t s0 = grp ? s.ends[grp - 1] : 0, e0 = s.ends[grp];
      if (e0 == s0) {  // empty group: amax 0 for every row
        const float e = scale_from_amax_bits(0u, p.pow2);
#pragma unroll
        for (int qq = 0; qq < kQ; ++qq) {
          const int32_t n = n0 + lane + 32 * qq;
          if (n < p.N) p.scales[static_cast<size_t>(n) * p.G + grp] = e;
        }
        continue;
      }
      if (np > 1) {
        const int32_t w = windows_of(s0, e0);
        const int32_t wa = part * w / np, wb = (part + 1) * w / np;
        x0 = (s0 & ~7) + wa * kTm;
        lo = s0 - x0;  // below 0 past part 0
        hi = min(e0, (s0 & ~7) + wb * kTm) - x0;
        nst = wb - wa;
        sidx = s.sb[grp] * static_cast<int32_t>(p.bands) + n0 / kTn;
      } else {
        x0 = s0 & ~7;
        lo = s0 - x0;
        hi = e0 - x0;
        nst = (hi + kTm - 1) / kTm;
      }
    }
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
      if (kSplit) {
        U.sidx = sidx;
        U.parts = np;
        U.part = part;
      }
      U.x0 = x0;
      U.lo = lo;
      U.hi = hi;
      U.nst = nst;
      U.resident = nst <= kFit ? 1 : 0;
      U.hold = p.skip_arrival && u == 0u;
      U.a_done = 0u;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.u_full[us]);
    ++useq;
    // the previous unit's scales, now that this unit's pass A may run
    if (kSplit) {
      if (pend && !split_scales(s, p, useq - 2, lane)) return;
      pend = sidx >= 0;
    }
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
template <bool kSplit>
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
    if (kSplit && U.sidx >= 0) {
      // a part of a split unit: its maxima join the unit's words at once;
      // the descriptor warp takes the scales once every part is in
      merge_part(p.split + static_cast<size_t>(U.sidx) * kSplitWords, U.amax, !hold, lane);
      return true;
    }
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

template <bool kSplit>
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
      if (!pass_a<kSplit>(s, cu, hold, j, p, w, lane, wait_ns)) return;
      if (pending && !pass_b(s, pv, pv.first, j, p, w, lane, wait_ns)) return;
      pv = cu;
      pending = true;
    } else {
      if (pending && !pass_b(s, pv, pv.first, j, p, w, lane, wait_ns)) return;
      pending = false;
      g += static_cast<uint32_t>(cu.nst);
      if (!pass_a<kSplit>(s, cu, hold, j, p, w, lane, wait_ns)) return;
      const uint32_t base = g;  // the windows come again
      g += static_cast<uint32_t>(cu.nst);
      if (!pass_b(s, cu, base, j, p, w, lane, wait_ns)) return;
    }
  }
}

template <bool kSplit>
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
    descriptor_warp<kSplit>(s, p, lane);
  else if (warp == kLoaderWarp)
    loader_warp(s, &amap, p, lane);
  else
    consumer_warp<kSplit>(s, p, warp, lane);

  // The last block to finish returns the counters to zero, so that the next
  // call on this workspace may skip its clear (GQ_WORKSPACE_ZEROED); the
  // split words return to zero with their last read.  Every block gets
  // here, also after a bounded wait expired, and has made its last claim
  // before its arrival is counted.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int32_t clear = 0;
    if (atomicAdd(p.ticket + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.ticket, 0u);
      atomicExch(p.ticket + 1, 0u);
      if (kSplit) {
        // after an expired wait, split words may be left behind: clear them
        clear = ld_volatile_u32(p.err) != 0u ? 1 : 0;
        atomicExch(p.ticket + 2, 0u);
        atomicExch(p.ticket + 3, 0u);
      }
    }
    if (kSplit) s.clear_all = clear;
  }
  if (kSplit) {
    __syncthreads();
    if (s.clear_all)
      for (uint64_t i = threadIdx.x; i < p.split_words; i += blockDim.x) p.split[i] = 0u;
  }
}

// ---------------------------------------------------------------- host --
gq_status setup(DeviceInfo& info) {
  gq_status st = check_cuda(
      cudaFuncSetAttribute(rowwise_kernel<false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)),
      "rowwise_t: set shared memory size");
  if (st != GQ_OK) return st;
  st = check_cuda(cudaFuncSetAttribute(rowwise_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes)),
                  "rowwise_t: set shared memory size");
  if (st != GQ_OK) return st;
  int occ = 0;
  st = check_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &occ, rowwise_kernel<true>, kThreads, kSmemBytes),
                  "rowwise_t: occupancy");
  if (st != GQ_OK) return st;
  if (occ < 1) return fail(GQ_ERR_UNSUPPORTED, "rowwise_t kernel does not fit an SM");
  info.rowwise_ctas_per_sm = occ;
  return GQ_OK;
}

size_t workspace_bytes(int64_t N, int64_t Mg, int64_t G) {
  // a split unit's group has more than kSplitOver windows: at least
  // kSplitOver * kTm - 6 tokens (window 0 starts up to 7 tokens early)
  const int64_t bands = (N + kTn - 1) / kTn;
  const int64_t max_groups = std::min<int64_t>(G, Mg / (kSplitOver * kTm - 6));
  return kHeaderBytes + static_cast<size_t>(bands * max_groups) * kSplitWords * 4;
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
  // tickets: one per unit, or per part of a split unit; a part has at
  // least kFit / 2 windows and a group of s tokens at most s / kTm + 2, so
  // the groups give fewer than G + (Mg / kTm + 2 G) / (kFit / 2) parts
  const int64_t tickets = bands * (G + (Mg / kTm + 2 * static_cast<int64_t>(G)) / (kFit / 2));
  const int64_t max_ctas = static_cast<int64_t>(info.sm_count) * info.rowwise_ctas_per_sm;
  const int grid = static_cast<int>(tickets < max_ctas ? tickets : max_ctas);
  // the counter ends below tickets + (kAhead + 1) * grid
  if (tickets + (kAhead + 1) * static_cast<int64_t>(grid) >= (int64_t(1) << 32))
    return fail(GQ_ERR_UNSUPPORTED, "rowwise_t: (N / 64) x n_groups too large");
  const size_t ws_bytes = workspace_bytes(N, Mg, G);
  p.offs = offs;
  p.ticket = static_cast<uint32_t*>(ws);  // first word of the header
  p.split = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + kHeaderBytes);
  p.split_words = (ws_bytes - kHeaderBytes) / 4;
  p.max_split = static_cast<int32_t>(p.split_words / kSplitWords);
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
  p.no_split = dbg.no_split;
  p.pow2 = (flags & GQ_SCALE_POW2) != 0;

  if (!(flags & GQ_WORKSPACE_ZEROED)) {
    st = check_cuda(cudaMemsetAsync(ws, 0, ws_bytes, stream), "rowwise_t: clear the workspace");
    if (st != GQ_OK) return st;
  }
  // A plain launch: units are claimed in order by running blocks and never
  // wait for another block; split units are used only when the kernel has
  // found every block of the grid resident (at most one per SM).  The build
  // that can split is taken where groups average kSplitAvg tokens or more;
  // the other reads every unit of more than kFit windows twice, which at
  // shorter groups is faster.
  if (Mg / G >= kSplitAvg)
    rowwise_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(amap, p);
  else
    rowwise_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(amap, p);
  return check_cuda(cudaGetLastError(), "rowwise_t: launch");
}

}  // namespace rowwise
}  // namespace gq
