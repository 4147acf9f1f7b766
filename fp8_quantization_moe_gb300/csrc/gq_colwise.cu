// gq_colwise.cu -- colwise per-token-group fp8 e4m3 scaling on sm_103a.
//
// X (M, K) bf16 row-major; token groups are row ranges [s_g, e_g); one scale
// per (group, column).  This is the per-token-group scaling "along dim0" of
// pytorch/ao #2668 ("use smaller block sizes for per group scaling kernels
// to improve perf", intro); that page's lesson -- the grid was too small to
// fill the SMs -- is answered here by a persistent grid of one block per SM
// whose pipelines claim small pieces of work from global counters.
//
// Work is cut along the groups.  A strip is (group g, column slab d): the
// group's rows by kW = 128 columns; every scale of a strip depends on that
// strip alone.  A strip of at most kResRows = 320 rows is "resident": one
// block loads it once, folds its column maxima, computes its scales and
// casts it out of shared memory (one HBM read, no other block involved).  A
// longer strip is cut into tiles of kTileRows = 768 rows (fewer for small
// problems, so that every block gets several; the last tile of a strip
// shorter) and goes through two phases:
//   phase A -- a block folds a tile's column maxima, adds them to the
//     strip's amax words in global memory (one atomicMax per column) and
//     counts the tile on the strip's counter (a release reduction);
//   phase B -- in halves of a phase-A tile (kBSplit: so that a finished
//     strip is re-read by more blocks at once and leaves L2 sooner), a
//     block loads the rows again -- from L2: phase-A loads carry an L2
//     evict_last hint -- and, once the strip's counter shows all its
//     phase-A tiles (an acquire load), reads the strip's amax words,
//     computes its 128 scales (448 / max(amax, 1e-12), IEEE division) and
//     casts them.
//
// Each block runs two independent pipelines.  Both take work from global
// counters in the same order -- slab by slab, strips in group order, tiles
// in row order: the phase-one pipeline takes "items" (a resident strip, or
// a phase-A tile), the phase-B pipeline takes phase-B tiles.  Phase one
// never waits for other blocks, except that an item may not start before
// the phase-B tiles up to `limit` tiles behind it have been taken -- the
// phase-A data in flight, and so what L2 must hold until phase B re-reads
// it, stays bounded (`limit`: the longest strip's phase-B tile count plus
// 2.5 slabs of phase-B tiles, or 1.75 phase-A tiles per block where 2.5
// slabs come to less than 1.25 of them); `limit` exceeds the longest
// strip's phase-B tile count, so the strips of those phase-B tiles precede
// the item and are all claimed, and the wait always ends.  Phase B waits
// only for strips whose phase-A tiles are all claimed.  Claims are made by running blocks, in order, and each
// block works through its claims in order, so every wait ends whichever
// blocks are resident (the launch needs no co-residency).
//
// Block roles (22 warps).  Phase one: a scheduler warp claims items (one
// ahead) and publishes a context per item in a ring of two -- few, so
// that a claimed item is soon loaded and its strip soon complete; a
// producer warp loads each item's stages -- 32 rows x 128 columns, 8 KB,
// one TMA box -- into a ring of stage buffers; twelve consumer warps fold
// (and for resident strips cast) them.  Phase B: a scheduler warp claims
// tiles (two ahead) for a ring of two contexts; two scale warps, context
// i to warp i % 2, decode the tile into its context (the producer warp
// then loads it), wait for the strip and turn its amax words into the
// scales; four consumer warps cast.  Stage v of a pipeline's stream goes to
// its consumer warp v % 12 (phase one) or v % 4 (phase B).  Lane l of a
// consumer warp owns the 16-byte column chunk l % 16 (8 columns) of stage
// rows l / 16, l / 16 + 2, ...:
// every shared-memory access reads whole 256-byte rows (no swizzle
// needed), a warp store writes two 128-byte output rows.
//   fold: |x| folded with max.xorsign.abs.bf16x2, one shuffle joins the two
//     row halves, shared-memory atomics join the warps' maxima in the
//     context;
//   cast: each lane takes its chunk's eight scales from the context,
//     multiplies in IEEE fp32 (mul.rn.f32x2) and packs with
//     cvt.rn.satfinite.e4m3x2.
// While one warp builds the plan at the start, the producer warp prefetches
// the block's share of the first column slab's rows into L2 (TMA prefetches:
// no shared memory, nothing to wait for), so that the first items' loads,
// which the plan and the first claims delay by microseconds, find L2.
// The last phase-B read of a strip returns its amax words and counter to
// zero, and the last block to finish returns the work counters to zero, so
// a workspace is left ready for the next call.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace colwise {

constexpr int kRows = 32;                       // rows per stage (one TMA box)
constexpr int kTileStages = 24;                 // stages per two-phase tile (at most)
constexpr int kTileRows = kTileStages * kRows;  // rows per two-phase tile (at most)
constexpr int kResStages = 10;                  // a strip of up to this many stages is resident
constexpr int kResRows = kResStages * kRows;
constexpr int kTileStep = 8 * kRows;  // 256 rows: the phase-A tile ladder's step, the least tile
constexpr int kStages = 12;                     // stage ring of each pipeline
constexpr int kCtx = 2;                         // contexts of the phase-B pipeline
constexpr int kCtxA = 2;                        // contexts of the phase-one pipeline
constexpr int kAhead = 2;                       // phase-B claims made before they are needed
constexpr int kConsA = 12;                      // consumer warps of the phase-one pipeline
constexpr int kConsB = 4;                       // consumer warps of the phase-B pipeline
constexpr int kHelpers = 2;                     // phase-B context i: scale warp i % 2
// warps
constexpr int kConsA0 = 0;                      // 0 .. 11
constexpr int kConsB0 = kConsA;                 // 12 .. 15
constexpr int kProdA = kConsA + kConsB;         // 16
constexpr int kProdB = kProdA + 1;              // 17
constexpr int kSchedA = kProdA + 2;             // 18
constexpr int kSchedB = kProdA + 3;             // 19
constexpr int kScale0 = kProdA + 4;             // 20, 21
constexpr int kThreads = (kScale0 + kHelpers) * 32;
constexpr int kRowBytes = kW * 2;
constexpr int kStageBytes = kRows * kRowBytes;
constexpr int kBSplit = 2;  // phase-B tiles per phase-A tile (when they stay >= kTileStep rows)
constexpr int kWarmSlabs = 1;  // column slabs prefetched into L2 at the start
constexpr int kLeadQuarters = 10;  // phase-A lead: the longest strip + 2.5 slabs of phase-B tiles
constexpr int kShortLeadEighths = 14;  // the lead where slabs are short: 1.75 phase-A tiles per block
static_assert(kW == 128, "lane maps assume 128-column slabs");
static_assert(kResStages <= kStages, "a resident strip fits the ring");
static_assert(kStages % kConsA == 0 && kStages % kConsB == 0 && kStages <= 32,
              "stage waits stay within one phase");
static_assert(kCtx % kHelpers == 0, "a context always has the same scale warp");
static_assert(kCtxA <= kCtx, "both pipelines' contexts live in Pipe::ctx[kCtx]");

constexpr int32_t kTypeA = 0;     // phase A of a tile of a long strip
constexpr int32_t kTypeB = 1;     // phase B of a tile of a long strip
constexpr int32_t kTypeR = 2;     // a resident strip, both phases
constexpr int32_t kTypeStop = -1;

// workspace header words
constexpr int kHeadA = 0;       // phase-one items claimed
constexpr int kHeadB = 1;       // phase-B tiles claimed
constexpr int kBTaken = 2;      // phase-B tiles whose strip was found complete
constexpr int kFinished = 3;    // blocks finished
constexpr int kHeadWords = 4;

struct Ctx {
  int32_t type;
  uint32_t bidx;     // phase B: the tile claimed for this context
  int32_t g, d, k;   // group, slab, tile of the strip
  int32_t row0;      // first row of the tile
  int32_t rows;      // rows of the tile
  int32_t nsub;      // stages
  int32_t ntiles;    // tiles of the strip
  int32_t hold;      // test hook: the tile is never counted
  uint32_t f_cnt;    // stages folded
  alignas(16) uint32_t amax[kW];  // column maxima, fp32 bit patterns
  alignas(16) float scale[kW];
};

// The facts of a call that every block derives from the offsets.
struct Plan {
  int32_t nsl;       // column slabs
  int32_t ts;        // phase-one items per slab
  int32_t tb;        // phase-B tiles per slab
  int32_t limit;     // phase-A tiles allowed ahead of the phase-B tiles taken
  uint32_t total_a;  // phase-one items
  uint32_t total_b;  // phase-B tiles
};

// A pipeline's shared state.  The stage ring comes first and every Pipe
// starts on a 1024-byte boundary: TMA destinations must be aligned.
struct alignas(1024) Pipe {
  uint8_t tile[kStages][kStageBytes];
  Ctx ctx[kCtx];
  uint64_t full[kStages];   // stage loaded (TMA bytes)
  uint64_t empty[kStages];  // stage released
  uint64_t hdr[kCtx];       // context published (scheduler)
  uint64_t ready[kCtx];     // scales in the context
  uint64_t claimed[kCtx];   // phase B: tile claimed (scheduler)
  uint64_t freed[kCtx];     // context no longer needed
};

struct Smem {
  Pipe a, b;  // first members: 1024-byte aligned
  Plan plan;
  int32_t clear_all;
  int32_t ends[kMaxGroups];
  int32_t ip[kMaxGroups + 1];  // phase-one items of a slab before group g
  int32_t bp[kMaxGroups + 1];  // phase-B tiles of a slab before group g
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack
static_assert(sizeof(Pipe) % 1024 == 0 && offsetof(Smem, b) % 1024 == 0,
              "both stage rings start on 1024-byte boundaries");
static_assert(kStageBytes % 1024 == 0, "every stage buffer starts on a 1024-byte boundary");
static_assert(kSmemBytes <= 227 * 1024, "fits one SM's shared memory");

struct Params {
  const int32_t* offs;  // nullptr: groups of `uniform` rows each
  int32_t uniform;
  uint32_t* head;   // workspace header (kHeadWords counters)
  uint32_t* strip;  // per (group, slab): phase-A tiles counted + phase-B reads
  uint32_t* amax;   // (G, K) fp32 bit patterns
  uint8_t* out;
  float* scales;
  unsigned* err;
  int32_t M, K, G;
  int32_t tile_rows;   // rows per two-phase tile: kTileRows, or less for small problems
  int32_t tile_rows_b; // rows per phase-B tile: tile_rows / b_split
  int32_t b_split;     // phase-B tiles per phase-A tile (kBSplit, or 1)
  int32_t forced_lag;  // > 0: the phase-A lead in slabs of phase-B tiles
  uint64_t timeout_ns;
  uint64_t clear_words;  // 32-bit words from `strip` to the end of the workspace
  int32_t skip_arrival;
  bool pow2;       // scales rounded down to powers of two
  bool scales16;   // the scales base is 16-byte aligned (rows are: K % 16 == 0)
  bool two_phase;  // no resident strips (GQ_TWO_PHASE)
};

// Four scales of one row of the (G, K) scale matrix, at a column that is a
// multiple of 4.
__device__ __forceinline__ void store_scales4(const Params& p, int g, int32_t col, float4 v) {
  float* dst = p.scales + static_cast<size_t>(g) * p.K + col;
  if (p.scales16) {
    *reinterpret_cast<float4*>(dst) = v;
  } else {
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
  }
}

__device__ __forceinline__ float4 scales_of(uint4 a, bool pow2) {
  return make_float4(scale_from_amax_bits(a.x, pow2), scale_from_amax_bits(a.y, pow2),
                     scale_from_amax_bits(a.z, pow2), scale_from_amax_bits(a.w, pow2));
}

__device__ __forceinline__ uint4 ld_cg_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// 2-D tiled TMA prefetch of one box into L2 (no shared memory, nothing to
// wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.2d.L2.global.tile.L2::cache_hint [%0, {%1, %2}], %3;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}


// ------------------------------------------------------------------ plan --
// Built by one warp from the offsets: the group-end table, and per group its
// phase-one items and phase-B tiles in a slab (prefix sums ip, bp), then the
// item and tile counts and the throttle limit.
__device__ __forceinline__ void build_plan(Smem& s, const Params& p, int lane) {
  build_ends(p.offs, p.uniform, p.G, p.M, s.ends, lane);
  __syncwarp();
  int32_t ci = 0, cb = 0, maxnt = 0;
  for (int base = 0; base < p.G; base += 32) {
    const int g = base + lane;
    int32_t items = 0, bt = 0;
    if (g < p.G) {
      const int32_t rows = s.ends[g] - (g ? s.ends[g - 1] : 0);
      const int32_t nt = (rows + p.tile_rows - 1) / p.tile_rows;
      const int32_t ntb = (rows + p.tile_rows_b - 1) / p.tile_rows_b;
      const bool resident = rows <= kResRows && !p.two_phase;
      items = resident ? (rows > 0 ? 1 : 0) : nt;
      bt = resident ? 0 : ntb;
    }
    int32_t xi = items, xb = bt;  // inclusive scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t yi = __shfl_up_sync(0xffffffffu, xi, o);
      const int32_t yb = __shfl_up_sync(0xffffffffu, xb, o);
      if (lane >= o) {
        xi += yi;
        xb += yb;
      }
    }
    if (g < p.G) {
      s.ip[g] = ci + xi - items;
      s.bp[g] = cb + xb - bt;
    }
    ci += __shfl_sync(0xffffffffu, xi, 31);
    cb += __shfl_sync(0xffffffffu, xb, 31);
    maxnt = max(maxnt, bt);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxnt = max(maxnt, __shfl_xor_sync(0xffffffffu, maxnt, o));
  if (lane == 0) {
    s.ip[p.G] = ci;
    s.bp[p.G] = cb;
    const int32_t nsl = (p.K + kW - 1) / kW;
    // the lead: kLeadQuarters / 4 slabs of phase-B tiles, but never less
    // than about one phase-A tile per block in flight, which phase one needs
    // to keep every block busy (a slab of few tiles -- few rows, or uniform groups --
    // would otherwise starve it); where that floor binds, the lead is
    // counted in tiles per block, kShortLeadEighths / 8 of them, which
    // holds about as many bytes in L2 as 2.5 slabs of a 65536-row input
    const int64_t quarters = p.forced_lag > 0 ? 4 * static_cast<int64_t>(p.forced_lag) : kLeadQuarters;
    int64_t lead = quarters * cb / 4;
    if (p.forced_lag <= 0) {
      const int64_t per_block = static_cast<int64_t>(gridDim.x) * p.b_split;
      const int64_t floor_lead = 5 * per_block / 4;
      if (lead < floor_lead) lead = max(floor_lead, kShortLeadEighths * per_block / 8);
    }
    int64_t limit = static_cast<int64_t>(maxnt) + lead;
    if (limit > (int64_t(1) << 30)) limit = int64_t(1) << 30;
    s.plan.nsl = nsl;
    s.plan.ts = ci;
    s.plan.tb = cb;
    s.plan.limit = static_cast<int32_t>(limit);
    s.plan.total_a = static_cast<uint32_t>(static_cast<int64_t>(nsl) * ci);
    s.plan.total_b = static_cast<uint32_t>(static_cast<int64_t>(nsl) * cb);
  }
}

// Largest g in [0, n) with pre[g] <= j, for a nondecreasing pre with
// pre[0] <= j; a whole warp searches 32 probes at a time.
__device__ __forceinline__ int find_group(const int32_t* pre, int n, int32_t j, int lane) {
  int lo = 0, span = n;
  while (span > 1) {
    const int step = (span + 31) >> 5;
    const int idx = lo + lane * step;
    const bool le = idx < lo + span && pre[idx] <= j;
    const unsigned m = __ballot_sync(0xffffffffu, le);  // a prefix of the lanes, lane 0 set
    const int nlo = lo + (31 - __clz(m)) * step;
    span = min(step, lo + span - nlo);
    lo = nlo;
  }
  return lo;
}

// The context fields of tile k of strip (g, d).
__device__ __forceinline__ void fill_ctx(Ctx& c, const Smem& s, int32_t tile_rows, int32_t type,
                                         int g, int32_t d, int32_t k, int32_t hold) {
  const int32_t sg = g ? s.ends[g - 1] : 0;
  const int32_t row0 = sg + k * tile_rows;
  const int32_t rows = min(tile_rows, s.ends[g] - row0);
  c.type = type;
  c.g = g;
  c.d = d;
  c.k = k;
  c.row0 = row0;
  c.rows = rows;
  c.nsub = (rows + kRows - 1) / kRows;
  c.ntiles = (s.ends[g] - sg + tile_rows - 1) / tile_rows;
  c.hold = hold;
  c.f_cnt = 0;
}

// ----------------------------------------------------- phase-one scheduler --
__device__ __forceinline__ void sched_a(Smem& s, const Params& p, int lane) {
  Pipe& P = s.a;
  const Plan pl = s.plan;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  const uint32_t ts = static_cast<uint32_t>(pl.ts);
  // lane 0 claims one item ahead.  Items are claimed late on purpose: a
  // claimed item waits in this block until it is loaded, and the strip it
  // belongs to completes only when its last item is folded, so few items in
  // flight per block keep strips completing soon after their loads.
  uint32_t q0 = lane == 0 ? claim_ticket(p.head + kHeadA) : 0u;
  uint32_t taken = 0;  // phase-B tiles taken, as last read
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % kCtxA;
    Ctx& c = P.ctx[ci];
    const uint32_t fresh = ld_volatile_u32(p.head + kBTaken);  // used after the decode
    if (!mbar_wait(&P.freed[ci], ((seq / kCtxA) & 1) ^ 1u, wait_ns, p.err)) return;
    const uint32_t t = __shfl_sync(0xffffffffu, q0, 0);
    if (lane == 0 && t < pl.total_a) q0 = claim_ticket(p.head + kHeadA);
    if (t >= pl.total_a) {
      if (lane == 0) {
        c.type = kTypeStop;
        mbar_arrive(&P.hdr[ci]);
      }
      return;
    }
    const uint32_t d = t / ts, j = t - d * ts;
    const int g = find_group(s.ip, p.G, static_cast<int32_t>(j), lane);
    const int32_t k = static_cast<int32_t>(j) - s.ip[g];
    const bool resident = s.bp[g + 1] == s.bp[g];
    // the throttle: phase-B tiles before this item, less the limit, must be taken
    const int64_t before =
        static_cast<int64_t>(d) * pl.tb + s.bp[g] + (resident ? 0 : static_cast<int64_t>(k) * p.b_split);
    const int64_t need = before - pl.limit;
    taken = max(taken, fresh);
    if (need > static_cast<int64_t>(taken)) {
      const uint64_t t0 = global_timer_ns();
      for (;;) {
        taken = ld_volatile_u32(p.head + kBTaken);
        if (static_cast<int64_t>(taken) >= need) break;
        if (ld_volatile_u32(p.err) != 0u || global_timer_ns() - t0 > p.timeout_ns) {
          if (lane == 0) atomicOr(p.err, kErrDepTimeout);
          break;
        }
        __nanosleep(32);
      }
    }
    if (lane == 0)
      // a resident strip is one item, of up to kResRows rows (more than the
      // least tile)
      fill_ctx(c, s, resident ? kResRows : p.tile_rows, resident ? kTypeR : kTypeA, g,
               static_cast<int32_t>(d), k,
               p.skip_arrival && !resident && d == 0 && k == 0);
    sts128(smem_addr(&c.amax[4 * lane]), make_uint4(0, 0, 0, 0));
    __syncwarp();
    if (lane == 0) mbar_arrive(&P.hdr[ci]);
  }
}

// ------------------------------------------------------- phase-B scheduler --
// Claims phase-B tiles in order and hands each to the next context; the
// context's scale warp decodes it, so that several contexts are prepared
// side by side.
__device__ __forceinline__ void sched_b(Smem& s, const Params& p, int lane) {
  Pipe& P = s.b;
  const uint32_t total = s.plan.total_b;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t q[kAhead];
#pragma unroll
  for (int a = 0; a < kAhead; ++a) q[a] = lane == 0 ? claim_ticket(p.head + kHeadB) : 0u;
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % kCtx;
    if (!mbar_wait(&P.freed[ci], ((seq / kCtx) & 1) ^ 1u, wait_ns, p.err)) return;
    const uint32_t h = __shfl_sync(0xffffffffu, q[0], 0);
#pragma unroll
    for (int a = 0; a + 1 < kAhead; ++a) q[a] = q[a + 1];
    if (lane == 0 && h < total) q[kAhead - 1] = claim_ticket(p.head + kHeadB);
    const bool stop = h >= total;
    // a stop for each scale warp (each walks its own contexts); the
    // consumers and the producer stop at the first
    for (int j = 0; j < (stop ? kHelpers : 1); ++j) {
      const int cj = (seq + j) % kCtx;
      if (j > 0 && !mbar_wait(&P.freed[cj], (((seq + j) / kCtx) & 1) ^ 1u, wait_ns, p.err))
        return;
      if (lane == 0) {
        P.ctx[cj].bidx = h;
        mbar_arrive(&P.claimed[cj]);
      }
    }
    if (stop) return;
  }
}

// --------------------------------------------------------------- producer --
// Loads the stages of each published context of a pipeline, in order, lanes
// side by side.
template <int NCTX>
__device__ __forceinline__ void producer(Pipe& P, const CUtensorMap* xmap, const Params& p,
                                         int lane) {
  const uint64_t pol_keep = policy_evict_last();   // phase A: read again in phase B
  const uint64_t pol_once = policy_evict_first();  // phase B, resident strips
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t g = 0;  // stages loaded
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % NCTX;
    bool ok = mbar_wait(&P.hdr[ci], (seq / NCTX) & 1, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;
    const Ctx& c = P.ctx[ci];
    const int32_t type = c.type;
    if (type == kTypeStop) break;
    const int nsub = c.nsub;
    // at most kStages loads side by side: a slot's previous load must have
    // been issued (and its own wait passed) before a lane waits on its
    // release, or the barrier's parity could stand two phases behind
    for (int kb = 0; kb < nsub; kb += kStages) {
      const int k = kb + lane;
      if (lane < kStages && k < nsub) {
        const uint32_t L = g + static_cast<uint32_t>(k);
        const int st = static_cast<int>(L % kStages);
        ok = mbar_wait(&P.empty[st], ((L / kStages) & 1) ^ 1u, wait_ns, p.err);
        if (ok) {
          mbar_arrive_expect_tx(&P.full[st], kStageBytes);
          tma_load_2d(P.tile[st], xmap, c.d * kW, c.row0 + k * kRows, &P.full[st],
                      type == kTypeA ? pol_keep : pol_once);
        }
      }
      if (__any_sync(0xffffffffu, !ok)) break;
    }
    if (__any_sync(0xffffffffu, !ok)) break;
    g += static_cast<uint32_t>(nsub);
  }
  // no load may still be in flight when the block exits
  if (lane == 0)
    for (uint32_t L = g > static_cast<uint32_t>(kStages) ? g - kStages : 0u; L < g; ++L)
      mbar_wait(&P.full[L % kStages], (L / kStages) & 1, wait_ns, p.err);
}

// ------------------------------------------------------------- consumers --
// Column maxima of the first `rb` rows of a stage, joined into the context
// with shared-memory atomics.
__device__ __forceinline__ void fold_stage(Ctx& c, uint32_t tile, int rb, int lane) {
  const int kc = lane & 15;  // column chunk
  const int rl = lane >> 4;  // rows rl + 2 i
  const uint32_t base = tile + static_cast<uint32_t>(rl * kRowBytes + kc * 16);
  uint32_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
  if (rb == kRows) {
    uint4 v[kRows / 2];
#pragma unroll
    for (int i = 0; i < kRows / 2; ++i) v[i] = lds128(base + i * 2 * kRowBytes);
#pragma unroll
    for (int i = 0; i < kRows / 2; ++i) {
      acc0 = absmax_bf16x2(acc0, v[i].x);
      acc1 = absmax_bf16x2(acc1, v[i].y);
      acc2 = absmax_bf16x2(acc2, v[i].z);
      acc3 = absmax_bf16x2(acc3, v[i].w);
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < kRows / 2; ++i) {
      if (rl + 2 * i < rb) {
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
  const uint32_t dst = smem_addr(&c.amax[8 * kc + 4 * rl]);
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (m[e]) red_max_shared(dst + 4 * e, m[e]);
}

// The scaled cast of the first `rb` rows of stage v of the context's tile.
__device__ __forceinline__ void cast_stage(const Ctx& c, int v, uint32_t tile, int rb,
                                           const Params& p, int lane) {
  const int kc = lane & 15;  // column chunk
  const int rl = lane >> 4;  // rows rl + 2 i
  const int32_t c8 = c.d * kW + 8 * kc;
  if (c8 >= p.K) return;  // K % 16 == 0: a chunk is wholly inside or outside
  const float4 sa = *reinterpret_cast<const float4*>(&c.scale[8 * kc]);
  const float4 sb = *reinterpret_cast<const float4*>(&c.scale[8 * kc + 4]);
  const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
  const uint32_t base = tile + static_cast<uint32_t>(rl * kRowBytes + kc * 16);
  const size_t K2 = 2 * static_cast<size_t>(p.K);
  uint8_t* obase = p.out + static_cast<size_t>(c.row0 + v * kRows + rl) * p.K + c8;
  if (rb == kRows) {
    // loads first, then the casts and stores: sixteen independent chains
    uint4 x[kRows / 2];
#pragma unroll
    for (int i = 0; i < kRows / 2; ++i) x[i] = lds128(base + i * 2 * kRowBytes);
#pragma unroll
    for (int i = 0; i < kRows / 2; ++i)
      __stcs(reinterpret_cast<uint2*>(obase + i * K2), quant8(x[i], sc));
  } else {
#pragma unroll 1
    for (int i = 0; i < kRows / 2; ++i)
      if (rl + 2 * i < rb)
        __stcs(reinterpret_cast<uint2*>(obase + i * K2), quant8(lds128(base + i * 2 * kRowBytes), sc));
  }
}

// Waits until stage load L of a pipeline is in place.  Stages are released
// out of order, so the load kStages before L may not be consumed yet and
// the full barrier would still show its round: its release comes first.
// (Loads L - kStages and L - 2 kStages belong to the same consumer warp --
// kStages is a multiple of the consumer count -- which released them in order, so the
// empty barrier is never two phases behind here.)
__device__ __forceinline__ bool wait_stage(Pipe& P, uint32_t L, uint64_t wait_ns, unsigned* err) {
  const int st = static_cast<int>(L % kStages);
  bool ok = mbar_wait(&P.empty[st], ((L / kStages) & 1) ^ 1u, wait_ns, err);
  if (ok) ok = mbar_wait(&P.full[st], (L / kStages) & 1, wait_ns, err);
  return ok;
}

// Phase-one consumer warp w: folds its stages of each item; the warp that
// folds an item's last stage pushes a phase-A tile's maxima to the strip's
// amax words, or turns a resident strip's maxima into its scales; resident
// strips are then cast from the same stages, after all their folds.
__device__ __forceinline__ void consumer_a(Smem& s, const Params& p, int w, int lane) {
  Pipe& P = s.a;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t g = 0;  // stages of the stream so far (the producer's count)
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % kCtxA;
    const uint32_t par = (seq / kCtxA) & 1;
    bool ok = mbar_wait(&P.hdr[ci], par, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) return;
    Ctx& c = P.ctx[ci];
    const int32_t type = c.type;
    if (type == kTypeStop) return;
    const int nsub = c.nsub;
    const int v0 = (w + kConsA - static_cast<int>(g % kConsA)) % kConsA;
    uint32_t mine = 0;
    for (int v = v0; v < nsub; v += kConsA) {
      ok = wait_stage(P, g + v, wait_ns, p.err);
      if (__any_sync(0xffffffffu, !ok)) return;
      const uint32_t tile = pin(smem_addr(P.tile[(g + v) % kStages]));
      fold_stage(c, tile, min(kRows, c.rows - v * kRows), lane);
      if (type == kTypeA) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&P.empty[(g + v) % kStages]);
      }
      ++mine;
    }
    if (mine > 0) {
      __syncwarp();
      uint32_t prev = 0;
      if (lane == 0) prev = atom_add_acq_rel_cta_shared(smem_addr(&c.f_cnt), mine);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev + mine == static_cast<uint32_t>(nsub)) {  // the item's last stage folded
        __syncwarp();
        const uint4 a = lds128(smem_addr(&c.amax[4 * lane]));
        const int32_t col = c.d * kW + 4 * lane;
        if (type == kTypeA) {
          if (col < p.K) {
            uint32_t* dst = p.amax + static_cast<size_t>(c.g) * p.K + col;
            if (a.x) atomicMax(dst, a.x);
            if (a.y) atomicMax(dst + 1, a.y);
            if (a.z) atomicMax(dst + 2, a.z);
            if (a.w) atomicMax(dst + 3, a.w);
          }
        } else {
          const float4 sc = scales_of(a, p.pow2);
          *reinterpret_cast<float4*>(&c.scale[4 * lane]) = sc;
          if (col < p.K) store_scales4(p, c.g, col, sc);
        }
        __syncwarp();
        if (lane == 0) {
          if (type == kTypeA && !c.hold)  // count the tile (release: after the maxima)
            red_release_add(p.strip + static_cast<size_t>(c.g) * s.plan.nsl + c.d, 1u);
          mbar_arrive(&P.ready[ci]);
        }
      }
      if (type == kTypeR) {
        ok = mbar_wait(&P.ready[ci], par, wait_ns, p.err);
        if (__any_sync(0xffffffffu, !ok)) return;
        for (int v = v0; v < nsub; v += kConsA) {
          const uint32_t tile = pin(smem_addr(P.tile[(g + v) % kStages]));
          cast_stage(c, v, tile, min(kRows, c.rows - v * kRows), p, lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(&P.empty[(g + v) % kStages]);
        }
      }
    }
    g += static_cast<uint32_t>(nsub);
    __syncwarp();
    if (lane == 0) mbar_arrive(&P.freed[ci]);
  }
}

// Phase-B consumer warp w: casts its stages of each tile.
__device__ __forceinline__ void consumer_b(Smem& s, const Params& p, int w, int lane) {
  Pipe& P = s.b;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  uint32_t g = 0;
  for (int32_t seq = 0;; ++seq) {
    const int ci = seq % kCtx;
    const uint32_t par = (seq / kCtx) & 1;
    bool ok = mbar_wait(&P.hdr[ci], par, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) return;
    const Ctx& c = P.ctx[ci];
    if (c.type == kTypeStop) return;
    const int nsub = c.nsub;
    const int v0 = (w + kConsB - static_cast<int>(g % kConsB)) % kConsB;
    if (v0 < nsub) {
      ok = mbar_wait(&P.ready[ci], par, wait_ns, p.err);
      if (__any_sync(0xffffffffu, !ok)) return;
      for (int v = v0; v < nsub; v += kConsB) {
        ok = wait_stage(P, g + v, wait_ns, p.err);
        if (__any_sync(0xffffffffu, !ok)) return;
        const uint32_t tile = pin(smem_addr(P.tile[(g + v) % kStages]));
        cast_stage(c, v, tile, min(kRows, c.rows - v * kRows), p, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&P.empty[(g + v) % kStages]);
      }
    }
    g += static_cast<uint32_t>(nsub);
    __syncwarp();
    if (lane == 0) mbar_arrive(&P.freed[ci]);
  }
}

// ------------------------------------------------------------------ scale --
// The strip's last phase-B read returns its amax words and counter to zero:
// the counter ends at the strip's phase-A tiles plus its phase-B tiles
// (every phase-A tile, then every phase-B read).  A read's atomic is
// issued with it and its result examined one phase-B context later, so that
// its round trip is off the path.
struct StripRead {
  uint32_t* word = nullptr;
  uint32_t* am = nullptr;  // this lane's four amax words (nullptr: outside K)
  uint32_t target = 0;
  uint32_t old = 0;        // lane 0: the counter before this read
};

__device__ __forceinline__ void finish_read(StripRead& r, int lane) {
  if (r.word == nullptr) return;
  const uint32_t old = __shfl_sync(0xffffffffu, r.old, 0);
  if (old + 1u == r.target) {
    if (r.am != nullptr) *reinterpret_cast<uint4*>(r.am) = make_uint4(0, 0, 0, 0);
    if (lane == 0) *r.word = 0u;
  }
  r.word = nullptr;
}

// Scale warp i prepares phase-B contexts i, i + kHelpers, ...: it decodes
// the claimed tile into the context, waits until the strip's counter shows
// all its phase-A tiles (acquire), publishes the context (the producer then
// loads the tile) and turns the strip's amax words into its scales; the
// strip's first tile writes them out.
__device__ __forceinline__ void scale_warp(Smem& s, const Params& p, int i, int lane) {
  Pipe& P = s.b;
  const Plan pl = s.plan;
  const uint64_t wait_ns = 4 * p.timeout_ns;
  // empty groups: no rows, amax 0 -- their scales, spread over the blocks
  const float e = scale_from_amax_bits(0u, p.pow2);
  for (int g = i; g < p.G; g += kHelpers) {
    if (s.ends[g] != (g ? s.ends[g - 1] : 0)) continue;
    for (int32_t col = (blockIdx.x * 32 + lane) * 4; col < p.K; col += gridDim.x * 128)
      store_scales4(p, g, col, make_float4(e, e, e, e));
  }
  StripRead pend;
  for (int32_t seq = i;; seq += kHelpers) {
    const int ci = seq % kCtx;
    const uint32_t par = (seq / kCtx) & 1;
    bool ok = mbar_wait(&P.claimed[ci], par, wait_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;
    Ctx& c = P.ctx[ci];
    const uint32_t h = c.bidx;
    if (h >= pl.total_b) {
      if (lane == 0) {
        c.type = kTypeStop;
        mbar_arrive(&P.hdr[ci]);
      }
      break;
    }
    const uint32_t d = h / static_cast<uint32_t>(pl.tb);
    const uint32_t j = h - d * static_cast<uint32_t>(pl.tb);
    const int g = find_group(s.bp, p.G, static_cast<int32_t>(j), lane);
    if (lane == 0)
      fill_ctx(c, s, p.tile_rows_b, kTypeB, g, static_cast<int32_t>(d), static_cast<int32_t>(j) - s.bp[g],
               0);
    __syncwarp();
    // the tile is published (and loaded) only once its strip is complete:
    // loaded earlier, it could come from HBM ahead of phase A, and it would
    // hold stage buffers while it waits
    uint32_t* word = p.strip + static_cast<size_t>(g) * pl.nsl + d;
    const int32_t strip_rows = s.ends[g] - (g ? s.ends[g - 1] : 0);
    const uint32_t target = static_cast<uint32_t>((strip_rows + p.tile_rows - 1) / p.tile_rows);
    const uint32_t reads = static_cast<uint32_t>(c.ntiles);  // phase-B tiles of the strip
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      const uint32_t v = ld_acquire_u32(word);
      if (__all_sync(0xffffffffu, v >= target)) break;
      if (ld_volatile_u32(p.err) != 0u || global_timer_ns() - t0 > p.timeout_ns) {
        if (lane == 0) atomicOr(p.err, kErrDepTimeout);
        break;  // the kernel still finishes; the call reports GQ_ERR_TIMEOUT
      }
      __nanosleep(32);
    }
    if (lane == 0) {
      mbar_arrive(&P.hdr[ci]);
      atomicAdd(p.head + kBTaken, 1u);
    }
    const int32_t col = static_cast<int32_t>(d) * kW + 4 * lane;
    uint32_t* am = p.amax + static_cast<size_t>(g) * p.K + col;
    const uint4 a = col < p.K ? ld_cg_v4(am) : make_uint4(0, 0, 0, 0);
    const float4 sc = scales_of(a, p.pow2);
    *reinterpret_cast<float4*>(&c.scale[4 * lane]) = sc;
    if (c.k == 0 && col < p.K) store_scales4(p, g, col, sc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&P.ready[ci]);
    // count this read (acquire-release: every lane's amax read is ordered
    // before it), then settle the previous one
    uint32_t old = 0;
    if (lane == 0) old = atom_add_acq_rel_gpu(word, 1u);
    finish_read(pend, lane);
    pend.word = word;
    pend.am = col < p.K ? am : nullptr;
    pend.target = target + reads;  // the counter's final value
    pend.old = old;
    __syncwarp();
    if (lane == 0) mbar_arrive(&P.freed[ci]);
  }
  finish_read(pend, lane);
}

__global__ void __launch_bounds__(kThreads, 1)
    colwise_kernel(const __grid_constant__ CUtensorMap xmap, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    Pipe* pipes[2] = {&s.a, &s.b};
    for (Pipe* P : pipes) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&P->full[i], 1);
        mbar_init(&P->empty[i], 1);
      }
      for (int i = 0; i < kCtx; ++i) {
        mbar_init(&P->hdr[i], 1);
        mbar_init(&P->ready[i], 1);
        mbar_init(&P->claimed[i], 1);
      }
    }
    for (int i = 0; i < kCtx; ++i) {
      mbar_init(&s.a.freed[i], kConsA);
      mbar_init(&s.b.freed[i], kConsB + 1);  // + the context's scale warp
    }
    fence_mbar_init();
  }
  if (warp == kSchedA) build_plan(s, p, lane);
  if (warp == kProdA) {
    if (lane == 0) prefetch_tensormap(&xmap);
    // while the plan is built: this block's share of the first kWarmSlabs
    // column slabs, the first items' rows, prefetched into L2
    const int32_t per = (p.M + static_cast<int32_t>(gridDim.x) - 1) / static_cast<int32_t>(gridDim.x);
    const int32_t r0 = static_cast<int32_t>(blockIdx.x) * per;
    const int32_t r1 = min(r0 + per, p.M);
    const uint64_t pol = policy_evict_last();
    for (int d = 0; d < kWarmSlabs && d * kW < p.K; ++d)
      for (int32_t r = r0 + lane * kRows; r < r1; r += 32 * kRows)
        tma_prefetch_2d(&xmap, d * kW, r, pol);
  }
  __syncthreads();

  if (warp < kConsB0)
    consumer_a(s, p, warp - kConsA0, lane);
  else if (warp < kProdA)
    consumer_b(s, p, warp - kConsB0, lane);
  else if (warp == kProdA)
    producer<kCtxA>(s.a, &xmap, p, lane);
  else if (warp == kProdB)
    producer<kCtx>(s.b, &xmap, p, lane);
  else if (warp == kSchedA)
    sched_a(s, p, lane);
  else if (warp == kSchedB)
    sched_b(s, p, lane);
  else
    scale_warp(s, p, warp - kScale0, lane);

  // The last block to finish returns the header counters to zero (every
  // block has made its last claim before it is counted); if a wait gave up
  // anywhere, it also clears the strip counters and amax words, which a
  // cut-short launch may have left behind.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int32_t clear = 0;
    if (atomicAdd(p.head + kFinished, 1u) == gridDim.x - 1) {
      clear = ld_volatile_u32(p.err) != 0u ? 1 : 0;
      for (int i = 0; i < kHeadWords; ++i) atomicExch(p.head + i, 0u);
    }
    s.clear_all = clear;
  }
  __syncthreads();
  if (s.clear_all)
    for (uint64_t i = threadIdx.x; i < p.clear_words; i += blockDim.x) p.strip[i] = 0u;
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
  // items and tiles are counted in 32 bits: at most one item per kTileStep
  // rows or group, per slab
  const int64_t items = ((K + kW - 1) / kW) * ((M + kTileStep - 1) / kTileStep + G);
  if (items >= (int64_t(1) << 31))
    return fail(GQ_ERR_UNSUPPORTED, "colwise: (M / 256 + n_groups) x (K / 128) too large");
  CUtensorMap xmap;
  gq_status st = encode_tiled_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(x), static_cast<uint64_t>(K),
                                 static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(K) * 2, kW, kRows,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;

  const WorkspaceLayout L = colwise_workspace(K, G);
  uint8_t* w = static_cast<uint8_t*>(ws);
  Params p;
  p.offs = offs;
  p.uniform = uniform;
  p.head = reinterpret_cast<uint32_t*>(w);
  p.strip = reinterpret_cast<uint32_t*>(w + L.counters);
  p.amax = reinterpret_cast<uint32_t*>(w + L.amax);
  p.out = static_cast<uint8_t*>(out);
  p.scales = scales;
  p.err = info.err_word;
  p.M = M;
  p.K = K;
  p.G = G;
  // the largest tile that still gives every block about four tiles per phase
  const int64_t max_ctas = static_cast<int64_t>(info.sm_count) * info.colwise_ctas_per_sm;
  p.tile_rows = kTileStep;
  for (int32_t rows = kTileRows; rows > kTileStep; rows -= kTileStep)
    if (((K + kW - 1) / kW) * static_cast<int64_t>(M) / rows >= 4 * max_ctas) {
      p.tile_rows = rows;
      break;
    }
  p.b_split = p.tile_rows % kBSplit == 0 && p.tile_rows / kBSplit >= kTileStep ? kBSplit : 1;
  p.tile_rows_b = p.tile_rows / p.b_split;
  p.forced_lag = dbg.lag[GQ_KIND_COLWISE];
  p.timeout_ns = dbg.timeout_ns;
  p.clear_words = (L.total - L.counters) / 4;
  p.skip_arrival = dbg.skip_arrival;
  p.pow2 = (flags & GQ_SCALE_POW2) != 0;
  p.scales16 = (reinterpret_cast<uintptr_t>(scales) & 15) == 0;
  p.two_phase = (flags & GQ_TWO_PHASE) != 0;

  const int grid = static_cast<int>(items < max_ctas ? items : max_ctas);
  if (!(flags & GQ_WORKSPACE_ZEROED)) {
    st = check_cuda(cudaMemsetAsync(ws, 0, L.total, stream), "colwise: clear workspace");
    if (st != GQ_OK) return st;
  }
  // A plain launch: blocks need not be resident together.  Every wait is on
  // work that a running block has claimed -- items, tiles and phase-B reads
  // are claimed from counters in order, and each block works through its
  // claims in order -- so the kernel progresses whichever blocks run.
  colwise_kernel<<<grid, kThreads, kSmemBytes, stream>>>(xmap, p);
  return check_cuda(cudaGetLastError(), "colwise: launch");
}

}  // namespace colwise
}  // namespace gq
