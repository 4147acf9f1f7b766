// gq_device.cuh -- device building blocks shared by the two quantization
// kernels: inline-PTX wrappers (mbarrier, TMA, cp.async, L2 policies, e4m3
// convert), bounded waits, the group-end table, tile headers and the ticket
// schedule.
//
// Execution model (both kernels).  A persistent grid, launched cooperatively
// so that every CTA is resident, of CTAs with three roles: a producer warp
// that fills a ring of 16 KB shared-memory stages by TMA, eight consumer
// warps that each work on every stage independently, and a signal lane.
//
// Work comes in super tiles of kSub stages (4 x 64 = 256 consecutive tokens
// of one column slab or row band).  Each super tile is visited twice: in
// phase A its |x| maxima are folded into per-(group, column) or per-(row,
// group) amax words with atomicMax; in phase B, once every phase-A super
// tile its amax words depend on is done, it is re-read, scaled and cast.
// Tiles that share amax words form a "dependency group" (a column slab for
// colwise, a row band for rowwise_t).  Tickets follow a fixed order in which
// phase A of dependency group d+L precedes phase B of group d (L = the lag),
// so that by the time phase B of a group comes up its phase-A tiles are long
// finished and its bytes still sit in L2 (loaded with evict_last): HBM sees
// one read of the input.  CTA c takes tickets c, c + grid, c + 2 grid, ...
// in that order.
//
// Per ticket the producer writes a context -- the super tile's header (its
// group segments) and, in phase B, the amax words of its first segments,
// copied with cp.async -- and loads the kSub stages.  Consumer warps carry
// per-segment state (maxima, scales) across the stages of a super tile, so
// the per-segment work -- reductions, atomics, divisions -- is paid once per
// 256 tokens.
//
// The signal lane runs an event loop with two jobs.  (1) Finished phase-A
// super tiles reach it through a small ring of shared-memory slots; it
// publishes them on the groups' done counters with release reductions, so
// the memory fence that publishing implies never stalls a consumer.  (2) It
// walks the CTA's own ticket sequence ahead of the producer and, for each
// dependency group a phase-B ticket will need, polls the group's done counter
// (acquire) and then raises a shared-memory flag (release); the producer
// waits on the flag, so the global round trips of dependency checks leave
// its critical path.
//
// Progress: all CTAs are resident and each takes its tickets in increasing
// order, so the smallest unfinished ticket can always advance -- its phase-A
// dependencies have smaller tickets -- and the schedule cannot deadlock; the
// signal lane never blocks on a dependency while completions wait in its
// ring.  Every wait is nonetheless bounded in time.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gq {

// -------------------------------------------------------------- constants --
constexpr float kFp8Max = 448.0f;  // fp8_dtype_max of the pages' kernel
constexpr float kEps = 1e-12f;     // EPS of the pages' kernel
constexpr int kMaxGroups = 1024;   // GQ_MAX_GROUPS

// error-word bits
constexpr unsigned kErrDepTimeout = 1u;   // a dependency-group wait expired
constexpr unsigned kErrMbarTimeout = 2u;  // an mbarrier wait expired

// ------------------------------------------------------------ tile header --
// Header of a super tile, written by the producer warp into a context and
// read by the consumers once the super tile's first stage is full.  Segment
// bounds are relative to lo.
template <int kMaxSeg>
struct alignas(16) TileHdr {
  int32_t phase;   // 0 = A (amax), 1 = B (scale + cast), -1 = stop
  int32_t dg;      // dependency group
  int32_t lo, hi;  // token range [lo, hi) of the super tile, clamped to the extent
  int32_t own_lo, own_hi;  // groups whose scales phase B of this tile writes
  int32_t nseg;            // nonempty group segments inside [lo, hi)
  int32_t nsub;            // stages (64-token sub-tiles) of the super tile
  int16_t seg_g[kMaxSeg];
  uint16_t seg_lo[kMaxSeg];
  uint16_t seg_hi[kMaxSeg];
};

// ---------------------------------------------------------- PTX wrappers --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Blocks for up to kSuspendNs (or until the phase completes) and reports
// whether the phase with the given parity has completed; a waiting thread
// sleeps instead of spinning, leaving issue slots to the working warps.
constexpr uint32_t kSuspendNs = 100000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Arrival that also announces `bytes` of asynchronous transfers to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// after `timeout_ns`, records kErrMbarTimeout and returns false.  Callers pass
// a limit several times the dependency-wait limit: a stage can only be late
// because a dependency wait is in progress, and those give up first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t timeout_ns,
                                          unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrMbarTimeout);
      return false;
    }
  }
  return true;
}

// 16-byte copy global -> shared (L2 only); reads src_bytes (0 or 16) and
// zero-fills the rest.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src,
                                            uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

// Makes the current phase of `bar` also wait for the completion of every
// cp.async this thread has issued (adds one pending arrival now, which the
// copies' completion performs).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m))
               : "memory");
}

// 2-D tiled TMA load global -> shared, completing on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map,
                                            int32_t x, int32_t y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
      "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled TMA store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map,
                                             const void* src, int32_t x,
                                             int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_"
      "hint [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (a following TMA store).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier among `nthreads` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so
// that they all take the same branch afterwards.
__device__ __forceinline__ bool named_bar_any(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ldmatrix x4 transposed: four 8x8 b16 matrices; lane l supplies the row
// address of row (l & 7) of matrix (l >> 3).  Lane l receives, for matrix j,
// the b16 pair at stored rows 2*(l&3) and 2*(l&3)+1 of column (l >> 2).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0,
                                              uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

// max(|a|, |b|) per bf16 lane (the sign of the result is the xor of the
// signs and is discarded by the caller).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest magnitude in a bf16x2 accumulator, as the fp32 bit pattern of the
// bf16 value (sign cleared).  For non-negative floats the bit patterns order
// like the values, so atomicMax on them is a max of amax.
__device__ __forceinline__ uint32_t amax_bits_of(uint32_t acc) {
  const uint32_t lo = acc & 0x7FFFu, hi = (acc >> 16) & 0x7FFFu;
  return (lo > hi ? lo : hi) << 16;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

// Two fp32 -> packed e4m3x2, round-to-nearest-even, saturating to +-448
// (`lo` lands in the low byte).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

// scale = 448 / max(amax, 1e-12), IEEE fp32 round-to-nearest division.
__device__ __forceinline__ float scale_from_amax_bits(uint32_t bits) {
  const float a = __uint_as_float(bits);
  return __fdiv_rn(kFp8Max, fmaxf(a, kEps));
}

__device__ __forceinline__ uint32_t ld_cg_u32(const uint32_t* p) {
  return __ldcg(p);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Release reduction: every write that happens before it (in this thread or,
// through synchronisation, in others) is visible to whoever acquires the
// counter value it produces.
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const unsigned* p) {
  return *reinterpret_cast<const volatile unsigned*>(p);
}

__device__ __forceinline__ void st_release_cta_s32(int32_t* p, int32_t v) {
  asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v)
               : "memory");
}

__device__ __forceinline__ int32_t ld_acquire_cta_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];"
               : "=r"(v)
               : "r"(smem_addr(p))
               : "memory");
  return v;
}

// ------------------------------------------------------ group-end table --
// ends[g] = min(extent, max(0, offs[0..g]))  -- the running maximum clamped
// to the extent.  Computed by one warp; `ends` is shared memory.
__device__ __forceinline__ void build_ends(const int32_t* __restrict__ offs,
                                           int n_groups, int32_t extent,
                                           int32_t* ends, int lane) {
  int32_t carry = 0;
  for (int base = 0; base < n_groups; base += 32) {
    const int g = base + lane;
    int32_t v = g < n_groups ? __ldg(offs + g) : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v = max(v, o);
    }
    v = max(v, carry);
    carry = __shfl_sync(0xffffffffu, v, 31);
    if (g < n_groups) ends[g] = min(v, extent);
  }
}

// The header of the tile with token range [lo, hi), built by one warp from
// the group-end table: the nonempty group segments in the tile and the range
// of groups whose scales the tile owns (the groups starting inside it; the
// last tile of the token extent also owns those starting at or after its
// start).  Groups are examined 32 at a time, from the block that holds the
// first group ending at or after lo (found by probing the block ends).
template <int kMaxSeg>
__device__ __forceinline__ void build_header_warp(TileHdr<kMaxSeg>& h,
                                                  const int32_t* ends, int n,
                                                  int32_t lo, int32_t hi,
                                                  bool last, int lane) {
  int b0 = 0;
  if (n > 32) {  // n <= 1024: one probe per block end
    const int pe = 32 * lane + 31;
    const unsigned m = __ballot_sync(0xffffffffu, pe >= n || ends[pe] >= lo);
    b0 = m ? __ffs(m) - 1 : 32;  // 32: no group ends at or after lo
  }
  const unsigned lt = (1u << lane) - 1u;
  int ns = 0, own_lo = n, own_hi = 0;
  for (int b = b0; 32 * b < n; ++b) {
    const int g = 32 * b + lane;
    const bool valid = g < n;
    const int32_t s = valid ? (g ? ends[g - 1] : 0) : 0;
    const int32_t e = valid ? ends[g] : 0;
    const bool seg = valid && s < hi && e > lo && s < e;
    const bool own = valid && s >= lo && (last || s < hi);
    const unsigned ms = __ballot_sync(0xffffffffu, seg);
    const unsigned mo = __ballot_sync(0xffffffffu, own);
    if (seg) {
      const int pos = ns + __popc(ms & lt);
      if (pos < kMaxSeg) {
        h.seg_g[pos] = static_cast<int16_t>(g);
        h.seg_lo[pos] = static_cast<uint16_t>(max(s, lo) - lo);
        h.seg_hi[pos] = static_cast<uint16_t>(min(e, hi) - lo);
      }
    }
    ns += __popc(ms);
    if (mo) {  // owned groups are contiguous
      own_lo = min(own_lo, 32 * b + __ffs(mo) - 1);
      own_hi = 32 * b + 32 - __clz(mo);
    }
    // starts are nondecreasing: once a start reaches hi, no later group has
    // a segment here, and only the last tile owns groups starting later
    if (!last && __ballot_sync(0xffffffffu, valid && s < hi) != 0xffffffffu) break;
  }
  if (lane == 0) {
    h.lo = lo;
    h.hi = hi;
    h.nseg = min(ns, kMaxSeg);
    h.own_lo = own_hi > 0 ? own_lo : 0;
    h.own_hi = own_hi;
  }
}

// ---------------------------------------------------------- ticket order --
struct Schedule {
  int32_t units;   // tiles per dependency group (>= 1)
  int32_t groups;  // dependency groups (>= 1)
  int32_t lag;     // 1 <= lag <= groups
};

// Tickets come in blocks of `units` (one dependency group, one phase), in
// the order
//   A(0) .. A(L-1), then A(L), B(0), A(L+1), B(1), ..., A(G-1), B(G-1-L),
//   then B(G-L) .. B(G-1).
// Block b holds tickets b * units .. b * units + units - 1; the unit is the
// ticket's place in its block.  Returns the phase (0 = A, 1 = B) and group.
__device__ __forceinline__ void decode_block(int32_t b, const Schedule& s,
                                             int32_t& phase, int32_t& dg) {
  if (b < s.lag) {
    phase = 0;
    dg = b;
    return;
  }
  const int32_t i = b - s.lag;
  const int32_t pairs = s.groups - s.lag;
  if (i < 2 * pairs) {
    phase = i & 1;
    dg = (i & 1) ? (i >> 1) : s.lag + (i >> 1);
  } else {
    phase = 1;
    dg = pairs + (i - 2 * pairs);
  }
}

// Walks tickets first, first + stride, first + 2 stride, ... as (block,
// unit) pairs without a division per step.
struct TicketWalk {
  int32_t block, unit;
  int32_t q, r;  // stride = q * units + r
  __device__ __forceinline__ TicketWalk(uint32_t first, uint32_t stride,
                                        int32_t units) {
    block = static_cast<int32_t>(first / static_cast<uint32_t>(units));
    unit = static_cast<int32_t>(first % static_cast<uint32_t>(units));
    q = static_cast<int32_t>(stride / static_cast<uint32_t>(units));
    r = static_cast<int32_t>(stride % static_cast<uint32_t>(units));
  }
  __device__ __forceinline__ void next(int32_t units) {
    block += q;
    unit += r;
    if (unit >= units) {
      unit -= units;
      ++block;
    }
  }
};

// Two fp32 products in one instruction, each rounded to nearest even like
// __fmul_rn (no flush of subnormals).
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"((static_cast<uint64_t>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x)),
        "l"((static_cast<uint64_t>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x)));
  return make_float2(__uint_as_float(static_cast<uint32_t>(d)),
                     __uint_as_float(static_cast<uint32_t>(d >> 32)));
}

// Eight bf16 (one 16-byte chunk) times eight scales -> eight e4m3 bytes
// (lowest column in the lowest byte).
__device__ __forceinline__ uint2 quant8(uint4 v, const float* sc) {
  const float2 p0 = mul_f32x2(make_float2(bf16_lo(v.x), bf16_hi(v.x)), make_float2(sc[0], sc[1]));
  const float2 p1 = mul_f32x2(make_float2(bf16_lo(v.y), bf16_hi(v.y)), make_float2(sc[2], sc[3]));
  const float2 p2 = mul_f32x2(make_float2(bf16_lo(v.z), bf16_hi(v.z)), make_float2(sc[4], sc[5]));
  const float2 p3 = mul_f32x2(make_float2(bf16_lo(v.w), bf16_hi(v.w)), make_float2(sc[6], sc[7]));
  return make_uint2(cvt_e4m3x2(p0.x, p0.y) | (cvt_e4m3x2(p1.x, p1.y) << 16),
                    cvt_e4m3x2(p2.x, p2.y) | (cvt_e4m3x2(p3.x, p3.y) << 16));
}

// ----------------------------------------------------------- signal ring --
// Consumer warps -> signal lane: one slot per finished phase-A tile.  A
// slot's full barrier counts one arrival per consumer warp (each after
// __syncwarp, which orders that warp's amax atomics before it); its empty
// barrier one arrival by the signal lane.
template <int kSlots>
struct SigRing {
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  int32_t dg[kSlots];
};

constexpr int32_t kSigEnd = -1;   // the consumers are done
constexpr int32_t kSigSkip = -2;  // a completion withheld (test hook)

template <int kSlots>
__device__ __forceinline__ void sig_init(SigRing<kSlots>& r, int consumer_warps) {
  for (int i = 0; i < kSlots; ++i) {
    mbar_init(&r.full[i], consumer_warps);
    mbar_init(&r.empty[i], 1);
  }
}

// Called by every consumer thread, in step (consumer warps never drift a
// whole ring apart: they meet at a barrier on every tile).  Hands over a
// finished phase-A tile of dependency group dg >= 0, kSigSkip or kSigEnd.
template <int kSlots>
__device__ __forceinline__ void sig_post(SigRing<kSlots>& r, int32_t dg, int t,
                                         int lane, uint32_t& seq,
                                         uint64_t timeout_ns, unsigned* err) {
  const int slot = static_cast<int>(seq % kSlots);
  const uint32_t par = (seq / kSlots) & 1u;
  ++seq;
  if (t == 0) {
    mbar_wait(&r.empty[slot], par ^ 1u, timeout_ns, err);
    r.dg[slot] = dg;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&r.full[slot]);
}

// Dependency readiness, written by the signal lane, read by the producer.
struct DepFlag {
  int32_t ready;  // every dependency group <= ready that this CTA needs is complete
  int32_t fail;   // 1 once the signal lane gave up waiting
};

// The next dependency group > last that a phase-B ticket of the walk needs
// (-1 when the walk is exhausted); the walk advances past that ticket.
__device__ __forceinline__ int32_t next_b_group(TicketWalk& tw, const Schedule& s,
                                                int32_t last) {
  const int32_t blocks = 2 * s.groups;
  for (; tw.block < blocks; tw.next(s.units)) {
    int32_t phase, dg;
    decode_block(tw.block, s, phase, dg);
    if (phase == 1 && dg > last) {
      tw.next(s.units);
      return dg;
    }
  }
  return -1;
}

// The signal lane's event loop.  (1) Takes the posted slots in order -- all
// that are posted each time round -- and adds each run of equal groups to
// that group's done counter with one release reduction.  (2) Walks the
// CTA's tickets ahead of the producer: for the next dependency group a
// phase-B ticket needs, probes its done counter (acquire) once per round and,
// when it has reached `target`, publishes the group in f.ready (release).
// It never blocks on a dependency, so this CTA's own completions keep
// flowing.  Returns after kSigEnd.  Gives up a dependency after timeout_ns
// (kErrDepTimeout, f.fail = 1) and the ring after idle_ns without any event.
template <int kSlots>
__device__ __forceinline__ void signal_lane(SigRing<kSlots>& r, DepFlag& f,
                                            uint32_t* done, const Schedule& sched,
                                            uint32_t target, uint64_t timeout_ns,
                                            uint64_t idle_ns, unsigned* err) {
  TicketWalk tw(blockIdx.x, gridDim.x, sched.units);
  int32_t want = next_b_group(tw, sched, -1);
  uint32_t seq = 0;
  uint64_t t_event = global_timer_ns(), t_want = t_event;
  for (;;) {
    bool progress = false, stop = false;
    int32_t run_dg = -1;
    uint32_t run = 0;
    for (int n = 0; n < kSlots; ++n) {
      const int slot = static_cast<int>(seq % kSlots);
      if (!mbar_test_wait(&r.full[slot], (seq / kSlots) & 1u)) break;
      const int32_t dg = r.dg[slot];
      mbar_arrive(&r.empty[slot]);
      ++seq;
      progress = true;
      if (dg == kSigEnd) {
        stop = true;
        break;
      }
      if (dg >= 0) {
        if (dg != run_dg) {
          if (run) red_release_add(done + run_dg, run);
          run_dg = dg;
          run = 0;
        }
        ++run;
      }
    }
    if (run) red_release_add(done + run_dg, run);
    if (stop) return;
    const uint64_t now = global_timer_ns();
    if (want >= 0) {
      if (ld_acquire_u32(done + want) >= target) {
        st_release_cta_s32(&f.ready, want);
        want = next_b_group(tw, sched, want);
        t_want = now;
        progress = true;
      } else if (ld_volatile_u32(err) != 0u || now - t_want > timeout_ns) {
        if (ld_volatile_u32(err) == 0u) atomicOr(err, kErrDepTimeout);
        st_release_cta_s32(&f.fail, 1);
        want = -1;
      }
    }
    if (progress) {
      t_event = now;
    } else {
      if (now - t_event > idle_ns) {
        atomicOr(err, kErrMbarTimeout);
        st_release_cta_s32(&f.fail, 1);
        return;
      }
      __nanosleep(want >= 0 ? 64 : 256);
    }
  }
}

// Producer side: waits until f.ready >= dg.  False when the signal lane gave
// up, an error is recorded elsewhere, or timeout_ns passes.
__device__ __forceinline__ bool wait_dep_flag(DepFlag& f, int32_t dg,
                                              uint64_t timeout_ns, unsigned* err) {
  if (ld_acquire_cta_s32(&f.ready) >= dg) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (ld_acquire_cta_s32(&f.ready) >= dg) return true;
    if (ld_acquire_cta_s32(&f.fail) != 0) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrDepTimeout);
      return false;
    }
    __nanosleep(32);
  }
}

}  // namespace gq
