// gq_device.cuh -- device building blocks shared by the two quantization
// kernels: inline-PTX wrappers (mbarrier, TMA, cp.async, L2 policies, e4m3
// convert), bounded waits, the group-end table, tile headers and the ticket
// schedule.
//
// Execution model (both kernels).  A persistent grid, launched cooperatively
// so that every CTA is resident, of CTAs with four roles: a context warp, a
// producer warp, consumer warps and a signal lane.
//
// Work comes in tickets: super tiles of kSub stages (256 consecutive tokens
// of one column slab or row band; a stage is 8 KB).  Each super tile is
// visited twice: in phase A the |x| maxima of its stages are folded into
// per-(group, column) or per-(row, group) amax words with atomicMax; in
// phase B, once every phase-A super tile its amax words depend on is done,
// it is re-read, scaled and cast.  Tiles that share amax words form a
// "dependency group" (a column slab for colwise, a row band for rowwise_t).
// Tickets are numbered in an order in which phase A of dependency group d+L
// precedes phase B of group d (L = the lag), so that by the time phase B of
// a group comes up its phase-A tiles are finished and its bytes still sit in
// L2 (loaded with evict_last): HBM sees one read of the input.  CTAs claim
// tickets from a global counter, so tickets are taken roughly in that order
// whatever the pace of each CTA.
//
// The context warp claims the CTA's tickets, one ahead, and writes a context
// per ticket into a small ring: first the ticket itself (published at once,
// so that the producer can start loading), then -- in phase B after the
// dependency group is complete -- the super tile's header (its group
// segments) and the amax words of its first segments, copied with cp.async.
// The producer warp follows the published tickets and loads their stages,
// in order, into a shared ring of stage buffers with TMA, tagging each with
// its ticket and place.  A consumer warp takes the next loaded stage (a
// shared counter), whichever ticket it belongs to, and does all the work of
// that stage alone, with no barrier among warps, so the per-stage
// bookkeeping (the waits, the segment walk, the scale divisions) is paid
// once per 8 KB.  In phase A the warps fold their stage maxima into the
// context with shared-memory atomics; the warp that finishes a super tile's
// last stage (an acquire-release counter in the context tells it) adds them
// to the global amax words, one atomicMax per (segment, column or row), and
// posts the super tile to the signal lane.
//
// The signal lane runs an event loop with two jobs.  (1) Finished phase-A
// super tiles reach it through a small ring of shared-memory slots; it
// publishes them on the groups' done counters with release reductions, so
// the memory fence that publishing implies never stalls a consumer.  (2)
// When the context warp waits for a dependency group, it polls the group's
// done counter (acquire) and then raises a shared-memory flag (release).
//
// Progress: all CTAs are resident and each processes its tickets in
// increasing order, so the smallest unfinished ticket can always advance --
// its phase-A dependencies have smaller tickets, claimed by running CTAs;
// within a CTA, stages are loaded and claimed in ticket order, so the stages
// of a ticket never wait behind those of a later one -- and the schedule
// cannot deadlock; the signal lane never blocks on a dependency while
// completions wait in its ring.  Every wait is nonetheless bounded in time.
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
// Header of a super tile, written by the context warp into a context and
// read by the consumers once the context is full.  Segment
// bounds are relative to lo.
template <int kMaxSeg>
struct alignas(16) TileHdr {
  int32_t phase;   // 0 = A (amax), 1 = B (scale + cast)
  int32_t dg;      // dependency group
  int32_t lo, hi;  // token range [lo, hi) of the super tile, clamped to the extent
  int32_t own_lo, own_hi;  // groups whose scales phase B of this tile writes
  int32_t nseg;            // nonempty group segments inside [lo, hi)
  int32_t nsub;            // stages of the super tile (a short last tile has fewer)
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

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;"
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

// Returns v unchanged, but the compiler must assume it changed here: the
// addresses of the pure shared loads below are derived from a value pinned
// after the stage's full barrier, so those loads cannot be issued before the
// wait.  (They cannot sink past the stage's release either: their values
// feed stores and atomics that precede it.)
__device__ __forceinline__ uint32_t pin(uint32_t v) {
  asm volatile("" : "+r"(v)::"memory");
  return v;
}

// Shared-memory atomic max (u32) and acquire-release add at CTA scope.
__device__ __forceinline__ void red_max_shared(uint32_t addr, uint32_t v) {
  asm volatile("red.shared.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_cta_shared(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// 16-byte shared load; pure, so the compiler may overlap it with other work.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(addr));
  return v;
}

// ldmatrix x4 transposed: four 8x8 b16 matrices; lane l supplies the row
// address of row (l & 7) of matrix (l >> 3).  Lane l receives, for matrix j,
// the b16 pair at stored rows 2*(l&3) and 2*(l&3)+1 of column (l >> 2).
// Pure, like lds128.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0,
                                              uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm(
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

// scale = 448 / max(amax, 1e-12), IEEE fp32 round-to-nearest division.
__device__ __forceinline__ float scale_from_amax_bits(uint32_t bits) {
  const float a = __uint_as_float(bits);
  return __fdiv_rn(kFp8Max, fmaxf(a, kEps));
}

// The same scale, rounded down to a power of two when `pow2` is set
// (round_scales_to_power_of_2): the scale is a positive normal fp32
// (448 / 3.4e38 > 2^-126), so clearing its mantissa leaves 2^floor(log2 s).
__device__ __forceinline__ float scale_from_amax_bits(uint32_t bits, bool pow2) {
  const float s = scale_from_amax_bits(bits);
  return pow2 ? __uint_as_float(__float_as_uint(s) & 0xFF800000u) : s;
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
// to the extent; with offs == nullptr, groups of `uniform` tokens each:
// ends[g] = min(extent, (g + 1) * uniform).  Computed by one warp; `ends` is
// shared memory.
__device__ __forceinline__ void build_ends(const int32_t* __restrict__ offs, int32_t uniform,
                                           int n_groups, int32_t extent,
                                           int32_t* ends, int lane) {
  if (offs == nullptr) {
    for (int g = lane; g < n_groups; g += 32)
      ends[g] = static_cast<int32_t>(
          min(static_cast<int64_t>(g + 1) * uniform, static_cast<int64_t>(extent)));
    return;
  }
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

// Four e4m3 bytes from two bf16x2 words w0 = (x0, x1), w1 = (x2, x3) and
// four scales: byte i = e4m3(fp32(x_i * s_i)), x0 in the lowest byte.  The
// products are IEEE fp32 multiplies rounded to nearest even (mul.rn.f32x2,
// no flush of subnormals); the cast rounds to nearest even and saturates to
// +-448 (cvt.rn.satfinite).  A bf16 value is the upper half of its fp32.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float s0,
                                          float s1, float s2, float s3) {
  uint32_t out;
  asm("{\n\t"
      ".reg .b32 a0, a1, a2, a3;\n\t"
      ".reg .b64 x0, x1, k0, k1, y0, y1;\n\t"
      ".reg .b16 h0, h1;\n\t"
      "shl.b32 a0, %1, 16;\n\t"
      "and.b32 a1, %1, 0xFFFF0000;\n\t"
      "shl.b32 a2, %2, 16;\n\t"
      "and.b32 a3, %2, 0xFFFF0000;\n\t"
      "mov.b64 x0, {a0, a1};\n\t"
      "mov.b64 x1, {a2, a3};\n\t"
      "mov.b64 k0, {%3, %4};\n\t"
      "mov.b64 k1, {%5, %6};\n\t"
      "mul.rn.f32x2 y0, x0, k0;\n\t"
      "mul.rn.f32x2 y1, x1, k1;\n\t"
      "mov.b64 {a0, a1}, y0;\n\t"
      "mov.b64 {a2, a3}, y1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, a3, a2;\n\t"
      "mov.b32 %0, {h0, h1};\n\t"
      "}"
      : "=r"(out)
      : "r"(w0), "r"(w1), "f"(s0), "f"(s1), "f"(s2), "f"(s3));
  return out;
}

// Eight bf16 (one 16-byte chunk) times eight scales -> eight e4m3 bytes
// (lowest column in the lowest byte).
__device__ __forceinline__ uint2 quant8(uint4 v, const float* sc) {
  return make_uint2(quant4(v.x, v.y, sc[0], sc[1], sc[2], sc[3]),
                    quant4(v.z, v.w, sc[4], sc[5], sc[6], sc[7]));
}

// ----------------------------------------------------------- signal ring --
// Consumer warps -> signal lane: one slot per finished phase-A super tile, taken
// in the order of a shared claim counter.  A slot's full barrier counts the
// posting warp's lane-0 arrival (after __syncwarp, which orders the warp's
// amax atomics before it); its empty barrier the signal lane's.  Only the
// warp that flushes a super tile's maxima posts it.
template <int kSlots>
struct SigRing {
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  int32_t dg[kSlots];
  uint32_t head;  // next slot sequence number to claim
};

constexpr int32_t kSigEnd = -1;   // a consumer warp is done
constexpr int32_t kSigSkip = -2;  // a completion withheld (test hook)

template <int kSlots>
__device__ __forceinline__ void sig_init(SigRing<kSlots>& r) {
  for (int i = 0; i < kSlots; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], 1);
  }
  r.head = 0;
}

// Called by a whole consumer warp: hands over a finished phase-A super tile of
// dependency group dg >= 0, kSigSkip or kSigEnd.  At most one post per warp
// is outstanding and there are fewer warps than slots, so a claimed slot's
// previous round is the one its empty barrier last completed.
template <int kSlots>
__device__ __forceinline__ void sig_post(SigRing<kSlots>& r, int32_t dg, int lane,
                                         uint64_t timeout_ns, unsigned* err) {
  __syncwarp();
  if (lane == 0) {
    const uint32_t seq = atomicAdd(&r.head, 1u);
    const int slot = static_cast<int>(seq % kSlots);
    mbar_wait(&r.empty[slot], ((seq / kSlots) & 1u) ^ 1u, timeout_ns, err);
    r.dg[slot] = dg;
    mbar_arrive(&r.full[slot]);
  }
  __syncwarp();
}

// Dependency readiness, shared by the context warp and the signal lane.
struct DepFlag {
  int32_t want;   // dependency group the context warp waits for (-1: none)
  int32_t ready;  // largest dependency group seen complete (-1: none)
  int32_t fail;   // 1 once the signal lane gave up waiting
};

__device__ __forceinline__ void dep_init(DepFlag& f) {
  f.want = -1;
  f.ready = -1;
  f.fail = 0;
}

// The signal lane's event loop.  (1) Takes the posted slots in order -- all
// that are posted each time round -- and adds each run of equal groups to
// that group's done counter with one release reduction.  (2) When the
// context warp waits for a dependency group (f.want), probes the group's done
// counter (acquire) once per round and, when it has reached `target`,
// publishes the group in f.ready (release).  It never blocks on a
// dependency, so this CTA's own completions keep flowing.  Returns after
// `posters` kSigEnd posts.  Gives up a dependency after timeout_ns
// (kErrDepTimeout, f.fail = 1) and the ring after idle_ns without any event.
template <int kSlots>
__device__ __forceinline__ void signal_lane(SigRing<kSlots>& r, DepFlag& f,
                                            uint32_t* done, uint32_t target, int posters,
                                            uint64_t timeout_ns, uint64_t idle_ns,
                                            unsigned* err) {
  uint32_t seq = 0;
  int ended = 0;
  int32_t ready = -1, watched = -1;
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
        if (++ended == posters) {
          stop = true;
          break;
        }
        continue;
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
    const int32_t want = *reinterpret_cast<volatile int32_t*>(&f.want);
    if (want != watched) {
      watched = want;
      t_want = now;
    }
    if (want > ready) {
      if (ld_acquire_u32(done + want) >= target) {
        ready = want;
        st_release_cta_s32(&f.ready, want);
        progress = true;
      } else if (ld_volatile_u32(err) != 0u || now - t_want > timeout_ns) {
        if (ld_volatile_u32(err) == 0u) atomicOr(err, kErrDepTimeout);
        st_release_cta_s32(&f.fail, 1);
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
      __nanosleep(want > ready ? 64 : 256);
    }
  }
}

// Context-warp side: announces dependency group dg and waits until it is
// complete.  False when the signal lane gave up, an error is recorded
// elsewhere, or timeout_ns passes.
__device__ __forceinline__ bool wait_dep_flag(DepFlag& f, int32_t dg,
                                              uint64_t timeout_ns, unsigned* err) {
  if (ld_acquire_cta_s32(&f.ready) >= dg) return true;
  *reinterpret_cast<volatile int32_t*>(&f.want) = dg;
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

// Tickets are claimed from a global counter, in increasing order; ticket t
// is unit t % units of block t / units.
__device__ __forceinline__ uint32_t claim_ticket(uint32_t* counter) {
  return atomicAdd(counter, 1u);
}

}  // namespace gq
