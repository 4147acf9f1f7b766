// gq_device.cuh -- device building blocks shared by the two quantization
// kernels: inline-PTX wrappers (mbarrier, TMA, L2 policies, e4m3 convert),
// bounded waits, the group-end table, and the ticket schedule.
//
// Execution model (both kernels).  A persistent grid of CTAs, each with one
// producer warp and kConsumerWarps consumer warps.  The work is a list of
// tiles of the input.  A tile is visited twice: in phase A its |x| maxima
// are folded into per-(group, column) or per-(row, group) amax words with
// atomicMax; in phase B, once every phase-A tile its amax words depend on is
// done, it is re-read, scaled and cast.  Tiles that share amax words form a
// "dependency group" (a column slab for colwise, a row band for rowwise_t).
// Tickets are claimed with one atomicAdd per tile in a fixed order in which
// phase A of dependency group d+L precedes phase B of group d (L = the lag),
// so that by the time phase B of a group is claimed, its phase-A tiles are
// long finished and its bytes still sit in L2 (loaded with evict_last):
// HBM sees one read of the input.  Every CTA processes the tickets it claims
// in increasing order, so the smallest unfinished ticket can always make
// progress: the schedule cannot deadlock, even when not all CTAs are
// resident.  The wait for a dependency group is nonetheless bounded in time.
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
// Written by the producer lane into shared memory next to each stage; read by
// the consumers after the stage's full barrier completes.
template <int kMaxSeg>
struct alignas(16) TileHdr {
  int32_t phase;   // 0 = A (amax), 1 = B (scale + cast), -1 = no more work
  int32_t dg;      // dependency group
  int32_t lo, hi;  // token range [lo, hi) of the tile, clamped to the extent
  int32_t own_lo, own_hi;  // groups whose scales phase B of this tile writes
  int32_t nseg;            // nonempty group segments inside [lo, hi)
  int32_t last;            // 1 if the tile is the last of its group dim
  int32_t seg_g[kMaxSeg];
  int32_t seg_lo[kMaxSeg];  // relative to lo
  int32_t seg_hi[kMaxSeg];
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

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
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

__device__ __forceinline__ uint32_t ld_volatile_u32(const unsigned* p) {
  return *reinterpret_cast<const volatile unsigned*>(p);
}

// Waits until *counter >= target.  Bounded: after `timeout_ns` it records
// kErrDepTimeout and returns; it also returns at once when another block has
// already recorded an error, so one lost signal cannot stall every block for
// the full timeout.
__device__ __forceinline__ void wait_counter(const uint32_t* counter,
                                             uint32_t target,
                                             uint64_t timeout_ns,
                                             unsigned* err) {
  if (ld_acquire_u32(counter) >= target) return;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_u32(counter) < target) {
    if (ld_volatile_u32(err) != 0u) return;
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrDepTimeout);
      return;
    }
    __nanosleep(64);
  }
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

// First g in [0, n) with ends[g] > t (n if none).
__device__ __forceinline__ int first_end_above(const int32_t* ends, int n,
                                               int32_t t) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ends[mid] > t)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

// First g in [0, n) whose start (g ? ends[g-1] : 0) is >= t (n if none).
// Starts are nondecreasing in g.
__device__ __forceinline__ int first_start_at_or_above(const int32_t* ends,
                                                       int n, int32_t t) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int32_t st = mid ? ends[mid - 1] : 0;
    if (st >= t)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

// Fills the segment part of a tile header for the token range [lo, hi).
template <int kMaxSeg>
__device__ __forceinline__ void fill_segments(TileHdr<kMaxSeg>& h,
                                              const int32_t* ends, int n,
                                              int32_t lo, int32_t hi,
                                              bool last) {
  h.lo = lo;
  h.hi = hi;
  h.last = last ? 1 : 0;
  h.own_lo = first_start_at_or_above(ends, n, lo);
  h.own_hi = last ? n : first_start_at_or_above(ends, n, hi);
  int ns = 0;
  for (int g = first_end_above(ends, n, lo); g < n; ++g) {
    const int32_t s = g ? ends[g - 1] : 0;
    if (s >= hi) break;
    const int32_t a = max(s, lo), b = min(ends[g], hi);
    if (b > a && ns < kMaxSeg) {
      h.seg_g[ns] = g;
      h.seg_lo[ns] = a - lo;
      h.seg_hi[ns] = b - lo;
      ++ns;
    }
  }
  h.nseg = ns;
}

// ---------------------------------------------------------- ticket order --
struct Schedule {
  int32_t units;   // tiles per dependency group (>= 1)
  int32_t groups;  // dependency groups (>= 1)
  int32_t lag;     // 1 <= lag <= groups
};

struct Ticket {
  int32_t phase;  // 0 = A, 1 = B
  int32_t dg;     // dependency group
  int32_t unit;   // tile within the group
};

// Order of blocks of `units` tickets:
//   A(0) .. A(L-1), then A(L), B(0), A(L+1), B(1), ..., A(G-1), B(G-1-L),
//   then B(G-L) .. B(G-1).
__device__ __forceinline__ Ticket decode_ticket(uint32_t t, const Schedule& s) {
  Ticket k;
  const int32_t b = static_cast<int32_t>(t / static_cast<uint32_t>(s.units));
  k.unit = static_cast<int32_t>(t % static_cast<uint32_t>(s.units));
  if (b < s.lag) {
    k.phase = 0;
    k.dg = b;
    return k;
  }
  const int32_t i = b - s.lag;
  const int32_t pairs = s.groups - s.lag;
  if (i < 2 * pairs) {
    if ((i & 1) == 0) {
      k.phase = 0;
      k.dg = s.lag + (i >> 1);
    } else {
      k.phase = 1;
      k.dg = i >> 1;
    }
  } else {
    k.phase = 1;
    k.dg = pairs + (i - 2 * pairs);
  }
  return k;
}

}  // namespace gq
