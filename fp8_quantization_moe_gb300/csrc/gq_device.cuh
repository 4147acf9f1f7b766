// gq_device.cuh -- device building blocks shared by the kernels of
// libgqfp8: inline-PTX wrappers (mbarrier, TMA loads and stores, cp.async,
// L2 cache policies, shared-memory loads, ldmatrix, bf16 |x| maxima, the
// e4m3 convert), bounded waits, the scale of an amax, and the group-end
// table.  Each kernel describes its own execution model in its file:
//   gq_colwise.cu  (group, slab) strips: resident strips in one pass, longer
//                  ones in two phases through L2, tickets from a counter;
//   gq_rowwise.cu  (row band, group) units held in shared memory between
//                  their two passes, one HBM read; a unit far longer than
//                  the ring is cut into parts that several blocks take;
//   gq_mxfp8.cu    a plain coalesced stream;
//   gq_wgrad.cu    a tcgen05 grouped GEMM.
//
// Every wait on another warp or block is bounded by %globaltimer: on expiry
// the waiter records a bit in the per-device error word and returns false,
// so a kernel ends instead of hanging and the host reports GQ_ERR_TIMEOUT.
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

// Tickets are claimed from a global counter, in increasing order.
__device__ __forceinline__ uint32_t claim_ticket(uint32_t* counter) {
  return atomicAdd(counter, 1u);
}

}  // namespace gq
