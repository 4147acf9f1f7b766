// gq_wgrad.cu -- grouped grad_weight GEMM from the two quantized operands,
// on the sm_103a tensor cores (tcgen05, TMEM accumulators, TMA operands).
//
// The MoE backward pass needs, per token group g = [s_g, e_g) (pytorch/ao
// #2668, MoE fp8 training test: grad_weight = grad_output_t @ input),
//   out[g][n][k] = sum over t in g of (qa_t[t][n] / sa[n][g]) * (qx[t][k] / sx[g][k])
// where qa_t (T, N) e4m3 row-major is the rowwise_t result (grad_output_t as
// a column-major operand) with scales sa (N, G), and qx (T, K) e4m3 row-major
// is the colwise result of the layer input with scales sx (G, K).  The
// scales are constant over a group's tokens, so the tensor cores form the
// plain e4m3 sums and the epilogue divides once:
//   out[g][n][k] = bf16( acc[n][k] * (1 / sa[n][g]) * (1 / sx[g][k]) ).
//
// Tiles are (group, 128 rows n, 256 columns k); a persistent grid takes them
// in a fixed order, each block every gridDim-th.  Warp roles:
//   warp 0 (one lane): TMA loads of the tile's token chunks -- 128 tokens x
//     128 n of qa_t and 2 x (128 tokens x 128 k) of qx, 48 KB, 128-byte
//     swizzle; a group's last chunk only as many 32-token slices as it
//     needs -- into a ring of kStages stages;
//   warp 1: allocates the 512 TMEM columns (two accumulators of 256 fp32
//     columns, so that a tile's epilogue overlaps the next tile's MMAs);
//     zeroes the token rows of a group's last chunk that lie past its end;
//     one lane issues tcgen05.mma kind::f8f6f4 (M = 128, N = 256, K = 32,
//     both operands MN-major: the token index is the contraction index and
//     the operands are contiguous along n and k) and commits each stage back
//     to the producer and each finished accumulator to the epilogue;
//   warps 2-9: two per TMEM lane quarter (32 rows n), each taking half of
//     the tile's columns; each reads its lanes with tcgen05.ld, 32 columns
//     at a time, scales (the scales of a tile are loaded two tiles ahead),
//     rounds to bf16, stages the 32 rows' 64-byte runs in shared memory and
//     stores them eight rows per instruction.
// A group with no tokens gets zeros from the epilogue without any MMA.
// Every wait is bounded; on expiry the error word is set, the warp leaves
// its loop (as a whole: the lanes agree through __all_sync), the others
// time out in turn, loads and MMAs still in flight are waited for, and the
// TMEM is freed before the block exits.
#include <cuda_bf16.h>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace wgrad {

constexpr int kBM = 128;     // rows n of a tile (the MMA's M)
constexpr int kHalfN = 128;  // columns k per swizzle atom (128 e4m3 bytes), one TMA box
constexpr int kBN = 2 * kHalfN;  // columns k of a tile (the MMA's N)
constexpr int kBK = 128;    // tokens per stage
constexpr int kSubK = 32;   // tokens per MMA (kind::f8f6f4)
constexpr int kStages = 4;
constexpr int kABytes = kBK * kBM;         // 16 KB
constexpr int kBHalfBytes = kBK * kHalfN;  // 16 KB
constexpr int kStageBytes = kABytes + 2 * kBHalfBytes;
// Stage layout: the two qx boxes (k 0-127, k 128-255), then the qa_t box.
constexpr int kBOff = 0;
constexpr int kAOff = 2 * kBHalfBytes;
static_assert(kABytes == kBHalfBytes, "three operand blocks of 16 KB, back to back");
constexpr int kAccCols = kBN;              // fp32 TMEM columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kEpiWarps = 8;                // two per TMEM lane quarter
constexpr int kEpiCols = kBN / 2;           // accumulator columns per epilogue warp
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kChunk = 32;                  // accumulator columns per epilogue step: 64-byte runs
constexpr int kStageRow = kChunk * 2;       // staged bf16 row (no padding: XOR-swizzled parts)
static_assert(kTmemCols == 512, "two accumulators fill the TMEM");
static_assert(kBM == 128 && kHalfN == 128 && kBK % kSubK == 0, "MMA shape");

struct Smem {
  uint8_t stage[kStages][kStageBytes];  // 1024-byte aligned (swizzle atoms)
  uint64_t full[kStages];     // stage loaded (TMA bytes)
  uint64_t empty[kStages];    // stage consumed (MMA commit)
  uint64_t acc_full[2];       // accumulator complete (MMA commit)
  uint64_t acc_empty[2];      // accumulator read (one arrival per epilogue warp)
  uint64_t drain;             // the MMA warp's last commit
  uint32_t tmem_base;
  int32_t ends[kMaxGroups];
  alignas(16) float rx[kEpiWarps][kEpiCols];  // per epilogue warp: 1/sx of its columns
  alignas(16) uint8_t rows[kEpiWarps][32 * kStageRow];  // per epilogue warp: 32 staged row runs
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "fits one SM's shared memory");

struct Params {
  const float* sa;       // (N, G)
  const float* sx;       // (G, K)
  uint16_t* out;         // bf16 (G, N, K)
  const int32_t* offs;
  unsigned* err;
  int32_t T, N, K, G;
  int32_t tiles_n, tiles_k;
  int64_t tiles;
  uint64_t timeout_ns;
  int32_t skip_arrival;  // test hook: block 0 never frees its first accumulator
};

// ------------------------------------------------------------ tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// The mbarrier gets one arrival once every tcgen05 operation this thread
// has issued so far is complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
// D (TMEM) = A * B (+ D if accumulate), e4m3 x e4m3 -> fp32.
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr)
               : "memory");
}
// Waits for this thread's TMEM loads; the registers pass through the asm so
// that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) : : "memory");
}

// 16-byte shared load ordered after the warp's preceding shared stores
// (volatile, with a memory clobber).
__device__ __forceinline__ uint4 lds128_ordered(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Shared-memory matrix descriptor of one operand sub-tile: MN-major, 128-byte
// swizzle; a swizzle atom is 8 token rows x 128 bytes (128 e4m3 values along
// M or N), atoms along the token index 1024 bytes apart, atoms along M or N
// `lbo` bytes apart.  Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29: for swizzled MN-major operands the stride between
// atoms along M or N), stride byte offset >> 4 (32-45: the stride between
// 8-row groups along the token index), descriptor version 1 (46-47), base
// offset 0 (49-51: atoms are 1024-byte aligned), swizzle mode 2 = 128 bytes
// (61-63).
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr, uint32_t lbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(1024u >> 4) << 32) | (uint64_t(1) << 46) |
         (uint64_t(2) << 61);
}

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3
// (bits 7-9, 10-12 = 0), A and B MN-major (bits 15, 16), N >> 3 (17-22),
// M >> 4 (24-28).  M = 128, N = 256: one MMA covers the whole tile.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 15) | (1u << 16) |
                            (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);
static_assert((kBN >> 3) < 64 && (kBM >> 4) < 32, "descriptor field widths");

struct TileId {
  int32_t g, n0, k0, t0, tg;  // group, first row, first column, first token, tokens
};

constexpr int kScaleLoads = kEpiCols / 32;  // sx values per lane and tile

__device__ __forceinline__ TileId tile_of(const Params& p, const int32_t* ends, int64_t i) {
  const int64_t per_group = static_cast<int64_t>(p.tiles_n) * p.tiles_k;
  TileId t;
  t.g = static_cast<int32_t>(i / per_group);
  const int32_t r = static_cast<int32_t>(i % per_group);
  t.n0 = (r % p.tiles_n) * kBM;
  t.k0 = (r / p.tiles_n) * kBN;
  t.t0 = t.g > 0 ? ends[t.g - 1] : 0;
  t.tg = ends[t.g] - t.t0;
  return t;
}

// The raw scales epilogue lane `lane` of quarter q, column half hc, needs
// for tile i: sx of columns k0 + kEpiCols hc + lane + 32 m and sa of row
// n0 + 32 q + lane; 1.0 for columns past K, rows past N and tiles past the
// last, so that every reciprocal stays finite.
__device__ __forceinline__ void load_scales(const Params& p, const int32_t* ends, int64_t i, int q,
                                            int hc, int lane, float (&x)[kScaleLoads], float& a) {
  if (i >= p.tiles) {
#pragma unroll
    for (int m = 0; m < kScaleLoads; ++m) x[m] = 1.0f;
    a = 1.0f;
    return;
  }
  const TileId t = tile_of(p, ends, i);
  const float* sxg = p.sx + static_cast<int64_t>(t.g) * p.K;
#pragma unroll
  for (int m = 0; m < kScaleLoads; ++m) {
    const int32_t k = t.k0 + kEpiCols * hc + lane + 32 * m;
    x[m] = k < p.K ? __ldg(sxg + k) : 1.0f;
  }
  const int32_t n = t.n0 + 32 * q + lane;
  a = n < p.N ? __ldg(p.sa + static_cast<int64_t>(n) * p.G + t.g) : 1.0f;
}

__global__ void __launch_bounds__(kThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap amap,
                 const __grid_constant__ CUtensorMap xmap,
                 const __grid_constant__ CUtensorMap amap32,
                 const __grid_constant__ CUtensorMap xmap32, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = 4 * p.timeout_ns;

  if (warp == 0) {
    build_ends(p.offs, 0, p.G, p.T, s.ends, lane);
    if (lane == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(&s.acc_full[b], 1);
        mbar_init(&s.acc_empty[b], kEpiWarps);
      }
      mbar_init(&s.drain, 1);
      fence_mbar_init();
      prefetch_tensormap(&amap);
      prefetch_tensormap(&xmap);
      prefetch_tensormap(&amap32);
      prefetch_tensormap(&xmap32);
    }
  } else if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ loads --
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      uint32_t it = 0;
      bool ok = true;
      for (int64_t i = blockIdx.x; ok && i < p.tiles; i += gridDim.x) {
        const TileId t = tile_of(p, s.ends, i);
        for (int32_t c = 0; ok && c < t.tg; c += kBK, ++it) {
          const int st = static_cast<int>(it % kStages);
          ok = mbar_wait(&s.empty[st], ((it / kStages) & 1) ^ 1u, wait_ns, p.err);
          if (!ok) break;
          uint8_t* base = s.stage[st];
          const int32_t rem = min(t.tg - c, kBK);
          if (rem == kBK) {
            mbar_arrive_expect_tx(&s.full[st], kStageBytes);
            tma_load_2d(base + kBOff, &xmap, t.k0, t.t0 + c, &s.full[st], pol);
            tma_load_2d(base + kBOff + kBHalfBytes, &xmap, t.k0 + kHalfN, t.t0 + c, &s.full[st],
                        pol);
            tma_load_2d(base + kAOff, &amap, t.n0, t.t0 + c, &s.full[st], pol);
          } else {
            // a group's last, partial chunk: only the 32-token slices the
            // MMAs will read
            const int nsub = (rem + kSubK - 1) / kSubK;
            mbar_arrive_expect_tx(&s.full[st], static_cast<uint32_t>(nsub * 3 * kSubK * 128));
            for (int u = 0; u < nsub; ++u) {
              const int32_t y = t.t0 + c + u * kSubK;
              const int off = u * kSubK * 128;
              tma_load_2d(base + kBOff + off, &xmap32, t.k0, y, &s.full[st], pol);
              tma_load_2d(base + kBOff + kBHalfBytes + off, &xmap32, t.k0 + kHalfN, y, &s.full[st],
                          pol);
              tma_load_2d(base + kAOff + off, &amap32, t.n0, y, &s.full[st], pol);
            }
          }
        }
      }
      // the block must not exit while a load is still writing its memory
      for (uint32_t u = it > kStages ? it - kStages : 0; u < it; ++u)
        mbar_wait(&s.full[u % kStages], (u / kStages) & 1, wait_ns, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs --
    uint32_t it = 0, tc = 0;
    bool ok = true;
    bool issued = false;
    for (int64_t i = blockIdx.x; ok && i < p.tiles; i += gridDim.x) {
      const TileId t = tile_of(p, s.ends, i);
      if (t.tg <= 0) continue;
      const int b = static_cast<int>(tc & 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&s.acc_empty[b], ((tc >> 1) & 1) ^ 1u, wait_ns, p.err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(b * kAccCols);
      for (int32_t c = 0; c < t.tg; c += kBK, ++it) {
        const int st = static_cast<int>(it % kStages);
        ok = __all_sync(0xffffffffu, mbar_wait(&s.full[st], (it / kStages) & 1, wait_ns, p.err));
        if (!ok) break;
        const int32_t rem = min(t.tg - c, kBK);  // tokens of the group in this chunk
        const int32_t used = (rem + kSubK - 1) / kSubK * kSubK;
        uint8_t* base = s.stage[st];
        if (rem < used) {
          // rows rem .. used-1 hold tokens of the next group (or the fill):
          // zero them in all three operand blocks (a whole 128-byte row is
          // one swizzle row, so the swizzle does not matter)
          const int n16 = (used - rem) * 8;
          for (int j = lane; j < 3 * n16; j += 32) {
            const int blk = j / n16, w = j % n16;  // block 0, 1: qx halves; 2: qa_t
            const uint32_t off = static_cast<uint32_t>(blk * kBHalfBytes + rem * 128 + w * 16);
            sts128(smem_addr(base + off), make_uint4(0u, 0u, 0u, 0u));
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_addr(base + kAOff);
          const uint32_t b0 = smem_addr(base + kBOff);
          for (int32_t j = 0; j < used; j += kSubK) {
            const uint32_t off = static_cast<uint32_t>(j * 128);  // 32 rows = 4 atoms
            const uint32_t acc = (c > 0 || j > 0) ? 1u : 0u;
            // A: one atom along n; B: two atoms along k, one box apart
            tc_mma_e4m3(d, operand_desc(a0 + off, 1024u), operand_desc(b0 + off, kBHalfBytes),
                        kIdesc, acc);
          }
          tc_commit(&s.empty[st]);
          issued = true;
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&s.acc_full[b]);
      ++tc;
    }
    // every MMA this warp issued is complete before the TMEM is freed
    issued = __shfl_sync(0xffffffffu, issued, 0);
    if (issued) {
      if (lane == 0) tc_commit(&s.drain);
      mbar_wait(&s.drain, 0, wait_ns, p.err);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    // Lane l of epilogue warp (q, hc) owns row n0 + 32 q + l of the tile and
    // the columns [kEpiCols hc, kEpiCols (hc + 1)).  Per step of 32 columns
    // it reads its row's accumulators, scales them, packs bf16 and writes
    // the row's 64-byte run into the warp's staging rows; the warp then
    // stores the 32 runs, eight rows per instruction.  (One lane per row,
    // each writing its own row, runs at three quarters of the rate: every
    // store instruction would touch 32 lines.)  The four 16-byte parts of a
    // staged run are XOR-swizzled by (row / 2) % 4, so that both the
    // row-wise writes and the part-wise reads are free of bank conflicts.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    const int hc = ew / 4;   // column half
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float* rx = s.rx[ew];
    const uint32_t stage_rows = smem_addr(s.rows[ew]);
    const uint32_t my_row = stage_rows + static_cast<uint32_t>(lane * kStageRow);
    const uint32_t my_swz = static_cast<uint32_t>((lane >> 1) & 3);
    // the store side: lane j takes part j % 4 of rows 8 it + j / 4
    const int part = lane & 3;
    // The scales of a tile are loaded two tiles ahead: under the TMA traffic
    // their latency is several microseconds, which would otherwise stall
    // every tile's epilogue.
    uint32_t tc = 0;
    bool ok = true;
    float x0[kScaleLoads], x1[kScaleLoads], x2[kScaleLoads];
    float a0, a1, a2;
    load_scales(p, s.ends, blockIdx.x, q, hc, lane, x0, a0);
    load_scales(p, s.ends, blockIdx.x + static_cast<int64_t>(gridDim.x), q, hc, lane, x1, a1);
    for (int64_t i = blockIdx.x; ok && i < p.tiles; i += gridDim.x) {
      load_scales(p, s.ends, i + 2 * static_cast<int64_t>(gridDim.x), q, hc, lane, x2, a2);
      const TileId t = tile_of(p, s.ends, i);
      const int32_t k0 = t.k0 + kEpiCols * hc;
      const int32_t nbase = t.n0 + 32 * q;
      const bool empty_group = t.tg <= 0;
      __syncwarp();  // the previous tile's readers of rx are done
      // 1/sx of the warp's columns (0 past K), 1/sa of this lane's row
#pragma unroll
      for (int m = 0; m < kScaleLoads; ++m)
        rx[lane + 32 * m] = k0 + lane + 32 * m < p.K ? __frcp_rn(x0[m]) : 0.0f;
      const float ra = nbase + lane < p.N ? __frcp_rn(a0) : 0.0f;
#pragma unroll
      for (int m = 0; m < kScaleLoads; ++m) {
        x0[m] = x1[m];
        x1[m] = x2[m];
      }
      a0 = a1;
      a1 = a2;
      const int b = static_cast<int>(tc & 1);
      if (!empty_group) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&s.acc_full[b], (tc >> 1) & 1, wait_ns, p.err));
        if (!ok) break;
        tc_fence_after();
      }
      __syncwarp();  // rx visible to the warp
      // TMEM loads run one step ahead of the math (h[0] / h[1] alternate)
      const uint32_t tacc =
          tmem + lane_base + static_cast<uint32_t>(b * kAccCols + kEpiCols * hc);
      uint32_t h[2][32];
      if (!empty_group) tmem_ld32(tacc, h[0]);
      uint8_t* orow0 = reinterpret_cast<uint8_t*>(p.out) +
                       ((static_cast<int64_t>(t.g) * p.N + nbase) * p.K + k0) * 2 + part * 16;
#pragma unroll
      for (int st = 0; st < kEpiCols / kChunk; ++st) {
        uint32_t(&hc_)[32] = h[st & 1];
        uint32_t w[16];
        if (!empty_group) {
          tmem_ld_wait(hc_);
          if (st + 1 < kEpiCols / kChunk)
            tmem_ld32(tacc + static_cast<uint32_t>((st + 1) * kChunk), h[(st + 1) & 1]);
          const float* rxc = rx + st * kChunk;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(
                __uint_as_float(hc_[2 * e]) * ra * rxc[2 * e],
                __uint_as_float(hc_[2 * e + 1]) * ra * rxc[2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&v);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = 0u;
        }
        const int32_t kc = k0 + st * kChunk;
        if (kc >= p.K) continue;  // warp-uniform: the rest of the row is past K
#pragma unroll
        for (int c = 0; c < 4; ++c)
          sts128(my_row + ((static_cast<uint32_t>(c) ^ my_swz) << 4),
                 make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]));
        __syncwarp();
        // K % 16 == 0: an 8-column part is wholly inside or outside
        const bool k_ok = kc + part * 8 < p.K;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int row = 8 * it + (lane >> 2);
          const uint32_t src = stage_rows + static_cast<uint32_t>(row * kStageRow) +
                               ((static_cast<uint32_t>(part) ^ ((row >> 1) & 3)) << 4);
          const uint4 v = lds128_ordered(src);
          if (nbase + row < p.N && k_ok)
            *reinterpret_cast<uint4*>(orow0 + static_cast<int64_t>(row) * p.K * 2 + st * kChunk * 2) = v;
        }
        __syncwarp();  // staging rows free for the next step
      }
      if (!empty_group) {
        tmem_ld_wait(h[(kEpiCols / kChunk - 1) & 1]);  // no TMEM load outlives the tile
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !(p.skip_arrival && blockIdx.x == 0 && tc == 0))
          mbar_arrive(&s.acc_empty[b]);
        ++tc;
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

gq_status setup(DeviceInfo& info) {
  (void)info;
  return check_cuda(cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes)),
                    "grouped_wgrad: shared memory size");
}

gq_status launch(const DeviceInfo& info, const DebugKnobs& dbg, const void* qa_t, const float* sa,
                 const void* qx, const float* sx, int32_t T, int32_t N, int32_t K,
                 const int32_t* offs, int32_t G, void* out, cudaStream_t stream) {
  // 128-token boxes for full chunks, 32-token boxes for a group's last one
  CUtensorMap amap, xmap, amap32, xmap32;
  const struct {
    CUtensorMap* map;
    const void* base;
    int32_t inner;
    uint32_t rows;
  } maps[4] = {{&amap, qa_t, N, kBK}, {&xmap, qx, K, kBK}, {&amap32, qa_t, N, kSubK},
               {&xmap32, qx, K, kSubK}};
  for (const auto& m : maps) {
    const gq_status st = encode_tiled_2d(m.map, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                         const_cast<void*>(m.base), static_cast<uint64_t>(m.inner),
                                         static_cast<uint64_t>(T), static_cast<uint64_t>(m.inner),
                                         128, m.rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GQ_OK) return st;
  }
  Params p;
  p.sa = sa;
  p.sx = sx;
  p.out = static_cast<uint16_t*>(out);
  p.offs = offs;
  p.err = info.err_word;
  p.T = T;
  p.N = N;
  p.K = K;
  p.G = G;
  p.tiles_n = (N + kBM - 1) / kBM;
  p.tiles_k = (K + kBN - 1) / kBN;
  p.tiles = static_cast<int64_t>(p.tiles_n) * p.tiles_k * G;
  p.timeout_ns = dbg.timeout_ns;
  p.skip_arrival = dbg.skip_arrival;
  const int64_t grid = p.tiles < info.sm_count ? p.tiles : info.sm_count;
  wgrad_kernel<<<static_cast<int>(grid), kThreads, kSmemBytes, stream>>>(amap, xmap, amap32, xmap32,
                                                                         p);
  return check_cuda(cudaGetLastError(), "grouped_wgrad: launch");
}

}  // namespace wgrad
}  // namespace gq
