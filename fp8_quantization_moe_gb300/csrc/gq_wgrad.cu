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
//     swizzle -- into a ring of kStages stages;
//   warp 1: allocates the 512 TMEM columns (two accumulators of 256 fp32
//     columns, so that a tile's epilogue overlaps the next tile's MMAs);
//     zeroes the token rows of a group's last chunk that lie past its end;
//     one lane issues tcgen05.mma kind::f8f6f4 (M = 128, N = 128, K = 32,
//     both operands MN-major: the token index is the contraction index and
//     the operands are contiguous along n and k) and commits each stage back
//     to the producer and each finished accumulator to the epilogue;
//   warps 2-5: each reads its 32 TMEM lanes (rows n) with tcgen05.ld, scales,
//     rounds to bf16 and stores its rows' 512-byte runs of the tile.
// A group with no tokens gets zeros from the epilogue without any MMA.
// Every wait is bounded; on expiry the error word is set, the warp leaves
// its loop (as a whole: the lanes agree through __all_sync), the others time out in turn, loads and MMAs still in flight are
// waited for, and the TMEM is freed before the block exits.
#include <cuda_bf16.h>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace wgrad {

constexpr int kBM = 128;    // rows n of a tile (the MMA's M)
constexpr int kHalfN = 128;  // columns k per MMA (the MMA's N)
constexpr int kBN = 2 * kHalfN;  // columns k of a tile
constexpr int kBK = 128;    // tokens per stage
constexpr int kSubK = 32;   // tokens per MMA (kind::f8f6f4)
constexpr int kStages = 4;
constexpr int kABytes = kBK * kBM;         // 16 KB
constexpr int kBHalfBytes = kBK * kHalfN;  // 16 KB
constexpr int kStageBytes = kABytes + 2 * kBHalfBytes;
constexpr int kAccCols = kBN;              // fp32 TMEM columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kEpiWarps) * 32;
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
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

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

// Shared-memory matrix descriptor of one operand sub-tile: MN-major, 128-byte
// swizzle, exactly one swizzle atom (128 bytes = 128 e4m3 values) along
// M or N, groups of 8 token rows 1024 bytes apart.  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (16-29; the stride between
// atoms along M/N, never used with one atom), stride byte offset >> 4
// (32-45), descriptor version 1 (46-47), base offset 0 (49-51: atoms are
// 1024-byte aligned), swizzle mode 2 = 128 bytes (61-63).
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(1024u >> 4) << 16) |
         (static_cast<uint64_t>(1024u >> 4) << 32) | (uint64_t(1) << 46) |
         (uint64_t(2) << 61);
}

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3
// (bits 7-9, 10-12 = 0), A and B MN-major (bits 15, 16), N >> 3 (17-22),
// M >> 4 (24-28).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 15) | (1u << 16) |
                            (static_cast<uint32_t>(kHalfN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);

struct TileId {
  int32_t g, n0, k0, t0, tg;  // group, first row, first column, first token, tokens
};

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

__global__ void __launch_bounds__(kThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap amap,
                 const __grid_constant__ CUtensorMap xmap, const Params p) {
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
          mbar_arrive_expect_tx(&s.full[st], kStageBytes);
          tma_load_2d(base, &amap, t.n0, t.t0 + c, &s.full[st], pol);
          tma_load_2d(base + kABytes, &xmap, t.k0, t.t0 + c, &s.full[st], pol);
          tma_load_2d(base + kABytes + kBHalfBytes, &xmap, t.k0 + kHalfN, t.t0 + c, &s.full[st],
                      pol);
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
            const int blk = j / n16, w = j % n16;
            const uint32_t off = static_cast<uint32_t>(blk * kABytes + rem * 128 + w * 16);
            sts128(smem_addr(base + off), make_uint4(0u, 0u, 0u, 0u));
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_addr(base);
          const uint32_t b0 = a0 + kABytes;
          const uint32_t b1 = b0 + kBHalfBytes;
          for (int32_t j = 0; j < used; j += kSubK) {
            const uint32_t off = static_cast<uint32_t>(j * 128);  // 32 rows = 4 atoms
            const uint32_t acc = (c > 0 || j > 0) ? 1u : 0u;
            tc_mma_e4m3(d, operand_desc(a0 + off), operand_desc(b0 + off), kIdesc, acc);
            tc_mma_e4m3(d + kHalfN, operand_desc(a0 + off), operand_desc(b1 + off), kIdesc, acc);
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
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    uint32_t tc = 0;
    bool ok = true;
    for (int64_t i = blockIdx.x; ok && i < p.tiles; i += gridDim.x) {
      const TileId t = tile_of(p, s.ends, i);
      const int32_t n = t.n0 + 32 * q + lane;
      const bool row_ok = n < p.N;
      uint16_t* orow = p.out + (static_cast<int64_t>(t.g) * p.N + n) * p.K;
      if (t.tg <= 0) {
        if (row_ok)
          for (int32_t k = t.k0; k < t.k0 + kBN && k < p.K; k += 8)
            __stcs(reinterpret_cast<uint4*>(orow + k), make_uint4(0u, 0u, 0u, 0u));
        continue;
      }
      const int b = static_cast<int>(tc & 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&s.acc_full[b], (tc >> 1) & 1, wait_ns, p.err));
      if (!ok) break;
      tc_fence_after();
      const float ra = row_ok ? __frcp_rn(__ldg(p.sa + static_cast<int64_t>(n) * p.G + t.g)) : 0.0f;
      const float* sxg = p.sx + static_cast<int64_t>(t.g) * p.K;
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(b * kAccCols + ch * 32), r);
        tmem_ld_wait(r);
        const int32_t kc = t.k0 + ch * 32;
        if (!row_ok || kc >= p.K) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int32_t k = kc + 8 * v;
          if (k >= p.K) break;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(r[8 * v + 2 * e]) * ra * __frcp_rn(__ldg(sxg + k + 2 * e));
            const float x1 = __uint_as_float(r[8 * v + 2 * e + 1]) * ra * __frcp_rn(__ldg(sxg + k + 2 * e + 1));
            const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
            w[e] = *reinterpret_cast<const uint32_t*>(&h);
          }
          __stcs(reinterpret_cast<uint4*>(orow + k), make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.acc_empty[b]);
      ++tc;
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
  CUtensorMap amap, xmap;
  gq_status st = encode_tiled_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(qa_t),
                                 static_cast<uint64_t>(N), static_cast<uint64_t>(T),
                                 static_cast<uint64_t>(N), kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;
  st = encode_tiled_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(qx),
                       static_cast<uint64_t>(K), static_cast<uint64_t>(T),
                       static_cast<uint64_t>(K), kHalfN, kBK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;
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
  const int64_t grid = p.tiles < info.sm_count ? p.tiles : info.sm_count;
  wgrad_kernel<<<static_cast<int>(grid), kThreads, kSmemBytes, stream>>>(amap, xmap, p);
  return check_cuda(cudaGetLastError(), "grouped_wgrad: launch");
}

}  // namespace wgrad
}  // namespace gq
