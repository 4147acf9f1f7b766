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
// kernel: tiles come in by TMA with 128-byte rows, the transpose happens in
// shared memory (ldmatrix .trans), and the fp8 result leaves by TMA stores
// of 32-byte row runs of A^T.
//
// Tiles are kTn = 128 rows of A x kTm = 64 token columns (16 KB), staged
// with the 128-byte TMA swizzle so that row-wise and column-wise
// shared-memory accesses are bank-conflict free.  A row band (kTn rows, all
// Mg columns) is one dependency group.  See gq_device.cuh for the schedule.
// In phase B the producer lanes bring the amax words of the tile's 128 rows
// for each of its first kSegA segments into the stage.
//
// The eight consumer warps work on each stage independently:
//   phase A: warp w takes rows 16w .. 16w + 15; lane l folds |x| of row
//     16w + l % 16 over columns 32 (l / 16) .. + 31 of each group segment
//     with max.xorsign.abs.bf16x2, one shuffle joins the two column halves,
//     and 16 lanes issue one atomicMax each, into amax words laid out (G, N)
//     so that the 16 atomics of a warp hit one 64-byte run;
//   phase B: warp w takes the 32 x 32 block of rows 32 (w % 4) .. + 31 and
//     columns 32 (w / 4) .. + 31: per segment a lane computes the scale of
//     one row (448 / max(amax, 1e-12), IEEE division) and gathers the eight
//     it needs by shuffles; ldmatrix.x4.trans gives every lane the pairs
//     (n, n+1) of one column m, which are multiplied in fp32 (mul.rn.f32x2)
//     and packed with cvt.rn.satfinite.e4m3x2 into bytes of A^T; one shuffle
//     between neighbouring lanes assembles 4-byte runs of an output row; the
//     warp's 32 x 32-byte block of A^T leaves by its own TMA store.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace rowwise {

constexpr int kStages = 5;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 64;  // + producer warp + signal warp
constexpr int kSigSlots = 16;
constexpr int kTileBytes = kTn * kTm * 2;  // bf16 in
constexpr int kBlk = 32;                   // phase-B block: 32 rows x 32 columns
constexpr int kOutBytes = kBlk * kBlk;     // e4m3 out per warp and buffer
constexpr int kSegA = 4;  // segments whose amax words ride in the stage
static_assert(kTm * 2 == 128 && kTn == 128, "128-byte swizzled rows in");
static_assert(kTn == 32 * 4, "one 16-byte amax chunk per producer lane");
static_assert(kConsumerWarps * kBlk * kBlk == kTn * kTm, "warps tile the stage");
static_assert(kSigSlots > kStages, "a warp cannot lap the signal ring");

using Hdr = TileHdr<kTm>;

struct Smem {
  uint8_t tile[kStages][kTileBytes];  // 1024-byte aligned (swizzle atom)
  uint8_t outt[kConsumerWarps][2][kOutBytes];
  alignas(16) uint32_t amax[kStages][kSegA][kTn];  // phase B amax words
  Hdr hdr[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t ends_ready;
  SigRing<kSigSlots> sig;
  int32_t ends[kMaxGroups];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Params {
  const int32_t* offs;
  uint8_t* out_t;
  float* scales;
  uint32_t* done;  // one word per row band
  uint32_t* amax;  // (G, N) fp32 bit patterns
  unsigned* err;
  int32_t N, Mg, G;
  Schedule sched;
  uint64_t timeout_ns;
  int32_t skip_arrival;
};

// Shared-memory address of 16-byte chunk c (8 token columns) of tile row r
// (128-byte TMA swizzle: the chunk index is xor-ed with r % 8).
__device__ __forceinline__ uint32_t chunk_addr(uint32_t tile, int r, int c) {
  return tile + static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// The producer warp: group-end table, then per ticket header + loads.
__device__ __forceinline__ void producer(Smem& s, const CUtensorMap* amap,
                                         const Params& p, int lane) {
  build_ends(p.offs, p.G, p.Mg, s.ends, lane);
  __syncwarp();
  if (lane == 0) mbar_arrive(&s.ends_ready);

  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  const int32_t units = p.sched.units;
  const int32_t blocks = 2 * p.sched.groups;
  int32_t ready_dg = -1;  // bands <= ready_dg are complete
  int st = 0;
  uint32_t ph = 0;
  for (TicketWalk tw(blockIdx.x, gridDim.x, units);; tw.next(units)) {
    Hdr& h = s.hdr[st];
    if (!mbar_wait(&s.empty[st], ph ^ 1u, 4 * p.timeout_ns, p.err)) return;
    bool stop = tw.block >= blocks;
    int32_t phase = 0, dg = 0;
    if (!stop) decode_block(tw.block, p.sched, phase, dg);
    if (!stop && phase == 1 && dg > ready_dg) {
      bool ok = true;
      if (lane == 0)
        ok = wait_counter(p.done + dg, static_cast<uint32_t>(units), p.timeout_ns,
                          p.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) {
        ld_acquire_u32(p.done + dg);  // every lane acquires before reading amax
        ready_dg = dg;
      }
      stop = !ok;
    }
    if (stop) {
      if (lane == 0) {
        h.phase = -1;
        mbar_arrive(&s.full[st]);
      }
      return;
    }
    const int32_t n0 = dg * kTn;
    const int32_t m0 = tw.unit * kTm;
    build_header_warp(h, s.ends, p.G, m0, min(m0 + kTm, p.Mg), tw.unit == units - 1,
                      lane);
    __syncwarp();
    if (phase == 1) {
      const int n = min(static_cast<int>(h.nseg), kSegA);
      const int32_t row = n0 + 4 * lane;
      for (int j = 0; j < n; ++j)
        cp_async_16(smem_addr(&s.amax[st][j][4 * lane]),
                    p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + (row < p.N ? row : 0),
                    row < p.N ? 16u : 0u);
      cp_async_mbar_arrive(&s.full[st]);
    }
    if (lane == 0) {
      h.phase = phase;
      h.dg = dg;
      h.unit = tw.unit;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(&s.full[st], kTileBytes);
      tma_load_2d(s.tile[st], amap, m0, n0, &s.full[st], phase == 0 ? pol_a : pol_b);
    }
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
}

// Phase A, warp w: per segment, the |x| maxima of rows 16w .. 16w + 15; then
// the tile goes to the signal lane.
__device__ __forceinline__ void phase_a(Smem& s, const Hdr& h, uint32_t tile,
                                        const Params& p, int warp, int lane,
                                        uint32_t& sig_seq) {
  const int r = 16 * warp + (lane & 15);  // tile row
  const int hc = lane >> 4;               // column half: chunks 4 hc .. 4 hc + 3
  const int32_t n = h.dg * kTn + r;
  const int nseg = h.nseg;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    uint32_t acc = 0;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int c = 4 * hc + cc;
      const int lo = c * 8, hi = lo + 8;
      if (hi <= a || lo >= b) continue;
      const uint4 v = lds128(chunk_addr(tile, r, c));
      if (lo >= a && hi <= b) {
        acc = absmax_bf16x2(acc, v.x);
        acc = absmax_bf16x2(acc, v.y);
        acc = absmax_bf16x2(acc, v.z);
        acc = absmax_bf16x2(acc, v.w);
      } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int col = lo + e;
          if (col >= a && col < b) {
            const uint32_t half = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
            acc = absmax_bf16x2(acc, half);
          }
        }
      }
    }
    acc = absmax_bf16x2(acc, __shfl_xor_sync(0xffffffffu, acc, 16));
    const uint32_t m = amax_bits_of(acc);
    if (lane < 16 && m != 0u && n < p.N)
      atomicMax(p.amax + static_cast<size_t>(h.seg_g[j]) * p.N + n, m);
  }
  sig_post(s.sig, (p.skip_arrival && h.dg == 0 && h.unit == 0) ? kSigSkip : h.dg,
           warp * 32 + lane, lane, sig_seq, 4 * p.timeout_ns, p.err);
}

// Phase B, warp w: scale, cast and transpose its 32 x 32 block into its
// output buffer, then store the block of A^T.
__device__ __forceinline__ void phase_b(Smem& s, const Hdr& h, int st,
                                        uint32_t tile, const CUtensorMap* omap,
                                        const Params& p, int warp, int lane,
                                        uint32_t& ob, uint64_t pol_out) {
  const int rq = warp & 3;   // rows 32 rq .. 32 rq + 31
  const int hc = warp >> 2;  // columns 32 hc .. 32 hc + 31
  const int32_t n0 = h.dg * kTn;
  const int32_t nrow = n0 + kBlk * rq + lane;  // the row whose scales this lane computes
  const bool row_in = nrow < p.N;
  const int q = lane & 3;
  const bool odd = (lane & 1) != 0;
  const int mcol = lane >> 2;  // column within an 8-column chunk
  const uint32_t lrow = tile + static_cast<uint32_t>(kBlk * rq + lane) * 128u;
  uint8_t* obuf = s.outt[warp][ob];
  const uint32_t obase = smem_addr(obuf);
  if (lane == 0) bulk_wait_read<1>();  // the store that last read obuf is done
  __syncwarp();

  // owned groups without columns: amax 0
  if (hc == 0) {
    for (int g = h.own_lo; g < h.own_hi; ++g) {
      const int32_t gs = g ? s.ends[g - 1] : 0;
      if (row_in && s.ends[g] == gs)
        p.scales[static_cast<size_t>(nrow) * p.G + g] = scale_from_amax_bits(0u);
    }
  }

  const int nseg = h.nseg;
  const int wlo = kBlk * hc, whi = wlo + kBlk;  // this warp's columns
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    if (b <= wlo || a >= whi) continue;  // no column of this warp
    const int g = h.seg_g[j];
    const uint32_t bits =
        j < kSegA ? s.amax[st][j][kBlk * rq + lane]
                  : (row_in ? ld_cg_u32(p.amax + static_cast<size_t>(g) * p.N + nrow) : 0u);
    const float sc = scale_from_amax_bits(bits);
    // the group starts inside the tile at column a: the warps holding
    // column a write its scales
    if (hc == (a >> 5) && row_in && g >= h.own_lo && g < h.own_hi)
      p.scales[static_cast<size_t>(nrow) * p.G + g] = sc;
    float sv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sv[2 * i] = __shfl_sync(0xffffffffu, sc, 8 * i + 2 * q);
      sv[2 * i + 1] = __shfl_sync(0xffffffffu, sc, 8 * i + 2 * q + 1);
    }
    const int c_first = max(a, wlo) >> 3;
    const int c_last = (min(b, whi) - 1) >> 3;
    for (int c = c_first; c <= c_last; ++c) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4_trans(lrow + ((((c ^ lane) & 7)) << 4), r0, r1, r2, r3);
      const int m = c * 8 + mcol;  // token column within the tile
      // pair i: rows 8i + 2q (+1) of the block, column m -> 2 bytes of A^T
      const float2 f0 = mul_f32x2(make_float2(bf16_lo(r0), bf16_hi(r0)), make_float2(sv[0], sv[1]));
      const float2 f1 = mul_f32x2(make_float2(bf16_lo(r1), bf16_hi(r1)), make_float2(sv[2], sv[3]));
      const float2 f2 = mul_f32x2(make_float2(bf16_lo(r2), bf16_hi(r2)), make_float2(sv[4], sv[5]));
      const float2 f3 = mul_f32x2(make_float2(bf16_lo(r3), bf16_hi(r3)), make_float2(sv[6], sv[7]));
      const uint32_t p0 = cvt_e4m3x2(f0.x, f0.y), p1 = cvt_e4m3x2(f1.x, f1.y);
      const uint32_t p2 = cvt_e4m3x2(f2.x, f2.y), p3 = cvt_e4m3x2(f3.x, f3.y);
      // even lanes keep pairs 0,1 and take the odd neighbour's; odd lanes
      // keep pairs 2,3 -- each lane ends with two 4-byte runs of row m
      const uint32_t send = odd ? (p0 | (p1 << 16)) : (p2 | (p3 << 16));
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
      if (m >= a && m < b) {
        const int nb = 2 * (q & 2);  // first row of the 4-run
        uint32_t wa, wb;
        int na, nb2;
        if (!odd) {
          wa = p0 | ((recv & 0xFFFFu) << 16);  // rows nb + 0..3
          wb = p1 | ((recv >> 16) << 16);      // rows nb + 8 + 0..3
          na = nb;
          nb2 = nb + 8;
        } else {
          wa = (recv >> 16) | (p3 << 16);      // rows nb + 24 + 0..3
          wb = (recv & 0xFFFFu) | (p2 << 16);  // rows nb + 16 + 0..3
          na = nb + 24;
          nb2 = nb + 16;
        }
        const uint32_t rowb = obase + static_cast<uint32_t>((m - wlo) * kBlk);
        sts32(rowb + na, wa);
        sts32(rowb + nb2, wb);
      }
    }
  }
  fence_proxy_async_smem();
  __syncwarp();

  // store the block: rows m0 + wlo .. of A^T that lie in the tile
  const int32_t m0 = h.lo;
  const int width = h.hi - m0;  // tokens in the tile
  if (wlo >= width) return;
  const int32_t cover = min(h.hi, p.G > 0 ? s.ends[p.G - 1] : 0) - m0;
  if (min(whi, width) <= cover) {
    if (lane == 0) {
      tma_store_2d(omap, obuf, n0 + kBlk * rq, m0 + wlo, pol_out);
      bulk_commit();
    }
    ob ^= 1u;
  } else if (cover > wlo) {
    // tokens past the last group end must stay untouched: plain stores of
    // the covered output rows only
    const int rows = cover - wlo;
    for (int i = lane; i < 2 * rows; i += 32) {
      const int ml = i >> 1, hb = i & 1;
      const int32_t nn = n0 + kBlk * rq + 16 * hb;
      if (nn < p.N) {
        const uint4 v = lds128(obase + static_cast<uint32_t>(ml * kBlk + 16 * hb));
        *reinterpret_cast<uint4*>(p.out_t + static_cast<size_t>(m0 + wlo + ml) * p.N + nn) = v;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    rowwise_kernel(const __grid_constant__ CUtensorMap amap,
                   const __grid_constant__ CUtensorMap omap, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kConsumerWarps);
    }
    mbar_init(&s.ends_ready, 1);
    sig_init(s.sig, kConsumerWarps);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps + 1) {
    if (lane == 0) sig_loop(s.sig, p.done, 8 * p.timeout_ns, p.err);
    return;
  }
  if (warp == kConsumerWarps) {
    if (lane == 0) prefetch_tensormap(&amap);
    producer(s, &amap, p, lane);
    return;
  }

  if (lane == 0) prefetch_tensormap(&omap);
  mbar_wait(&s.ends_ready, 0u, 4 * p.timeout_ns, p.err);
  const uint64_t pol_out = policy_evict_first();
  int st = 0;
  uint32_t ph = 0;
  uint32_t ob = 0;
  uint32_t sig_seq = 0;
  for (;;) {
    const bool ok = mbar_wait(&s.full[st], ph, 4 * p.timeout_ns, p.err);
    if (__any_sync(0xffffffffu, !ok)) break;  // the warp leaves together
    const Hdr& h = s.hdr[st];
    const int phase = h.phase;
    if (phase < 0) break;
    const uint32_t tile = smem_addr(s.tile[st]);
    if (phase == 0)
      phase_a(s, h, tile, p, warp, lane, sig_seq);
    else
      phase_b(s, h, st, tile, &omap, p, warp, lane, ob, pol_out);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
  sig_post(s.sig, kSigEnd, warp * 32 + lane, lane, sig_seq, 4 * p.timeout_ns, p.err);
  if (lane == 0) bulk_wait<0>();  // this warp's TMA stores done before exit
}

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
  CUtensorMap amap, omap;
  gq_status st = encode_tiled_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 const_cast<void*>(a), static_cast<uint64_t>(Mg),
                                 static_cast<uint64_t>(N),
                                 static_cast<uint64_t>(Mg) * 2, kTm, kTn,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;
  st = encode_tiled_2d(&omap, CU_TENSOR_MAP_DATA_TYPE_UINT8, out_t,
                       static_cast<uint64_t>(N), static_cast<uint64_t>(Mg),
                       static_cast<uint64_t>(N), kBlk, kBlk,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;

  Params p;
  p.sched.units = (Mg + kTm - 1) / kTm;
  p.sched.groups = (N + kTn - 1) / kTn;
  const int64_t total = 2ll * p.sched.units * p.sched.groups;
  const int64_t max_ctas =
      static_cast<int64_t>(info.sm_count) * info.rowwise_ctas_per_sm;
  const int grid = static_cast<int>(total < max_ctas ? total : max_ctas);
  p.sched.lag = schedule_lag(dbg.lag[GQ_KIND_ROWWISE_T], p.sched.units,
                             p.sched.groups, grid, kStages);

  const WorkspaceLayout L =
      workspace_layout(p.sched.groups, static_cast<int64_t>(N) * G);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.offs = offs;
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
  // cooperative: the static ticket order needs every CTA resident
  void* args[] = {&amap, &omap, &p};
  return check_cuda(
      cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(rowwise_kernel),
                                  dim3(grid), dim3(kThreads), args, kSmemBytes,
                                  stream),
      "rowwise_t: launch");
}

}  // namespace rowwise
}  // namespace gq
