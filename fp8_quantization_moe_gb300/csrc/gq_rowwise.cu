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
// shared memory (ldmatrix .trans), and the fp8 tile leaves by a TMA store
// with 128-byte rows of A^T.
//
// Tiles are kTn = 128 rows of A x kTm = 64 token columns (16 KB in, 8 KB
// out), both staged with the 128-byte TMA swizzle so that row-wise and
// column-wise shared-memory accesses are bank-conflict free.  A row band
// (kTn rows, all Mg columns) is one dependency group.  See gq_device.cuh for
// the schedule.
//
// Phase A: consumer thread t owns row t of the tile and folds |x| of each
// group segment with max.xorsign.abs.bf16x2; one atomicMax per (row, group)
// and tile.  Phase B: per (row, group) scales go to shared memory; each warp
// takes 32 rows and walks the tile's 8-column chunks: ldmatrix.x4.trans gives
// every lane the pairs (n, n+1) of one column m, which are multiplied in fp32
// and packed with cvt.rn.satfinite.e4m3x2 into bytes of A^T; one shuffle
// between neighbouring lanes assembles 4-byte runs of an output row, which
// are stored into the swizzled output tile.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace rowwise {

constexpr int kStages = 5;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kTileBytes = kTn * kTm * 2;  // bf16 in
constexpr int kOutBytes = kTm * kTn;       // e4m3 out
constexpr int kSegCache = 8;               // segments whose scales fit at once
static_assert(kConsumers == kTn, "phase A: one consumer thread per tile row");
static_assert(kTm * 2 == 128 && kTn == 128, "128-byte swizzled rows in and out");

using Hdr = TileHdr<kTm>;

struct Smem {
  uint8_t tile[kStages][kTileBytes];  // 1024-byte aligned (swizzle atom)
  uint8_t outt[2][kOutBytes];
  Hdr hdr[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t ends_ready;
  int32_t ends[kMaxGroups];
  alignas(16) float sc[kSegCache][kTn];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Params {
  const int32_t* offs;
  uint8_t* out_t;
  float* scales;
  uint32_t* ticket;
  uint32_t* done;  // one word per row band
  uint32_t* amax;  // (N, G) fp32 bit patterns
  unsigned* err;
  int32_t N, Mg, G;
  Schedule sched;
  uint64_t timeout_ns;
  int32_t skip_arrival;
};

// Byte offset of (row r, byte column c) in a tile of 128-byte rows stored
// with the 128-byte TMA swizzle: the 16-byte chunk index is xor-ed with r % 8.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((((c >> 4) ^ r) & 7) << 4) + (c & 15));
}

__device__ __forceinline__ void producer(Smem& s, const CUtensorMap* amap,
                                         const Params& p) {
  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  const uint32_t total = 2u * static_cast<uint32_t>(p.sched.units) *
                         static_cast<uint32_t>(p.sched.groups);
  bool ends_ok = false;
  int st = 0;
  uint32_t ph = 0;
  for (;;) {
    if (!mbar_wait(&s.empty[st], ph ^ 1u, 4 * p.timeout_ns, p.err)) return;
    const uint32_t t = atomicAdd(p.ticket, 1u);
    Hdr& h = s.hdr[st];
    if (t >= total) {
      h.phase = -1;
      mbar_arrive(&s.full[st]);
      return;
    }
    const Ticket k = decode_ticket(t, p.sched);
    const int32_t n0 = k.dg * kTn;
    const int32_t m0 = k.unit * kTm;
    mbar_expect_tx(&s.full[st], kTileBytes);
    tma_load_2d(s.tile[st], amap, m0, n0, &s.full[st],
                k.phase == 0 ? pol_a : pol_b);
    if (!ends_ok) {
      if (!mbar_wait(&s.ends_ready, 0u, 4 * p.timeout_ns, p.err)) return;
      ends_ok = true;
    }
    h.phase = k.phase;
    h.dg = k.dg;
    fill_segments(h, s.ends, p.G, m0, min(m0 + kTm, p.Mg),
                  k.unit == p.sched.units - 1);
    mbar_arrive(&s.full[st]);
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
}

// Phase A: row t of the tile, |x| maxima per group segment.
__device__ __forceinline__ void phase_a(const Hdr& h, uint32_t tile,
                                        const Params& p, int t) {
  const int32_t n = h.dg * kTn + t;
  const int nseg = h.nseg;
  const uint32_t row = tile + static_cast<uint32_t>(t) * 128u;
  for (int j = 0; j < nseg; ++j) {
    const int a = h.seg_lo[j], b = h.seg_hi[j];
    uint32_t acc = 0;
#pragma unroll
    for (int c = 0; c < kTm / 8; ++c) {
      const int lo = c * 8, hi = lo + 8;
      if (hi <= a || lo >= b) continue;
      const uint4 v = lds128(row + ((((c ^ t) & 7)) << 4));
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
    const uint32_t m = amax_bits_of(acc);
    if (m != 0u && n < p.N)
      atomicMax(p.amax + static_cast<size_t>(n) * p.G + h.seg_g[j], m);
  }
  named_bar(1, kConsumers);
  if (t == 0) {
    const bool skip = p.skip_arrival && h.dg == 0 && h.lo == 0;
    __threadfence();
    if (!skip) atomicAdd(p.done + h.dg, 1u);
  }
}

// Phase B: scale, cast and transpose the tile into outt, then store it.
__device__ __forceinline__ void phase_b(Smem& s, const Hdr& h, uint32_t tile,
                                        const CUtensorMap* omap,
                                        const Params& p, int t, int warp,
                                        int lane, uint32_t& ob,
                                        uint64_t pol_out) {
  const int32_t n0 = h.dg * kTn;
  const int32_t nrow = n0 + t;  // row of A owned for scales
  if (t == 0) {
    wait_counter(p.done + h.dg, static_cast<uint32_t>(p.sched.units),
                 p.timeout_ns, p.err);
    bulk_wait_read<1>();  // the store that last read outt[ob] has finished
  }
  named_bar(1, kConsumers);

  if (nrow < p.N) {
    for (int g = h.own_lo; g < h.own_hi; ++g) {
      const size_t i = static_cast<size_t>(nrow) * p.G + g;
      p.scales[i] = scale_from_amax_bits(ld_cg_u32(p.amax + i));
    }
  }

  uint8_t* outt = s.outt[ob];
  const uint32_t obase = smem_addr(outt);
  const int nseg = h.nseg;
  const int q = lane & 3;
  const bool odd = (lane & 1) != 0;
  const int mcol = lane >> 2;  // column within an 8-column chunk
  const uint32_t lrow = tile + static_cast<uint32_t>(warp * 32 + lane) * 128u;

  for (int jb = 0; jb < nseg; jb += kSegCache) {
    const int je = min(nseg, jb + kSegCache);
    if (jb > 0) named_bar(1, kConsumers);  // previous batch done with sc
    for (int j = jb; j < je; ++j) {
      s.sc[j - jb][t] =
          nrow < p.N ? scale_from_amax_bits(ld_cg_u32(
                           p.amax + static_cast<size_t>(nrow) * p.G + h.seg_g[j]))
                     : 0.0f;
    }
    named_bar(1, kConsumers);
    const int c_first = h.seg_lo[jb] >> 3;
    const int c_last = (h.seg_hi[je - 1] - 1) >> 3;
    int js_cached = -1;
    float sv[8];
    for (int c = c_first; c <= c_last; ++c) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4_trans(lrow + ((((c ^ lane) & 7)) << 4), r0, r1, r2, r3);
      const int m = c * 8 + mcol;  // token column within the tile
      int js = -1;
      for (int j = jb; j < je; ++j)
        if (m >= h.seg_lo[j] && m < h.seg_hi[j]) js = j - jb;
      if (js >= 0 && js != js_cached) {
        js_cached = js;
        const float* scr = s.sc[js] + warp * 32 + 2 * q;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = *reinterpret_cast<const float2*>(scr + 8 * i);
          sv[2 * i] = f.x;
          sv[2 * i + 1] = f.y;
        }
      }
      // pair i: rows warp*32 + 8i + 2q (+1) of A, column m -> 2 bytes of A^T
      const uint32_t p0 = cvt_e4m3x2(__fmul_rn(bf16_lo(r0), sv[0]), __fmul_rn(bf16_hi(r0), sv[1]));
      const uint32_t p1 = cvt_e4m3x2(__fmul_rn(bf16_lo(r1), sv[2]), __fmul_rn(bf16_hi(r1), sv[3]));
      const uint32_t p2 = cvt_e4m3x2(__fmul_rn(bf16_lo(r2), sv[4]), __fmul_rn(bf16_hi(r2), sv[5]));
      const uint32_t p3 = cvt_e4m3x2(__fmul_rn(bf16_lo(r3), sv[6]), __fmul_rn(bf16_hi(r3), sv[7]));
      // even lanes keep pairs 0,1 and take the odd neighbour's; odd lanes
      // keep pairs 2,3 -- each lane ends with two 4-byte runs of row m
      const uint32_t send = odd ? (p0 | (p1 << 16)) : (p2 | (p3 << 16));
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
      if (js >= 0) {
        const int nb = warp * 32 + 2 * (q & 2);  // first row of the 4-run
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
        sts32(obase + swz128(m, na), wa);
        sts32(obase + swz128(m, nb2), wb);
      }
    }
  }
  fence_proxy_async_smem();
  named_bar(1, kConsumers);

  const int32_t m0 = h.lo;
  const int32_t cover = min(h.hi, p.G > 0 ? s.ends[p.G - 1] : 0) - m0;
  if (cover >= h.hi - m0) {
    if (t == 0) {
      tma_store_2d(omap, outt, n0, m0, pol_out);
      bulk_commit();
    }
  } else if (cover > 0) {
    // tokens past the last group end must stay untouched: plain stores of
    // the covered output rows only
    for (int i = t; i < cover * (kTn / 16); i += kConsumers) {
      const int m = i / (kTn / 16);
      const int k = i % (kTn / 16);
      if (n0 + 16 * k < p.N) {
        const uint4 v = lds128(obase + static_cast<uint32_t>(m * 128 + ((((k ^ m) & 7)) << 4)));
        *reinterpret_cast<uint4*>(p.out_t + static_cast<size_t>(m0 + m) * p.N + n0 +
                                  16 * k) = v;
      }
    }
  }
  ob ^= 1u;
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
    mbar_init(&s.ends_ready, 32);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tensormap(&amap);
      producer(s, &amap, p);
    }
    return;
  }

  if (warp == 0) {
    build_ends(p.offs, p.G, p.Mg, s.ends, lane);
    __syncwarp();
    mbar_arrive(&s.ends_ready);
  }
  // consumers read ends (coverage of the last group) in phase B
  named_bar(1, kConsumers);

  const int t = threadIdx.x;
  if (t == 0) prefetch_tensormap(&omap);
  const uint64_t pol_out = policy_evict_first();
  int st = 0;
  uint32_t ph = 0;
  uint32_t ob = 0;
  for (;;) {
    const bool ok = mbar_wait(&s.full[st], ph, 4 * p.timeout_ns, p.err);
    if (named_bar_any(1, kConsumers, !ok)) break;  // all consumers agree
    const Hdr& h = s.hdr[st];
    const int phase = h.phase;
    if (phase < 0) break;
    const uint32_t tile = smem_addr(s.tile[st]);
    if (phase == 0)
      phase_a(h, tile, p, t);
    else
      phase_b(s, h, tile, &omap, p, t, warp, lane, ob, pol_out);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
  if (t == 0) bulk_wait<0>();  // outstanding TMA stores done before exit
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
                       static_cast<uint64_t>(N), kTn, kTm,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;

  Params p;
  p.sched.units = (Mg + kTm - 1) / kTm;
  p.sched.groups = (N + kTn - 1) / kTn;
  const int64_t total = 2ll * p.sched.units * p.sched.groups;
  const int64_t max_ctas =
      static_cast<int64_t>(info.sm_count) * info.rowwise_ctas_per_sm;
  const int grid = static_cast<int>(total < max_ctas ? total : max_ctas);
  int64_t lag = (2ll * grid + p.sched.units - 1) / p.sched.units;
  if (lag < 1) lag = 1;
  if (lag > p.sched.groups) lag = p.sched.groups;
  p.sched.lag = static_cast<int32_t>(lag);

  const WorkspaceLayout L =
      workspace_layout(p.sched.groups, static_cast<int64_t>(N) * G);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.offs = offs;
  p.out_t = static_cast<uint8_t*>(out_t);
  p.scales = scales;
  p.ticket = reinterpret_cast<uint32_t*>(w);
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
  rowwise_kernel<<<grid, kThreads, kSmemBytes, stream>>>(amap, omap, p);
  return check_cuda(cudaGetLastError(), "rowwise_t: launch");
}

}  // namespace rowwise
}  // namespace gq
