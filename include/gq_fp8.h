/*
 * gq_fp8.h -- C ABI of libgqfp8: per-token-group fp8 e4m3 quantization for
 * the grouped GEMMs of MoE fp8 training, on GB300 (sm_103a).
 *
 * The method comes from two pytorch/ao pull-request pages:
 *   [moe training] "use smaller block sizes for per group scaling kernels to
 *       improve perf" (#2668): intro (the per-token-group scaling kernel along
 *       dim0, and its "grid too small" finding) and the kernel arguments in
 *       its torch.compile failure report (fp8_dtype_max = 448.0,
 *       fp8_dtype_min = -448.0, EPS = 1e-12);
 *   [moe fp8 training] "test and bench new faster method for per group
 *       rowwise scaling" (#2863): Summary (per-group rowwise scaling for the
 *       backward grad_weight = grad_output_t @ input GEMM, computed through
 *       the transpose so that global accesses stay coalesced).
 *
 * For a token group g = [s_g, e_g) and each column (colwise) or row
 * (rowwise):
 *     amax  = max |x| over the group's tokens (0 when the group is empty)
 *     scale = 448 / max(amax, 1e-12)                      IEEE fp32 division
 *     q     = e4m3(fp32(x * scale))                       fp32 multiply, then
 *             round-to-nearest-even, saturating to +-448
 * The stored scale is that multiplier; dequantization divides by it.
 *
 * Token groups.  `offs` holds n_groups int32 END offsets on the device:
 * group 0 is [0, offs[0]), group g is [offs[g-1], offs[g]).  Contract:
 * nondecreasing, offs[n_groups-1] <= extent (M for colwise, Mg for
 * rowwise_t).  The library never reads offs on the host (that would need a
 * device synchronisation); the kernels read each end as the running maximum
 * of offs[0..g] clamped to [0, extent], so out-of-contract offsets cannot
 * cause an out-of-bounds access.  Tokens past the last end belong to no
 * group: their output bytes are left untouched.  Groups need not be
 * multiples of 16 tokens (the MoE training test aligns them to 16; these
 * kernels do not rely on it).
 *
 * Memory.  Every pointer is device memory that the caller allocates and
 * owns; the library allocates nothing and does not synchronise the host on
 * the quantization calls, which are asynchronous on `stream` (a
 * cudaStream_t; NULL is the legacy default stream).  Outputs and the
 * workspace must stay valid until the stream's work completes.  Concurrent
 * calls must use distinct workspaces.  The library keeps per-device state
 * (launch set-up, the device addresses of its own __device__ arrays) for the
 * life of the process, so no gq_* call may follow a cudaDeviceReset of that
 * device in the same process.
 *
 * Errors.  Every condition the host can check returns a status before any
 * work is enqueued; nothing aborts.  Failures of the CUDA runtime during
 * set-up or launch return GQ_ERR_CUDA, with detail in gq_last_error().  A
 * kernel that waits on another thread block gives up after a bounded time
 * (default 1 s): it then records GQ_ERR_TIMEOUT in a per-device error word,
 * finishes without hanging, and gq_check_device_error() reports it.
 */
#ifndef GQ_FP8_H
#define GQ_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* gq_stream_t;

typedef enum gq_status {
  GQ_OK = 0,
  GQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment,
                             workspace too small */
  GQ_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle:
                             n_groups > GQ_MAX_GROUPS, K % 16, N % 16,
                             Mg % 8, an extent >= 2^31, no sm_103 device */
  GQ_ERR_CUDA = 3,        /* CUDA runtime failure (see gq_last_error) */
  GQ_ERR_TIMEOUT = 4      /* a bounded cross-block wait expired on the GPU */
} gq_status;

#define GQ_KIND_COLWISE 0
#define GQ_KIND_ROWWISE_T 1
#define GQ_MAX_GROUPS 1024

/*
 * Workspace size in bytes for one call.
 *   kind GQ_KIND_COLWISE:   rows = M, cols = K.
 *   kind GQ_KIND_ROWWISE_T: rows = N, cols = Mg.
 * Colwise: a work counter, a finished-blocks counter, one counter per
 * (group, 128-column slab) strip and the per-(group, column) running amax
 * words.  Rowwise_t: a 256-byte header (a work counter, a finished-blocks
 * counter, and two words with which the blocks settle whether all of them
 * are resident), then 68 words per (64-row band, group) unit that may be
 * split across blocks -- a group of 4090 tokens or more, so at most
 * min(n_groups, Mg / 4090) per band: calls whose groups average 2048
 * tokens or more cut such units (more than 64 windows of 64 tokens) into
 * parts that several blocks take, which join their row maxima there; a
 * call does so only when it finds every one of its blocks resident (at
 * most one per SM), and otherwise runs those units whole, as the shorter
 * ones.  The call clears what it uses itself, so the contents on entry do
 * not matter (with GQ_WORKSPACE_ZEROED the call skips the clear; see
 * there).  Returns 0 when no workspace is needed (empty problems) and for
 * invalid arguments.
 */
size_t gq_workspace_bytes(int kind, int64_t rows, int64_t cols,
                          int32_t n_groups);

/*
 * Colwise per-token-group scaling: groups run along dim0 (the token rows),
 * one scale per (group, column).  The dim0 kernel of pytorch/ao #2668.
 *
 *   x        bf16 [M, K] row-major, 16-byte aligned base.       (input)
 *   M, K     M >= 0 tokens; K >= 0 columns, K % 16 == 0.
 *   offs     int32 [n_groups] end offsets along M, device.      (input)
 *   n_groups 1 <= n_groups <= GQ_MAX_GROUPS.
 *   out      e4m3 bytes [M, K] row-major, 16-byte aligned.       (output)
 *            out[r][k] = q(x[r][k]) for every r inside a group.
 *   scales   fp32 [n_groups, K] row-major, 4-byte aligned.       (output)
 *            Every entry is written, empty groups included
 *            (448 / 1e-12 rounded to fp32).
 *   workspace, workspace_bytes: at least gq_workspace_bytes(GQ_KIND_COLWISE,
 *            M, K, n_groups) bytes, 256-byte aligned (may be NULL when that
 *            is 0).
 *   stream   the CUDA stream to run on.
 */
gq_status gq_fp8_colwise(const void* x, int64_t M, int64_t K,
                         const int32_t* offs, int32_t n_groups, void* out,
                         float* scales, void* workspace,
                         size_t workspace_bytes, gq_stream_t stream);

/*
 * Rowwise per-token-group scaling with transposed output: groups run along
 * dim1 (the Mg token columns of A), one scale per (row, group), and the fp8
 * result is written as A^T -- the operand layout the backward grad_weight
 * GEMM of pytorch/ao #2863 consumes.
 *
 *   a        bf16 [N, Mg] row-major, 16-byte aligned base.      (input)
 *   N, Mg    N >= 0 rows, N % 16 == 0; Mg >= 0 tokens, Mg % 8 == 0.
 *   offs     int32 [n_groups] end offsets along Mg, device.     (input)
 *   n_groups 1 <= n_groups <= GQ_MAX_GROUPS.
 *   out_t    e4m3 bytes [Mg, N] row-major, 16-byte aligned.      (output)
 *            out_t[m][n] = q(a[n][m]) for every token m inside a group.
 *   scales   fp32 [N, n_groups] row-major, 4-byte aligned.       (output)
 *            Every entry is written, empty groups included.
 *   workspace, workspace_bytes: at least gq_workspace_bytes(
 *            GQ_KIND_ROWWISE_T, N, Mg, n_groups) bytes, 256-byte aligned.
 *   stream   the CUDA stream to run on.
 */
gq_status gq_fp8_rowwise_t(const void* a, int64_t N, int64_t Mg,
                           const int32_t* offs, int32_t n_groups, void* out_t,
                           float* scales, void* workspace,
                           size_t workspace_bytes, gq_stream_t stream);

/*
 * Options of the _ex calls (a bit mask; unknown bits are GQ_ERR_INVALID_ARG).
 *   GQ_SCALE_POW2  round every scale down to a power of two,
 *                  s = 2^floor(log2(448 / max(amax, 1e-12))) -- the
 *                  round_scales_to_power_of_2 option of the kernel in
 *                  pytorch/ao #2668 (kernel arguments in its torch.compile
 *                  failure report).  The cast multiplies by s as usual; the
 *                  product is then exact, and the scale no larger than the
 *                  plain one, so in a group column (row) whose amax is at
 *                  least 1e-12 the largest |q| lies in [224, 448].
 */
#define GQ_SCALE_POW2 1u
/*
 *   GQ_WORKSPACE_ZEROED  the caller states that the workspace holds
 *                  zeros where this call uses it -- zero-filled once, or
 *                  left so by an earlier call of the same library on it
 *                  that completed: every colwise, expert_dim1 and rowwise_t
 *                  launch returns the part of its workspace it used to zero
 *                  before it ends, also after a bounded wait expired -- and
 *                  the call skips its own clear (one device operation less
 *                  per call).
 */
#define GQ_WORKSPACE_ZEROED 2u
/*
 *   GQ_TWO_PHASE   (colwise and expert_dim1 only; GQ_ERR_INVALID_ARG for
 *                  rowwise_t) every (group, 128-column slab) strip goes
 *                  through the two-phase path -- amax tiles, then a second
 *                  read for the cast -- also strips of at most 320 rows,
 *                  which are otherwise loaded once and cast out of shared
 *                  memory.  Results are identical; the option exists to
 *                  test and time the two-phase path on any shape.
 */
#define GQ_TWO_PHASE 4u

/*
 * gq_fp8_colwise / gq_fp8_rowwise_t with option flags; the calls above are
 * these with flags = 0.  Arguments, layouts and errors as above.
 */
gq_status gq_fp8_colwise_ex(const void* x, int64_t M, int64_t K,
                            const int32_t* offs, int32_t n_groups, void* out,
                            float* scales, uint32_t flags, void* workspace,
                            size_t workspace_bytes, gq_stream_t stream);
gq_status gq_fp8_rowwise_t_ex(const void* a, int64_t N, int64_t Mg,
                              const int32_t* offs, int32_t n_groups, void* out_t,
                              float* scales, uint32_t flags, void* workspace,
                              size_t workspace_bytes, gq_stream_t stream);

/*
 * Scaling of stacked expert weights along dim1: the "fused reduction kernel
 * along dim1 for 3d expert weights" of the pytorch/ao #2863 page's PR stack
 * (#2865).  Each expert's (K, N) matrix is scaled per column, the amax taken
 * over its K rows: exactly gq_fp8_colwise on the (E * K, N) stack with E
 * token groups of K rows each, without an offsets array.
 *
 *   w        bf16 [E, K, N] row-major, 16-byte aligned.          (input)
 *   E, K, N  1 <= E <= GQ_MAX_GROUPS experts; K >= 0; N >= 0, N % 16 == 0;
 *            E * K < 2^31.
 *   out      e4m3 bytes [E, K, N] row-major, 16-byte aligned.    (output)
 *   scales   fp32 [E, N] row-major: scale of expert e, column n. (output)
 *   flags    0, GQ_SCALE_POW2, GQ_WORKSPACE_ZEROED or both.
 *   workspace, workspace_bytes: at least gq_workspace_bytes(GQ_KIND_COLWISE,
 *            E * K, N, E) bytes, 256-byte aligned.
 *   stream   the CUDA stream to run on.
 */
gq_status gq_fp8_expert_dim1(const void* w, int64_t E, int64_t K, int64_t N, void* out,
                             float* scales, uint32_t flags, void* workspace,
                             size_t workspace_bytes, gq_stream_t stream);

/*
 * Scaling of stacked expert weights per row: the "fp8 rowwise kernels for
 * expert weights" of the pytorch/ao #2668 page's PR stack (#2696).  Each
 * expert's (N, K) matrix is scaled per row, the amax taken over the row's
 * K elements: scale[e][n] = 448 / max(amax, 1e-12) (IEEE fp32; rounded down
 * to a power of two with GQ_SCALE_POW2), out[e][n][k] = e4m3(fp32(w[e][n][k]
 * * scale[e][n])), round-to-nearest-even, saturating.  With K = 0 every
 * scale is 448 / 1e-12.
 *
 *   w        bf16 [E, N, K] row-major, 16-byte aligned.          (input)
 *   E, N, K  E >= 1, N >= 0, K >= 0, each below 2^31; K % 8 == 0.
 *   out      e4m3 bytes [E, N, K] row-major, 16-byte aligned.    (output)
 *   scales   fp32 [E, N] row-major: scale of expert e, row n.    (output)
 *   flags    0 or GQ_SCALE_POW2.
 *   stream   the CUDA stream to run on.  No workspace.
 */
gq_status gq_fp8_expert_rowwise(const void* w, int64_t E, int64_t N, int64_t K, void* out,
                                float* scales, uint32_t flags, gq_stream_t stream);

/*
 * mxfp8 cast along dim0 (pytorch/ao page "[mxfp8 moe training] fix mxfp8
 * a2a bench script; set mxfp8 a2a scaling type to RCEIL", Summary: the
 * dim0_mxfp8_floor cast benchmark and the RCEIL scaling type).  Every 32
 * consecutive elements of a row form a block sharing one power-of-two scale
 * 2^E, stored as the e8m0 byte E + 127; q = e4m3(fp32(x * 2^-E)), saturating
 * round-to-nearest-even.
 *   mode GQ_MX_FLOOR:  E = floor(log2(amax)) - 8 (the exponent of 448);
 *   mode GQ_MX_RCEIL:  E = ceil(log2(fp32(amax / 448))).
 * E is clamped to [-127, 127]; a block with amax 0 gets E = -127 (byte 0).
 *
 *   x        bf16 [M, K] row-major, 16-byte aligned.             (input)
 *   M, K     M >= 0, K >= 0, K % 32 == 0.
 *   out      e4m3 bytes [M, K] row-major, 16-byte aligned.       (output)
 *   scales   e8m0 bytes [M, K / 32] row-major.                   (output)
 *   stream   the CUDA stream to run on.  No workspace.
 */
#define GQ_MX_FLOOR 0
#define GQ_MX_RCEIL 1
gq_status gq_mxfp8_dim0(const void* x, int64_t M, int64_t K, void* out, uint8_t* scales,
                        int mode, gq_stream_t stream);

/*
 * The grad_weight GEMM of the MoE backward pass, one product per token group,
 * from the two quantized operands (pytorch/ao page "[moe training] use
 * smaller block sizes for per group scaling kernels to improve perf", MoE
 * fp8 training test: grad_weight = grad_output_t @ input, token groups):
 *
 *   out[g][n][k] = bf16( acc * (1 / sa[n][g]) * (1 / sx[g][k]) ),
 *   acc = sum over tokens t of group g of e4m3(qa_t[t][n]) * e4m3(qx[t][k]),
 *
 * acc accumulated in fp32 on the tensor cores (order unspecified),
 * reciprocals and products in IEEE fp32, bf16 by round-to-nearest-even.
 *
 *   qa_t     e4m3 [T, N] row-major (the gq_fp8_rowwise_t output: grad_output_t
 *            as a column-major (N, T) operand), 16-byte aligned.  (input)
 *   sa       fp32 [N, n_groups], the scales that produced qa_t.  (input)
 *   qx       e4m3 [T, K] row-major (the gq_fp8_colwise output of the layer
 *            input), 16-byte aligned.                            (input)
 *   sx       fp32 [n_groups, K], the scales that produced qx.    (input)
 *   T, N, K  >= 0, N % 16 == 0 and K % 16 == 0, each below 2^31.
 *   offs     device int32 [n_groups], END offsets along T (as for the other
 *            calls: running maximum, clamped to [0, T]); tokens past the last
 *            end belong to no group.                             (input)
 *   n_groups 1 .. GQ_MAX_GROUPS.
 *   out      bf16 [n_groups, N, K] row-major, 16-byte aligned; a group with
 *            no tokens gets zeros.                               (output)
 *   stream   the CUDA stream to run on.  No workspace.
 * Returns GQ_ERR_INVALID_ARG for a NULL or misaligned pointer, a negative
 * size or n_groups out of range; GQ_ERR_UNSUPPORTED for N or K not a
 * multiple of 16 or an extent of 2^31 or more.
 */
gq_status gq_grouped_wgrad(const void* qa_t, const float* sa, const void* qx, const float* sx,
                           int64_t T, int64_t N, int64_t K, const int32_t* offs,
                           int32_t n_groups, void* out, gq_stream_t stream);

/*
 * Colwise scaling with no allocation at all, not even a caller workspace.
 * The pytorch/ao pages have no counterpart to this entry point; it exists for
 * callers that cannot obtain device memory at the point where they quantize
 * -- a plugin running inside another runtime that owns the whole device heap
 * and lends out no workspace, or a hot path that must not call
 * cudaMalloc / cudaFree because those can synchronise the device.
 *
 * Arguments, layouts and results are those of gq_fp8_colwise without the
 * workspace.  The scratch lives in one fixed array of
 * GQ_NOALLOC_SCRATCH_BYTES inside the library's device memory, present on
 * every GPU that loads the library until the process exits.
 *   - Limit: gq_workspace_bytes(GQ_KIND_COLWISE, M, K, n_groups) must be at
 *     most GQ_NOALLOC_SCRATCH_BYTES (about n_groups * K <= 261,900);
 *     larger calls return GQ_ERR_UNSUPPORTED before enqueueing anything.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, that device current); make that first call
 *     before any stream capture.  Only a successful lookup is kept: if it
 *     fails (GQ_ERR_CUDA), the next call on that device tries again.
 *   - Each call clears the part of the array it uses (cudaMemsetAsync on
 *     `stream`), so leftovers of an earlier call do not matter.
 *   - All calls on a device share the array: calls whose GPU work may
 *     overlap (other streams, other host threads) race and corrupt each
 *     other's results.  Issue them on one stream, or order them.
 */
#define GQ_NOALLOC_SCRATCH_BYTES (1u << 20)
gq_status gq_fp8_colwise_noalloc(const void* x, int64_t M, int64_t K,
                                 const int32_t* offs, int32_t n_groups,
                                 void* out, float* scales, gq_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns GQ_ERR_TIMEOUT if any kernel since the last check gave up a
 * bounded wait, GQ_ERR_CUDA if the stream reports an error, else GQ_OK.
 * Not for the hot path: it blocks the host.
 */
gq_status gq_check_device_error(gq_stream_t stream);

/* Static English text for a status code. */
const char* gq_status_string(gq_status status);

/* Detail for the calling thread's last non-OK status ("" if none). */
const char* gq_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gq_version(void);

/*
 * Test hooks.  wait_timeout_ns sets the limit after which a waiting kernel
 * gives up (0 restores the 1 s default).  flags (other bits are
 * GQ_ERR_INVALID_ARG):
 *   bit 0  the next launches omit a completion signal, so that its waiters
 *          must time out and report GQ_ERR_TIMEOUT -- colwise: the count of
 *          the first phase-A tile of every two-phase strip of the first
 *          column slab (waiters: other thread blocks); rowwise_t: the
 *          amax-complete signal of the (first row band, first group) unit
 *          (waiters: the warps that would cast it), or, in a call that
 *          splits units, the count of the first split unit's first part
 *          (waiters: the other parts); grouped_wgrad: the release of thread
 *          block 0's first TMEM accumulator (waiter: the block's MMA warp);
 *   bit 1  rowwise_t never splits units across blocks (results are the
 *          same; the path a call takes when it does not find all of its
 *          blocks resident).
 * Process-wide; not thread-safe with concurrent calls.
 */
gq_status gq_debug_set(int flags, int64_t wait_timeout_ns);

/*
 * Tuning knob for the phase interleave of `kind`.  The colwise kernel
 * visits every tile of a group strip longer than 320 rows twice -- phase A
 * (amax) and phase B (scale + cast) -- and gives phase A a lead of `lag`
 * column slabs (128 columns each): phase A of slab d + lag is scheduled
 * alongside phase B of slab d.  A longer lead keeps phase B from waiting on
 * unfinished amax words; a shorter one keeps the re-read tiles in L2.
 * lag = 0 restores the automatic choice; larger values are clamped to the
 * number of slabs.  Results do not depend on it.
 * GQ_KIND_ROWWISE_T is accepted and has no effect: that kernel has no
 * cross-block schedule.  Process-wide; not thread-safe with concurrent
 * calls.  Returns GQ_ERR_INVALID_ARG for an unknown kind or a negative lag.
 */
gq_status gq_set_lag(int kind, int32_t lag);

#ifdef __cplusplus
}
#endif

#endif /* GQ_FP8_H */
