/*
 * tq.h -- C ABI of libtq: ternary weights after a 128-point block
 * Walsh-Hadamard rotation, on one GB300 GPU (sm_103a).
 *
 * The method (pages are named by address; none carries a title):
 *   offline   w' = W . blockdiag(H_128)/sqrt(128) along K, then per group of
 *             128 weights s = fp16(mean |w'|), t = clamp(rint(w'/s), -1, 1),
 *             packed as 2-bit codes or as five base-3 digits per byte
 *             (mhpq.cn/news/1159370 sec. 1.1, 1.3, 2.2, 3.1);
 *   run time  x' = blockdiag(H_128)/sqrt(128) . x along K (the rotation is
 *             absorbed on the activation side, mhpq.cn/news/1159370 sec. 2.3;
 *             zwxr.cn/news/303439, activation-side Hadamard), and
 *             y[m][n] = sum_g s[n][g] * sum_{k in g} t[n][k] * x'[m][k]
 *             accumulated in fp32 (fusion of transform and ternary matmul:
 *             mhpq.cn/news/1159370 sec. 3.3; dpshk.com/news/5289456 sec. 4.2).
 *
 * H[i][j] = (-1)^popcount(i & j) (dpshk.com/news/5289456 sec. 2.1).  The
 * transform runs butterfly stages h = 1, 2, 4, ..., 64 in fp32 and then
 * multiplies by c = RN_fp32(1/sqrt(128)) (xxqk.cn/news/652513 sec. 2).
 *
 * Layouts (row-major, leading dimensions in ELEMENTS of the pointed-to type):
 *   W      [N][ldw]   weights, fp32 or bf16          (N outputs, K inputs)
 *   x      [M][ldx]   activations, bf16 (fp32 also accepted by tq_fwht128)
 *   y      [M][ldy]   fp32 outputs
 *   scales [N][lds]   fp16 bit patterns, one per group of 128 (G = K/128)
 *   codes2 [N][ld2]   2-bit codes: code = t + 1 in bits 2*(k%4) of byte k/4
 *   codes3 [N][ld3]   base-3 bytes: byte j = sum_{i<5} (t[5j+i] + 1) * 3^i;
 *                     trits past K count as t = 0; bytes from ceil(K/5)
 *                     to tq_packed_ld(K, TQ_PACK_BASE3) are written as 0,
 *                     bytes past that (up to ld3) are not touched
 *
 * Every call:
 *   - takes DEVICE pointers owned by the caller (except where noted) and
 *     allocates no memory;
 *   - is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream); results are valid once the stream reaches that point;
 *   - validates its arguments on the host first and returns a status; a
 *     non-OK status means nothing was launched;
 *   - is thread-safe.  The library keeps per-device read-only setup and
 *     a few process-wide device status words (see tq_device_fault): a
 *     kernel that gives up a bounded wait sets a bit there, and
 *     tq_device_fault reads and clears them for every caller at once, so
 *     in a process with several host threads one thread's call may report
 *     (and clear) another thread's event.
 * Pointers must be 16-byte aligned and every row must start 16-byte aligned
 * (ld * element size % 16 == 0), else TQ_ERR_ALIGN.  K must be a positive
 * multiple of 128, else TQ_ERR_SHAPE.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TQ_API __attribute__((visibility("default")))
#else
#define TQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1, /* NULL pointer, bad enum, negative size         */
  TQ_ERR_SHAPE = 2,       /* K % 128 != 0, M out of range, ld too small    */
  TQ_ERR_ALIGN = 3,       /* pointer or row not 16-byte aligned            */
  TQ_ERR_UNSUPPORTED = 4, /* dtype/format combination not provided         */
  TQ_ERR_CUDA = 5,        /* a CUDA launch or query failed                 */
  TQ_ERR_RANGE = 6,       /* activations out of the representable range   */
  TQ_ERR_TIMEOUT = 7      /* a kernel gave up a bounded wait (see below)   */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

typedef enum { TQ_PACK_2BIT = 1, TQ_PACK_BASE3 = 2, TQ_PACK_BOTH = 3 } tq_pack;

/* cudaStream_t, passed through untouched. */
typedef void *tq_stream;

/* Human-readable name of a status code (static storage). */
TQ_API const char *tq_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
TQ_API int tq_version(void);

/* Minimum leading dimension in bytes of one packed layout for K inputs:
 * K/4 for TQ_PACK_2BIT; ceil(K/5) rounded up to 16 for TQ_PACK_BASE3.
 * Returns -1 for a bad K or format. */
TQ_API int64_t tq_packed_ld(int64_t K, int fmt);

/* Block FWHT-128 along K of `rows` rows:
 *   y[r][128g + i] = c * sum_j H[i][j] x[r][128g + j]
 * computed in fp32 (stages h = 1..64, then * c) and rounded once to yt.
 * xt in {TQ_F32, TQ_BF16}; yt in {TQ_F32, TQ_BF16, TQ_F16}.  With an fp32
 * output the result is bit-identical to the staged fp32 definition.
 * x == y is allowed when xt == yt and ldx == ldy (in place); other
 * overlaps are undefined.  rows == 0 is a no-op. */
TQ_API tq_status tq_fwht128(const void *x, int xt, int64_t ldx, void *y, int yt, int64_t ldy,
                     int64_t rows, int64_t K, tq_stream stream);

/* Offline quantise + pack (mhpq.cn/news/1159370 sec. 1.1 absmean
 * ternarisation, sec. 1.3 fp16 scale per 128, sec. 3.1 packing):
 * for every row n and group g, w' = FWHT-128 of W[n][128g .. 128g+127]
 * (fp32, as tq_fwht128), sum |w'| by the halving tree (h = 64 .. 1),
 * s = fp16_RN(sum * 2^-7), t = clamp(rint(w' / s), -1, 1) with IEEE
 * division and ties to even (t = 0 when s == 0).  Codes and scales are
 * bit-exact with that definition.  wt in {TQ_F32, TQ_BF16}.  fmt selects
 * which of codes2 / codes3 are written (the other may be NULL); scales is
 * always written.  ld2 >= K/4, ld3 >= tq_packed_ld(K, TQ_PACK_BASE3),
 * lds >= K/128 (fp16 elements, lds * 2 % 16 == 0 not required). */
TQ_API tq_status tq_quantize_pack(const void *W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt,
                           uint8_t *codes2, int64_t ld2, uint8_t *codes3, int64_t ld3,
                           uint16_t *scales, int64_t lds, tq_stream stream);

/* Decode GEMV / skinny GEMM, 1 <= M <= 16, FWHT of x fused into the kernel
 * (no workspace):  y[m][n] = sum_g s[n][g] sum_{k in g} t[n][k] x'[m][k]
 * with x' = FWHT-128(x) in fp32, then carried at reduced precision: on the
 * tensor-memory kernel (tq_gemv_path) as three e4m3 pieces per element under
 * a power-of-two scale per group and row of x (within max(2^-12 |x'|, 2^-15
 * max|x'|) of it, the maximum over the element's group), on the mma.sync
 * kernel rounded to fp16; products and sums in fp32.  fmt is TQ_PACK_2BIT or
 * TQ_PACK_BASE3 (codes laid out as above); x is bf16.  Accuracy against the
 * fp64 definition: relative L2 error <= 2e-3.  N == 0 is a no-op.  y must
 * not overlap the inputs.  The tensor-memory kernel adds its partial sums in
 * a fixed order (repeated calls give identical bits); the mma.sync kernel
 * does not. */
TQ_API tq_status tq_gemv(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                  int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                  tq_stream stream);

/* tq_gemv with flags (0 = exactly tq_gemv).
 *   TQ_GEMV_WEIGHTS_READY  codes and scales were completely written before
 *       the work that precedes this call on `stream` started (inference
 *       weights written once, long before).  The kernel may then start
 *       streaming them while that preceding work is still finishing
 *       (programmatic dependent launch); x is still read only after it has
 *       finished.  Without the flag every input waits for it.
 *   TQ_GEMV_TEST_STALL (for testing the failure path, not for production
 *       use): the first CTA of the tensor-memory kernel never issues the
 *       copy of its first stage of codes, so its pipeline waits run out, and
 *       every bounded wait of the launch gives up after about 20 ms instead
 *       of about 2 s.  The launch winds down as after a real stall (no trap,
 *       no fault, the context stays usable); tq_device_fault then returns
 *       TQ_ERR_TIMEOUT and the rows of y of the stalled CTA's cluster are not
 *       written.  TQ_ERR_UNSUPPORTED when the shape takes the mma.sync
 *       kernel (which has no waits).
 *   TQ_GEMV_X_ROTATED  x is already rotated: fp32 x' = FWHT-128(x), M rows
 *       of ldx floats (4-byte aligned), as tq_gemv_rotate_next writes it for
 *       the next layer; it is read instead of bf16 x and not rotated again.
 *       Tensor-memory kernel only (TQ_ERR_UNSUPPORTED otherwise).
 * Unknown flag bits: TQ_ERR_INVALID_ARG.  Everything else as tq_gemv. */
enum { TQ_GEMV_WEIGHTS_READY = 1, TQ_GEMV_X_ROTATED = 2, TQ_GEMV_TEST_STALL = 0x100 };
TQ_API tq_status tq_gemv_ex(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                            int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                            unsigned int flags, tq_stream stream);

/* tq_gemv_ex that also hands its output to the next layer already rotated
 * (the activation transform fused into the producer of x, dpshk.com/news/
 * 5289456 sec. 4.2, mhpq.cn/news/1159370 sec. 3.3, for decode): besides y it
 * writes x'_next = FWHT-128(y) in fp32 into xnext (M rows of ldxn >= N
 * floats, 4-byte aligned), computed from the fp32 y in the staged order --
 * the x of a following tq_gemv_ex(..., TQ_GEMV_X_ROTATED) whose x is this
 * call's y (K_next = N).  N must be a multiple of 128.  In the cluster
 * reduction rank 0 then adds the partial sums of all rows of its tiles (it
 * needs whole groups), so the call may plan a different K split than
 * tq_gemv_ex.  flags: TQ_GEMV_WEIGHTS_READY, TQ_GEMV_X_ROTATED (x is itself
 * a previous call's xnext), TQ_GEMV_TEST_STALL.  Tensor-memory kernel only
 * (TQ_ERR_UNSUPPORTED otherwise).  xnext must not overlap x or y. */
TQ_API tq_status tq_gemv_rotate_next(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales,
                                     int64_t lds, int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M,
                                     float *y, int64_t ldy, unsigned int flags, float *xnext, int64_t ldxn,
                                     tq_stream stream);

/* Which kernel tq_gemv runs for a shape (introspection; launches nothing):
 *   TQ_GEMV_TENSOR_MEMORY  2-bit or base-3 codes, any M, when one CTA's share
 *                          of the rotated activations fits in shared memory
 *                          (a K slice of up to 16 CTAs of a cluster; 2-bit:
 *                          K up to about 280 thousand at M <= 2, 150
 *                          thousand at M = 16; base-3 about two thirds of
 *                          that; when the rows of x do not fit one launch
 *                          they are split evenly over up to four launches):
 *                          weights unpacked to fp8 in tensor memory,
 *                          activations as three e4m3 pieces, tcgen05 MMAs;
 *   TQ_GEMV_MMA_SYNC       everything else (larger K): fp16 x' in shared
 *                          memory, weights as fp16 on mma.sync (16-row
 *                          tiles).
 * Queries device properties of the current device on first use.  Returns
 * -TQ_ERR_INVALID_ARG / -TQ_ERR_SHAPE for arguments tq_gemv would reject
 * with those codes. */
enum { TQ_GEMV_TENSOR_MEMORY = 1, TQ_GEMV_MMA_SYNC = 2, TQ_GEMV_CUDA_CORES = 3 };
TQ_API int tq_gemv_path(int64_t N, int64_t K, int64_t M, int fmt);

/* The tensor-memory kernel's work split for a shape (introspection; launches
 * nothing).  *ctas_per_cluster (1, 2, 3, 4, 6, 7, 8, or 16 where no smaller
 * cluster fits the activations): the CTAs of a thread-block cluster that
 * split the K groups of its tiles and add their partial sums in distributed
 * shared memory; *clusters: the clusters of a launch, each
 * owning a range of 128-row tiles; *launches (1 .. 4): the launches the rows
 * of x are split over (the split reported is the first launch's, which takes
 * M / launches rows, rounded down).  chained != 0 plans tq_gemv_rotate_next
 * (N a multiple of 128).  fmt: TQ_PACK_2BIT or TQ_PACK_BASE3.  Returns TQ_OK;
 * TQ_ERR_UNSUPPORTED when the shape takes another kernel (tq_gemv_path);
 * TQ_ERR_INVALID_ARG for a null output or bad format; TQ_ERR_SHAPE as
 * tq_gemv_path, or a chained N that is not a multiple of 128.  Queries the
 * current device as tq_gemv_path does. */
TQ_API tq_status tq_gemv_plan(int64_t N, int64_t K, int64_t M, int fmt, int chained, int *ctas_per_cluster,
                              int *clusters, int *launches);

/* Bytes of caller-provided workspace tq_gemm needs for M x K activations:
 * a status word and the rotated activations in fp16 (256 + 2 M K bytes,
 * rounded up to 256), then 40 MiB for the fp32 partial tiles of a last wave
 * of tiles that the GEMM splits along K (see tq_gemm). */
TQ_API size_t tq_gemm_workspace_bytes(int64_t M, int64_t K);

/* Prefill GEMM, M >= 1 (tensor cores: tcgen05 MMA with fp16 operands and
 * fp32 accumulation in tensor memory):  same formula as tq_gemv.  Runs the
 * FWHT-128 of x into the workspace (fp16, overflow recorded in the status
 * word), then the GEMM, on `stream`.  When the output tiles leave a short
 * last wave on the GPU's SMs, those tiles are computed in K segments whose
 * partial sums go to the workspace and are added in a fixed order by a second
 * kernel (results are identical from call to call).  fmt is TQ_PACK_2BIT.
 * ws_bytes must be >= tq_gemm_workspace_bytes(M, K).  y must not overlap the
 * inputs. */
TQ_API tq_status tq_gemm(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                  int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                  void *workspace, size_t ws_bytes, tq_stream stream);

/* tq_gemm with flags.  TQ_GEMM_REUSE_ROTATED: the workspace already holds the
 * rotated activations of this same x (same M, K and values), left there by
 * the previous tq_gemm / tq_gemm_ex call on `workspace` -- e.g. the gate
 * projection before the up projection of a feed-forward block, which read
 * the same x.  The FWHT pre-pass is skipped and x is not read; the status
 * word keeps what the earlier call recorded (its fp16-overflow bit describes
 * the same x').  Whether x matches is the caller's contract: it is not
 * checked; with a workspace that holds no x' of this M and K the output is
 * meaningless, but every access stays inside the workspace.  x is still
 * validated like any argument, though not read.
 *
 * TQ_GEMM_TEST_STALL (for testing the failure path, not for production
 * use): the first CTA of the GEMM never issues the copy of its first stage
 * of activations, so its pipeline waits run out, and every bounded wait of
 * the launch gives up after about 20 ms instead of about 2 s.  The launch
 * winds down as after a real stall (no trap, no fault, the context stays
 * usable); tq_gemm_check_range then returns TQ_ERR_TIMEOUT and y is not
 * meaningful.
 *
 * Unknown flag bits return TQ_ERR_INVALID_ARG. */
enum { TQ_GEMM_REUSE_ROTATED = 1, TQ_GEMM_TEST_STALL = 0x100 };
TQ_API tq_status tq_gemm_ex(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                  int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                  void *workspace, size_t ws_bytes, unsigned int flags, tq_stream stream);

/* tq_gemm_ex that also hands its output to the next layer already rotated
 * (the activation transform fused into the producer of x: dpshk.com/news/
 * 5289456 sec. 4.2, mhpq.cn/news/1159370 sec. 3.3).  Besides y it writes
 * FWHT-128(y), computed in fp32 from the accumulators in the staged order and
 * rounded once to fp16, into next_ws -- the rotated activations of a
 * following tq_gemm_ex(..., TQ_GEMM_REUSE_ROTATED) on next_ws whose x is this
 * call's y (M rows, K_next = N), which then skips its pre-pass -- and records
 * their fp16 overflow in next_ws's status word (cleared first; read with
 * tq_gemm_check_range(next_ws)).  The fp16 x' comes from the fp32 y, not from
 * y rounded to bf16 as the plain chain would give it.  N must be a multiple
 * of 128 and next_ws_bytes >= tq_gemm_workspace_bytes(M, N); the output
 * tiles are then whole 128-column groups.  When a short last wave is split
 * along K (y 16-byte aligned, ldy % 4 == 0), the x' of those tiles is
 * computed after the fix-up from the finished fp32 y by the same staged
 * transform (bit-identical); otherwise the last wave is not split.  next_ws
 * must not overlap workspace.  Flags and everything else as tq_gemm_ex. */
TQ_API tq_status tq_gemm_rotate_next(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales,
                                     int64_t lds, int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M,
                                     float *y, int64_t ldy, void *workspace, size_t ws_bytes, unsigned int flags,
                                     void *next_ws, size_t next_ws_bytes, tq_stream stream);

/* Synchronises `stream`, then reads the status word the last tq_gemm left in
 * `workspace`: TQ_ERR_RANGE if a rotated activation overflowed fp16 (the
 * output is then not meaningful), else TQ_OK. */
TQ_API tq_status tq_gemm_check_range(const void *workspace, tq_stream stream);

/* Prefill GEMM that allocates nothing and needs no workspace argument.  The
 * published method has no counterpart; this entry exists for callers that cannot
 * allocate device memory themselves (code that runs inside a fixed memory
 * pool or arena, or plugins that may only use the buffers their host hands
 * them).  It computes exactly what tq_gemm computes, with the same kernels,
 * but takes the workspace from a fixed scratch array inside the library:
 *   - the array holds the rotated activations for M * K <= 16,777,216
 *     (e.g. 2048 x 8192); larger M * K returns TQ_ERR_SHAPE;
 *   - it lives in device memory of every GPU that loads the library, until
 *     the process exits (about 32 MiB per GPU);
 *   - every call looks up the array's device address with the device
 *     current (a host-side query); the first call on a device also loads the
 *     library's module there (set-up), so make that first call before any
 *     stream capture;
 *   - every call shares the one array and it keeps the last call's contents
 *     (the call clears the status word it uses); calls whose work overlaps
 *     on the GPU (different streams, or different host threads on the same
 *     device) race on it and must be serialised by the caller;
 *   - a bounded wait of the GEMM that ran out is recorded in the array's
 *     status word and reported by tq_device_fault (TQ_ERR_TIMEOUT);
 *   - an fp16 overflow of the rotated activations is NOT reported on this
 *     path (tq_gemm reports it through tq_gemm_check_range): the output may
 *     then hold inf or NaN.  With bf16 inputs this needs a 128-block of x
 *     whose 2-norm exceeds 65504.
 * No cudaMalloc, cudaFree or other allocating call is made.  Arguments,
 * layouts and other errors as for tq_gemm. */
TQ_API tq_status tq_gemm_noalloc(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                                 int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                                 tq_stream stream);

/* ------------------------------------------------------------------------
 * Layout variants: the ranked follow-ons of the method, each a parameter of
 * the same path.
 *   block   FWHT block size along K: 64, 128 or 256 (H_n from the popcount
 *           rule or the Sylvester recursion for any power of two,
 *           dpshk.com/news/5289456 sec. 2.1; block size against caches,
 *           xxqk.cn/news/652513 sec. 2.2).  The transform runs the stages
 *           h = 1 .. block/2 in fp32 and multiplies by RN_fp32(1/sqrt(block))
 *           (exactly 1/8 and 1/16 for 64 and 256).
 *   group   weights per fp16 scale: 128 or 256 (mhpq.cn/news/1159370 sec.
 *           1.4: 16/256 = 0.0625 bit of scale per weight); the absmean sum is
 *           the halving tree over the group (h = group/2 .. 1), times
 *           1/group.
 *   flags   TQ_LAYOUT_RESIDUAL: the residual two-pass ternarisation
 *           (xxqk.cn/news/652513 sec. 3, residual calibrator): after the
 *           first pass (s1, t1) the residual r = w' - s1 t1 (a zero trit
 *           dequantises to 0) is rotated by the same block transform and
 *           ternarised with scales s2 of its own.  Since the normalised
 *           transform is its own inverse, the residual pass meets the
 *           unrotated activations:
 *             y = sum s1 sum t1 x' + sum s2 sum t2 x.
 * {128, 128, 0} is the method itself; a NULL layout means that.  K must be a
 * multiple of max(block, group).  A layout's codes hold Keff = K trits per
 * row (2K with TQ_LAYOUT_RESIDUAL: the first pass's, then the residual
 * pass's), packed over all Keff as for the plain layout; its scales hold
 * K/group per row (twice with the residual pass: the s1, then the s2). */
typedef struct {
  int32_t block;
  int32_t group;
  uint32_t flags;
} tq_layout;
enum { TQ_LAYOUT_RESIDUAL = 1 };

/* Minimum leading dimensions of a layout's codes (bytes, fmt TQ_PACK_2BIT or
 * TQ_PACK_BASE3) and scales (elements); -1 for bad arguments. */
TQ_API int64_t tq_layout_codes_ld(int64_t K, int fmt, const tq_layout *lay);
TQ_API int64_t tq_layout_scales_ld(int64_t K, const tq_layout *lay);

/* tq_fwht128 at block size 64, 128 or 256 (K a multiple of block); same
 * arguments, dtypes, exactness and in-place rule. */
TQ_API tq_status tq_fwht(const void *x, int xt, int64_t ldx, void *y, int yt, int64_t ldy, int64_t rows,
                         int64_t K, int block, tq_stream stream);

/* tq_quantize_pack under a layout.  ld2 >= tq_layout_codes_ld(K, 2-bit),
 * ld3 >= tq_layout_codes_ld(K, base-3), lds >= tq_layout_scales_ld(K).  Codes
 * and scales are bit-exact with the definition.  A layout other than
 * {128, 128, 0} runs a general kernel that keeps a row's trits in shared
 * memory: TQ_ERR_UNSUPPORTED when Keff exceeds about 190 thousand. */
TQ_API tq_status tq_quantize_pack_layout(const void *W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt,
                                         uint8_t *codes2, int64_t ld2, uint8_t *codes3, int64_t ld3,
                                         uint16_t *scales, int64_t lds, const tq_layout *lay, tq_stream stream);

/* tq_gemv_ex under a layout: K is the activations' K; codes hold Keff.  A
 * layout other than {128, 128, 0} runs on the tensor-memory kernel only
 * (TQ_ERR_UNSUPPORTED where that kernel does not take the shape).  Flags as
 * tq_gemv_ex. */
TQ_API tq_status tq_gemv_layout(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                                int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                                const tq_layout *lay, unsigned int flags, tq_stream stream);

/* Workspace of tq_gemm_layout: as tq_gemm_workspace_bytes with the rotated
 * activations of both passes (M x Keff fp16). */
TQ_API size_t tq_gemm_workspace_bytes_layout(int64_t M, int64_t K, const tq_layout *lay);

/* tq_gemm_ex under a layout: the pre-pass writes x' (block transform) and,
 * with the residual pass, x itself beside it, both fp16 with the overflow
 * check; the GEMM then runs over Keff.  Flags as tq_gemm_ex. */
TQ_API tq_status tq_gemm_layout(const uint8_t *codes, int64_t ldc, int fmt, const uint16_t *scales, int64_t lds,
                                int64_t N, int64_t K, const void *x, int64_t ldx, int64_t M, float *y, int64_t ldy,
                                void *workspace, size_t ws_bytes, const tq_layout *lay, unsigned int flags,
                                tq_stream stream);

/* ---- 2:4-sparse ternary weights (mhpq.cn/news/1159370 sec. 1.2: two of
 * every four weights kept at regular positions, the kept ones ternarised;
 * sec. 1.1: the absmean rule).  Per quad of four consecutive k of a rotated
 * group w' = FWHT-128(w), the two largest |w'| are kept (a tie goes to the
 * lower index); the group's fp16 scale is the round-to-nearest mean |w'| of
 * its 64 kept weights (halving-tree sum in k order, times 2^-6); a kept
 * weight's trit is clamp(rint(w' / scale), -1, 1), a pruned one's is 0.
 *
 * Codes, one tensor holding mask and trits (row-major, ldc bytes per row,
 * 24 per group of 128: 1.5 bits per weight, plus 0.125 of scale): quad j of
 * a group has pattern p in 0..5 (its kept positions i0 < i1 in the order
 * (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)) and code c = 9 p + 3 (t[i0] + 1) +
 * (t[i1] + 1) < 54; the low nibble of c is nibble j % 2 of byte j / 2 of the
 * group, its two high bits are bits 2 (j % 4) of byte 16 + j / 4.  Scales
 * fp16 [N][K/128], row stride lds elements. */

/* Bytes of codes per row: 24 K / 128; -1 unless K is a positive multiple of 128. */
TQ_API int64_t tq_sparse24_ld(int64_t K);

/* Quantise + pack W (wt TQ_F32 or TQ_BF16, [N][K], ldw elements, 16-byte
 * aligned rows) into the 2:4 codes and scales.  Codes and scales are
 * bit-exact with the definition above (fp32 staged FWHT-128, IEEE division).
 * Requires K % 128 == 0, ldc >= tq_sparse24_ld(K), ldc % 4 == 0 and a 4-byte
 * aligned codes pointer (the codes are written as 32-bit words),
 * lds >= K/128, 2-byte aligned scales.  One launch; no allocation. */
TQ_API tq_status tq_quantize_pack_sparse24(const void *W, int wt, int64_t N, int64_t K, int64_t ldw,
                                           uint8_t *codes, int64_t ldc, uint16_t *scales, int64_t lds,
                                           tq_stream stream);

/* Workspace of tq_gemv_sparse24: the fp32 FWHT-128 of x ([M][K], rounded up
 * to 256 bytes) and, when the K groups are split into several slices, fp32
 * partial sums [slices][M][N].  The split depends on the shape only: enough
 * slices that M x (slice groups) x 516 bytes fit 96 KiB, and, for a short N,
 * up to ceil(512 / ceil(N / 32)) slices of at least 8 groups, the groups per
 * slice rounded up to a multiple of 8 where that still fits.  0 for bad
 * arguments. */
TQ_API size_t tq_gemv_sparse24_workspace_bytes(int64_t N, int64_t K, int64_t M);

/* y [M][N] fp32 = sum_g s[n][g] sum_{k in g} t[n][k] x'[m][k] over the 2:4
 * codes, x bf16 [M][K] (16-byte aligned rows), M = 1..16.  Two kernels:
 *   - the tensor-memory GEMV of tq_gemv (TQ_GEMV_TENSOR_MEMORY, see
 *     tq_gemv_sparse24_path) when the codes are 16-byte aligned with
 *     ldc % 16 == 0 and K / 128 is even and at least 4: each quad's code
 *     expands through a table into its four weights as fp8 bytes in tensor
 *     memory (the pruned ones as zeros), x' is carried as the three e4m3
 *     pieces of tq_gemv, and one launch does the rest (the workspace is not
 *     used);
 *   - otherwise (TQ_GEMV_CUDA_CORES) a pre-pass writes x' = FWHT-128(x) in
 *     fp32 to the workspace, a decode kernel adds only the kept weights
 *     (sign-select adds, fp32 accumulation, each group's sum scaled by its
 *     fp16 scale), and, when K is split, a third kernel adds the slices in
 *     order.
 * Results are identical from call to call.  ws_bytes >=
 * tq_gemv_sparse24_workspace_bytes(N, K, M) in both cases; the workspace must
 * not overlap the other arguments.  The codes are read as 32-bit words at
 * least: 4-byte aligned codes pointer and ldc % 4 == 0.  Codes outside 0..53
 * are read as a quad of zeros. */
TQ_API tq_status tq_gemv_sparse24(const uint8_t *codes, int64_t ldc, const uint16_t *scales, int64_t lds,
                                  int64_t N, int64_t K, const uint16_t *x, int64_t ldx, int64_t M, float *y,
                                  int64_t ldy, void *workspace, size_t ws_bytes, tq_stream stream);

/* Which kernel tq_gemv_sparse24 runs for a shape whose codes are 16-byte
 * aligned with ldc % 16 == 0 (introspection; launches nothing; queries the
 * current device on first use): TQ_GEMV_TENSOR_MEMORY or TQ_GEMV_CUDA_CORES.
 * -TQ_ERR_INVALID_ARG / -TQ_ERR_SHAPE for arguments tq_gemv_sparse24 would
 * reject with those codes. */
TQ_API int tq_gemv_sparse24_path(int64_t N, int64_t K, int64_t M);

/* Prefill GEMM of the 2:4 codes: tq_gemm on the tcgen05 tensor cores with
 * the 2:4 codes, M >= 1 rows of bf16 x.  The pruned weights are expanded
 * into the dense fp16 weight tiles in shared memory (dense kind::f16 MMAs;
 * the 2:4 sparse MMA form is not used), so the time is that of tq_gemm plus
 * the code expansion.  Same workspace (tq_gemm_workspace_bytes(M, K)), the
 * same fp16 x' overflow report through tq_gemm_check_range, the same
 * accuracy and repeatability.  The codes are read as 8-byte words: 8-byte
 * aligned codes pointer and ldc % 8 == 0. */
TQ_API tq_status tq_gemm_sparse24(const uint8_t *codes, int64_t ldc, const uint16_t *scales, int64_t lds,
                                  int64_t N, int64_t K, const uint16_t *x, int64_t ldx, int64_t M, float *y,
                                  int64_t ldy, void *workspace, size_t ws_bytes, tq_stream stream);

/* Failure detection.  Every wait inside a kernel (pipeline barriers between
 * the warps that copy weights and the warps that compute) is bounded by a
 * wall-clock limit of about 2 s.  A kernel whose wait runs out stops early,
 * lets its in-flight copies land, records the event in a device status word
 * and exits, so the CUDA context stays usable; its outputs are then not
 * meaningful.  This call synchronises the device, returns TQ_ERR_TIMEOUT if
 * any kernel recorded such an event since the previous call (and clears the
 * record); else TQ_ERR_RANGE if a tensor-memory GEMV met a group of rotated
 * activations outside what its fp8 pieces represent (max |x'| of the group
 * at least 2^108 or infinite, or positive but below 2^-93: those groups'
 * products saturate or flush, and y is not meaningful); else TQ_OK;
 * TQ_ERR_CUDA if the device could not be queried. */
TQ_API tq_status tq_device_fault(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
