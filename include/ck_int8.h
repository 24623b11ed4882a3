/*
 * ck_int8.h -- C ABI of the INT8 quantized linear layer for one NVIDIA GB300 (sm_103a).
 *
 *   y[m,n] = out( float(acc[m,n]) * x_scale[m] * w_scale[n] (+ bias[n]) ),  out = bf16, fp16 or fp32
 *   acc[m,n] = sum_k q[m,k] * w[n,k]            exact int32
 *   q = clamp(rint(v / x_scale), -127, 127),  x_scale = max|v| / 127
 *   v = x (TENSORWISE, PER_ROW) or x @ H (CONVROT)
 *
 * Sources (comfy-kitchen pages):
 *   - issue #280 "INT8 linears on sm_121 (GB10 / DGX Spark) run at ~37% of tensor-core
 *     peak via cutlass_int8_dequant; a fused-dequant Triton GEMM reaches ~88%,
 *     bit-identical", sections "Kernel used" (int32 accumulator over K; fp32 epilogue
 *     acc * x_scale[m] * w_scale[n] (+ bias[n]) -> output dtype; int64 offsets) and
 *     "Exactness" (same operation order; tensor-wide scales; no-bias calls);
 *   - issue #278 "int8_linear silently falls back to a DP4A-emulated INT8 GEMM on Volta
 *     (sm_70) ...", section "2. quantize_int8_rowwise raises instead of falling back"
 *     (the per-row quantize op) and "Suggested fix" (ConvRot: stored weight
 *     W_rot = W @ H^T, activation rotated online x_rot = x @ H, no inverse rotation);
 *   - issue #136 "INT8 GEMM kernels index the output in int32: illegal memory access
 *     once m*n >= 2**31", sections "Summary" and "Suggested fix" (64-bit addressing);
 *     section "Minimal reproduction" gives the call int8_linear(x, w, ws, out_dtype)
 *     with x bf16 [m,k], w int8 [n,k], ws fp32 [n].
 *
 * Conventions shared by every entry point
 *   - All tensors are dense row-major device buffers owned by the caller.  The library
 *     keeps no pointer after a call returns and allocates no device memory per call.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *     runs asynchronously; no entry point synchronises the host except
 *     ck_device_error() and ck_selftest_wait_timeout().
 *   - Every entry point returns a ck_status_t.  On a non-OK status nothing was
 *     enqueued (argument and device checks run first) unless the status is
 *     CK_ERR_CUDA from a launch; ck_last_error() then describes the failure.
 *   - Sizes are int64; every device address is computed in 64 bits, so M*N, M*K and
 *     N*K may exceed 2^31.  Each single dimension must stay below 2^31 (tensor-copy
 *     coordinates are 32-bit).
 *   - Requirements (CK_ERR_INVALID_ARG otherwise): M, N, K >= 1; K % 16 == 0;
 *     N % 8 == 0; K <= 131072 (so |acc| <= 127*127*K fits int32); every pointer
 *     16-byte aligned; CONVROT needs K % 128 == 0.  M == 0 is accepted and does nothing
 *     (after the shape checks); the buffers sized by M may then be NULL.
 *   - Device: compute capability 10.3 (GB300) only, else CK_ERR_UNSUPPORTED_DEVICE.
 *     There is no fallback path of any kind.
 *   - CUDA graphs: every entry point except ck_quantize_int8_tensorwise_noalloc (whose
 *     capture is not covered here) and ck_int8_linear_host (refused) may be captured (cudaStreamBeginCapture) and the
 *     graph replayed with new data in the same buffers; the results equal uncaptured
 *     calls.  Make one uncaptured call per device first (it sets kernel attributes and
 *     looks up the library's device symbols).  Under capture, ck_int8_linear in
 *     tensorwise mode runs its quantize as two launches plus a separate weight widening
 *     (the single launch exchanges block maxima under a per-call tag, which a replay would
 *     repeat), and no GEMM splits its last wave along K (the split's arrival counters are
 *     tagged the same way): same results, a few microseconds slower per call.
 *   - Bounded waits: kernels whose threads wait on each other give up after 2 s instead
 *     of hanging, record a bit in a device error word and exit normally; the entry point
 *     that enqueued them has long returned CK_OK by then.  ck_device_error() reads that
 *     word: a caller that must know a result is sound checks it after synchronizing.
 */
#ifndef CK_INT8_H
#define CK_INT8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CK_TENSORWISE = 0, /* one x_scale for the whole activation, one w_scale          */
    CK_PER_ROW = 1,    /* x_scale per activation row, w_scale per output channel     */
    CK_CONVROT = 2     /* like CK_PER_ROW on x @ H; w is the pre-rotated W @ H^T      */
} ck_mode_t;

/* Output element type of the dequant epilogue (the out_dtype of int8_linear).  The fp32
 * value is the same for every type; bf16 and fp16 round it to nearest even (fp16
 * overflows to +-inf, keeps subnormals); fp32 stores it as is. */
typedef enum {
    CK_OUT_BF16 = 0,
    CK_OUT_F16 = 1,
    CK_OUT_F32 = 2
} ck_dtype_t;

typedef enum {
    CK_OK = 0,
    CK_ERR_INVALID_ARG = 1,
    CK_ERR_UNSUPPORTED_DEVICE = 2,
    CK_ERR_CUDA = 3,
    CK_ERR_TIMEOUT = 4
} ck_status_t;

/* Per-row activation quantize (issue #278, quantize_int8_rowwise).
 *   x:       bf16 [M,K] device, read only.
 *   rotate:  0 = none; 1 = ConvRot, v = x @ H with H block-diagonal of the normalized
 *            128x128 Sylvester Hadamard matrix (needs K % 128 == 0), evaluated as an
 *            fp32 fast Walsh-Hadamard transform (spans 1..64 ascending, then times
 *            fp32(1/sqrt(128))); v is never rounded to bf16.
 *   q:       int8 [M,K] device, written: clamp(rint(v / x_scale[m]), -127, 127), rint
 *            rounding half to even, v / x_scale one correctly rounded fp32 division.
 *   x_scale: fp32 [M] device, written: max_k |v[m,k]| / 127 (fp32 division).  A row
 *            whose scale is 0 gets q = 0. */
int ck_quantize_int8_rowwise(const void *x, int64_t M, int64_t K, int rotate, int8_t *q, float *x_scale,
                             void *stream);

/* Tensorwise activation quantize (issue #280, "INT8 tensorwise linears"; tensor-wide
 * scales): x_scale[0] = max_{m,k} |x| / 127, q as above with that single scale.
 *   workspace: device scratch of at least ck_quantize_tensorwise_workspace_size()
 *   bytes (per-block partial maxima); its content on entry does not matter. */
size_t ck_quantize_tensorwise_workspace_size(void);
int ck_quantize_int8_tensorwise(const void *x, int64_t M, int64_t K, int8_t *q, float *x_scale,
                                void *workspace, size_t workspace_bytes, void *stream);

/* Tensorwise quantize for callers that cannot allocate device memory.  The pages have no
 * counterpart of this entry point.  It serves code that may not touch an allocator while
 * it runs: real-time loops that reserve their whole memory budget up front (an
 * allocation can block, or fail on a fragmented heap, at a moment they cannot afford),
 * hosts whose own memory manager must account for every byte on the device, and plugins
 * inside such hosts, which see only the buffers they are handed.  It computes exactly
 * what ck_quantize_int8_tensorwise computes, but keeps its partial maxima in a 16 KiB
 * array built into the library (present on every GPU that loads it, until the process
 * exits) instead of a caller workspace, and calls no allocation routine.
 *   x, q, x_scale: as for ck_quantize_int8_tensorwise (caller-owned device buffers).
 *   Limit: M*K <= 134,217,728 values, else CK_ERR_INVALID_ARG (nothing enqueued).
 *   The first call in a CUDA context looks up the array's device address there and keeps
 *   it; make that first call before any stream capture begins.  After a device reset the
 *   next call looks it up again.  All calls share the array, which keeps the last call's
 *   contents (nothing in it has to start at zero: a call reads only slots it wrote
 *   itself), so calls that overlap on the GPU (other streams or threads) race and may
 *   return a wrong scale: serialize them. */
int ck_quantize_int8_tensorwise_noalloc(const void *x, int64_t M, int64_t K, int8_t *q, float *x_scale,
                                        void *stream);

/* Bytes of device workspace ck_int8_linear needs for this problem (>= 0).  The
 * workspace holds the quantized activation and the weight as bf16 integers (the
 * tensor-core operand format), the activation scales and the tensorwise partial maxima. */
size_t ck_int8_linear_workspace_size(int64_t M, int64_t N, int64_t K, int mode);

/* Where ck_int8_linear leaves, in the caller's workspace, the activation quantize of its
 * last call (issue #278, section "2. quantize_int8_rowwise raises instead of falling
 * back": the codes q and the scales; issue #280, "Exactness": tensor-wide scales):
 *   *codes_offset:   byte offset of q as bf16 integers [M,K] row-major (every value an
 *                    integer in [-127, 127], exact in bf16; a zero may carry either sign);
 *   *x_scale_offset: byte offset of x_scale fp32 [M] (CK_PER_ROW, CK_CONVROT) or [1]
 *                    (CK_TENSORWISE).
 * The layout depends only on (M, N, K, mode), so a test can read what the layer's own
 * preparation kernel computed and compare it with a reference bit for bit.  Host only:
 * nothing is enqueued.  CK_ERR_INVALID_ARG for a bad mode, negative sizes or NULL
 * outputs. */
int ck_int8_linear_workspace_views(int64_t M, int64_t N, int64_t K, int mode, size_t *codes_offset,
                                   size_t *x_scale_offset);

/* The INT8 linear layer (issue #136 repro API int8_linear(x, w, ws, out_dtype) with
 * the optional bias of issue #280):
 *   x:       bf16 [M,K] activations, device.
 *   w:       int8 [N,K] weights, device; values in [-127, 127].  For CK_CONVROT this is
 *            the pre-rotated, per-row quantized W @ H^T, used as is.
 *   w_scale: fp32 [N] (CK_PER_ROW, CK_CONVROT) or fp32 [1] (CK_TENSORWISE).
 *   bias:    bf16 [N] or NULL.
 *   residual: [M,N] of out_dtype or NULL, added after the bias (issue #280, "Kernel
 *            used", mentions residual-fused calls); may be y itself (in-place update).
 *   y:       [M,N] of out_dtype (a ck_dtype_t), written.
 *            y = out((((float(acc) * xs) * ws) + bias) + residual) with every fp32
 *            operation rounded separately, in that order, and out the rounding of
 *            ck_dtype_t.
 *   workspace/workspace_bytes: device scratch of ck_int8_linear_workspace_size() bytes.
 * No int32 intermediate is ever written to device memory.  An out_dtype outside
 * ck_dtype_t gives CK_ERR_INVALID_ARG.
 * In CK_TENSORWISE mode the preparation kernel's blocks exchange their maxima and wait
 * for each other (bounded, 2 s).  A block that gives up makes x_scale NaN, so every
 * element of y is NaN rather than plausible, and sets a bit in the device error word:
 * ck_device_error() is how a caller learns of it. */
int ck_int8_linear(const void *x, const int8_t *w, const float *w_scale, const void *bias, const void *residual,
                   void *y, int64_t M, int64_t N, int64_t K, int mode, int out_dtype, void *workspace,
                   size_t workspace_bytes, void *stream);

/* The layer with the weight's GEMM operand prepared once, for callers that run a layer
 * many times and can hold 2 B per weight on the device: the int8 weight (issue #136's w,
 * int8 [N,K]) widened to its bf16 codes (every value an integer in [-127, 127], exact in
 * bf16), which ck_int8_linear would otherwise redo in every call's preparation launch.
 *   ck_int8_weight_codes: w int8 [N,K] device (read) -> w_codes bf16 [N,K] device
 *     (written; caller-owned, N*K*2 bytes).  K % 16 == 0.
 *   ck_int8_linear_codes: exactly ck_int8_linear (same arguments, same results bit for
 *     bit) with w_codes in place of w; its workspace,
 *     ck_int8_linear_codes_workspace_size(M, N, K, mode) bytes, holds no widened weight. */
int ck_int8_weight_codes(const int8_t *w, int64_t N, int64_t K, void *w_codes, void *stream);
size_t ck_int8_linear_codes_workspace_size(int64_t M, int64_t N, int64_t K, int mode);
int ck_int8_linear_codes(const void *x, const void *w_codes, const float *w_scale, const void *bias,
                         const void *residual, void *y, int64_t M, int64_t N, int64_t K, int mode, int out_dtype,
                         void *workspace, size_t workspace_bytes, void *stream);

/* The same layer with the activation read from and the output written to HOST memory
 * (issue #136's int8_linear(x, w, ws, out_dtype) called on host tensors; the weight,
 * its scales and the bias stay resident on the device):
 *   x_host:  bf16 [M,K] host memory, read.  y_host: [M,N] of out_dtype host memory,
 *            written.  Page-locked (pinned) host memory lets the copies overlap the
 *            kernels; pageable memory gives the same result with the copies serialized.
 *   w, w_scale, bias, mode, out_dtype: as for ck_int8_linear (device memory); no residual.
 *   slab_rows: rows per pipeline slab (0: about 64 MB of output per slab).  The call
 *            cuts M into slabs and overlaps, on two internal copy streams of the current
 *            context (made on its first call there) and the caller's stream, the copy of
 *            slab i+1 to the device, the kernels of slab i and the copy of slab i-1 back.
 *            CK_TENSORWISE copies all of x first (its one scale needs every value).
 *   workspace: ck_int8_linear_host_workspace_size(M, N, K, mode, out_dtype, slab_rows)
 *            bytes of device memory (two activation and two output slab buffers, the
 *            codes, the widened weight).
 * y_host is complete once the caller's stream has completed past this call (the stream
 * waits for the last copy).  The results equal ck_int8_linear's bit for bit.  Cannot be
 * captured into a CUDA graph (CK_ERR_INVALID_ARG). */
size_t ck_int8_linear_host_workspace_size(int64_t M, int64_t N, int64_t K, int mode, int out_dtype,
                                          int64_t slab_rows);
int ck_int8_linear_host(const void *x_host, const int8_t *w, const float *w_scale, const void *bias, void *y_host,
                        int64_t M, int64_t N, int64_t K, int mode, int out_dtype, int64_t slab_rows, void *workspace,
                        size_t workspace_bytes, void *stream);

/* ConvRot weight preparation (issue #278, "Suggested fix": the stored weight is
 * W_rot = W @ H^T; since H is symmetric, row n of it is row n of W times H), quantized
 * per output row, once per layer:
 *   W:       fp32 [N,K] device, read only; K % 128 == 0.
 *   w:       int8 [N,K] device, written: clamp(rint(v / w_scale[n]), -127, 127) with v the
 *            rotated row (the same fp32 block transform as ck_quantize_int8_rowwise's
 *            rotation), one IEEE fp32 division, rint half to even.
 *   w_scale: fp32 [N] device, written: max_k |v[n,k]| / 127.
 * The result is the w / w_scale that ck_int8_linear takes in CK_CONVROT mode. */
int ck_convrot_prepare_weight(const float *W, int64_t N, int64_t K, int8_t *w, float *w_scale, void *stream);

/* The 16-bit-activation path of the same layer (issue #278, "Suggested fix": the INT8
 * weight dequantized on the fly, the GEMM on 16-bit tensor cores, the weight keeping its
 * INT8 footprint; for ConvRot the activation rotated online and the weight used as
 * stored, in the rotated basis).  No activation quantize:
 *   y[m,n] = out( (fp32( sum_k a[m,k] * w[n,k] ) * w_scale[n] + bias[n]) + residual[m,n] )
 *   a = x (CK_TENSORWISE, CK_PER_ROW) or bf16_rne(x @ H) (CK_CONVROT, K % 128 == 0; the
 *   fp32 block transform of ck_quantize_int8_rowwise, rounded once).
 * The codes are exact in bf16; the sum over all of K is accumulated in fp32 by the tensor
 * cores (rounding order not specified: error at most about K * 2^-24 * sum_k |a w|),
 * then scaled, biased and rounded to out_dtype like ck_int8_linear's epilogue.
 *   x, w, w_scale (fp32 [1] for CK_TENSORWISE, else [N]), bias, residual, y, out_dtype:
 *   as for ck_int8_linear.  workspace: ck_w8a16_linear_workspace_size() bytes (the widened
 *   weight, and the rotated activation for ConvRot). */
size_t ck_w8a16_linear_workspace_size(int64_t M, int64_t N, int64_t K, int mode);
int ck_w8a16_linear(const void *x, const int8_t *w, const float *w_scale, const void *bias, const void *residual,
                    void *y, int64_t M, int64_t N, int64_t K, int mode, int out_dtype, void *workspace,
                    size_t workspace_bytes, void *stream);

/* GEMM + fused dequant on an already-quantized activation (the second half of
 * ck_int8_linear): q int8 [M,K], x_scale fp32 [M] (or [1] if scalar_scales), w int8
 * [N,K], w_scale fp32 [N] (or [1]), bias bf16 [N] or NULL, residual [M,N] of out_dtype
 * or NULL (may be y), y [M,N] of out_dtype (a ck_dtype_t).
 * workspace: ck_int8_gemm_workspace_size(M, N, K) bytes. */
size_t ck_int8_gemm_workspace_size(int64_t M, int64_t N, int64_t K);
int ck_int8_gemm_dequant(const int8_t *q, const float *x_scale, const int8_t *w, const float *w_scale,
                         const void *bias, const void *residual, void *y, int64_t M, int64_t N, int64_t K,
                         int scalar_scales, int out_dtype, void *workspace, size_t workspace_bytes, void *stream);

/* The raw int32 accumulators acc[m,n] = sum_k q[m,k] w[n,k] of the same GEMM engine,
 * written to acc int32 [M,N] (for exactness checks; the fused path never writes them).
 * workspace: ck_int8_gemm_workspace_size(M, N, K) bytes. */
int ck_int8_gemm_s32(const int8_t *q, const int8_t *w, int32_t *acc, int64_t M, int64_t N, int64_t K,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Launch profiling, for benchmarks.  Between ck_profile_begin() and ck_profile_end()
 * the library counts the kernels it enqueues from the calling host thread, by kind
 * (0 = activation quantize, 1 = int8 -> bf16 operand widening, 2 = GEMM with fused
 * epilogue).  With with_events != 0 it also brackets each launch with two CUDA events on
 * the kernel's own stream (the kernels are unchanged, but the events separate
 * consecutive kernels, so launch overlap between them is lost while timing).
 * ck_profile_end() waits for the events and fills, for each kind k < nkinds,
 * ms[k] = summed device milliseconds (0 without events) and launches[k] = number of
 * kernel launches.  Both arrays are host memory owned by the caller. */
int ck_profile_begin(int with_events);
int ck_profile_end(double *ms, int64_t *launches, int nkinds);

/* The GEMM launch configuration ck_int8_linear / ck_int8_gemm_* would use for an
 * M x N x K problem on the current device (the tile choice of issue #280, "Kernel used",
 * made per launch here): *bn = tile width in output columns (a multiple of 32, at most
 * 256), *cta_pair = 1 if two CTAs share a 256-row tile (tcgen05 cta_group::2) else 0
 * (128-row tiles), *resident_units = how many pairs / CTAs run at once (may be NULL),
 * *k_split = into how many K-slices each unit of the last partial wave is split over
 * otherwise idle pairs / CTAs (1 = none; may be NULL).  Split slices add their exact
 * int32 partial sums, so the result does not depend on the split.
 * The environment variables CK_GEMM_BN=<width>, CK_GEMM_PAIR=0 / 1 (single CTAs / pairs
 * only) and CK_GEMM_SPLIT=1 (no split) / <s> (s slices where possible) override the
 * choice for A/B timing; the query reports the result.  Host memory outputs; no work is
 * enqueued. */
int ck_gemm_tile_config(int64_t M, int64_t N, int64_t K, int *bn, int *cta_pair, int64_t *resident_units,
                        int *k_split);

/* Text of the last non-OK status returned on this host thread ("" if none). */
const char *ck_last_error(void);

/* Synchronises the current device, returns the device error word the kernels set
 * when a bounded wait gave up (0 = none; bit meanings in the csrc sources) and, if
 * `clear`, resets it.  Returns -1 if the word could not be read. */
int ck_device_error(int clear);

/* Failure-detection self-test: launches one block that waits on a barrier nothing
 * will ever complete, with a wait limit of timeout_ns.  The wait gives up, records
 * the error and the block exits normally; the call synchronises and returns
 * CK_ERR_TIMEOUT when that happened as designed (and clears the bit), CK_OK if the
 * wait unexpectedly completed, CK_ERR_CUDA on a CUDA error. */
int ck_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CK_INT8_H */
