/*
 * fp8mp.h -- C ABI of libfp8mp, the GB300 (sm_103a) hot path of an FP8
 * delayed-scaling linear layer used in mixed-precision training.
 *
 * Pages this interface follows (title -- site):
 *   [TE-FP8]  "Transformer Engine으로 FP8 사용하기" -- coniverse.tistory.com
 *   [MP]      "LLM) Mixed-Precision 개념 및 학습 방법 알아보기"
 *             -- data-newbie.tistory.com
 *   [PT-FP8]  "Các kiểu dữ liệu FP8 gốc của PyTorch ..." (PyTorch native FP8
 *             data types) -- hotroai.com
 *   [H100-Q]  "Как работает FP8 quantization на H100 (Transformer Engine)?"
 *             -- aivaro.ru
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout. Every matrix is row-major and dense (leading dimension = number of
 *   columns). M = tokens, K = in_features, N = out_features; the weight W is
 *   N x K, as a linear layer stores it.
 * Pointers. Every tensor argument is a DEVICE pointer of the current CUDA
 *   device, owned by the caller, which must keep it alive until the work on
 *   `stream` has finished. The library allocates no device memory and keeps
 *   no pointer after a call returns. Tensor pointers must be 16-byte aligned.
 * Stream. `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream). Every call only enqueues work on it and returns; no call
 *   synchronises with the host, and no data-dependent decision (the overflow
 *   skip of mp_master_step, the scale update) leaves the device.
 * Aliasing. Inputs are read-only; outputs must not overlap inputs, except
 *   the in-place state of mp_master_step and delayed_scaling_update.
 * Return value. 0 on success, otherwise a negative code:
 *   FP8MP_ERR_INVALID (-1): a required pointer is NULL or not 16-byte
 *     aligned, a size is negative or too large, an enum is out of range, or
 *     a GEMM dimension is not a multiple of 16 ([TE-FP8] "주의!" restricts
 *     FP8 linears to shapes whose dimensions divide by 16). Nothing was
 *     enqueued.
 *   FP8MP_ERR_DEVICE (-2): the current device is not an sm_103 GPU.
 *   FP8MP_ERR_LAUNCH (-3): a CUDA call or kernel launch failed.
 *   FP8MP_ERR_TIMEOUT (-4): returned by fp8mp_check(): a bounded wait inside
 *     a kernel ran out (a GEMM's wedged pipeline, the master step's grid
 *     barrier); that kernel's output is undefined, the CUDA context stays
 *     usable.
 *   fp8mp_last_error() then describes the failure (thread-local).
 * Launch. Kernels are launched with programmatic stream serialization: one
 *   may be scheduled while the previous kernel on the stream drains, and it
 *   waits for that kernel to complete before it touches global memory, so
 *   stream order holds as usual. Environment switches, read by the library:
 *   FP8MP_PDL=0 (once per process) launches plainly; FP8MP_GEMM_ENGINE=pair
 *   or single (per call) forces a GEMM tile engine; FP8MP_FUSED_MASTER=0
 *   (per call) runs the self-scanning master steps as three launches.
 */
#ifndef FP8MP_H
#define FP8MP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* FP8 formats ([TE-FP8] "Introduction to FP8"; [PT-FP8] finfo table).
 * E4M3: largest finite 448, no infinities; E5M2: largest finite 57344. */
typedef enum { FP8MP_E4M3 = 0, FP8MP_E5M2 = 1 } fp8mp_fmt;

/* High-precision element types of inputs and outputs. */
typedef enum { FP8MP_F32 = 0, FP8MP_BF16 = 1 } fp8mp_dtype;

/* amax_compute_algo of the DelayedScaling recipe ([TE-FP8] "FP8
 * 사용방안(recipe)"): the largest amax of the history, or the newest one. */
typedef enum { FP8MP_AMAX_MAX = 0, FP8MP_AMAX_MOST_RECENT = 1 } fp8mp_algo;

enum {
    FP8MP_OK = 0,
    FP8MP_ERR_INVALID = -1,
    FP8MP_ERR_DEVICE = -2,
    FP8MP_ERR_LAUNCH = -3,
    FP8MP_ERR_TIMEOUT = -4
};

/* Largest history a meta may have (floats per tensor). */
#define FP8MP_MAX_HISTORY 8192

/*
 * Per-tensor FP8 bookkeeping ([TE-FP8] "Scaling factor 선택 전략": each FP8
 * tensor keeps its own factor and a record of past amaxes; [H100-Q]
 * section 3). All four pointers are device pointers to fp32 values.
 * Initial state expected by delayed_scaling_update: history all 0,
 * scale = scale_inv = 1, cur_amax = 0.
 */
typedef struct fp8mp_meta {
    float *amax_history; /* [history_len], newest amax at index 0 */
    float *scale;        /* 1 value: multiplies the tensor before the cast */
    float *scale_inv;    /* 1 value: 1 / scale, multiplies GEMM results */
    float *cur_amax;     /* 1 value: amax of the current step; the casts and
                            the forward GEMM raise it with an atomic max */
    int32_t history_len; /* 1 .. FP8MP_MAX_HISTORY */
    int32_t fmt;         /* fp8mp_fmt of the tensor this meta scales */
} fp8mp_meta;

/*
 * fp8_quantize -- scaled, saturating round-to-nearest-even cast of a bf16 or
 * fp32 matrix to FP8, with the tensor's amax and an optional transposed copy.
 *
 * Defines ([H100-Q] section 3, steps 2-3; [TE-FP8] "Scaling factor 선택 전략"):
 *   out[r, c]   = sat_rne_fmt(fl32(x[r, c]) * scale[0])      (one fp32 multiply)
 *   out_t[c, r] = out[r, c]                                  (when out_t != NULL)
 *   *amax       = max(*amax, max_{r,c} |x[r, c]|)           (when amax != NULL)
 * Saturation: finite values beyond the format and +-Inf become +-largest
 * finite; NaN becomes 0x7F; subnormal FP8 results are kept (no flush).
 * The amax is over the UNSCALED input, NaN elements ignored; it is merged
 * into *amax with an atomic max, so *amax must hold a value >= +0 (the scale
 * update leaves 0 there).
 *
 * x      [rows x cols] of x_dtype (FP8MP_F32 or FP8MP_BF16).
 * scale  device pointer to one fp32 value (the tensor's meta->scale).
 * out    [rows x cols] bytes, required.
 * out_t  [cols x rows] bytes or NULL. When given, rows and cols must be
 *        multiples of 16; without it any rows x cols is accepted.
 * amax   device fp32 or NULL.
 * rows == 0 or cols == 0 is a no-op returning 0.
 */
int fp8_quantize(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                 const float *scale, uint8_t *out, uint8_t *out_t, float *amax, void *stream);

/* Flags of fp8_quantize_ex. */
#define FP8MP_OVERLAP_PREVIOUS 1u
/* fp8_linear_bwd_rowmajor_ex: signal in dw_nonfinite when dW is stored. */
#define FP8MP_SIGNAL_DW_DONE 2u
/* mp_master_step(_adam)_prescanned_ex: wait for that signal (with
 * FP8MP_OVERLAP_PREVIOUS). */
#define FP8MP_WAIT_DW_DONE 4u

/*
 * fp8_quantize_ex -- fp8_quantize with flags. The results are exactly
 * fp8_quantize's; the flags only change how the work is scheduled.
 *
 * FP8MP_OVERLAP_PREVIOUS: the caller guarantees that the work enqueued on
 *   `stream` before this call neither writes nor reads x, out, out_t or
 *   *amax (for example the dY cast of a layer's backward pass enqueued right
 *   after its forward GEMM, when dY does not come from that GEMM). The
 *   cast's blocks then do not wait for the previous kernel to finish: they
 *   start as soon as it lets the next kernel be scheduled (the library's
 *   GEMMs do so at the start of their mainloop) and run in the SM resources
 *   it leaves free. The call as a whole still completes only after the
 *   previous kernel, so everything enqueued after it sees the writes of
 *   both. Without programmatic launch (FP8MP_PDL=0) the flag has no effect.
 * Other flag bits: FP8MP_ERR_INVALID.
 */
int fp8_quantize_ex(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                    const float *scale, uint8_t *out, uint8_t *out_t, float *amax, uint32_t flags, void *stream);

/*
 * fp8_quantize_current -- the same cast under just-in-time ("current")
 * scaling ([TE-FP8] "Scaling factor 선택 전략", the just-in-time strategy:
 * the factor comes from the amax of the tensor being cast, measured each
 * time, instead of from the history). Three passes on `stream`:
 *   *amax = max_{r,c} |x[r, c]|                  (over the unscaled input)
 *   if *amax > 0 and finite: s = fl32(fmt_max / *amax) * 2^-margin, and
 *      *scale = s when s is finite and > 0 (else *scale keeps its value);
 *   *scale_inv = fl32(1 / *scale)
 *   out = sat_rne_fmt(fl32(x) * *scale); out_t = its transpose (optional)
 * This is delayed scaling with a one-entry history applied before the cast.
 * Arguments as fp8_quantize, plus: margin 0..126; scale (in/out, device fp32,
 * the fallback when the amax is zero or not finite); scale_inv and amax
 * (out, device fp32; *amax is overwritten, not max-merged).
 * Without out_t the three passes are one cooperative launch (after a
 * one-thread kernel that zeroes *amax and *scale_inv, the latter then
 * counting the blocks at a bounded grid barrier): every block casts the
 * share it measured, whose second read comes from L2 when x fits there. If
 * the device cannot run that grid at once, the three passes run as separate
 * launches. Traffic: the amax pass reads x once more (bf16: 5 B/elem; with
 * the transposed copy 6 B/elem).
 */
int fp8_quantize_current(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                         int32_t margin, float *scale, float *scale_inv, float *amax, uint8_t *out,
                         uint8_t *out_t, void *stream);

/*
 * fp8_quantize_dbias -- fp8_quantize of a layer's output gradient dY, with
 * its transposed copy, that also returns the bias gradient of the linear
 * layer ([TE-FP8] the te.Linear(768, 768, bias=True) example under "FP8
 * 사용방안(recipe)" and its backward under "Backward Pass 처리"; the bias
 * gradient of y = x W^T + b is the column sum of dY):
 *   out, out_t, *amax    exactly as fp8_quantize (out_t may be NULL: a
 *                        layer whose backward reads dY8 row-major through
 *                        fp8_linear_bwd_rowmajor needs no transposed copy);
 *   dbias[c] = sum_r x[r, c]  over the unscaled input, fp32 accumulation in
 *                             a fixed order (deterministic, set by the shape
 *                             alone): the rows are split among k CTAs per
 *                             128-column strip, k = max(1, min(ceil(rows/128),
 *                             152 / ceil(cols/128))), CTA j taking the 128-row
 *                             tiles j, j + k, ...; each CTA adds, per column,
 *                             its tiles' rows in 4-row runs (each run in row
 *                             order, runs tile after tile), combines the four
 *                             runs of each 16 rows pairwise ((a + b) + (c + d))
 *                             and the eight 16-row sums in order; the strip's
 *                             k CTA sums are added in order of j; rounded once
 *                             to dbias_dtype.
 * One launch: each CTA writes its column sums to the workspace and counts
 * itself in a per-strip word there; the last CTA of a strip to finish adds
 * the strip's sums, writes dbias, and sets the words it used back to zero.
 * Without a transposed copy, when 2 <= k <= 8 and the device holds every
 * strip's k CTAs as one thread-block cluster at once, CTA 0 of each strip
 * reads the others' sums from their shared memory instead (the same sums,
 * bit for bit; the workspace is not touched); at k = 1 a CTA writes dbias
 * itself.
 * workspace  device scratch of at least fp8_quantize_dbias_workspace_bytes
 *            (rows, cols) bytes, 16-byte aligned, owned by the caller. It
 *            must be ZERO-FILLED before its first use (e.g. cudaMemset or
 *            torch.zeros); every call leaves the bytes it used zero again,
 *            so one workspace serves later calls of any shape that fits
 *            without clearing. Calls that share a workspace must not overlap
 *            on the GPU (keep them on one stream).
 * rows, cols multiples of 16; rows == 0 gives dbias = 0.
 */
int fp8_quantize_dbias(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                       const float *scale, uint8_t *out, uint8_t *out_t, float *amax, void *dbias,
                       int32_t dbias_dtype, float *workspace, int64_t workspace_bytes, void *stream);

/* Workspace bytes fp8_quantize_dbias needs: k * cols * 4 for the CTAs'
 * column sums (k as above) plus ceil(cols / 128) * 4 for the strips' arrival
 * counters, rounded up to a multiple of 16; -1 for a negative or too large
 * shape. */
int64_t fp8_quantize_dbias_workspace_bytes(int64_t rows, int64_t cols);

/* Floats in the fixed scratch array of fp8_quantize_dbias_noalloc (4 MiB). */
#define FP8MP_NOALLOC_DBIAS_SCRATCH_FLOATS (1 << 20)

/*
 * fp8_quantize_dbias_noalloc -- fp8_quantize_dbias for callers that cannot
 * allocate device memory. The pages have no counterpart: this entry point
 * exists for callers that are not allowed to call cudaMalloc -- code running
 * inside a framework whose memory pool owns the device, plugin code handed
 * only input and output pointers, and latency-critical paths that cannot
 * take the implicit device synchronisation of cudaMalloc / cudaFree.
 *
 * Same arguments and results as fp8_quantize_dbias, minus the workspace:
 * the per-tile column sums and the strips' arrival counters live in a
 * file-scope device array of FP8MP_NOALLOC_DBIAS_SCRATCH_FLOATS floats
 * inside the library, which every GPU that loads the library holds until
 * the process exits. The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   - Limit: fp8_quantize_dbias_workspace_bytes(rows, cols) <=
 *     4 * FP8MP_NOALLOC_DBIAS_SCRATCH_FLOATS (any rows with cols up to
 *     1040432); larger shapes return FP8MP_ERR_INVALID with a message
 *     naming the limit.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for
 *     the life of the process; make that first call before any stream
 *     capture. The cache does not survive cudaDeviceReset: after a reset of
 *     a device that has called this function, do not call it again in that
 *     process.
 *   - The array starts zero-filled (the loader clears it) and every call
 *     leaves it zero again, which is what the counters need. Calls whose
 *     work overlaps on the GPU (other streams, other threads) race on the
 *     array: serialise them, e.g. on one stream.
 */
int fp8_quantize_dbias_noalloc(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                               const float *scale, uint8_t *out, uint8_t *out_t, float *amax, void *dbias,
                               int32_t dbias_dtype, void *stream);

/*
 * fp8_linear_fwd -- forward FP8 GEMM of a linear layer, E4M3 x E4M3.
 *
 * Defines ([PT-FP8] the torch._scaled_mm listing: two FP8 operands, their
 * scales, an optional bias and the output amax; [MP] "Accumulation into
 * FP32"; [H100-Q] section 3, step 4: the product is divided by the scales):
 *   y[m, n] = (sum_k x8[m, k] * w8[n, k]) * sinv_x[0] * sinv_w[0] + bias[n]
 * accumulated in fp32 on the tensor cores, rounded once to y_dtype.
 *   *y_amax = max(*y_amax, max |y as stored|)                (when y_amax != NULL)
 * NaN elements are left out of the amax (an E4M3 NaN code in x8 or w8 makes
 * NaN outputs); an output that overflows to +-Inf counts as Inf.
 *
 * x8  [M x K] E4M3 codes;  w8 [N x K] E4M3 codes (the weight, K contiguous).
 * sinv_x, sinv_w  device pointers to one fp32 each (metas' scale_inv).
 * bias  [N] of bias_dtype, or NULL.   y  [M x N] of y_dtype.
 * M, N, K multiples of 16. M == 0 or N == 0: no-op. K == 0: y = bias (or 0).
 */
int fp8_linear_fwd(const uint8_t *x8, const uint8_t *w8, int64_t M, int64_t N, int64_t K,
                   const float *sinv_x, const float *sinv_w, const void *bias, int32_t bias_dtype,
                   void *y, int32_t y_dtype, float *y_amax, void *stream);

/*
 * fp8_linear_fwd_fp8out -- fp8_linear_fwd whose output is written directly as
 * FP8 codes for the next layer ([PT-FP8] the torch._scaled_mm listing with
 * out_dtype=e4m3_type, returning the output and its amax). With y computed
 * in fp32 exactly as fp8_linear_fwd computes it before rounding:
 *   y8[m, n] = sat_rne_{y_fmt}(fl32(y[m, n] * y_scale[0]))
 *   *y_amax  = max(*y_amax, max |y|)     (fp32 y, unscaled: the amax delayed
 *                                         scaling records for that tensor)
 * y_scale is the consumer tensor's meta->scale. Saves the separate cast
 * pass of the next layer's input (its transposed copy is not produced).
 * Arguments otherwise as fp8_linear_fwd; y8 is [M x N] bytes.
 */
int fp8_linear_fwd_fp8out(const uint8_t *x8, const uint8_t *w8, int64_t M, int64_t N, int64_t K,
                          const float *sinv_x, const float *sinv_w, const void *bias, int32_t bias_dtype,
                          const float *y_scale, int32_t y_fmt, uint8_t *y8, float *y_amax, void *stream);

/*
 * fp8_linear_dgrad -- input gradient of the linear layer (HYBRID recipe:
 * E5M2 gradient against the E4M3 weight; [TE-FP8] "Introduction to FP8" and
 * "FP8 사용방안(recipe)", Format.HYBRID; "Backward Pass 처리").
 *   dx[m, k] = (sum_n dy8[m, n] * w8t[k, n]) * sinv_dy[0] * sinv_w[0]
 *
 * dy8  [M x N] codes of dy_fmt (E5M2 under HYBRID, E4M3 allowed).
 * w8t  [K x N] E4M3 codes: the transposed copy fp8_quantize writes to out_t
 *      when casting the weight.
 * dx   [M x K] of dx_dtype.  M, N, K multiples of 16; N == 0 gives dx = 0.
 */
int fp8_linear_dgrad(const uint8_t *dy8, const uint8_t *w8t, int64_t M, int64_t N, int64_t K,
                     int32_t dy_fmt, const float *sinv_dy, const float *sinv_w, void *dx,
                     int32_t dx_dtype, void *stream);

/*
 * fp8_linear_wgrad -- weight gradient of the linear layer (HYBRID recipe as
 * above), contracting over the M tokens:
 *   dw[n, k] = (sum_m dy8t[n, m] * x8t[k, m]) * sinv_dy[0] * sinv_x[0]
 *
 * dy8t [N x M] codes of dy_fmt: the transposed copy of the output gradient.
 * x8t  [K x M] E4M3 codes: the transposed copy of the layer input.
 * dw   [N x K] of dw_dtype.  M, N, K multiples of 16; M == 0 gives dw = 0.
 */
int fp8_linear_wgrad(const uint8_t *dy8t, const uint8_t *x8t, int64_t M, int64_t N, int64_t K,
                     int32_t dy_fmt, const float *sinv_dy, const float *sinv_x, void *dw,
                     int32_t dw_dtype, void *stream);

/*
 * fp8_linear_bwd -- both backward GEMMs of the linear layer in one launch:
 * exactly fp8_linear_dgrad and fp8_linear_wgrad above on the same arguments
 * (same per-element sums in the same order, so the results are bitwise those
 * of the two separate calls):
 *   dx[m, k] = (sum_n dy8[m, n]  * w8t[k, n]) * sinv_dy[0] * sinv_w[0]
 *   dw[n, k] = (sum_m dy8t[n, m] * x8t[k, m]) * sinv_dy[0] * sinv_x[0]
 * The two GEMMs are independent ([TE-FP8] "Backward Pass 처리": the input
 * gradient and the weight gradient both come from the one output gradient),
 * so their output tiles share one persistent grid, which keeps every SM busy
 * through the tail of the shorter GEMM instead of idling at each launch's
 * last partial wave.
 *
 * dy8 [M x N] and dy8t [N x M]: codes of dy_fmt (the output gradient and its
 * transposed copy, as fp8_quantize writes them); w8t [K x N], x8t [K x M]:
 * E4M3 codes. dx [M x K] of dx_dtype, dw [N x K] of dw_dtype, both required
 * when non-empty and not overlapping. M, N, K multiples of 16. Empty cases
 * follow the separate calls: N == 0 gives dx = 0, M == 0 gives dw = 0.
 */
int fp8_linear_bwd(const uint8_t *dy8, const uint8_t *dy8t, const uint8_t *w8t, const uint8_t *x8t, int64_t M,
                   int64_t N, int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                   const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype, void *stream);

/*
 * fp8_linear_bwd_rowmajor -- the backward GEMMs of the linear layer from the
 * row-major FP8 copies the forward pass already has, with no transposed
 * copies: the same results as fp8_linear_dgrad / fp8_linear_wgrad
 *   dx[m, k] = (sum_n dy8[m, n] * w8[n, k]) * sinv_dy[0] * sinv_w[0]
 *   dw[n, k] = (sum_m dy8[m, n] * x8[m, k]) * sinv_dy[0] * sinv_x[0]
 * (each sum in fp32 on the tensor cores, rounded once to the output type),
 * both in one launch ([TE-FP8] "Backward Pass 처리"). The tensor cores read
 * w8 and x8, and for dw also dy8, along their rows (MN-major shared-memory
 * operands), so casts for this layer need no transposed outputs.
 *
 * dy8 [M x N] codes of dy_fmt; w8 [N x K] and x8 [M x K] E4M3 codes (the
 * forward's operands). dx [M x K] of dx_dtype or NULL (no input gradient,
 * e.g. a first layer); dw [N x K] of dw_dtype or NULL (frozen weight); they
 * must not overlap. M, N, K multiples of 16. N == 0 gives dx = 0, M == 0
 * gives dw = 0.
 *
 * dw_nonfinite  device int32 or NULL. When given (and dw is computed), the
 *   wgrad epilogue ORs 1 into it if any element of dw as stored is Inf or
 *   NaN: the overflow check of the dynamic loss scaler ([MP], the loss-scale
 *   procedure: inspect the gradients for Inf/NaN), made where the gradients
 *   are produced, so mp_master_step_prescanned need not read them again.
 *   The caller zeroes it before the first backward of a step (the
 *   prescanned master step leaves it at 0); further backward passes of the
 *   step (gradient accumulation) keep OR-ing into it.
 */
int fp8_linear_bwd_rowmajor(const uint8_t *dy8, const uint8_t *w8, const uint8_t *x8, int64_t M, int64_t N,
                            int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                            const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype,
                            int32_t *dw_nonfinite, void *stream);

/*
 * fp8_linear_bwd_rowmajor_ex -- fp8_linear_bwd_rowmajor with flags:
 *   0                     the call without _ex.
 *   FP8MP_SIGNAL_DW_DONE  (needs dw and dw_nonfinite) the launch also tells a
 *                         master step that runs beside it when dW is
 *                         complete: each epilogue warp, once its part of a
 *                         dW tile is stored and visible, ORs that part's
 *                         Inf/NaN flag into bit 0 of *dw_nonfinite and adds
 *                         1 << 16 to the word; the last part sets bit 30.
 *                         (Bits 1-15 are the prescanned master step's block
 *                         count; at most 16383 parts: dW of up to 2047 tiles
 *                         of 256 x 256.) The word must hold only bit 0 or
 *                         nothing before the call (the prescanned master step
 *                         leaves it 0), and its consumer must be
 *                         mp_master_step(_adam)_prescanned_ex, which resets
 *                         it; an empty dW sets bit 30 at once. The launch
 *                         runs the dW tiles first when dW's contraction (M)
 *                         is the longer one, so the signal comes while the
 *                         dX tiles are still being computed.
 * Other bits: FP8MP_ERR_INVALID.
 */
int fp8_linear_bwd_rowmajor_ex(const uint8_t *dy8, const uint8_t *w8, const uint8_t *x8, int64_t M, int64_t N,
                               int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                               const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype,
                               int32_t *dw_nonfinite, uint32_t flags, void *stream);

/*
 * delayed_scaling_update -- the DelayedScaling bookkeeping of one step for a
 * batch of tensors ([TE-FP8] "Scaling factor 선택 전략", "FP8 사용방안(recipe)":
 * amax_history_len, amax_compute_algo; [PT-FP8] amax and scale history
 * synchronised once per step after backward; [H100-Q] section 3, step 2, and
 * section 10). For each meta, in this order:
 *   1. history[j] = history[j-1] for j = L-1 .. 1; history[0] = cur_amax;
 *   2. a = max_j history[j] (FP8MP_AMAX_MAX) or history[0] (MOST_RECENT);
 *   3. if a > 0 and finite: s = fl32(fmt_max / a) * 2^-margin; the scale
 *      becomes s when s is finite and > 0, otherwise it keeps its value;
 *   4. scale_inv = fl32(1 / scale); cur_amax = 0.
 * fmt_max is 448 (E4M3) or 57344 (E5M2) after meta->fmt.
 *
 * metas   HOST array of n structs whose pointers are device pointers; read
 *         during the call only (the values travel as kernel parameters).
 * algo    fp8mp_algo.   margin  0 .. 126.   n == 0 is a no-op.
 */
int delayed_scaling_update(const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin,
                           void *stream);

/*
 * delayed_scaling_update_ex -- delayed_scaling_update that also keeps the
 * scale_inv each tensor had before the update:
 *   prev_scale_inv[i] = metas[i].scale_inv as it was on entry
 * prev_scale_inv  device float[n] (4-byte aligned) or NULL (then this is
 *   delayed_scaling_update). With it the update may run before the backward
 *   GEMMs of the step: they take their scale_inv factors from
 *   prev_scale_inv, which are the factors the step's casts used ([TE-FP8]
 *   "Scaling factor 선택 전략": the step's tensors are cast with the scale of
 *   the previous steps' history; the new scale applies from the next cast on),
 *   so the results are bitwise those of the update run after them.
 */
int delayed_scaling_update_ex(const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin,
                              float *prev_scale_inv, void *stream);

/*
 * mp_master_step -- one mixed-precision optimizer step on a flat parameter
 * buffer: loss unscale, overflow check with dynamic loss scaling, FP32
 * master-weight SGD-momentum update and E4M3 re-cast ([MP] "FP32 Master Copy
 * of Weights", "Mixed-Precision Training Iteration" steps 5-7, and the
 * dynamic loss-scale procedure: skip the update and lower S when a gradient
 * is Inf/NaN, raise S after a run of clean steps; [H100-Q] section 7).
 *   found_inf = any grad is Inf or NaN                        (pass 1)
 *   if found_inf: S = S * backoff; growth = 0; nothing else changes.
 *   else, for every i (fp32; fmaf is one correctly rounded fused op):
 *     u = fp32(grad[i]) * fl32(1 / S)
 *     momentum[i] = fmaf(momentum_coef, momentum[i], u)
 *     master[i]   = fmaf(-lr, momentum[i], master[i])
 *     w8[i]       = sat_rne_E4M3(master[i] * scale_w[0])
 *     *amax_w     = max(*amax_w, |master[i]|)
 *   then growth += 1; if growth >= growth_interval: S = S * growth_factor,
 *   growth = 0.
 *
 * grad_bf16 [n] bf16 bits (gradients of the loss multiplied by S).
 * master, momentum [n] fp32 (in place);  w8 [n] E4M3 codes (written).
 * scale_w   device fp32: the weight meta's scale (delayed: this step's).
 * amax_w    device fp32: the weight meta's cur_amax (atomic max target).
 * loss_scale device fp32 S;  growth_tracker device int32;  both in place.
 * found_inf device int32 written with 0 or 1 (the step's overflow flag).
 * growth_interval >= 1. n == 0 still counts a clean step.
 */
int mp_master_step(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum,
                   uint8_t *w8, const float *scale_w, float *amax_w, float *loss_scale,
                   int32_t *growth_tracker, int32_t *found_inf, float lr, float momentum_coef,
                   float backoff, float growth_factor, int32_t growth_interval, void *stream);

/*
 * mp_master_step_adam -- mp_master_step with an Adam update of the FP32
 * master weights ([PT-FP8]: the float8_experimental training loop uses
 * torch.optim.Adam; the loss-scale, skip and re-cast frame is [MP]'s as
 * above). Pass 1 and the skip rule are mp_master_step's; otherwise, per
 * element, each operation one correctly rounded fp32 operation:
 *   u  = fp32(grad[i]) * fl32(1 / S)
 *   b1t = fl32(beta_pows[0] * beta1),  b2t = fl32(beta_pows[1] * beta2)
 *   exp_avg[i]    = fmaf(beta1, exp_avg[i], fl32(1 - beta1) * u)
 *   exp_avg_sq[i] = fmaf(beta2, exp_avg_sq[i], fl32(1 - beta2) * fl32(u * u))
 *   master[i] = fmaf(-lr, (exp_avg[i] / fl32(1 - b1t)) /
 *                         (sqrt(exp_avg_sq[i] / fl32(1 - b2t)) + eps), master[i])
 *   w8[i], *amax_w as mp_master_step.
 * beta_pows  device float[2] = (beta1^(t-1), beta2^(t-1)), both 1 before the
 *            first step; advanced to (b1t, b2t) on clean steps only.
 * exp_avg, exp_avg_sq  [n] fp32, zero before the first step (in place).
 * Traffic: 2 + (2 + 12) + (12 + 1) = 29 bytes per parameter.
 */
int mp_master_step_adam(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                        float *exp_avg_sq, uint8_t *w8, const float *scale_w, float *amax_w,
                        float *loss_scale, int32_t *growth_tracker, int32_t *found_inf, float *beta_pows,
                        float lr, float beta1, float beta2, float eps, float backoff, float growth_factor,
                        int32_t growth_interval, void *stream);

/*
 * mp_master_step_prescanned, mp_master_step_adam_prescanned -- the two steps
 * above when the gradients' producer has already looked for Inf/NaN in them
 * (fp8_linear_bwd_rowmajor's dw_nonfinite): the same results bit for bit,
 * with found_inf taken from the flag instead of a scan of the gradients
 * (which saves a 2-byte-per-parameter pass and the grid barrier).
 *   grad_nonfinite  device int32, in/out: 1 iff some gradient element is
 *                   Inf or NaN, else 0 (the producer ORs 1 into a word that
 *                   was 0). During the launch the step counts its blocks in
 *                   the word's upper bits; it writes the flag into
 *                   *found_inf (whatever that held: no memset precedes
 *                   this step) and leaves the word at 0 for the next
 *                   producer. It must not be found_inf itself.
 * Other arguments and results as mp_master_step / mp_master_step_adam.
 */
int mp_master_step_prescanned(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum,
                              uint8_t *w8, const float *scale_w, float *amax_w, float *loss_scale,
                              int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite, float lr,
                              float momentum_coef, float backoff, float growth_factor, int32_t growth_interval,
                              void *stream);
int mp_master_step_adam_prescanned(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                                   float *exp_avg_sq, uint8_t *w8, const float *scale_w, float *amax_w,
                                   float *loss_scale, int32_t *growth_tracker, int32_t *found_inf,
                                   int32_t *grad_nonfinite, float *beta_pows, float lr, float beta1, float beta2,
                                   float eps, float backoff, float growth_factor, int32_t growth_interval,
                                   void *stream);

/*
 * mp_master_step_prescanned_ex, mp_master_step_adam_prescanned_ex -- the
 * prescanned steps with the new E4M3 copy of the weight written to another
 * buffer than the one the current step's GEMMs read, so that the update can
 * run while a GEMM still reads the current copy:
 *   w8_in   [n] E4M3 codes: the current copy, read only when the step is
 *           skipped (found_inf): then w8_out = w8_in, so w8_out always holds
 *           the copy the next step uses. NULL or equal to w8_out: in place,
 *           as the calls without _ex. Otherwise w8_in and w8_out must not
 *           overlap.
 *   w8_out  [n] E4M3 codes (written): the w8 of the calls without _ex.
 *   flags   0 or FP8MP_OVERLAP_PREVIOUS: the caller guarantees that the work
 *           enqueued on `stream` before this call, other than what completed
 *           before the last kernel started, neither writes nor reads anything
 *           this step reads or writes. The typical case is the dgrad GEMM
 *           (fp8_linear_bwd_rowmajor with dw = NULL) enqueued right after the
 *           wgrad GEMM that produced grad_bf16 and grad_nonfinite: it reads
 *           w8_in while the step writes w8_out. The step then starts without
 *           waiting for that GEMM, as one block per SM whose registers fit
 *           beside the GEMM's CTA, and still completes only after it. The
 *           kernel before that one (the wgrad GEMM) must have finished
 *           before the previous kernel started (the library's kernels wait
 *           for their predecessor before they let the next one start).
 *           Without programmatic launch (FP8MP_PDL=0) the flag has no
 *           effect.
 *           FP8MP_WAIT_DW_DONE (only with FP8MP_OVERLAP_PREVIOUS): the
 *           kernel running before this one is the backward GEMM launch that
 *           produces grad_bf16 and signals its completion
 *           (fp8_linear_bwd_rowmajor_ex with FP8MP_SIGNAL_DW_DONE, on the
 *           same word as grad_nonfinite). The step then starts beside that
 *           launch, each block waits (bounded, about 2 s) for bit 30 of
 *           *grad_nonfinite before it reads the flag and the gradients, and
 *           reads them through L2. A wait that runs out raises the flag
 *           fp8mp_check reports (FP8MP_ERR_TIMEOUT) and the step is skipped.
 *           Other bits: FP8MP_ERR_INVALID.
 * Every other argument and every result as the calls without _ex (w8 there
 * is w8_out here).
 */
int mp_master_step_prescanned_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum,
                                 const uint8_t *w8_in, uint8_t *w8_out, const float *scale_w, float *amax_w,
                                 float *loss_scale, int32_t *growth_tracker, int32_t *found_inf,
                                 int32_t *grad_nonfinite, float lr, float momentum_coef, float backoff,
                                 float growth_factor, int32_t growth_interval, uint32_t flags, void *stream);
int mp_master_step_adam_prescanned_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                                      float *exp_avg_sq, const uint8_t *w8_in, uint8_t *w8_out,
                                      const float *scale_w, float *amax_w, float *loss_scale,
                                      int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite,
                                      float *beta_pows, float lr, float beta1, float beta2, float eps, float backoff,
                                      float growth_factor, int32_t growth_interval, uint32_t flags, void *stream);

/*
 * mp_master_step_prescanned_scaling_ex, mp_master_step_adam_prescanned_scaling_ex
 * -- the _ex steps that also run the step's delayed-scaling update of up to
 * 8 tensors, as delayed_scaling_update does it ([TE-FP8] "Scaling factor
 * 선택 전략" and "FP8 사용방안(recipe)"; [H100-Q] section 3), so that the
 * update needs no launch of its own in the training step: the step's blocks
 * run it while they wait for the backward launch's dW signal.
 *   metas, n_metas   0..8 metas (NULL when 0), amax_algo and margin as for
 *                    delayed_scaling_update. The meta whose scale is scale_w
 *                    (if any) is the weight's: it must have amax_w as its
 *                    cur_amax, and the step casts the new weight copy with
 *                    its NEW scale (the update's), then adds the new copy's
 *                    amax to the zeroed cur_amax -- as delayed_scaling_update
 *                    followed by the _ex step would.
 *   flags            must be FP8MP_OVERLAP_PREVIOUS | FP8MP_WAIT_DW_DONE
 *                    (the step starts beside the backward launch that signals
 *                    dW's completion).
 * Histories, scales and cur_amax are written as the step starts; each
 * meta's scale_inv keeps its old value until the backward launch the step
 * started beside has completed, so that launch may read the metas' scale_inv
 * (the step's factors, as the snapshot of delayed_scaling_update_ex gives
 * them) while the update runs. Results equal, bit for bit, those of
 * delayed_scaling_update_ex enqueued before the backward launch followed by
 * the _ex step. Every other argument as the _ex calls; FP8MP_ERR_INVALID for
 * a bad meta, a bad count, two metas holding scale_w, a meta holding amax_w
 * but not scale_w, or other flags.
 */
int mp_master_step_prescanned_scaling_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum,
                                         const uint8_t *w8_in, uint8_t *w8_out, const float *scale_w,
                                         float *amax_w, float *loss_scale, int32_t *growth_tracker,
                                         int32_t *found_inf, int32_t *grad_nonfinite, float lr, float momentum_coef,
                                         float backoff, float growth_factor, int32_t growth_interval,
                                         const fp8mp_meta *metas, int32_t n_metas, int32_t amax_algo,
                                         int32_t margin, uint32_t flags, void *stream);
int mp_master_step_adam_prescanned_scaling_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                                              float *exp_avg_sq, const uint8_t *w8_in, uint8_t *w8_out,
                                              const float *scale_w, float *amax_w, float *loss_scale,
                                              int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite,
                                              float *beta_pows, float lr, float beta1, float beta2, float eps,
                                              float backoff, float growth_factor, int32_t growth_interval,
                                              const fp8mp_meta *metas, int32_t n_metas, int32_t amax_algo,
                                              int32_t margin, uint32_t flags, void *stream);

/*
 * fp8mp_check -- synchronises `stream`, then reports and clears the device
 * flags a kernel sets when one of its bounded waits runs out (a GEMM's
 * mbarrier wait, the master step's grid barrier): FP8MP_ERR_TIMEOUT if one
 * was set, FP8MP_ERR_LAUNCH on a CUDA error, else 0.
 */
int fp8mp_check(void *stream);

/*
 * fp8mp_selftest_timeout -- diagnostic of the failure path. Enqueues on
 * `stream` a one-thread kernel that waits, with the bounded wait the GEMM
 * kernels use, on an mbarrier nothing ever signals. After about 2 s the wait
 * gives up and raises the device timeout flag, the kernel returns normally,
 * and the next fp8mp_check(stream) returns FP8MP_ERR_TIMEOUT (and clears the
 * flag). No fault, trap or hang is involved; the context stays usable.
 * Returns 0 when enqueued.
 */
int fp8mp_selftest_timeout(void *stream);

/*
 * fp8mp_selftest_barrier_timeout -- the same diagnostic for the grid barrier
 * of mp_master_step / mp_master_step_adam (which run as one cooperative
 * launch): a one-block kernel arrives at a barrier that waits for two
 * arrivals; after about 2 s the wait gives up, raises the device flag and
 * the kernel returns normally; the next fp8mp_check(stream) returns
 * FP8MP_ERR_TIMEOUT. Returns 0 when enqueued.
 */
int fp8mp_selftest_barrier_timeout(void *stream);

/* Thread-local description of the last nonzero return ("" if none). */
const char *fp8mp_last_error(void);

/* Interface version (incremented on any ABI change). */
int32_t fp8mp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8MP_H */
