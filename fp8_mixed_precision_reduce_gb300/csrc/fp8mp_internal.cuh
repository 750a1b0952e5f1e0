// fp8mp_internal.cuh -- device helpers (inline PTX for sm_103a) and host
// plumbing shared by the libfp8mp translation units. Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/fp8mp.h"

namespace fp8mp {

// ---------------------------------------------------------------- host side

// Records a thread-local message and returns `code`.
int fail(int code, const char *fmt, ...);
// Clears the thread-local message.
void clear_error();

struct DeviceInfo {
    int device;
    int num_sms;
    int cc_major, cc_minor;
};
// Fills `info` for the current device; returns FP8MP_ERR_DEVICE if it is not
// an sm_103 GPU, FP8MP_ERR_LAUNCH on a CUDA error.
int current_device(DeviceInfo *info);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernels of the library are launched with programmatic stream
// serialization (programmatic dependent launch): a kernel may be scheduled
// while the previous kernel on the stream drains, runs what touches no
// global memory, and waits in griddepcontrol.wait for the previous grids to
// complete (and their writes to be visible) before any global load or store.
// FP8MP_PDL=0 in the environment launches them plainly (read once).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The same, in thread-block clusters of `cluster_x` consecutive CTAs
// (grid.x a multiple of it; 1 = no cluster attribute).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    if (cluster_x > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = cluster_x;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Zeroes one 32-bit word on the stream with a one-thread kernel launched like
// the library's others, so a programmatic-launch chain is not broken the way
// a memset node breaks it (the kernel waits for the previous grid first).
cudaError_t launch_zero_word(void *word, cudaStream_t s);

// Launchers (return FP8MP_* codes; arguments already validated).
int launch_quantize_current(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, int margin,
                            float *scale, float *scale_inv, float *amax, uint8_t *out, uint8_t *out_t,
                            cudaStream_t s, const DeviceInfo &dev);
// CTAs per 128-column strip of the bias-gradient cast (a function of the
// shape only, so the column sums' order is too): its workspace holds that
// many rows of column sums, then one arrival counter per strip.
int dbias_ctas_per_strip(int64_t rows, int64_t cols);
int launch_quantize_dbias(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, const float *scale,
                          uint8_t *out, uint8_t *out_t, float *amax, void *dbias, int dbias_dtype, float *ws,
                          cudaStream_t s, const DeviceInfo &dev);
// early: the cast's blocks start without waiting for the previous kernel on
// the stream (its buffers do not interact with it; FP8MP_OVERLAP_PREVIOUS).
int launch_quantize(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt,
                    const float *scale, uint8_t *out, uint8_t *out_t, float *amax,
                    cudaStream_t s, const DeviceInfo &dev, bool early = false);
// One GEMM out[rows_a x rows_b] = (A B^T) * sinv_a * sinv_b (+ bias) over a
// contraction of length kc. A is [rows_a x kc] (K-major) or, with a_mn,
// [kc x rows_a] (MN-major); likewise B with rows_b and b_mn.
struct GemmDesc {
    const uint8_t *a;
    int fmt_a;
    const uint8_t *b;
    int fmt_b;
    int64_t rows_a, rows_b, kc;
    const float *sinv_a, *sinv_b;
    const void *bias;
    int bias_dtype;
    void *out;
    int out_dtype;
    float *out_amax;
    const float *out_scale;  // non-null: FP8 output of out_fmt under *out_scale
    int out_fmt;
    int a_mn, b_mn;
    int32_t *out_nonfinite = nullptr;  // non-null (bf16 / fp32 output): |= 1 when a stored element is Inf or NaN
    // with out_nonfinite: also count each stored tile part in that word and
    // set kDoneBit once the whole output is stored (see the word's layout)
    bool signal_done = false;
};
// The overflow word of a gradient (fp8_linear_bwd_rowmajor's dw_nonfinite,
// the prescanned master step's grad_nonfinite), bit by bit: bit 0 the
// Inf/NaN flag; bits 1-15 the master step's block arrivals (2 each); bits
// 16-29 the GEMM's stored tile parts when it signals completion; bit 30 set
// once every part is stored; bit 31 set by the master step that runs the
// delayed-scaling update as well, once the weight's new scale is written.
// The prescanned master step resets it to 0.
constexpr uint32_t kArrivalShift = 1, kArrivalMask = 0x7FFFu;
constexpr uint32_t kPartShift = 16, kPartMask = 0x3FFFu;
constexpr uint32_t kDoneBit = 1u << 30;
constexpr uint32_t kMetaBit = 1u << 31;

// The delayed-scaling update of up to kMaxFoldMetas tensors run by the
// blocks of a master step (mp_master_step_prescanned_scaling_ex): the
// metas' arrays, which of them is the weight's (its new scale is the one the
// step casts with; -1 if none), the recipe's algorithm and margin.
constexpr int kMaxFoldMetas = 8;
struct FoldMeta {
    float *hist, *scale, *scale_inv, *cur_amax;
    int32_t len, fmt;
};
struct FoldBatch {
    FoldMeta m[kMaxFoldMetas];
    int32_t n, w_index, algo, margin;
};
// One-thread kernel that ORs kDoneBit into the word.
cudaError_t launch_signal_done(int32_t *word, cudaStream_t s);
// Runs 1 or 2 independent GEMMs in one persistent launch.
int launch_gemms(const GemmDesc *descs, int n, cudaStream_t s, const DeviceInfo &dev);
int launch_gemm(const uint8_t *a, int fmt_a, const uint8_t *b, int fmt_b, int64_t rows_a,
                int64_t rows_b, int64_t kc, const float *sinv_a, const float *sinv_b,
                const void *bias, int bias_dtype, void *out, int out_dtype, float *out_amax,
                cudaStream_t s, const DeviceInfo &dev, const float *out_scale = nullptr,
                int out_fmt = FP8MP_E4M3);
// Registers one warp of the persistent (pair) GEMM holds, as allocated (8
// per thread at a time), and in *warps its warps per CTA; 0 if the attribute
// query fails.
int gemm_warp_registers(int *warps);
// prev_scale_inv (n floats or NULL) receives each meta's scale_inv as it
// was before the update.
int launch_scale_update(const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin,
                        cudaStream_t s, float *prev_scale_inv = nullptr);
// w8_in: the current E4M3 copy when the new one goes to a different buffer
// w8 (copied there on a skipped step), NULL for in place. early (prescanned
// steps only): start without waiting for the previous kernel on the stream
// (FP8MP_OVERLAP_PREVIOUS), complete after it. wait_done (with early):
// that kernel produces the gradients and signals their completion in the
// word (FP8MP_WAIT_DW_DONE).
int launch_master_step(const uint16_t *g, int64_t n, float *w, float *v, uint8_t *w8,
                       const float *scale_w, float *amax_w, float *loss_scale, int32_t *growth,
                       int32_t *found_inf, float lr, float mu, float backoff, float growth_factor,
                       int32_t growth_interval, cudaStream_t s, const DeviceInfo &dev,
                       int32_t *grad_nonfinite = nullptr, const uint8_t *w8_in = nullptr, bool early = false,
                       bool wait_done = false, const FoldBatch *fold = nullptr);
int launch_adam_step(const uint16_t *g, int64_t n, float *w, float *m, float *v, uint8_t *w8, const float *scale_w,
                     float *amax_w, float *loss_scale, int32_t *growth, int32_t *found_inf, float *beta_pows,
                     float lr, float b1, float b2, float eps, float backoff, float growth_factor,
                     int32_t growth_interval, cudaStream_t s, const DeviceInfo &dev,
                     int32_t *grad_nonfinite = nullptr, const uint8_t *w8_in = nullptr, bool early = false,
                     bool wait_done = false, const FoldBatch *fold = nullptr);
// Enqueues the one-thread kernel whose bounded wait is meant to run out.
int launch_timeout_selftest(cudaStream_t s);
// Reads and clears the GEMM wait-timeout flag (after a stream sync).
int read_and_clear_timeout_flag(unsigned int *value);
// Enqueues the one-block kernel whose grid-barrier wait is meant to run out.
int launch_barrier_selftest(cudaStream_t s);
// Reads and clears the tiled casts' wait-timeout flag.
int read_and_clear_cast_timeout_flag(unsigned int *value);
// Reads and clears the fused master step's barrier-timeout flag.
int read_and_clear_master_timeout_flag(unsigned int *value);
const char *last_error_message();

// -------------------------------------------------------------- device side

// Waits until the grids this one depends on (the previous kernel on the
// stream) have completed and their memory is visible; returns at once when
// the kernel was launched without programmatic serialization.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream be scheduled (it still waits in
// pdl_wait for this grid to complete before touching memory). Every kernel
// of the library calls it only after its own pdl_wait has returned, so the
// next kernel starting means every kernel before this one has completed
// (which a kernel launched with FP8MP_OVERLAP_PREVIOUS relies on).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Largest finite value of each format.
__host__ __device__ constexpr float fmt_max(int fmt) { return fmt == FP8MP_E4M3 ? 448.0f : 57344.0f; }


__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

// The scale rule of delayed / current scaling: with a > 0 and finite,
// s = fl32(fmt_max / a) * 2^-margin (one IEEE division, one exact multiply by
// a power of two, margin 0..126); the new scale is s when s is finite and
// > 0, otherwise the old scale is kept.
__device__ __forceinline__ float scale_from_amax(float a, float old_scale, int fmt, int margin) {
    float sc = old_scale;
    if (a > 0.0f && isfinite(a)) {
        const float s = __fdiv_rn(fmt_max(fmt), a);
        const float s2 = __fmul_rn(s, __int_as_float((127 - margin) << 23));
        if (isfinite(s2) && s2 > 0.0f) sc = s2;
    }
    return sc;
}

// Two fp32 values -> two FP8 codes with round-to-nearest-even and
// saturation to the largest finite value (PTX cvt .satfinite). `lo` lands in
// the low byte. A NaN input is mapped to 0x7F explicitly.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == FP8MP_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    uint32_t v = r;
    if (lo != lo) v = (v & 0xFF00u) | 0x7Fu;
    if (hi != hi) v = (v & 0x00FFu) | 0x7F00u;
    return v;
}

// Four fp32 values -> four codes packed little-endian in a 32-bit word.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_quad(float a, float b, float c, float d) {
    return cvt_pair<FMT>(a, b) | (cvt_pair<FMT>(c, d) << 16);
}

// max that never lets a NaN win (the NaN operand is ignored).
__device__ __forceinline__ float max_ignore_nan(float acc, float v) { return v > acc ? v : acc; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide max of a non-negative value, then one atomic max into *dst by
// thread 0 (integer order equals float order for values >= +0).
__device__ __forceinline__ void block_amax_atomic(float v, float *dst) {
    __shared__ float red[32];
    v = warp_max(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        float t = lane < nw ? red[lane] : 0.0f;
        t = warp_max(t);
        if (lane == 0 && dst != nullptr) atomicMax(reinterpret_cast<int *>(dst), __float_as_int(t));
    }
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace fp8mp
