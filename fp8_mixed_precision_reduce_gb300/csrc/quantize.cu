// quantize.cu -- scaled, saturating round-to-nearest-even cast of bf16/fp32
// tensors to E4M3/E5M2 with the fused per-tensor amax, and the variant that
// also writes the transposed copy the backward GEMMs consume.
//
// Pages: "Как работает FP8 quantization на H100 (Transformer Engine)?"
// (aivaro.ru) section 3, steps 2-3 -- the amax of the tensor and the cast of
// the scaled tensor; "Transformer Engine으로 FP8 사용하기" (coniverse.tistory.com)
// "Scaling factor 선택 전략" -- the per-tensor amax delayed scaling records.
//
// Both kernels are HBM-bound streams (algorithmic bytes per element: input
// 2 or 4, output 1, transposed output 1). Loads and stores are 16 bytes wide
// and coalesced; the amax is a per-thread max, a warp-shuffle max and one
// atomic max per block.
#include "fp8mp_internal.cuh"

namespace fp8mp {
namespace {

constexpr int kThreads = 256;

// 16 consecutive input elements starting at element 16*chunk, widened to fp32.
template <bool BF16>
__device__ __forceinline__ void load16(const void *x, int64_t chunk, float f[16]) {
    if constexpr (BF16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(x) + 2 * chunk;
        const uint4 a = __ldcs(p), b = __ldcs(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(x) + 4 * chunk;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = __ldcs(p + i);
            f[4 * i] = v.x;
            f[4 * i + 1] = v.y;
            f[4 * i + 2] = v.z;
            f[4 * i + 3] = v.w;
        }
    }
}

// 8 consecutive elements of row `r` starting at column `c`.
template <bool BF16>
__device__ __forceinline__ void load8(const void *x, int64_t cols, int64_t r, int64_t c, float f[8]) {
    const int64_t e = r * cols + c;
    if constexpr (BF16) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) + e));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + e);
        const float4 a = __ldcs(p), b = __ldcs(p + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
}

template <bool BF16>
__device__ __forceinline__ float load1(const void *x, int64_t i) {
    if constexpr (BF16)
        return bf16_bits_to_f32(reinterpret_cast<const uint16_t *>(x)[i]);
    else
        return reinterpret_cast<const float *>(x)[i];
}

// The casts' conversion step. cvt .satfinite rounds to nearest even and
// saturates finite overflow and infinities to the largest finite code; a NaN
// input gives a NaN code (E4M3 S.1111.111, E5M2 S.11111.mm with mm != 0) and
// no other input does. So instead of testing every element for NaN the casts
// test the packed codes: nan_probe sets bit 7 of every byte that holds a NaN
// code (the byte's low 7 bits plus 1 (E4M3) or 3 (E5M2) reach 0x80 exactly
// then, and no carry crosses a byte), and the rare words with one get their
// NaN bytes rewritten to 0x7F -- the same codes cvt_quad gives.
template <int FMT>
__device__ __forceinline__ uint32_t nan_probe(uint32_t codes) {
    return (codes & 0x7F7F7F7Fu) + (FMT == FP8MP_E4M3 ? 0x01010101u : 0x03030303u);
}
template <int FMT>
__device__ __forceinline__ uint32_t canonical_nan(uint32_t codes) {
    const uint32_t nan_bytes = ((nan_probe<FMT>(codes) & 0x80808080u) >> 7) * 0xFFu;
    return (codes & ~nan_bytes) | (0x7F7F7F7Fu & nan_bytes);
}
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair_raw(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == FP8MP_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Four elements -> four codes (little-endian) under `scale`; their |x| joins
// the running amax (fmaxf ignores a NaN operand, and the running value, which
// starts at +0, is never NaN) and their codes join the NaN probe.
template <int FMT>
__device__ __forceinline__ uint32_t cast4(float f0, float f1, float f2, float f3, float scale, float &am,
                                          uint32_t &probe) {
    const uint32_t q = cvt_pair_raw<FMT>(__fmul_rn(f0, scale), __fmul_rn(f1, scale)) |
                       (cvt_pair_raw<FMT>(__fmul_rn(f2, scale), __fmul_rn(f3, scale)) << 16);
    probe |= nan_probe<FMT>(q);
    am = fmaxf(fmaxf(am, fabsf(f0)), fmaxf(fabsf(f1), fmaxf(fabsf(f2), fabsf(f3))));
    return q;
}
// Two bf16 words (four elements) -> four codes.
template <int FMT>
__device__ __forceinline__ uint32_t cast4_bf16(uint32_t w0, uint32_t w1, float scale, float &am, uint32_t &probe) {
    return cast4<FMT>(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u), __uint_as_float(w1 << 16),
                      __uint_as_float(w1 & 0xFFFF0000u), scale, am, probe);
}

// Row-major cast of a flat array of n elements: chunks of 16 elements give
// one 16-byte store; the n % 16 tail is done element by element. Eight
// blocks of 256 threads fit an SM (32 registers a thread).
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads, 8)
cast_rows_kernel(const void *__restrict__ x, int64_t n, const float *__restrict__ scale_p,
                 uint8_t *__restrict__ out, float *__restrict__ amax_p) {
    pdl_wait();
    pdl_launch_dependents();
    const float scale = __ldg(scale_p);
    float am = 0.0f;
    const int64_t nchunk = n >> 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunk; c += stride) {
        uint32_t o[4], probe = 0;
        if constexpr (BF16) {
            const uint4 *p = reinterpret_cast<const uint4 *>(x) + 2 * c;
            const uint4 a = __ldcs(p), b = __ldcs(p + 1);
            o[0] = cast4_bf16<FMT>(a.x, a.y, scale, am, probe);
            o[1] = cast4_bf16<FMT>(a.z, a.w, scale, am, probe);
            o[2] = cast4_bf16<FMT>(b.x, b.y, scale, am, probe);
            o[3] = cast4_bf16<FMT>(b.z, b.w, scale, am, probe);
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(x) + 4 * c;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 v = __ldcs(p + j);
                o[j] = cast4<FMT>(v.x, v.y, v.z, v.w, scale, am, probe);
            }
        }
        if (probe & 0x80808080u) {
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = canonical_nan<FMT>(o[j]);
        }
        reinterpret_cast<uint4 *>(out)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (blockIdx.x == gridDim.x - 1) {
        for (int64_t i = (nchunk << 4) + threadIdx.x; i < n; i += blockDim.x) {
            const float v = load1<BF16>(x, i);
            out[i] = static_cast<uint8_t>(cvt_pair<FMT>(__fmul_rn(v, scale), 0.0f) & 0xFFu);
            am = fmaxf(am, fabsf(v));
        }
    }
    if (amax_p != nullptr) block_amax_atomic(am, amax_p);
}

// Row-major + transposed cast of one 128 x 128 tile per block.
// Phase 1: each thread converts a 4-row x 8-column patch (16-byte loads),
// stores its row-major bytes, transposes the 4 x 8 bytes in registers into
// eight 4-byte column words and parks them in shared memory, where word
// (column cc, row-group g) sits at index cc * 32 + (g ^ 2 * ((cc >> 3) & 15))
// -- the XOR spreads one store instruction of a warp over all 32 banks.
// Phase 2: each thread reads 16 consecutive row bytes of one column (one
// 16-byte shared load, un-permuting the XOR) and writes them to out_t, so a
// warp writes four full 128-byte rows of out_t.
// With DBIAS the kernel also sums its 128 rows per column (fp32, fixed order:
// each thread its 8 rows in row order, then the 16 row groups in order) and
// writes the 128 column sums of its tile to ws[tile_row * cols + col]; then
// out_t may be NULL (no transposed copy: phase 2 is skipped).
template <int FMT, bool BF16, bool DBIAS>
__global__ void __launch_bounds__(kThreads)
cast_rows_t_kernel(const void *__restrict__ x, int64_t rows, int64_t cols, const float *__restrict__ scale_p,
                   uint8_t *__restrict__ out, uint8_t *__restrict__ out_t, float *__restrict__ amax_p,
                   float *__restrict__ ws) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ __align__(16) uint32_t sT[128 * 32];
    __shared__ float s_colsum[DBIAS ? 16 * 128 : 1];
    float csum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int64_t tiles_c = (cols + 127) >> 7;
    const int64_t r0 = (blockIdx.x / tiles_c) * 128, c0 = (blockIdx.x % tiles_c) * 128;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const float scale = __ldg(scale_p);
    float am = 0.0f;
    const int64_t c = c0 + 8 * tx;
    const int sw1 = 2 * tx;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int g = ty + 16 * it;  // 4-row group within the tile
        const int64_t r = r0 + 4 * g;
        if (c < cols && r < rows) {
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8];
                load8<BF16>(x, cols, r + q, c, f);
                uint32_t probe = 0;
                lo[q] = cast4<FMT>(f[0], f[1], f[2], f[3], scale, am, probe);
                hi[q] = cast4<FMT>(f[4], f[5], f[6], f[7], scale, am, probe);
                if (probe & 0x80808080u) {
                    lo[q] = canonical_nan<FMT>(lo[q]);
                    hi[q] = canonical_nan<FMT>(hi[q]);
                }
                if constexpr (DBIAS) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) csum[j] = __fadd_rn(csum[j], f[j]);
                }
                *reinterpret_cast<uint2 *>(out + (r + q) * cols + c) = make_uint2(lo[q], hi[q]);
            }
            // 4 x 4 byte transposes: word j holds column (c + j), rows r .. r+3.
            uint32_t wcol[8];
            {
                const uint32_t t0 = __byte_perm(lo[0], lo[1], 0x5140), t1 = __byte_perm(lo[0], lo[1], 0x7362);
                const uint32_t t2 = __byte_perm(lo[2], lo[3], 0x5140), t3 = __byte_perm(lo[2], lo[3], 0x7362);
                wcol[0] = __byte_perm(t0, t2, 0x5410);
                wcol[1] = __byte_perm(t0, t2, 0x7632);
                wcol[2] = __byte_perm(t1, t3, 0x5410);
                wcol[3] = __byte_perm(t1, t3, 0x7632);
            }
            {
                const uint32_t t0 = __byte_perm(hi[0], hi[1], 0x5140), t1 = __byte_perm(hi[0], hi[1], 0x7362);
                const uint32_t t2 = __byte_perm(hi[2], hi[3], 0x5140), t3 = __byte_perm(hi[2], hi[3], 0x7362);
                wcol[4] = __byte_perm(t0, t2, 0x5410);
                wcol[5] = __byte_perm(t0, t2, 0x7632);
                wcol[6] = __byte_perm(t1, t3, 0x5410);
                wcol[7] = __byte_perm(t1, t3, 0x7632);
            }
            if (out_t != nullptr) {
#pragma unroll
                for (int j = 0; j < 8; ++j) sT[(8 * tx + j) * 32 + (g ^ sw1)] = wcol[j];
            }
        }
    }
    if constexpr (DBIAS) {
#pragma unroll
        for (int j = 0; j < 8; ++j) s_colsum[ty * 128 + 8 * tx + j] = csum[j];
    }
    __syncthreads();
    if constexpr (DBIAS) {
        if (threadIdx.x < 128 && c0 + threadIdx.x < cols) {
            float t = 0.0f;
            for (int g = 0; g < 16; ++g) t = __fadd_rn(t, s_colsum[g * 128 + threadIdx.x]);
            ws[(r0 >> 7) * cols + c0 + threadIdx.x] = t;
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (out_t == nullptr) break;
        const int id = threadIdx.x + kThreads * i;  // 0 .. 1023
        const int cc = id >> 3, k = id & 7;          // tile column, 16-row chunk
        const int64_t col = c0 + cc, row = r0 + 16 * k;
        if (col < cols && row < rows) {
            const int sw = 2 * ((cc >> 3) & 15);
            const uint4 P = *reinterpret_cast<const uint4 *>(&sT[cc * 32 + ((4 * k) ^ (sw & ~3))]);
            const uint4 o = (sw & 2) ? make_uint4(P.z, P.w, P.x, P.y) : P;
            *reinterpret_cast<uint4 *>(out_t + col * rows + row) = o;
        }
    }
    if (amax_p != nullptr) block_amax_atomic(am, amax_p);
}

// dbias[n] = the sum over tile rows t of ws[t * cols + n], in a fixed order:
// each of a block's 8 row groups sums the tile rows g, g + 8, g + 16, ...
// in increasing order, then the 8 group sums are added in group order. A
// block covers 32 columns, so each warp reads 128 contiguous bytes of one
// tile row and a thread has tile_rows / 8 independent loads in flight.
constexpr int kReduceCols = 32, kReduceGroups = 8;
__global__ void __launch_bounds__(kReduceCols * kReduceGroups)
dbias_reduce_kernel(const float *__restrict__ ws, int64_t tile_rows, int64_t cols, void *__restrict__ dbias,
                    int bf16_out) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ float part[kReduceGroups][kReduceCols];
    const int tx = threadIdx.x % kReduceCols, g = threadIdx.x / kReduceCols;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kReduceCols + tx;
    float t = 0.0f;
    if (n < cols) {
#pragma unroll 4
        for (int64_t r = g; r < tile_rows; r += kReduceGroups) t = __fadd_rn(t, ws[r * cols + n]);
    }
    part[g][tx] = t;
    __syncthreads();
    if (g != 0 || n >= cols) return;
    t = part[0][tx];
    for (int j = 1; j < kReduceGroups; ++j) t = __fadd_rn(t, part[j][tx]);
    if (bf16_out)
        static_cast<__nv_bfloat16 *>(dbias)[n] = __float2bfloat16_rn(t);
    else
        static_cast<float *>(dbias)[n] = t;
}

template <int FMT, bool BF16>
int launch_typed(const void *x, int64_t rows, int64_t cols, const float *scale, uint8_t *out,
                 uint8_t *out_t, float *amax, cudaStream_t s, const DeviceInfo &dev, float *ws = nullptr) {
    if (out_t == nullptr && ws == nullptr) {
        const int64_t n = rows * cols;
        const int64_t nchunk = n >> 4;
        // up to 32 blocks per SM (8 resident): smaller shares let the block
        // scheduler even out the tail, measured faster than one resident wave
        int64_t blocks = (nchunk + kThreads - 1) / kThreads;
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 32;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        launch_kernel(cast_rows_kernel<FMT, BF16>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, x, n,
                      scale, out, amax);
    } else {
        const int64_t tiles = ((rows + 127) >> 7) * ((cols + 127) >> 7);
        if (tiles > 0x7FFFFFFF) return fail(FP8MP_ERR_INVALID, "fp8_quantize: tensor too large");
        if (ws != nullptr)
            launch_kernel(cast_rows_t_kernel<FMT, BF16, true>, dim3(static_cast<unsigned>(tiles)), dim3(kThreads), 0,
                          s, x, rows, cols, scale, out, out_t, amax, ws);
        else
            launch_kernel(cast_rows_t_kernel<FMT, BF16, false>, dim3(static_cast<unsigned>(tiles)), dim3(kThreads), 0,
                          s, x, rows, cols, scale, out, out_t, amax, nullptr);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

// amax pass of current scaling: max |x| over a flat array, one atomic max
// per block into *amax (zeroed by the caller's stream just before).
template <bool BF16>
__global__ void __launch_bounds__(kThreads)
amax_kernel(const void *__restrict__ x, int64_t n, float *__restrict__ amax_p) {
    pdl_wait();
    pdl_launch_dependents();
    float am = 0.0f;
    const int64_t nchunk = n >> 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunk; c += stride) {
        float f[16];
        load16<BF16>(x, c, f);
#pragma unroll
        for (int j = 0; j < 16; ++j) am = fmaxf(am, fabsf(f[j]));
    }
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t i = (nchunk << 4) + threadIdx.x; i < n; i += blockDim.x) am = fmaxf(am, fabsf(load1<BF16>(x, i)));
    block_amax_atomic(am, amax_p);
}

// scale and scale_inv from this tensor's amax (the current-scaling rule).
__global__ void current_scale_kernel(const float *__restrict__ amax, float *__restrict__ scale,
                                     float *__restrict__ scale_inv, int fmt, int margin) {
    pdl_wait();
    pdl_launch_dependents();
    const float sc = scale_from_amax(*amax, *scale, fmt, margin);
    *scale = sc;
    *scale_inv = __fdiv_rn(1.0f, sc);
}

}  // namespace

int launch_quantize_current(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, int margin,
                            float *scale, float *scale_inv, float *amax, uint8_t *out, uint8_t *out_t,
                            cudaStream_t s, const DeviceInfo &dev) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_current: memset failed: %s", cudaGetErrorString(e));
    const int64_t n = rows * cols;
    int64_t blocks = ((n >> 4) + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (x_dtype == FP8MP_BF16)
        launch_kernel(amax_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, x, n, amax);
    else
        launch_kernel(amax_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, x, n, amax);
    launch_kernel(current_scale_kernel, dim3(1), dim3(1), 0, s, amax, scale, scale_inv, fmt, margin);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_current: launch failed: %s", cudaGetErrorString(e));
    if (n == 0) return FP8MP_OK;
    return launch_quantize(x, x_dtype, rows, cols, fmt, scale, out, out_t, nullptr, s, dev);
}

int launch_quantize_dbias(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, const float *scale,
                          uint8_t *out, uint8_t *out_t, float *amax, void *dbias, int dbias_dtype, float *ws,
                          cudaStream_t s, const DeviceInfo &dev) {
    const bool bf16 = x_dtype == FP8MP_BF16;
    int rc;
    if (fmt == FP8MP_E4M3)
        rc = bf16 ? launch_typed<FP8MP_E4M3, true>(x, rows, cols, scale, out, out_t, amax, s, dev, ws)
                  : launch_typed<FP8MP_E4M3, false>(x, rows, cols, scale, out, out_t, amax, s, dev, ws);
    else
        rc = bf16 ? launch_typed<FP8MP_E5M2, true>(x, rows, cols, scale, out, out_t, amax, s, dev, ws)
                  : launch_typed<FP8MP_E5M2, false>(x, rows, cols, scale, out, out_t, amax, s, dev, ws);
    if (rc) return rc;
    const int64_t tile_rows = (rows + 127) >> 7;
    launch_kernel(dbias_reduce_kernel, dim3(static_cast<unsigned>((cols + kReduceCols - 1) / kReduceCols)),
                  dim3(kReduceCols * kReduceGroups), 0, s, ws, tile_rows, cols, dbias, dbias_dtype == FP8MP_BF16 ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_dbias: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

int launch_quantize(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, const float *scale,
                    uint8_t *out, uint8_t *out_t, float *amax, cudaStream_t s, const DeviceInfo &dev) {
    const bool bf16 = x_dtype == FP8MP_BF16;
    if (fmt == FP8MP_E4M3)
        return bf16 ? launch_typed<FP8MP_E4M3, true>(x, rows, cols, scale, out, out_t, amax, s, dev)
                    : launch_typed<FP8MP_E4M3, false>(x, rows, cols, scale, out, out_t, amax, s, dev);
    return bf16 ? launch_typed<FP8MP_E5M2, true>(x, rows, cols, scale, out, out_t, amax, s, dev)
                : launch_typed<FP8MP_E5M2, false>(x, rows, cols, scale, out, out_t, amax, s, dev);
}

}  // namespace fp8mp
