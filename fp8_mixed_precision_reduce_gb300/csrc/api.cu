// api.cu -- the extern "C" entry points of libfp8mp declared in
// include/fp8mp.h: argument validation, device check, error reporting, and
// dispatch to the kernels' launchers. No computation happens here.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fp8mp_internal.cuh"

namespace fp8mp {

namespace {
__global__ void zero_word_kernel(uint32_t *word) {
    pdl_wait();  // the previous kernel may still read or write the word
    *word = 0u;
    pdl_launch_dependents();
}
// Sets the completion bit of an overflow word (an empty output is complete).
__global__ void signal_done_kernel(uint32_t *word) {
    pdl_wait();
    pdl_launch_dependents();
    __threadfence();
    atomicOr(word, kDoneBit);
}
}  // namespace

cudaError_t launch_signal_done(int32_t *word, cudaStream_t s) {
    return launch_kernel(signal_done_kernel, dim3(1), dim3(1), 0, s, reinterpret_cast<uint32_t *>(word));
}

cudaError_t launch_zero_word(void *word, cudaStream_t s) {
    return launch_kernel(zero_word_kernel, dim3(1), dim3(1), 0, s, static_cast<uint32_t *>(word));
}


namespace {
thread_local char g_last_error[512] = {0};
}

const char *last_error_message() { return g_last_error; }

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_last_error[0] = 0; }

bool pdl_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("FP8MP_PDL");
        return !(v != nullptr && std::strcmp(v, "0") == 0);
    }();
    return on;
}

int current_device(DeviceInfo *info) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    // per-device attributes, queried once; the flag is published after the
    // data (release) and checked before reading it (acquire)
    static DeviceInfo cache[64];
    static std::atomic<bool> have[64];
    if (dev >= 0 && dev < 64 && have[dev].load(std::memory_order_acquire)) {
        *info = cache[dev];
    } else {
        DeviceInfo d;
        d.device = dev;
        e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return fail(FP8MP_ERR_LAUNCH, "cudaDeviceGetAttribute failed: %s", cudaGetErrorString(e));
        if (dev >= 0 && dev < 64 && !have[dev].load(std::memory_order_acquire)) {
            static std::mutex m;
            std::lock_guard<std::mutex> lock(m);
            if (!have[dev].load(std::memory_order_relaxed)) {
                cache[dev] = d;
                have[dev].store(true, std::memory_order_release);
            }
        }
        *info = d;
    }
    if (info->cc_major != 10 || info->cc_minor != 3)
        return fail(FP8MP_ERR_DEVICE, "device %d is sm_%d%d; libfp8mp is built for sm_103a only", info->device,
                    info->cc_major, info->cc_minor);
    return FP8MP_OK;
}

}  // namespace fp8mp

using namespace fp8mp;

namespace {

bool valid_fmt(int32_t f) { return f == FP8MP_E4M3 || f == FP8MP_E5M2; }
bool valid_dtype(int32_t d) { return d == FP8MP_F32 || d == FP8MP_BF16; }

#define REQUIRE(cond, ...)                                        \
    do {                                                          \
        if (!(cond)) return fail(FP8MP_ERR_INVALID, __VA_ARGS__); \
    } while (0)

int check_ptr(const void *p, const char *fn, const char *name, bool required) {
    if (p == nullptr) {
        if (required) return fail(FP8MP_ERR_INVALID, "%s: %s is NULL", fn, name);
        return FP8MP_OK;
    }
    if (!aligned16(p)) return fail(FP8MP_ERR_INVALID, "%s: %s is not 16-byte aligned", fn, name);
    return FP8MP_OK;
}

#define CHECK_PTR(p, required)                              \
    do {                                                    \
        const int rc_ = check_ptr((p), fn, #p, (required)); \
        if (rc_) return rc_;                                \
    } while (0)

// Scalars (scales, amax slots, S, counters) only need 4-byte alignment.
int check_scalar(const void *p, const char *fn, const char *name, bool required) {
    if (p == nullptr) {
        if (required) return fail(FP8MP_ERR_INVALID, "%s: %s is NULL", fn, name);
        return FP8MP_OK;
    }
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return fail(FP8MP_ERR_INVALID, "%s: %s is misaligned", fn, name);
    return FP8MP_OK;
}

#define CHECK_SCALAR(p, required)                              \
    do {                                                       \
        const int rc_ = check_scalar((p), fn, #p, (required)); \
        if (rc_) return rc_;                                   \
    } while (0)

int check_gemm_dims(const char *fn, int64_t M, int64_t N, int64_t K) {
    REQUIRE(M >= 0 && N >= 0 && K >= 0, "%s: negative dimension", fn);
    REQUIRE(M % 16 == 0 && N % 16 == 0 && K % 16 == 0,
            "%s: M, N and K must be multiples of 16 (got %lld, %lld, %lld)", fn, (long long)M, (long long)N,
            (long long)K);
    REQUIRE(M <= (1ll << 30) && N <= (1ll << 30) && K <= (1ll << 30), "%s: dimension above 2^30", fn);
    return FP8MP_OK;
}

}  // namespace

extern "C" {

int32_t fp8mp_version(void) { return 1; }

const char *fp8mp_last_error(void) { return last_error_message(); }

static int quantize_entry(const char *fn, const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                          const float *scale, uint8_t *out, uint8_t *out_t, float *amax, uint32_t flags,
                          void *stream) {
    clear_error();
    REQUIRE(valid_dtype(x_dtype), "%s: x_dtype %d is not FP8MP_F32 or FP8MP_BF16", fn, x_dtype);
    REQUIRE(valid_fmt(fmt), "%s: fmt %d is not FP8MP_E4M3 or FP8MP_E5M2", fn, fmt);
    REQUIRE((flags & ~static_cast<uint32_t>(FP8MP_OVERLAP_PREVIOUS)) == 0u, "%s: unknown flags 0x%x", fn, flags);
    REQUIRE(rows >= 0 && cols >= 0, "%s: negative size", fn);
    REQUIRE(rows <= (1ll << 40) / (cols > 0 ? cols : 1), "%s: tensor too large", fn);
    if (out_t != nullptr)
        REQUIRE(rows % 16 == 0 && cols % 16 == 0,
                "%s: with a transposed output rows and cols must be multiples of 16 (got %lld x %lld)", fn,
                (long long)rows, (long long)cols);
    if (rows == 0 || cols == 0) return FP8MP_OK;
    CHECK_PTR(x, true);
    CHECK_PTR(out, true);
    CHECK_PTR(out_t, false);
    CHECK_SCALAR(scale, true);
    CHECK_SCALAR(amax, false);
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return launch_quantize(x, x_dtype, rows, cols, fmt, scale, out, out_t, amax, static_cast<cudaStream_t>(stream),
                           dev, (flags & FP8MP_OVERLAP_PREVIOUS) != 0u);
}

int fp8_quantize(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt, const float *scale,
                 uint8_t *out, uint8_t *out_t, float *amax, void *stream) {
    return quantize_entry("fp8_quantize", x, x_dtype, rows, cols, fmt, scale, out, out_t, amax, 0u, stream);
}

int fp8_quantize_ex(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt, const float *scale,
                    uint8_t *out, uint8_t *out_t, float *amax, uint32_t flags, void *stream) {
    return quantize_entry("fp8_quantize_ex", x, x_dtype, rows, cols, fmt, scale, out, out_t, amax, flags, stream);
}

int fp8_quantize_current(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt, int32_t margin,
                         float *scale, float *scale_inv, float *amax, uint8_t *out, uint8_t *out_t, void *stream) {
    const char *fn = "fp8_quantize_current";
    clear_error();
    REQUIRE(valid_dtype(x_dtype), "%s: x_dtype %d is not FP8MP_F32 or FP8MP_BF16", fn, x_dtype);
    REQUIRE(valid_fmt(fmt), "%s: fmt %d is not FP8MP_E4M3 or FP8MP_E5M2", fn, fmt);
    REQUIRE(margin >= 0 && margin <= 126, "%s: margin %d outside 0..126", fn, margin);
    REQUIRE(rows >= 0 && cols >= 0, "%s: negative size", fn);
    REQUIRE(rows <= (1ll << 40) / (cols > 0 ? cols : 1), "%s: tensor too large", fn);
    if (out_t != nullptr)
        REQUIRE(rows % 16 == 0 && cols % 16 == 0,
                "%s: with a transposed output rows and cols must be multiples of 16 (got %lld x %lld)", fn,
                (long long)rows, (long long)cols);
    CHECK_SCALAR(scale, true);
    CHECK_SCALAR(scale_inv, true);
    CHECK_SCALAR(amax, true);
    if (rows > 0 && cols > 0) {
        CHECK_PTR(x, true);
        CHECK_PTR(out, true);
        CHECK_PTR(out_t, false);
    }
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    return launch_quantize_current(x, x_dtype, rows, cols, fmt, margin, scale, scale_inv, amax, out, out_t,
                                   static_cast<cudaStream_t>(stream), dev);
}

int64_t fp8_quantize_dbias_workspace_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return -1;
    if (rows > (1ll << 40) / (cols > 0 ? cols : 1)) return -1;
    // the column sums of each of the k CTAs of a strip, then one arrival
    // counter per 128-column strip
    const int64_t bytes = static_cast<int64_t>(dbias_ctas_per_strip(rows, cols)) * cols *
                              static_cast<int64_t>(sizeof(float)) +
                          ((cols + 127) / 128) * static_cast<int64_t>(sizeof(uint32_t));
    return (bytes + 15) & ~static_cast<int64_t>(15);
}

int fp8_quantize_dbias(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt, const float *scale,
                       uint8_t *out, uint8_t *out_t, float *amax, void *dbias, int32_t dbias_dtype, float *workspace,
                       int64_t workspace_bytes, void *stream) {
    const char *fn = "fp8_quantize_dbias";
    clear_error();
    REQUIRE(valid_dtype(x_dtype), "%s: x_dtype %d is not FP8MP_F32 or FP8MP_BF16", fn, x_dtype);
    REQUIRE(valid_dtype(dbias_dtype), "%s: dbias_dtype %d invalid", fn, dbias_dtype);
    REQUIRE(valid_fmt(fmt), "%s: fmt %d is not FP8MP_E4M3 or FP8MP_E5M2", fn, fmt);
    REQUIRE(rows >= 0 && cols >= 0, "%s: negative size", fn);
    REQUIRE(rows <= (1ll << 40) / (cols > 0 ? cols : 1), "%s: tensor too large", fn);
    REQUIRE(rows % 16 == 0 && cols % 16 == 0, "%s: rows and cols must be multiples of 16 (got %lld x %lld)", fn,
            (long long)rows, (long long)cols);
    REQUIRE(rows < (1ll << 31) && cols < (1ll << 31), "%s: rows and cols must be below 2^31", fn);
    if (cols == 0) return FP8MP_OK;
    CHECK_PTR(dbias, true);
    const int64_t need = fp8_quantize_dbias_workspace_bytes(rows, cols);
    if (rows > 0) {
        CHECK_PTR(x, true);
        CHECK_PTR(out, true);
        CHECK_PTR(out_t, false);
        CHECK_SCALAR(scale, true);
        CHECK_SCALAR(amax, false);
        CHECK_PTR(workspace, true);
        REQUIRE(workspace_bytes >= need, "%s: workspace of %lld bytes, %lld needed", fn, (long long)workspace_bytes,
                (long long)need);
    }
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    if (rows == 0) {
        const cudaError_t e =
            cudaMemsetAsync(dbias, 0, static_cast<size_t>(cols) * (dbias_dtype == FP8MP_BF16 ? 2 : 4),
                            static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: memset failed: %s", fn, cudaGetErrorString(e));
        return FP8MP_OK;
    }
    return launch_quantize_dbias(x, x_dtype, rows, cols, fmt, scale, out, out_t, amax, dbias, dbias_dtype, workspace,
                                 static_cast<cudaStream_t>(stream), dev);
}

int fp8_linear_fwd(const uint8_t *x8, const uint8_t *w8, int64_t M, int64_t N, int64_t K, const float *sinv_x,
                   const float *sinv_w, const void *bias, int32_t bias_dtype, void *y, int32_t y_dtype,
                   float *y_amax, void *stream) {
    const char *fn = "fp8_linear_fwd";
    clear_error();
    int rc = check_gemm_dims(fn, M, N, K);
    if (rc) return rc;
    REQUIRE(valid_dtype(y_dtype), "%s: y_dtype %d invalid", fn, y_dtype);
    REQUIRE(bias == nullptr || valid_dtype(bias_dtype), "%s: bias_dtype %d invalid", fn, bias_dtype);
    if (M == 0 || N == 0) return FP8MP_OK;
    CHECK_PTR(y, true);
    CHECK_PTR(bias, false);
    CHECK_SCALAR(y_amax, false);
    CHECK_SCALAR(sinv_x, true);
    CHECK_SCALAR(sinv_w, true);
    if (K > 0) {
        CHECK_PTR(x8, true);
        CHECK_PTR(w8, true);
    }
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    return launch_gemm(x8, FP8MP_E4M3, w8, FP8MP_E4M3, M, N, K, sinv_x, sinv_w, bias, bias_dtype, y, y_dtype,
                       y_amax, static_cast<cudaStream_t>(stream), dev);
}

int fp8_linear_fwd_fp8out(const uint8_t *x8, const uint8_t *w8, int64_t M, int64_t N, int64_t K, const float *sinv_x,
                          const float *sinv_w, const void *bias, int32_t bias_dtype, const float *y_scale,
                          int32_t y_fmt, uint8_t *y8, float *y_amax, void *stream) {
    const char *fn = "fp8_linear_fwd_fp8out";
    clear_error();
    int rc = check_gemm_dims(fn, M, N, K);
    if (rc) return rc;
    REQUIRE(valid_fmt(y_fmt), "%s: y_fmt %d invalid", fn, y_fmt);
    REQUIRE(bias == nullptr || valid_dtype(bias_dtype), "%s: bias_dtype %d invalid", fn, bias_dtype);
    if (M == 0 || N == 0) return FP8MP_OK;
    CHECK_PTR(y8, true);
    CHECK_PTR(bias, false);
    CHECK_SCALAR(y_amax, false);
    CHECK_SCALAR(y_scale, true);
    CHECK_SCALAR(sinv_x, true);
    CHECK_SCALAR(sinv_w, true);
    if (K > 0) {
        CHECK_PTR(x8, true);
        CHECK_PTR(w8, true);
    }
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    return launch_gemm(x8, FP8MP_E4M3, w8, FP8MP_E4M3, M, N, K, sinv_x, sinv_w, bias, bias_dtype, y8, FP8MP_F32,
                       y_amax, static_cast<cudaStream_t>(stream), dev, y_scale, y_fmt);
}

int fp8_linear_dgrad(const uint8_t *dy8, const uint8_t *w8t, int64_t M, int64_t N, int64_t K, int32_t dy_fmt,
                     const float *sinv_dy, const float *sinv_w, void *dx, int32_t dx_dtype, void *stream) {
    const char *fn = "fp8_linear_dgrad";
    clear_error();
    int rc = check_gemm_dims(fn, M, N, K);
    if (rc) return rc;
    REQUIRE(valid_fmt(dy_fmt), "%s: dy_fmt %d invalid", fn, dy_fmt);
    REQUIRE(valid_dtype(dx_dtype), "%s: dx_dtype %d invalid", fn, dx_dtype);
    if (M == 0 || K == 0) return FP8MP_OK;
    CHECK_PTR(dx, true);
    CHECK_SCALAR(sinv_dy, true);
    CHECK_SCALAR(sinv_w, true);
    if (N > 0) {
        CHECK_PTR(dy8, true);
        CHECK_PTR(w8t, true);
    }
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    return launch_gemm(dy8, dy_fmt, w8t, FP8MP_E4M3, M, K, N, sinv_dy, sinv_w, nullptr, FP8MP_F32, dx, dx_dtype,
                       nullptr, static_cast<cudaStream_t>(stream), dev);
}

int fp8_linear_wgrad(const uint8_t *dy8t, const uint8_t *x8t, int64_t M, int64_t N, int64_t K, int32_t dy_fmt,
                     const float *sinv_dy, const float *sinv_x, void *dw, int32_t dw_dtype, void *stream) {
    const char *fn = "fp8_linear_wgrad";
    clear_error();
    int rc = check_gemm_dims(fn, M, N, K);
    if (rc) return rc;
    REQUIRE(valid_fmt(dy_fmt), "%s: dy_fmt %d invalid", fn, dy_fmt);
    REQUIRE(valid_dtype(dw_dtype), "%s: dw_dtype %d invalid", fn, dw_dtype);
    if (N == 0 || K == 0) return FP8MP_OK;
    CHECK_PTR(dw, true);
    CHECK_SCALAR(sinv_dy, true);
    CHECK_SCALAR(sinv_x, true);
    if (M > 0) {
        CHECK_PTR(dy8t, true);
        CHECK_PTR(x8t, true);
    }
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    return launch_gemm(dy8t, dy_fmt, x8t, FP8MP_E4M3, N, K, M, sinv_dy, sinv_x, nullptr, FP8MP_F32, dw, dw_dtype,
                       nullptr, static_cast<cudaStream_t>(stream), dev);
}

int fp8_linear_bwd(const uint8_t *dy8, const uint8_t *dy8t, const uint8_t *w8t, const uint8_t *x8t, int64_t M,
                   int64_t N, int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                   const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype, void *stream) {
    const char *fn = "fp8_linear_bwd";
    clear_error();
    int rc = check_gemm_dims(fn, M, N, K);
    if (rc) return rc;
    REQUIRE(valid_fmt(dy_fmt), "%s: dy_fmt %d invalid", fn, dy_fmt);
    REQUIRE(valid_dtype(dx_dtype), "%s: dx_dtype %d invalid", fn, dx_dtype);
    REQUIRE(valid_dtype(dw_dtype), "%s: dw_dtype %d invalid", fn, dw_dtype);
    if (K == 0 || (M == 0 && N == 0)) return FP8MP_OK;
    CHECK_SCALAR(sinv_dy, true);
    if (M > 0) {
        CHECK_PTR(dx, true);
        CHECK_SCALAR(sinv_w, true);
    }
    if (N > 0) {
        CHECK_PTR(dw, true);
        CHECK_SCALAR(sinv_x, true);
    }
    if (M > 0 && N > 0) {
        CHECK_PTR(dy8, true);
        CHECK_PTR(dy8t, true);
        CHECK_PTR(w8t, true);
        CHECK_PTR(x8t, true);
        const uintptr_t a = reinterpret_cast<uintptr_t>(dx), b = reinterpret_cast<uintptr_t>(dw);
        const uintptr_t na = static_cast<uintptr_t>(M * K) * (dx_dtype == FP8MP_BF16 ? 2 : 4);
        const uintptr_t nb = static_cast<uintptr_t>(N * K) * (dw_dtype == FP8MP_BF16 ? 2 : 4);
        REQUIRE(a + na <= b || b + nb <= a, "%s: dx and dw overlap", fn);
    }
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    const GemmDesc d[2] = {
        {dy8, dy_fmt, w8t, FP8MP_E4M3, M, K, N, sinv_dy, sinv_w, nullptr, FP8MP_F32, dx, dx_dtype, nullptr, nullptr,
         FP8MP_E4M3, 0, 0},
        {dy8t, dy_fmt, x8t, FP8MP_E4M3, N, K, M, sinv_dy, sinv_x, nullptr, FP8MP_F32, dw, dw_dtype, nullptr, nullptr,
         FP8MP_E4M3, 0, 0}};
    return launch_gemms(d, 2, static_cast<cudaStream_t>(stream), dev);
}

static int bwd_rowmajor_entry(const char *fn, const uint8_t *dy8, const uint8_t *w8, const uint8_t *x8, int64_t M,
                              int64_t N, int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                              const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype,
                              int32_t *dw_nonfinite, uint32_t flags, void *stream) {
    clear_error();
    REQUIRE((flags & ~static_cast<uint32_t>(FP8MP_SIGNAL_DW_DONE)) == 0u, "%s: unknown flags 0x%x", fn, flags);
    if (flags & FP8MP_SIGNAL_DW_DONE)
        REQUIRE(dw != nullptr && dw_nonfinite != nullptr, "%s: FP8MP_SIGNAL_DW_DONE needs dw and dw_nonfinite", fn);
    int rc = check_gemm_dims(fn, M, N, K);
    if (rc) return rc;
    REQUIRE(valid_fmt(dy_fmt), "%s: dy_fmt %d invalid", fn, dy_fmt);
    REQUIRE(dx == nullptr || valid_dtype(dx_dtype), "%s: dx_dtype %d invalid", fn, dx_dtype);
    REQUIRE(dw == nullptr || valid_dtype(dw_dtype), "%s: dw_dtype %d invalid", fn, dw_dtype);
    const bool want_dx = dx != nullptr && M > 0 && K > 0;
    const bool want_dw = dw != nullptr && N > 0 && K > 0;
    const bool signal = (flags & FP8MP_SIGNAL_DW_DONE) != 0u;
    if (!want_dx && !want_dw && !signal) return FP8MP_OK;
    CHECK_PTR(dx, false);
    CHECK_PTR(dw, false);
    CHECK_SCALAR(dw_nonfinite, false);
    if (!want_dx && !want_dw) {  // an empty dW is complete at once
        DeviceInfo dev;
        rc = current_device(&dev);
        if (rc) return rc;
        const cudaError_t e = launch_signal_done(dw_nonfinite, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
        return FP8MP_OK;
    }
    CHECK_SCALAR(sinv_dy, true);
    if (want_dx) CHECK_SCALAR(sinv_w, true);
    if (want_dw) CHECK_SCALAR(sinv_x, true);
    if (M > 0 && N > 0) {
        CHECK_PTR(dy8, true);
        if (want_dx) CHECK_PTR(w8, true);
        if (want_dw) CHECK_PTR(x8, true);
    }
    if (want_dx && want_dw) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(dx), b = reinterpret_cast<uintptr_t>(dw);
        const uintptr_t na = static_cast<uintptr_t>(M * K) * (dx_dtype == FP8MP_BF16 ? 2 : 4);
        const uintptr_t nb = static_cast<uintptr_t>(N * K) * (dw_dtype == FP8MP_BF16 ? 2 : 4);
        REQUIRE(a + na <= b || b + nb <= a, "%s: dx and dw overlap", fn);
    }
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    GemmDesc d[2];
    int n = 0;
    // dgrad: A = dY8 [M x N] K-major, B = W8 [N x K] read MN-major (rows_b = K, kc = N)
    if (want_dx)
        d[n++] = {dy8, dy_fmt, w8, FP8MP_E4M3, M, K, N, sinv_dy, sinv_w, nullptr, FP8MP_F32, dx, dx_dtype, nullptr,
                  nullptr, FP8MP_E4M3, 0, 1};
    // wgrad: A = dY8 [M x N] read MN-major (rows_a = N, kc = M), B = X8 [M x K] read MN-major
    if (want_dw)
        d[n++] = {dy8,     dy_fmt,    x8,  FP8MP_E4M3, N,     K,       M,          sinv_dy, sinv_x, nullptr,
                  FP8MP_F32, dw,      dw_dtype, nullptr, nullptr, FP8MP_E4M3, 1, 1, dw_nonfinite,
                  signal};
    if (!want_dw && signal) {  // dx only: dW is empty, complete before the GEMM
        const cudaError_t e = launch_signal_done(dw_nonfinite, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    }
    return launch_gemms(d, n, static_cast<cudaStream_t>(stream), dev);
}

int fp8_linear_bwd_rowmajor(const uint8_t *dy8, const uint8_t *w8, const uint8_t *x8, int64_t M, int64_t N,
                            int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                            const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype,
                            int32_t *dw_nonfinite, void *stream) {
    return bwd_rowmajor_entry("fp8_linear_bwd_rowmajor", dy8, w8, x8, M, N, K, dy_fmt, sinv_dy, sinv_w, sinv_x, dx,
                              dx_dtype, dw, dw_dtype, dw_nonfinite, 0u, stream);
}

int fp8_linear_bwd_rowmajor_ex(const uint8_t *dy8, const uint8_t *w8, const uint8_t *x8, int64_t M, int64_t N,
                               int64_t K, int32_t dy_fmt, const float *sinv_dy, const float *sinv_w,
                               const float *sinv_x, void *dx, int32_t dx_dtype, void *dw, int32_t dw_dtype,
                               int32_t *dw_nonfinite, uint32_t flags, void *stream) {
    return bwd_rowmajor_entry("fp8_linear_bwd_rowmajor_ex", dy8, w8, x8, M, N, K, dy_fmt, sinv_dy, sinv_w, sinv_x,
                              dx, dx_dtype, dw, dw_dtype, dw_nonfinite, flags, stream);
}

static int scale_update_entry(const char *fn, const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin,
                              float *prev_scale_inv, void *stream) {
    clear_error();
    REQUIRE(n >= 0, "%s: negative count", fn);
    if (n == 0) return FP8MP_OK;
    REQUIRE(metas != nullptr, "%s: metas is NULL", fn);
    REQUIRE(algo == FP8MP_AMAX_MAX || algo == FP8MP_AMAX_MOST_RECENT, "%s: algo %d invalid", fn, algo);
    REQUIRE(margin >= 0 && margin <= 126, "%s: margin %d outside 0..126", fn, margin);
    CHECK_SCALAR(prev_scale_inv, false);
    for (int32_t i = 0; i < n; ++i) {
        const fp8mp_meta &m = metas[i];
        REQUIRE(m.history_len >= 1 && m.history_len <= FP8MP_MAX_HISTORY, "%s: meta %d history_len %d outside 1..%d",
                fn, i, m.history_len, FP8MP_MAX_HISTORY);
        REQUIRE(valid_fmt(m.fmt), "%s: meta %d fmt %d invalid", fn, i, m.fmt);
        REQUIRE(m.amax_history && m.scale && m.scale_inv && m.cur_amax, "%s: meta %d has a NULL pointer", fn, i);
    }
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    return launch_scale_update(metas, n, algo, margin, static_cast<cudaStream_t>(stream), prev_scale_inv);
}

int delayed_scaling_update(const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin, void *stream) {
    return scale_update_entry("delayed_scaling_update", metas, n, algo, margin, nullptr, stream);
}

int delayed_scaling_update_ex(const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin,
                              float *prev_scale_inv, void *stream) {
    return scale_update_entry("delayed_scaling_update_ex", metas, n, algo, margin, prev_scale_inv, stream);
}

// w8_in and the flags of the _ex forms: the current E4M3 copy (NULL or w8
// itself: in place) and FP8MP_OVERLAP_PREVIOUS.
static int check_w8_pair(const char *fn, const uint8_t *w8_in, const uint8_t *w8, int64_t n, uint32_t flags) {
    REQUIRE((flags & ~static_cast<uint32_t>(FP8MP_OVERLAP_PREVIOUS | FP8MP_WAIT_DW_DONE)) == 0u,
            "%s: unknown flags 0x%x", fn, flags);
    REQUIRE(!(flags & FP8MP_WAIT_DW_DONE) || (flags & FP8MP_OVERLAP_PREVIOUS),
            "%s: FP8MP_WAIT_DW_DONE needs FP8MP_OVERLAP_PREVIOUS", fn);
    CHECK_PTR(w8_in, false);
    if (w8_in != nullptr && w8_in != w8 && n > 0)
        REQUIRE(w8_in + n <= w8 || w8 + n <= w8_in, "%s: w8_in and w8_out overlap without being equal", fn);
    return FP8MP_OK;
}

// The metas of a master step that also runs the step's delayed-scaling
// update (the _scaling_ex entries): validated as delayed_scaling_update
// validates them, at most kMaxFoldMetas, the weight's meta found by its
// scale pointer (it must then also hold amax_w); the step must start beside
// the backward launch and wait for its dW signal.
static int build_fold(const char *fn, const fp8mp_meta *metas, int32_t n_metas, int32_t algo, int32_t margin,
                      const float *scale_w, const float *amax_w, uint32_t flags, FoldBatch *fb) {
    std::memset(fb, 0, sizeof *fb);
    fb->w_index = -1;
    REQUIRE(n_metas >= 0 && n_metas <= kMaxFoldMetas, "%s: n_metas = %d outside 0..%d", fn, n_metas, kMaxFoldMetas);
    REQUIRE(n_metas == 0 || metas != nullptr, "%s: metas is NULL", fn);
    REQUIRE(algo == FP8MP_AMAX_MAX || algo == FP8MP_AMAX_MOST_RECENT, "%s: algo %d invalid", fn, algo);
    REQUIRE(margin >= 0 && margin <= 126, "%s: margin %d outside 0..126", fn, margin);
    REQUIRE(flags == (FP8MP_OVERLAP_PREVIOUS | FP8MP_WAIT_DW_DONE),
            "%s: flags must be FP8MP_OVERLAP_PREVIOUS | FP8MP_WAIT_DW_DONE", fn);
    for (int32_t i = 0; i < n_metas; ++i) {
        const fp8mp_meta &m = metas[i];
        REQUIRE(m.history_len >= 1 && m.history_len <= FP8MP_MAX_HISTORY, "%s: meta %d history_len %d outside 1..%d",
                fn, i, m.history_len, FP8MP_MAX_HISTORY);
        REQUIRE(valid_fmt(m.fmt), "%s: meta %d fmt %d invalid", fn, i, m.fmt);
        REQUIRE(m.amax_history && m.scale && m.scale_inv && m.cur_amax, "%s: meta %d has a NULL pointer", fn, i);
        if (m.scale == scale_w) {
            REQUIRE(fb->w_index < 0, "%s: two metas hold scale_w", fn);
            REQUIRE(m.cur_amax == amax_w, "%s: the meta holding scale_w must hold amax_w as its cur_amax", fn);
            fb->w_index = i;
        }
        // the step adds to amax_w only after the weight's meta (found by
        // scale_w) has zeroed it: a meta holding amax_w under another scale
        // would zero it while the step's blocks add to it
        REQUIRE(m.cur_amax != amax_w || m.scale == scale_w, "%s: meta %d holds amax_w but not scale_w", fn, i);
        fb->m[i] = FoldMeta{m.amax_history, m.scale, m.scale_inv, m.cur_amax, m.history_len, m.fmt};
    }
    fb->n = n_metas;
    fb->algo = algo;
    fb->margin = margin;
    return FP8MP_OK;
}

static int master_step_entry(const char *fn, const uint16_t *grad_bf16, int64_t n, float *master,
                             float *momentum, uint8_t *w8, const float *scale_w, float *amax_w, float *loss_scale,
                             int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite, bool prescanned,
                             float lr, float momentum_coef, float backoff, float growth_factor,
                             int32_t growth_interval, void *stream, const uint8_t *w8_in = nullptr,
                             uint32_t flags = 0u, const FoldBatch *fold = nullptr) {
    clear_error();
    REQUIRE(n >= 0 && n <= (1ll << 40), "%s: n = %lld out of range", fn, (long long)n);
    REQUIRE(growth_interval >= 1, "%s: growth_interval must be >= 1", fn);
    CHECK_PTR(grad_bf16, n > 0);
    CHECK_PTR(master, n > 0);
    CHECK_PTR(momentum, n > 0);
    CHECK_PTR(w8, n > 0);
    {
        const int rc_ = check_w8_pair(fn, w8_in, w8, n, flags);
        if (rc_) return rc_;
    }
    CHECK_SCALAR(scale_w, true);
    CHECK_SCALAR(amax_w, true);
    CHECK_SCALAR(loss_scale, true);
    CHECK_SCALAR(growth_tracker, true);
    CHECK_SCALAR(found_inf, true);
    CHECK_SCALAR(grad_nonfinite, prescanned);
    REQUIRE(grad_nonfinite != found_inf, "%s: grad_nonfinite and found_inf must be different words", fn);
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    return launch_master_step(grad_bf16, n, master, momentum, w8, scale_w, amax_w, loss_scale, growth_tracker,
                              found_inf, lr, momentum_coef, backoff, growth_factor, growth_interval,
                              static_cast<cudaStream_t>(stream), dev, grad_nonfinite, w8_in,
                              (flags & FP8MP_OVERLAP_PREVIOUS) != 0u, (flags & FP8MP_WAIT_DW_DONE) != 0u, fold);
}

int mp_master_step(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum, uint8_t *w8,
                   const float *scale_w, float *amax_w, float *loss_scale, int32_t *growth_tracker,
                   int32_t *found_inf, float lr, float momentum_coef, float backoff, float growth_factor,
                   int32_t growth_interval, void *stream) {
    return master_step_entry("mp_master_step", grad_bf16, n, master, momentum, w8, scale_w, amax_w, loss_scale,
                             growth_tracker, found_inf, nullptr, false, lr, momentum_coef, backoff, growth_factor,
                             growth_interval, stream);
}

int mp_master_step_prescanned(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum, uint8_t *w8,
                              const float *scale_w, float *amax_w, float *loss_scale, int32_t *growth_tracker,
                              int32_t *found_inf, int32_t *grad_nonfinite, float lr, float momentum_coef,
                              float backoff, float growth_factor, int32_t growth_interval, void *stream) {
    return master_step_entry("mp_master_step_prescanned", grad_bf16, n, master, momentum, w8, scale_w, amax_w,
                             loss_scale, growth_tracker, found_inf, grad_nonfinite, true, lr, momentum_coef, backoff,
                             growth_factor, growth_interval, stream);
}

static int adam_step_entry(const char *fn, const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                           float *exp_avg_sq, uint8_t *w8, const float *scale_w, float *amax_w, float *loss_scale,
                           int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite, bool prescanned,
                           float *beta_pows, float lr, float beta1, float beta2, float eps, float backoff,
                           float growth_factor, int32_t growth_interval, void *stream,
                           const uint8_t *w8_in = nullptr, uint32_t flags = 0u, const FoldBatch *fold = nullptr) {
    clear_error();
    REQUIRE(n >= 0 && n <= (1ll << 40), "%s: n = %lld out of range", fn, (long long)n);
    REQUIRE(growth_interval >= 1, "%s: growth_interval must be >= 1", fn);
    REQUIRE(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f, "%s: betas must lie in [0, 1)", fn);
    CHECK_PTR(grad_bf16, n > 0);
    CHECK_PTR(master, n > 0);
    CHECK_PTR(exp_avg, n > 0);
    CHECK_PTR(exp_avg_sq, n > 0);
    CHECK_PTR(w8, n > 0);
    CHECK_SCALAR(scale_w, true);
    CHECK_SCALAR(amax_w, true);
    CHECK_SCALAR(loss_scale, true);
    CHECK_SCALAR(growth_tracker, true);
    CHECK_SCALAR(found_inf, true);
    CHECK_SCALAR(beta_pows, true);
    CHECK_SCALAR(grad_nonfinite, prescanned);
    REQUIRE(grad_nonfinite != found_inf, "%s: grad_nonfinite and found_inf must be different words", fn);
    {
        const int rc_ = check_w8_pair(fn, w8_in, w8, n, flags);
        if (rc_) return rc_;
    }
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    return launch_adam_step(grad_bf16, n, master, exp_avg, exp_avg_sq, w8, scale_w, amax_w, loss_scale,
                            growth_tracker, found_inf, beta_pows, lr, beta1, beta2, eps, backoff, growth_factor,
                            growth_interval, static_cast<cudaStream_t>(stream), dev, grad_nonfinite, w8_in,
                            (flags & FP8MP_OVERLAP_PREVIOUS) != 0u, (flags & FP8MP_WAIT_DW_DONE) != 0u, fold);
}

int mp_master_step_adam(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg, float *exp_avg_sq,
                        uint8_t *w8, const float *scale_w, float *amax_w, float *loss_scale, int32_t *growth_tracker,
                        int32_t *found_inf, float *beta_pows, float lr, float beta1, float beta2, float eps,
                        float backoff, float growth_factor, int32_t growth_interval, void *stream) {
    return adam_step_entry("mp_master_step_adam", grad_bf16, n, master, exp_avg, exp_avg_sq, w8, scale_w, amax_w,
                           loss_scale, growth_tracker, found_inf, nullptr, false, beta_pows, lr, beta1, beta2, eps,
                           backoff, growth_factor, growth_interval, stream);
}

int mp_master_step_adam_prescanned(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                                   float *exp_avg_sq, uint8_t *w8, const float *scale_w, float *amax_w,
                                   float *loss_scale, int32_t *growth_tracker, int32_t *found_inf,
                                   int32_t *grad_nonfinite, float *beta_pows, float lr, float beta1, float beta2,
                                   float eps, float backoff, float growth_factor, int32_t growth_interval,
                                   void *stream) {
    return adam_step_entry("mp_master_step_adam_prescanned", grad_bf16, n, master, exp_avg, exp_avg_sq, w8, scale_w,
                           amax_w, loss_scale, growth_tracker, found_inf, grad_nonfinite, true, beta_pows, lr, beta1,
                           beta2, eps, backoff, growth_factor, growth_interval, stream);
}

int mp_master_step_prescanned_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum,
                                 const uint8_t *w8_in, uint8_t *w8_out, const float *scale_w, float *amax_w,
                                 float *loss_scale, int32_t *growth_tracker, int32_t *found_inf,
                                 int32_t *grad_nonfinite, float lr, float momentum_coef, float backoff,
                                 float growth_factor, int32_t growth_interval, uint32_t flags, void *stream) {
    return master_step_entry("mp_master_step_prescanned_ex", grad_bf16, n, master, momentum, w8_out, scale_w, amax_w,
                             loss_scale, growth_tracker, found_inf, grad_nonfinite, true, lr, momentum_coef, backoff,
                             growth_factor, growth_interval, stream, w8_in, flags);
}

int mp_master_step_adam_prescanned_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                                      float *exp_avg_sq, const uint8_t *w8_in, uint8_t *w8_out,
                                      const float *scale_w, float *amax_w, float *loss_scale,
                                      int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite,
                                      float *beta_pows, float lr, float beta1, float beta2, float eps, float backoff,
                                      float growth_factor, int32_t growth_interval, uint32_t flags, void *stream) {
    return adam_step_entry("mp_master_step_adam_prescanned_ex", grad_bf16, n, master, exp_avg, exp_avg_sq, w8_out,
                           scale_w, amax_w, loss_scale, growth_tracker, found_inf, grad_nonfinite, true, beta_pows,
                           lr, beta1, beta2, eps, backoff, growth_factor, growth_interval, stream, w8_in, flags);
}

int mp_master_step_prescanned_scaling_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *momentum,
                                         const uint8_t *w8_in, uint8_t *w8_out, const float *scale_w,
                                         float *amax_w, float *loss_scale, int32_t *growth_tracker,
                                         int32_t *found_inf, int32_t *grad_nonfinite, float lr, float momentum_coef,
                                         float backoff, float growth_factor, int32_t growth_interval,
                                         const fp8mp_meta *metas, int32_t n_metas, int32_t amax_algo,
                                         int32_t margin, uint32_t flags, void *stream) {
    const char *fn = "mp_master_step_prescanned_scaling_ex";
    clear_error();
    FoldBatch fb;
    const int rc = build_fold(fn, metas, n_metas, amax_algo, margin, scale_w, amax_w, flags, &fb);
    if (rc) return rc;
    return master_step_entry(fn, grad_bf16, n, master, momentum, w8_out, scale_w, amax_w, loss_scale, growth_tracker,
                             found_inf, grad_nonfinite, true, lr, momentum_coef, backoff, growth_factor,
                             growth_interval, stream, w8_in, flags, &fb);
}

int mp_master_step_adam_prescanned_scaling_ex(const uint16_t *grad_bf16, int64_t n, float *master, float *exp_avg,
                                              float *exp_avg_sq, const uint8_t *w8_in, uint8_t *w8_out,
                                              const float *scale_w, float *amax_w, float *loss_scale,
                                              int32_t *growth_tracker, int32_t *found_inf, int32_t *grad_nonfinite,
                                              float *beta_pows, float lr, float beta1, float beta2, float eps,
                                              float backoff, float growth_factor, int32_t growth_interval,
                                              const fp8mp_meta *metas, int32_t n_metas, int32_t amax_algo,
                                              int32_t margin, uint32_t flags, void *stream) {
    const char *fn = "mp_master_step_adam_prescanned_scaling_ex";
    clear_error();
    FoldBatch fb;
    const int rc = build_fold(fn, metas, n_metas, amax_algo, margin, scale_w, amax_w, flags, &fb);
    if (rc) return rc;
    return adam_step_entry(fn, grad_bf16, n, master, exp_avg, exp_avg_sq, w8_out, scale_w, amax_w, loss_scale,
                           growth_tracker, found_inf, grad_nonfinite, true, beta_pows, lr, beta1, beta2, eps, backoff,
                           growth_factor, growth_interval, stream, w8_in, flags, &fb);
}

int fp8mp_selftest_timeout(void *stream) {
    clear_error();
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    return launch_timeout_selftest(static_cast<cudaStream_t>(stream));
}

int fp8mp_selftest_barrier_timeout(void *stream) {
    clear_error();
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    return launch_barrier_selftest(static_cast<cudaStream_t>(stream));
}

int fp8mp_check(void *stream) {
    clear_error();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "stream synchronize failed: %s", cudaGetErrorString(e));
    unsigned int flag = 0, mflag = 0, cflag = 0;
    int rc = read_and_clear_timeout_flag(&flag);
    if (rc) return rc;
    rc = read_and_clear_master_timeout_flag(&mflag);
    if (rc) return rc;
    rc = read_and_clear_cast_timeout_flag(&cflag);
    if (rc) return rc;
    if (flag) return fail(FP8MP_ERR_TIMEOUT, "a GEMM kernel's bounded wait expired; its output is undefined");
    if (cflag)
        return fail(FP8MP_ERR_TIMEOUT, "the bias-gradient cast's bounded wait expired; its outputs are undefined");
    if (mflag)
        return fail(FP8MP_ERR_TIMEOUT, "the master step's bounded grid barrier expired; the step's results are "
                                       "undefined");
    return FP8MP_OK;
}

}  // extern "C"
