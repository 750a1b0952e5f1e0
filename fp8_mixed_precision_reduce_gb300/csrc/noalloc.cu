// noalloc.cu -- fp8_quantize_dbias_noalloc: the fused gradient cast + bias
// gradient for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a host
// framework whose memory pool owns the device (a foreign allocation would
// fail or fragment it), plugin or extension code that is only handed input
// and output pointers, and latency-critical paths where the implicit device
// synchronisation of cudaMalloc / cudaFree is not acceptable. For them this
// entry point keeps the per-block partial column sums in a fixed scratch
// array compiled into the library instead of a caller-provided workspace.
//
// The scratch is the file-scope array below: 2^20 floats (4 MiB), held by
// every GPU that loads the library until the process exits. It holds the
// per-tile column sums and, after them, the column strips' arrival counters.
// The loader zero-fills it, and every call leaves what it used zero again,
// so the counters start at zero on every call. On the host its name is only
// a host-side stand-in, so the device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) on the first call on
// that device, and passed to the kernel. That cached address is not
// refreshed after cudaDeviceReset (the header says so).
#include <mutex>

#include "fp8mp_internal.cuh"

namespace fp8mp {
namespace {

static __device__ __align__(256) float g_dbias_scratch[FP8MP_NOALLOC_DBIAS_SCRATCH_FLOATS];

std::mutex g_scratch_mutex;
float *g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
int scratch_address(int device, float **out) {
    if (device < 0 || device >= 64) return fail(FP8MP_ERR_DEVICE, "device index %d out of range", device);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[device] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_dbias_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(FP8MP_ERR_LAUNCH, "cudaGetSymbolAddress of the scratch array failed: %s",
                        cudaGetErrorString(e));
        g_scratch_ptr[device] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[device];
    return FP8MP_OK;
}

}  // namespace
}  // namespace fp8mp

using namespace fp8mp;

extern "C" int fp8_quantize_dbias_noalloc(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t fmt,
                                          const float *scale, uint8_t *out, uint8_t *out_t, float *amax, void *dbias,
                                          int32_t dbias_dtype, void *stream) {
    const char *fn = "fp8_quantize_dbias_noalloc";
    clear_error();
    if (rows < 0 || cols < 0) return fail(FP8MP_ERR_INVALID, "%s: negative size", fn);
    // bound the shape before the size product can overflow (the workspace
    // size is -1 for a tensor beyond 2^40 elements)
    const int64_t need = fp8_quantize_dbias_workspace_bytes(rows, cols);
    const int64_t have = static_cast<int64_t>(FP8MP_NOALLOC_DBIAS_SCRATCH_FLOATS) * static_cast<int64_t>(sizeof(float));
    if (need < 0 || need > have)
        return fail(FP8MP_ERR_INVALID,
                    "%s: %lld x %lld needs %lld scratch bytes (ceil(rows/128) * cols floats and ceil(cols/128) "
                    "counters) but the fixed scratch array holds %lld; use fp8_quantize_dbias with a workspace",
                    fn, (long long)rows, (long long)cols, (long long)need, (long long)have);
    float *ws = nullptr;
    if (rows > 0 && cols > 0) {
        DeviceInfo dev;
        const int rc = current_device(&dev);
        if (rc) return rc;
        const int rs = scratch_address(dev.device, &ws);
        if (rs) return rs;
    }
    // The array is zero on entry (zero-filled at load, and every call leaves
    // what it used zero), as the workspace contract asks; the validated entry
    // point does the rest.
    return fp8_quantize_dbias(x, x_dtype, rows, cols, fmt, scale, out, out_t, amax, dbias, dbias_dtype, ws,
                              ws != nullptr ? have : 0, stream);
}
