// scale_update.cu -- the DelayedScaling bookkeeping of one training step for a
// batch of per-tensor metas, one thread block per tensor.
//
// Pages: "Transformer Engine으로 FP8 사용하기" (coniverse.tistory.com),
// "Scaling factor 선택 전략" (the factor of delayed scaling comes from a record
// of amaxes of earlier iterations) and "FP8 사용방안(recipe)" (DelayedScaling
// with amax_history_len and amax_compute_algo); "Как работает FP8
// quantization на H100 (Transformer Engine)?" (aivaro.ru), section 3 (the
// factor relates the amax to the format's largest value) and section 10
// (the HYBRID recipe with a 1024-long history).
//
// Arithmetic is plain IEEE fp32 with explicit round-to-nearest intrinsics:
// one division fmt_max / a, one multiply by the exact power of two
// 2^-margin, one division 1 / scale.
#include <cstring>

#include "fp8mp_internal.cuh"

namespace fp8mp {
namespace {

constexpr int kMetasPerLaunch = 32;
constexpr int kThreads = 256;

struct MetaArgs {
    float *hist;
    float *scale;
    float *scale_inv;
    float *cur_amax;
    float *prev_scale_inv;  // receives scale_inv as it was before the update, or NULL
    int32_t len;
    int32_t fmt;
};

struct MetaBatch {
    MetaArgs m[kMetasPerLaunch];
    int32_t algo;
    int32_t margin;
};

__global__ void __launch_bounds__(kThreads) scale_update_kernel(const __grid_constant__ MetaBatch b) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ float old_hist[];
    const MetaArgs &m = b.m[blockIdx.x];
    const int L = m.len;
    const float cur = *m.cur_amax;
    // the old scale (and scale_inv), loaded with the rest so the final step waits on nothing
    const float old_scale = threadIdx.x == 0 ? *m.scale : 0.0f;
    const float old_sinv = (threadIdx.x == 0 && m.prev_scale_inv != nullptr) ? *m.scale_inv : 0.0f;
    for (int j = threadIdx.x; j < L; j += blockDim.x) old_hist[j] = m.hist[j];
    __syncthreads();
    // roll by one, newest first, and take the max of the new window
    float mx = 0.0f;
    for (int j = threadIdx.x; j < L; j += blockDim.x) {
        const float h = (j == 0) ? cur : old_hist[j - 1];
        m.hist[j] = h;
        mx = max_ignore_nan(mx, h);
    }
    __shared__ float red[kThreads / 32];
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float all = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w) all = fmaxf(all, red[w]);
        const float a = (b.algo == FP8MP_AMAX_MAX) ? all : cur;
        const float sc = scale_from_amax(a, old_scale, m.fmt, b.margin);
        if (m.prev_scale_inv != nullptr) *m.prev_scale_inv = old_sinv;
        *m.scale = sc;
        *m.scale_inv = __fdiv_rn(1.0f, sc);
        *m.cur_amax = 0.0f;
    }
}

}  // namespace

int launch_scale_update(const fp8mp_meta *metas, int32_t n, int32_t algo, int32_t margin, cudaStream_t s,
                        float *prev_scale_inv) {
    for (int32_t first = 0; first < n; first += kMetasPerLaunch) {
        const int32_t cnt = (n - first < kMetasPerLaunch) ? (n - first) : kMetasPerLaunch;
        MetaBatch b;
        std::memset(&b, 0, sizeof b);
        int32_t max_len = 1;
        for (int32_t i = 0; i < cnt; ++i) {
            const fp8mp_meta &src = metas[first + i];
            b.m[i] = MetaArgs{src.amax_history, src.scale, src.scale_inv, src.cur_amax,
                              prev_scale_inv != nullptr ? prev_scale_inv + first + i : nullptr, src.history_len,
                              src.fmt};
            if (src.history_len > max_len) max_len = src.history_len;
        }
        b.algo = algo;
        b.margin = margin;
        // at most FP8MP_MAX_HISTORY floats = 32 KB, inside the default 48 KB
        const size_t smem = static_cast<size_t>(max_len) * sizeof(float);
        launch_kernel(scale_update_kernel, dim3(static_cast<unsigned>(cnt)), dim3(kThreads), smem, s, b);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(FP8MP_ERR_LAUNCH, "delayed_scaling_update: launch failed: %s", cudaGetErrorString(e));
    }
    return FP8MP_OK;
}

}  // namespace fp8mp
