// master_step.cu -- one mixed-precision optimizer step over a flat parameter
// buffer: overflow scan, loss unscale, FP32 master SGD-momentum update, E4M3
// re-cast of the weights and their amax, and the dynamic loss-scale update.
//
// Pages: "LLM) Mixed-Precision 개념 및 학습 방법 알아보기" (data-newbie.tistory.com),
// "FP32 Master Copy of Weights", "Mixed-Precision Training Iteration" (steps
// 5 and 7: multiply the weight gradients by 1/S, update the FP32 master) and
// the dynamic loss-scaling procedure (an Inf/NaN gradient lowers S and skips
// the update; a run of clean steps raises S); "Как работает FP8 quantization
// на H100 (Transformer Engine)?" (aivaro.ru) section 7 (FP32 master weights
// with FP8 forward/backward copies).
//
// Three launches on the caller's stream, no host round trip:
//   1. grad_scan_kernel: reads the bf16 gradients once (2 B/param) and sets
//      found_inf when any exponent field is all ones;
//   2. master_update_kernel: every block first reads found_inf and leaves if
//      it is set; otherwise one pass reads g, v, w (10 B/param) and writes
//      v, w, w8 (9 B/param), fusing the unscale, the momentum and master
//      updates, the E4M3 cast under the weight scale and the weight amax;
//   3. loss_scale_kernel: one thread updates S and the growth counter after
//      every block of pass 2 has read S.
#include "fp8mp_internal.cuh"

namespace fp8mp {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool has_nonfinite_bf16x2(uint32_t w) {
    const uint32_t t = (w & 0x7F807F80u) ^ 0x7F807F80u;  // a zero half <=> exponent all ones
    return (t & 0xFFFFu) == 0u || (t >> 16) == 0u;
}

__global__ void __launch_bounds__(kThreads)
grad_scan_kernel(const uint16_t *__restrict__ g, int64_t n, int32_t *__restrict__ found_inf) {
    pdl_wait();
    pdl_launch_dependents();
    bool bad = false;
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 d = __ldcs(g4 + i);
        bad |= has_nonfinite_bf16x2(d.x) | has_nonfinite_bf16x2(d.y) | has_nonfinite_bf16x2(d.z) |
               has_nonfinite_bf16x2(d.w);
    }
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t i = (nvec << 3) + threadIdx.x; i < n; i += blockDim.x) bad |= (g[i] & 0x7F80u) == 0x7F80u;
    if (__syncthreads_or(bad) && threadIdx.x == 0) *found_inf = 1;
}

struct Elem {
    float v, w;
};

__device__ __forceinline__ Elem update_one(float g, float v, float w, float inv_s, float mu, float neg_lr) {
    const float u = __fmul_rn(g, inv_s);
    const float vn = __fmaf_rn(mu, v, u);
    const float wn = __fmaf_rn(neg_lr, vn, w);
    return Elem{vn, wn};
}

__global__ void __launch_bounds__(kThreads)
master_update_kernel(const uint16_t *__restrict__ g, int64_t n, float *__restrict__ w, float *__restrict__ v,
                     uint8_t *__restrict__ w8, const float *__restrict__ scale_w, float *__restrict__ amax_w,
                     const float *__restrict__ loss_scale, const int32_t *__restrict__ found_inf, float lr,
                     float mu) {
    pdl_wait();
    pdl_launch_dependents();
    if (*reinterpret_cast<const volatile int32_t *>(found_inf) != 0) return;  // skipped step
    const float inv_s = __fdiv_rn(1.0f, *loss_scale);
    const float sw = *scale_w;
    const float neg_lr = -lr;
    float am = 0.0f;
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 gd = __ldcs(reinterpret_cast<const uint4 *>(g) + i);
        float4 *v4 = reinterpret_cast<float4 *>(v) + 2 * i;
        float4 *w4 = reinterpret_cast<float4 *>(w) + 2 * i;
        const float4 va = __ldcs(v4), vb = __ldcs(v4 + 1);
        const float4 wa = __ldcs(w4), wb = __ldcs(w4 + 1);
        const uint32_t gw[4] = {gd.x, gd.y, gd.z, gd.w};
        float gf[8], vf[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w},
                     wf[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            gf[2 * j] = __uint_as_float(gw[j] << 16);
            gf[2 * j + 1] = __uint_as_float(gw[j] & 0xFFFF0000u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const Elem e = update_one(gf[j], vf[j], wf[j], inv_s, mu, neg_lr);
            vf[j] = e.v;
            wf[j] = e.w;
            am = max_ignore_nan(am, fabsf(e.w));
        }
        __stcs(v4, make_float4(vf[0], vf[1], vf[2], vf[3]));
        __stcs(v4 + 1, make_float4(vf[4], vf[5], vf[6], vf[7]));
        __stcs(w4, make_float4(wf[0], wf[1], wf[2], wf[3]));
        __stcs(w4 + 1, make_float4(wf[4], wf[5], wf[6], wf[7]));
        const uint32_t q0 = cvt_quad<FP8MP_E4M3>(__fmul_rn(wf[0], sw), __fmul_rn(wf[1], sw), __fmul_rn(wf[2], sw),
                                                 __fmul_rn(wf[3], sw));
        const uint32_t q1 = cvt_quad<FP8MP_E4M3>(__fmul_rn(wf[4], sw), __fmul_rn(wf[5], sw), __fmul_rn(wf[6], sw),
                                                 __fmul_rn(wf[7], sw));
        reinterpret_cast<uint2 *>(w8)[i] = make_uint2(q0, q1);
    }
    if (blockIdx.x == gridDim.x - 1) {
        for (int64_t i = (nvec << 3) + threadIdx.x; i < n; i += blockDim.x) {
            const Elem e = update_one(bf16_bits_to_f32(g[i]), v[i], w[i], inv_s, mu, neg_lr);
            v[i] = e.v;
            w[i] = e.w;
            w8[i] = static_cast<uint8_t>(cvt_pair<FP8MP_E4M3>(__fmul_rn(e.w, sw), 0.0f) & 0xFFu);
            am = max_ignore_nan(am, fabsf(e.w));
        }
    }
    block_amax_atomic(am, amax_w);
}

__global__ void loss_scale_kernel(float *__restrict__ S, int32_t *__restrict__ growth,
                                  const int32_t *__restrict__ found_inf, float backoff, float growth_factor,
                                  int32_t interval) {
    pdl_wait();
    pdl_launch_dependents();
    if (*found_inf != 0) {
        *S = __fmul_rn(*S, backoff);
        *growth = 0;
    } else {
        int32_t gr = *growth + 1;
        if (gr >= interval) {
            *S = __fmul_rn(*S, growth_factor);
            gr = 0;
        }
        *growth = gr;
    }
}

// Adam variant of pass 2 (same skip rule). Per element, each operation one
// correctly rounded fp32 operation in this order:
//   u = g * fl32(1/S); m = fmaf(b1, m, (1-b1) * u); v = fmaf(b2, v, (1-b2) * (u*u))
//   w = fmaf(-lr, (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), w)
// with b^t = fl32(b^(t-1) * b) from the running powers in beta_pows.
__global__ void __launch_bounds__(kThreads)
adam_update_kernel(const uint16_t *__restrict__ g, int64_t n, float *__restrict__ w, float *__restrict__ m,
                   float *__restrict__ v, uint8_t *__restrict__ w8, const float *__restrict__ scale_w,
                   float *__restrict__ amax_w, const float *__restrict__ loss_scale,
                   const int32_t *__restrict__ found_inf, const float *__restrict__ beta_pows, float lr, float b1,
                   float b2, float eps) {
    pdl_wait();
    pdl_launch_dependents();
    if (*reinterpret_cast<const volatile int32_t *>(found_inf) != 0) return;  // skipped step
    const float inv_s = __fdiv_rn(1.0f, *loss_scale);
    const float sw = *scale_w;
    const float c1 = __fsub_rn(1.0f, b1), c2 = __fsub_rn(1.0f, b2);
    const float bc1 = __fsub_rn(1.0f, __fmul_rn(beta_pows[0], b1));
    const float bc2 = __fsub_rn(1.0f, __fmul_rn(beta_pows[1], b2));
    const float neg_lr = -lr;
    float am = 0.0f;
    auto one = [&](float gf, float &mi, float &vi, float &wi) {
        const float u = __fmul_rn(gf, inv_s);
        mi = __fmaf_rn(b1, mi, __fmul_rn(c1, u));
        vi = __fmaf_rn(b2, vi, __fmul_rn(c2, __fmul_rn(u, u)));
        const float mh = __fdiv_rn(mi, bc1);
        const float vh = __fdiv_rn(vi, bc2);
        const float den = __fadd_rn(__fsqrt_rn(vh), eps);
        wi = __fmaf_rn(neg_lr, __fdiv_rn(mh, den), wi);
        am = max_ignore_nan(am, fabsf(wi));
    };
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 gd = __ldcs(reinterpret_cast<const uint4 *>(g) + i);
        float4 *m4 = reinterpret_cast<float4 *>(m) + 2 * i;
        float4 *v4 = reinterpret_cast<float4 *>(v) + 2 * i;
        float4 *w4 = reinterpret_cast<float4 *>(w) + 2 * i;
        const float4 ma = __ldcs(m4), mb = __ldcs(m4 + 1);
        const float4 va = __ldcs(v4), vb = __ldcs(v4 + 1);
        const float4 wa = __ldcs(w4), wb = __ldcs(w4 + 1);
        const uint32_t gw[4] = {gd.x, gd.y, gd.z, gd.w};
        float mf[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        float vf[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        float wf[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float gf = (j & 1) ? __uint_as_float(gw[j >> 1] & 0xFFFF0000u) : __uint_as_float(gw[j >> 1] << 16);
            one(gf, mf[j], vf[j], wf[j]);
        }
        __stcs(m4, make_float4(mf[0], mf[1], mf[2], mf[3]));
        __stcs(m4 + 1, make_float4(mf[4], mf[5], mf[6], mf[7]));
        __stcs(v4, make_float4(vf[0], vf[1], vf[2], vf[3]));
        __stcs(v4 + 1, make_float4(vf[4], vf[5], vf[6], vf[7]));
        __stcs(w4, make_float4(wf[0], wf[1], wf[2], wf[3]));
        __stcs(w4 + 1, make_float4(wf[4], wf[5], wf[6], wf[7]));
        const uint32_t q0 = cvt_quad<FP8MP_E4M3>(__fmul_rn(wf[0], sw), __fmul_rn(wf[1], sw), __fmul_rn(wf[2], sw),
                                                 __fmul_rn(wf[3], sw));
        const uint32_t q1 = cvt_quad<FP8MP_E4M3>(__fmul_rn(wf[4], sw), __fmul_rn(wf[5], sw), __fmul_rn(wf[6], sw),
                                                 __fmul_rn(wf[7], sw));
        reinterpret_cast<uint2 *>(w8)[i] = make_uint2(q0, q1);
    }
    if (blockIdx.x == gridDim.x - 1) {
        for (int64_t i = (nvec << 3) + threadIdx.x; i < n; i += blockDim.x) {
            float mi = m[i], vi = v[i], wi = w[i];
            one(bf16_bits_to_f32(g[i]), mi, vi, wi);
            m[i] = mi;
            v[i] = vi;
            w[i] = wi;
            w8[i] = static_cast<uint8_t>(cvt_pair<FP8MP_E4M3>(__fmul_rn(wi, sw), 0.0f) & 0xFFu);
        }
    }
    block_amax_atomic(am, amax_w);
}

// Loss-scale update plus, on a clean step, beta_pows = (b1^t, b2^t).
__global__ void adam_bookkeeping_kernel(float *__restrict__ S, int32_t *__restrict__ growth,
                                        const int32_t *__restrict__ found_inf, float *__restrict__ beta_pows,
                                        float b1, float b2, float backoff, float growth_factor, int32_t interval) {
    pdl_wait();
    pdl_launch_dependents();
    if (*found_inf != 0) {
        *S = __fmul_rn(*S, backoff);
        *growth = 0;
    } else {
        beta_pows[0] = __fmul_rn(beta_pows[0], b1);
        beta_pows[1] = __fmul_rn(beta_pows[1], b2);
        int32_t gr = *growth + 1;
        if (gr >= interval) {
            *S = __fmul_rn(*S, growth_factor);
            gr = 0;
        }
        *growth = gr;
    }
}

}  // namespace

int launch_adam_step(const uint16_t *g, int64_t n, float *w, float *m, float *v, uint8_t *w8, const float *scale_w,
                     float *amax_w, float *loss_scale, int32_t *growth, int32_t *found_inf, float *beta_pows,
                     float lr, float b1, float b2, float eps, float backoff, float growth_factor,
                     int32_t growth_interval, cudaStream_t s, const DeviceInfo &dev) {
    cudaError_t e = cudaMemsetAsync(found_inf, 0, sizeof(int32_t), s);
    if (e != cudaSuccess)
        return fail(FP8MP_ERR_LAUNCH, "mp_master_step_adam: memset failed: %s", cudaGetErrorString(e));
    const int64_t nvec = n >> 3;
    int64_t blocks = (nvec + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (n > 0) {
        launch_kernel(grad_scan_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, g, n, found_inf);
        launch_kernel(adam_update_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, g, n, w, m, v,
                      w8, scale_w, amax_w, loss_scale, found_inf, beta_pows, lr, b1, b2, eps);
    }
    launch_kernel(adam_bookkeeping_kernel, dim3(1), dim3(1), 0, s, loss_scale, growth, found_inf, beta_pows, b1, b2,
                  backoff, growth_factor, growth_interval);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FP8MP_ERR_LAUNCH, "mp_master_step_adam: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

int launch_master_step(const uint16_t *g, int64_t n, float *w, float *v, uint8_t *w8, const float *scale_w,
                       float *amax_w, float *loss_scale, int32_t *growth, int32_t *found_inf, float lr, float mu,
                       float backoff, float growth_factor, int32_t growth_interval, cudaStream_t s,
                       const DeviceInfo &dev) {
    cudaError_t e = cudaMemsetAsync(found_inf, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "mp_master_step: memset failed: %s", cudaGetErrorString(e));
    const int64_t nvec = n >> 3;
    int64_t blocks = (nvec + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (n > 0) {
        launch_kernel(grad_scan_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, g, n, found_inf);
        launch_kernel(master_update_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, g, n, w, v, w8,
                      scale_w, amax_w, loss_scale, found_inf, lr, mu);
    }
    launch_kernel(loss_scale_kernel, dim3(1), dim3(1), 0, s, loss_scale, growth, found_inf, backoff, growth_factor,
                  growth_interval);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "mp_master_step: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

}  // namespace fp8mp
