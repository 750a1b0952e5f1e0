// master_step.cu -- one mixed-precision optimizer step over a flat parameter
// buffer: overflow scan, loss unscale, FP32 master update (SGD with momentum
// or Adam), E4M3 re-cast of the weights and their amax, and the dynamic
// loss-scale update.
//
// Pages: "LLM) Mixed-Precision 개념 및 학습 방법 알아보기" (data-newbie.tistory.com),
// "FP32 Master Copy of Weights", "Mixed-Precision Training Iteration" (steps
// 5 and 7: multiply the weight gradients by 1/S, update the FP32 master) and
// the dynamic loss-scaling procedure (an Inf/NaN gradient lowers S and skips
// the update; a run of clean steps raises S); "Как работает FP8 quantization
// на H100 (Transformer Engine)?" (aivaro.ru) section 7 (FP32 master weights
// with FP8 forward/backward copies); "Các kiểu dữ liệu FP8 gốc của PyTorch
// ..." (hotroai.com), the float8_experimental training loop (torch.optim.Adam).
//
// The step is three passes: scan the bf16 gradients for Inf/NaN (2 B/param);
// unless one was found, one fused pass per element (unscale, optimizer
// update, E4M3 cast under the weight scale, weight amax); then S and the
// growth counter (and Adam's beta powers) change by one thread, after every
// element has read S. Two ways to run it, same arithmetic (the per-element
// operations live once, in SgdOpt / AdamOpt):
//   fused (default): one cooperative launch. Each block scans its slice,
//     the blocks meet at a bounded grid barrier, each block updates its
//     slice (re-reading the gradients it scanned, kept in L2 by an
//     evict-last hint), and the last block to finish does the bookkeeping;
//   three launches (FP8MP_FUSED_MASTER=0): grad_scan_kernel, the update
//     kernel (every block leaves at once when found_inf is set), and a
//     one-thread bookkeeping kernel.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "fp8mp_internal.cuh"

namespace fp8mp {

__device__ unsigned int g_master_timeout_flag = 0;

namespace {

constexpr int kThreads = 256;
// Early (FP8MP_OVERLAP_PREVIOUS) grid: one block per SM, of as many warps
// (at most this many threads) as the registers a GEMM CTA leaves free allow.
constexpr int kEarlyMaxThreads = 768;
constexpr long long kBarrierLimitCycles = 4000000000ll;  // about 2 s at the SM clock

__device__ __forceinline__ bool has_nonfinite_bf16x2(uint32_t w) {
    const uint32_t t = (w & 0x7F807F80u) ^ 0x7F807F80u;  // a zero half <=> exponent all ones
    return (t & 0xFFFFu) == 0u || (t >> 16) == 0u;
}

// L2 policy: keep the lines (the fused step re-reads the gradients).
__device__ __forceinline__ uint64_t evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_with_policy(const uint4 *ptr, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr), "l"(pol)
                 : "memory");
    return r;
}

// Scans this thread's grid-stride share of the gradients (16-byte vectors,
// the n % 8 tail by the last block).
template <bool KEEP_IN_L2>
__device__ __forceinline__ bool scan_share(const uint16_t *__restrict__ g, int64_t n) {
    bool bad = false;
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
    uint64_t pol = 0;
    if constexpr (KEEP_IN_L2) pol = evict_last_policy();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        uint4 d;
        if constexpr (KEEP_IN_L2)
            d = ld_with_policy(g4 + i, pol);
        else
            d = __ldcs(g4 + i);
        bad |= has_nonfinite_bf16x2(d.x) | has_nonfinite_bf16x2(d.y) | has_nonfinite_bf16x2(d.z) |
               has_nonfinite_bf16x2(d.w);
    }
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t i = (nvec << 3) + threadIdx.x; i < n; i += blockDim.x) bad |= (g[i] & 0x7F80u) == 0x7F80u;
    return bad;
}

// Thread 0 of a block: counts the block's arrival (adds 2 to *word: bit 0 is
// left to the overflow flag) and waits, bounded by about 2 s, until the
// arrivals reach `expected`. Returns the word's last value, or -1 when the
// wait ran out (then the device timeout flag is set).
__device__ int32_t barrier_arrive_and_wait(int32_t *word, int32_t expected) {
    volatile int32_t *vw = word;
    __threadfence();
    atomicAdd(word, 2);
    const long long t0 = clock64();
    int32_t f;
    while (((f = *vw) >> 1) < expected) {
        if (clock64() - t0 > kBarrierLimitCycles) {
            atomicOr(&g_master_timeout_flag, 1u);
            return -1;
        }
        __nanosleep(128);
    }
    __threadfence();
    return f;
}

// ---------------------------------------------------------- optimizers

struct SgdArgs {
    float *w, *v;
    float lr, mu;
};

// SGD with momentum: u = g * fl32(1/S); v = fmaf(mu, v, u); w = fmaf(-lr, v, w).
struct SgdOpt {
    float *w, *v;
    float inv_s, mu, neg_lr;
    __device__ __forceinline__ float one(float g, float &vi, float wi) const {
        const float u = __fmul_rn(g, inv_s);
        vi = __fmaf_rn(mu, vi, u);
        return __fmaf_rn(neg_lr, vi, wi);
    }
    // 8 parameters starting at 8*i; returns the 8 new master weights in wf.
    __device__ __forceinline__ void vec8(int64_t i, const float gf[8], float wf[8]) const {
        float4 *v4 = reinterpret_cast<float4 *>(v) + 2 * i;
        float4 *w4 = reinterpret_cast<float4 *>(w) + 2 * i;
        const float4 va = __ldcs(v4), vb = __ldcs(v4 + 1);
        const float4 wa = __ldcs(w4), wb = __ldcs(w4 + 1);
        float vf[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        const float wo[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) wf[j] = one(gf[j], vf[j], wo[j]);
        __stcs(v4, make_float4(vf[0], vf[1], vf[2], vf[3]));
        __stcs(v4 + 1, make_float4(vf[4], vf[5], vf[6], vf[7]));
        __stcs(w4, make_float4(wf[0], wf[1], wf[2], wf[3]));
        __stcs(w4 + 1, make_float4(wf[4], wf[5], wf[6], wf[7]));
    }
    __device__ __forceinline__ float scalar(int64_t i, float g) const {
        float vi = v[i];
        const float wn = one(g, vi, w[i]);
        v[i] = vi;
        w[i] = wn;
        return wn;
    }
};

struct AdamArgs {
    float *w, *m, *v;
    float *beta_pows;
    float lr, b1, b2, eps;
};

// Adam: u = g * fl32(1/S); m = fmaf(b1, m, (1-b1) * u); v = fmaf(b2, v, (1-b2) * (u*u));
// w = fmaf(-lr, (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), w), each operation one correctly
// rounded fp32 operation in this order, with b^t = fl32(b^(t-1) * b) from the running powers.
struct AdamOpt {
    float *w, *m, *v;
    float inv_s, b1, b2, c1, c2, bc1, bc2, eps, neg_lr;
    __device__ __forceinline__ float one(float g, float &mi, float &vi, float wi) const {
        const float u = __fmul_rn(g, inv_s);
        mi = __fmaf_rn(b1, mi, __fmul_rn(c1, u));
        vi = __fmaf_rn(b2, vi, __fmul_rn(c2, __fmul_rn(u, u)));
        const float mh = __fdiv_rn(mi, bc1);
        const float vh = __fdiv_rn(vi, bc2);
        const float den = __fadd_rn(__fsqrt_rn(vh), eps);
        return __fmaf_rn(neg_lr, __fdiv_rn(mh, den), wi);
    }
    __device__ __forceinline__ void vec8(int64_t i, const float gf[8], float wf[8]) const {
        float4 *m4 = reinterpret_cast<float4 *>(m) + 2 * i;
        float4 *v4 = reinterpret_cast<float4 *>(v) + 2 * i;
        float4 *w4 = reinterpret_cast<float4 *>(w) + 2 * i;
        const float4 ma = __ldcs(m4), mb = __ldcs(m4 + 1);
        const float4 va = __ldcs(v4), vb = __ldcs(v4 + 1);
        const float4 wa = __ldcs(w4), wb = __ldcs(w4 + 1);
        float mf[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        float vf[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        const float wo[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) wf[j] = one(gf[j], mf[j], vf[j], wo[j]);
        __stcs(m4, make_float4(mf[0], mf[1], mf[2], mf[3]));
        __stcs(m4 + 1, make_float4(mf[4], mf[5], mf[6], mf[7]));
        __stcs(v4, make_float4(vf[0], vf[1], vf[2], vf[3]));
        __stcs(v4 + 1, make_float4(vf[4], vf[5], vf[6], vf[7]));
        __stcs(w4, make_float4(wf[0], wf[1], wf[2], wf[3]));
        __stcs(w4 + 1, make_float4(wf[4], wf[5], wf[6], wf[7]));
    }
    __device__ __forceinline__ float scalar(int64_t i, float g) const {
        float mi = m[i], vi = v[i];
        const float wn = one(g, mi, vi, w[i]);
        m[i] = mi;
        v[i] = vi;
        w[i] = wn;
        return wn;
    }
};

__device__ __forceinline__ SgdOpt make_opt(const SgdArgs &a, float inv_s) {
    SgdOpt o;
    o.w = a.w;
    o.v = a.v;
    o.inv_s = inv_s;
    o.mu = a.mu;
    o.neg_lr = -a.lr;
    return o;
}
__device__ __forceinline__ AdamOpt make_opt(const AdamArgs &a, float inv_s) {
    AdamOpt o;
    o.w = a.w;
    o.m = a.m;
    o.v = a.v;
    o.inv_s = inv_s;
    o.b1 = a.b1;
    o.b2 = a.b2;
    o.c1 = __fsub_rn(1.0f, a.b1);
    o.c2 = __fsub_rn(1.0f, a.b2);
    o.bc1 = __fsub_rn(1.0f, __fmul_rn(a.beta_pows[0], a.b1));
    o.bc2 = __fsub_rn(1.0f, __fmul_rn(a.beta_pows[1], a.b2));
    o.eps = a.eps;
    o.neg_lr = -a.lr;
    return o;
}

// This thread's grid-stride share of an n-byte copy (16-byte vectors, the
// n % 16 tail by the last block).
__device__ __forceinline__ void copy_share(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int64_t n) {
    const int64_t nvec = n >> 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride)
        reinterpret_cast<uint4 *>(dst)[i] = __ldcs(reinterpret_cast<const uint4 *>(src) + i);
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t i = (nvec << 4) + threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

// The update pass over this thread's grid-stride share: the optimizer, the
// E4M3 re-cast of the new master weights under *scale_w, their max |w|.
// CG: the gradients are read through L2 only (ld.global.cg): a step that
// starts before their producer has finished must not see lines its SM's L1
// kept from an earlier kernel.
template <class Opt, bool CG = false>
__device__ __forceinline__ float update_share(const Opt &opt, const uint16_t *__restrict__ g, int64_t n,
                                              uint8_t *__restrict__ w8, float sw) {
    float am = 0.0f;
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 gd = CG ? __ldcg(reinterpret_cast<const uint4 *>(g) + i) : __ldcs(reinterpret_cast<const uint4 *>(g) + i);
        const uint32_t gw[4] = {gd.x, gd.y, gd.z, gd.w};
        float gf[8], wf[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            gf[2 * j] = __uint_as_float(gw[j] << 16);
            gf[2 * j + 1] = __uint_as_float(gw[j] & 0xFFFF0000u);
        }
        opt.vec8(i, gf, wf);
#pragma unroll
        for (int j = 0; j < 8; ++j) am = max_ignore_nan(am, fabsf(wf[j]));
        const uint32_t q0 = cvt_quad<FP8MP_E4M3>(__fmul_rn(wf[0], sw), __fmul_rn(wf[1], sw), __fmul_rn(wf[2], sw),
                                                 __fmul_rn(wf[3], sw));
        const uint32_t q1 = cvt_quad<FP8MP_E4M3>(__fmul_rn(wf[4], sw), __fmul_rn(wf[5], sw), __fmul_rn(wf[6], sw),
                                                 __fmul_rn(wf[7], sw));
        reinterpret_cast<uint2 *>(w8)[i] = make_uint2(q0, q1);
    }
    if (blockIdx.x == gridDim.x - 1) {
        for (int64_t i = (nvec << 3) + threadIdx.x; i < n; i += blockDim.x) {
            const float wn = opt.scalar(i, bf16_bits_to_f32(CG ? __ldcg(g + i) : g[i]));
            w8[i] = static_cast<uint8_t>(cvt_pair<FP8MP_E4M3>(__fmul_rn(wn, sw), 0.0f) & 0xFFu);
            am = max_ignore_nan(am, fabsf(wn));
        }
    }
    return am;
}

// S and the growth counter after a step with overflow flag `found`.
__device__ __forceinline__ void loss_scale_update(float *S, int32_t *growth, int found, float backoff,
                                                  float growth_factor, int32_t interval) {
    if (found) {
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

struct NoExtra {
    __device__ void clean_step() const {}
};
// Adam's beta powers advance on clean steps only.
struct AdamExtra {
    float *beta_pows;
    float b1, b2;
    __device__ void clean_step() const {
        beta_pows[0] = __fmul_rn(beta_pows[0], b1);
        beta_pows[1] = __fmul_rn(beta_pows[1], b2);
    }
};

struct StepCommon {
    const uint16_t *g;
    int64_t n;
    uint8_t *w8;
    const uint8_t *w8_in;  // the current copy when w8 is another buffer, else NULL (in place)
    const float *scale_w;
    float *amax_w;
    float *loss_scale;
    int32_t *growth;
    int32_t *found_inf;
    float backoff, growth_factor;
    int32_t interval;
};

// ------------------------------------------------ three-launch version

__global__ void __launch_bounds__(kThreads)
grad_scan_kernel(const uint16_t *__restrict__ g, int64_t n, int32_t *__restrict__ found_inf) {
    pdl_wait();
    pdl_launch_dependents();
    const bool bad = scan_share<false>(g, n);
    if (__syncthreads_or(bad) && threadIdx.x == 0) *found_inf = 1;
}

template <class Opt, class Args>
__global__ void __launch_bounds__(kThreads) update_kernel(const StepCommon c, const Args a) {
    pdl_wait();
    pdl_launch_dependents();
    if (*reinterpret_cast<const volatile int32_t *>(c.found_inf) != 0) return;  // skipped step
    const Opt opt = make_opt(a, __fdiv_rn(1.0f, *c.loss_scale));
    const float am = update_share(opt, c.g, c.n, c.w8, *c.scale_w);
    block_amax_atomic(am, c.amax_w);
}

template <class Extra>
__global__ void bookkeeping_kernel(const StepCommon c, const Extra x) {
    pdl_wait();
    pdl_launch_dependents();
    const int found = *c.found_inf != 0;
    if (!found) x.clean_step();
    loss_scale_update(c.loss_scale, c.growth, found, c.backoff, c.growth_factor, c.interval);
}

// ---------------------------------------------------- fused version

// found_inf is 0 on entry (the launcher zeroes it on the stream first).
// While the kernel runs, bit 0 of found_inf is the overflow flag (atomicOr)
// and the bits above count block arrivals (atomicAdd of 2, which never
// carries into bit 0): gridDim.x arrivals close the scan, 2 * gridDim.x the
// step. The last block to arrive does the bookkeeping and leaves found_inf
// holding the flag alone (0 or 1). The launch is cooperative, so every
// block is resident and the barrier completes; its wait is still bounded
// (about 2 s), after which the block sets a device flag that fp8mp_check()
// reports and skips the update (the step's results are then undefined).
template <class Opt, class Args, class Extra>
__global__ void __launch_bounds__(kThreads) fused_step_kernel(const StepCommon c, const Args a, const Extra x) {
    __shared__ int s_skip;
    const bool bad = __syncthreads_or(scan_share<true>(c.g, c.n));
    if (threadIdx.x == 0) {
        if (bad) atomicOr(c.found_inf, 1);
        const int32_t f = barrier_arrive_and_wait(c.found_inf, static_cast<int32_t>(gridDim.x));
        s_skip = f < 0 ? 1 : (f & 1);  // a timed-out barrier skips the update
    }
    __syncthreads();
    float am = 0.0f;
    if (!s_skip) {
        const Opt opt = make_opt(a, __fdiv_rn(1.0f, *c.loss_scale));
        am = update_share(opt, c.g, c.n, c.w8, *c.scale_w);
    }
    block_amax_atomic(am, c.amax_w);  // a skipped block adds +0: no change
    if (threadIdx.x == 0) {
        __threadfence();
        const int32_t prev = atomicAdd(c.found_inf, 2);
        if ((prev >> 1) == 2 * static_cast<int32_t>(gridDim.x) - 1) {
            __threadfence();
            const int found = prev & 1;
            if (!found) x.clean_step();
            loss_scale_update(c.loss_scale, c.growth, found, c.backoff, c.growth_factor, c.interval);
            *c.found_inf = found;
        }
    }
}

// FP8MP_FUSED_MASTER=0 selects the three-launch version (read per call, so
// tests can run both).
// The step when the gradients' producer has already looked for Inf/NaN
// (*grad_nonfinite is 1 iff it found one, else 0, e.g. the wgrad GEMM
// epilogue's flag): no scan pass and no barrier, so a plain launch, and no
// memset before it. Each block reads bit 0 of the flag word and adds 2 to
// the word when it is done (the count never touches bit 0); the last block
// does the bookkeeping, writes found_inf and resets the word to 0 for the
// next producer.
//
// With c.w8_in the new E4M3 copy goes to another buffer than the current
// one, and a skipped step copies the current one there. EARLY
// (FP8MP_OVERLAP_PREVIOUS): the caller guarantees that the kernel still
// running before this one on the stream neither writes nor reads anything
// the step touches (for example the dgrad GEMM of the same backward pass,
// which reads the current E4M3 copy while the step writes the other one), so
// the blocks start without waiting for it; block 0 waits for it at its very
// end, so the grid completes after it. What the step reads from the kernels
// before that one (the wgrad GEMM's dW and flag, the scale update's scale)
// is complete: the previous kernel let this one start only after its own
// wait on them had returned. The early grid is one block per SM,
// sized to fit beside a CTA of the GEMM (whose shared memory leaves room for
// one more block): every block runs from the start, so the whole update
// overlaps the GEMM instead of the few blocks that find room first.
//
// One tensor's delayed-scaling update by a whole block, as
// scale_update_kernel computes it (roll the history one place, newest at
// index 0; the max of the new window, or the newest amax with the
// most-recent algorithm; the scale from it), without staging the history in
// shared memory, of which a block beside a GEMM CTA has almost none: the
// history moves one place towards its end in chunks of blockDim elements,
// the highest chunk first, every old value of a chunk read before any of the
// chunk is written (a block barrier between), so nothing is overwritten
// before it is read. Returns the new scale in thread 0.
__device__ float fold_meta_update(const FoldMeta &m, int algo, int margin, float *red) {
    const int L = m.len;
    const int T = static_cast<int>(blockDim.x);
    const float cur = __ldcg(m.cur_amax);
    float mx = 0.0f;
    for (int base = ((L - 1) / T) * T; base >= 0; base -= T) {
        const int j = base + static_cast<int>(threadIdx.x);
        float v = 0.0f;
        if (j < L) v = (j == 0) ? cur : __ldcg(m.hist + j - 1);
        __syncthreads();
        if (j < L) {
            m.hist[j] = v;
            mx = max_ignore_nan(mx, v);
        }
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    float sc = 0.0f;
    if (threadIdx.x == 0) {
        float all = 0.0f;
        for (int w = 0; w < T / 32; ++w) all = fmaxf(all, red[w]);
        const float a = (algo == FP8MP_AMAX_MAX) ? all : cur;
        sc = scale_from_amax(a, __ldcg(m.scale), m.fmt, margin);
    }
    return sc;
}

// WAIT (with EARLY; FP8MP_WAIT_DW_DONE): the gradients' producer is the
// kernel still running (a backward GEMM launch that signals completion, its
// dW tiles first): thread 0 of each block waits, bounded by about 2 s, for
// the word's completion bit before the flag is read, and the gradients are
// read through L2 only. A wait that runs out raises the device timeout flag
// and the block updates nothing.
//
// FOLD (with EARLY and WAIT; mp_master_step_prescanned_scaling_ex): the
// blocks also run the step's delayed-scaling update of fb's metas, block b
// the metas b, b + gridDim.x, ..., before they wait for the gradients: each
// history rolled and each new scale and zeroed amax written at once, the
// weight's scale followed by bit 31 of the word, which every block waits
// for too before it casts with that scale (and adds to the weight's amax,
// zeroed just before). The new scale_inv values, which the still running
// backward GEMMs read in their old form, are written only after the block's
// griddepcontrol.wait at its end. Every result is that of the update
// launched before the backward with the scale_inv snapshot.
template <class Opt, class Args, class Extra, bool EARLY, bool WAIT, bool FOLD>
__global__ void __launch_bounds__(EARLY ? kEarlyMaxThreads : kThreads, EARLY ? 1 : 0)
prescanned_step_kernel(const StepCommon c, const Args a, const Extra x, int32_t *grad_nonfinite,
                       const __grid_constant__ FoldBatch fb) {
    if constexpr (!EARLY) {
        pdl_wait();
        pdl_launch_dependents();
    }
    __shared__ int s_skip;
    __shared__ float s_sinv[kMaxFoldMetas];  // FOLD: the new scale_inv of the metas this block updated
    if constexpr (FOLD) {
        __shared__ float s_red[32];
#pragma unroll 1
        for (int k = 0; k < kMaxFoldMetas; ++k) {
            const int mi = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
            if (mi >= fb.n) break;
            const FoldMeta &m = fb.m[mi];
            const float sc = fold_meta_update(m, fb.algo, fb.margin, s_red);
            if (threadIdx.x == 0) {
                *m.scale = sc;
                *m.cur_amax = 0.0f;
                s_sinv[k] = __fdiv_rn(1.0f, sc);
                if (mi == fb.w_index) {
                    __threadfence();  // the scale and the zeroed amax before the bit
                    atomicOr(reinterpret_cast<unsigned int *>(grad_nonfinite), kMetaBit);
                }
            }
            __syncthreads();  // s_red is free for the next meta
        }
    }
    if (threadIdx.x == 0) {
        if constexpr (WAIT) {
            const long long t0 = clock64();
            uint32_t w;
            int skip = 1;
            for (;;) {
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(w) : "l"(grad_nonfinite) : "memory");
                if ((w & kDoneBit) && (!FOLD || fb.w_index < 0 || (w & kMetaBit))) {
                    skip = (w & 1u) != 0;
                    break;
                }
                if (clock64() - t0 > kBarrierLimitCycles) {
                    atomicOr(&g_master_timeout_flag, 1u);
                    break;
                }
                __nanosleep(256);
            }
            s_skip = skip;
        } else {
            s_skip = (*reinterpret_cast<volatile int32_t *>(grad_nonfinite) & 1) != 0;
        }
    }
    __syncthreads();
    float am = 0.0f;
    if (!s_skip) {
        const Opt opt = make_opt(a, __fdiv_rn(1.0f, *c.loss_scale));
        am = update_share<Opt, WAIT>(opt, c.g, c.n, c.w8, FOLD ? __ldcg(c.scale_w) : *c.scale_w);
    } else if (c.w8_in != nullptr && c.w8_in != c.w8) {
        copy_share(c.w8_in, c.w8, c.n);  // skipped: the next copy is the current one
    }
    block_amax_atomic(am, c.amax_w);
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(reinterpret_cast<unsigned int *>(grad_nonfinite), 1u << kArrivalShift);
        if (((prev >> kArrivalShift) & kArrivalMask) == gridDim.x - 1) {
            __threadfence();
            const int found = s_skip;
            if (!found) x.clean_step();
            loss_scale_update(c.loss_scale, c.growth, found, c.backoff, c.growth_factor, c.interval);
            *c.found_inf = found;
            *grad_nonfinite = 0;
        }
    }
    if constexpr (FOLD) {
        if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < fb.n) {
            pdl_wait();  // the backward launch, which reads the old scale_inv, is complete
            for (int k = 0; k < kMaxFoldMetas; ++k) {
                const int mi = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
                if (mi >= fb.n) break;
                *fb.m[mi].scale_inv = s_sinv[k];
            }
        }
    }
    if constexpr (EARLY) {  // the next kernel may start once this wait has returned (as for the casts)
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            pdl_wait();
            pdl_launch_dependents();
        }
    }
}

// Diagnostic of the barrier's failure path: one block arrives at a barrier
// that waits for two arrivals, so the bounded wait runs out after about 2 s,
// raises the device flag and returns; the kernel ends normally.
__device__ int32_t g_selftest_word = 0;
__global__ void barrier_selftest_kernel() {
    if (threadIdx.x == 0) {
        g_selftest_word = 0;
        barrier_arrive_and_wait(&g_selftest_word, 2);
    }
}

bool fused_enabled() {
    const char *v = std::getenv("FP8MP_FUSED_MASTER");
    return !(v != nullptr && std::strcmp(v, "0") == 0);
}

// Resident blocks per SM of the fused kernel (SGD, Adam) per device, queried
// once; a query that raced with another thread's stores the same value.
struct FusedGrid {
    std::atomic<int> blocks_per_sm[2];
};
FusedGrid g_fused[64];

// Threads of an early block: as many warps as fit in the register file
// beside one CTA of the GEMM. The file is split between the SM's four
// schedulers, and the warps of a CTA are dealt to them in turn, so the
// bound is per scheduler: its quarter of the file, less the registers of the
// GEMM warps it holds (at most ceil(warps / 4)), over the registers of one
// warp of this kernel (allocated 8 per thread at a time), times four.
// Queried once per optimizer.
std::atomic<int> g_early_threads[4];  // [which + 2 * FOLD]

template <class Opt, class Args, class Extra, bool FOLD>
int early_block_threads(int which, const DeviceInfo &dev) {
    which += FOLD ? 2 : 0;
    int t = g_early_threads[which].load(std::memory_order_relaxed);
    if (t >= 32) return t;
    cudaFuncAttributes fa;
    int file = 0;
    if (cudaFuncGetAttributes(&fa, prescanned_step_kernel<Opt, Args, Extra, true, true, FOLD>) != cudaSuccess ||
        cudaDeviceGetAttribute(&file, cudaDevAttrMaxRegistersPerMultiprocessor, dev.device) != cudaSuccess)
        return 0;
    int gemm_warps = 0;
    const int gemm_warp = gemm_warp_registers(&gemm_warps);
    if (gemm_warp <= 0) return 0;
    const int per_warp = 32 * ((fa.numRegs + 7) & ~7);
    const int free_per_scheduler = file / 4 - ((gemm_warps + 3) / 4) * gemm_warp;
    int warps = 4 * (free_per_scheduler > 0 ? free_per_scheduler / per_warp : 0);
    if (warps > kEarlyMaxThreads / 32) warps = kEarlyMaxThreads / 32;
    if (warps < 4) warps = 4;  // no room beside the GEMM: the blocks wait for it, still one per SM
    t = warps * 32;
    g_early_threads[which].store(t, std::memory_order_relaxed);
    return t;
}

template <class Opt, class Args, class Extra>
int launch_step(const StepCommon &c, const Args &a, const Extra &x, int which, cudaStream_t s, const DeviceInfo &dev,
                const char *fn, int32_t *grad_nonfinite = nullptr, bool early = false, bool wait_done = false,
                const FoldBatch *fold = nullptr) {
    FoldBatch none;
    std::memset(&none, 0, sizeof none);
    none.w_index = -1;
    cudaError_t e = cudaSuccess;
    if (grad_nonfinite == nullptr) {  // the scanning steps count arrivals in found_inf: zero it
        e = launch_zero_word(c.found_inf, s);
        if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    }
    const int64_t nvec = c.n >> 3;
    int64_t blocks = (nvec + kThreads - 1) / kThreads;
    if (blocks < 1) blocks = 1;
    if (grad_nonfinite != nullptr) {
        // up to 32 blocks per SM (6 resident for SGD, 3 for Adam): smaller
        // shares let the block scheduler even out the tail, measured faster
        // than a grid of resident blocks
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 32;
        if (blocks > cap) blocks = cap;
        if (early) {
            const bool folded = fold != nullptr && wait_done;
            const int threads = folded ? early_block_threads<Opt, Args, Extra, true>(which, dev)
                                       : early_block_threads<Opt, Args, Extra, false>(which, dev);
            if (threads < 32) return fail(FP8MP_ERR_LAUNCH, "%s: kernel attribute query failed", fn);
            int64_t eb = (nvec + threads - 1) / threads;
            eb = eb < 1 ? 1 : (eb > dev.num_sms ? dev.num_sms : eb);
            if (folded)
                e = launch_kernel(prescanned_step_kernel<Opt, Args, Extra, true, true, true>,
                                  dim3(static_cast<unsigned>(eb)), dim3(threads), 0, s, c, a, x, grad_nonfinite,
                                  *fold);
            else if (wait_done)
                e = launch_kernel(prescanned_step_kernel<Opt, Args, Extra, true, true, false>,
                                  dim3(static_cast<unsigned>(eb)), dim3(threads), 0, s, c, a, x, grad_nonfinite,
                                  none);
            else
                e = launch_kernel(prescanned_step_kernel<Opt, Args, Extra, true, false, false>,
                                  dim3(static_cast<unsigned>(eb)), dim3(threads), 0, s, c, a, x, grad_nonfinite,
                                  none);
        } else {
            e = launch_kernel(prescanned_step_kernel<Opt, Args, Extra, false, false, false>,
                              dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, c, a, x, grad_nonfinite,
                              none);
        }
        if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
        return FP8MP_OK;
    }
    if (c.n > 0 && fused_enabled()) {
        std::atomic<int> &cached = g_fused[dev.device & 63].blocks_per_sm[which];
        int per_sm = cached.load(std::memory_order_relaxed);
        if (per_sm < 1) {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_step_kernel<Opt, Args, Extra>, kThreads,
                                                              0);
            if (e != cudaSuccess || per_sm < 1)
                return fail(FP8MP_ERR_LAUNCH, "%s: occupancy query failed: %s", fn, cudaGetErrorString(e));
            cached.store(per_sm, std::memory_order_relaxed);
        }
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * per_sm;
        if (blocks > cap) blocks = cap;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(kThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, fused_step_kernel<Opt, Args, Extra>, c, a, x);
        if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
        return FP8MP_OK;
    }
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (c.n > 0) {
        launch_kernel(grad_scan_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, c.g, c.n,
                      c.found_inf);
        launch_kernel(update_kernel<Opt, Args>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, c, a);
    }
    launch_kernel(bookkeeping_kernel<Extra>, dim3(1), dim3(1), 0, s, c, x);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    return FP8MP_OK;
}

}  // namespace

int launch_adam_step(const uint16_t *g, int64_t n, float *w, float *m, float *v, uint8_t *w8, const float *scale_w,
                     float *amax_w, float *loss_scale, int32_t *growth, int32_t *found_inf, float *beta_pows,
                     float lr, float b1, float b2, float eps, float backoff, float growth_factor,
                     int32_t growth_interval, cudaStream_t s, const DeviceInfo &dev, int32_t *grad_nonfinite,
                     const uint8_t *w8_in, bool early, bool wait_done, const FoldBatch *fold) {
    const StepCommon c = {g, n, w8, w8_in, scale_w, amax_w, loss_scale, growth, found_inf, backoff, growth_factor,
                          growth_interval};
    const AdamArgs a = {w, m, v, beta_pows, lr, b1, b2, eps};
    const AdamExtra x = {beta_pows, b1, b2};
    return launch_step<AdamOpt>(c, a, x, 1, s, dev, grad_nonfinite ? "mp_master_step_adam_prescanned"
                                                                   : "mp_master_step_adam",
                                grad_nonfinite, early, wait_done, fold);
}

int launch_master_step(const uint16_t *g, int64_t n, float *w, float *v, uint8_t *w8, const float *scale_w,
                       float *amax_w, float *loss_scale, int32_t *growth, int32_t *found_inf, float lr, float mu,
                       float backoff, float growth_factor, int32_t growth_interval, cudaStream_t s,
                       const DeviceInfo &dev, int32_t *grad_nonfinite, const uint8_t *w8_in, bool early,
                       bool wait_done, const FoldBatch *fold) {
    const StepCommon c = {g, n, w8, w8_in, scale_w, amax_w, loss_scale, growth, found_inf, backoff, growth_factor,
                          growth_interval};
    const SgdArgs a = {w, v, lr, mu};
    return launch_step<SgdOpt>(c, a, NoExtra{}, 0, s, dev,
                               grad_nonfinite ? "mp_master_step_prescanned" : "mp_master_step", grad_nonfinite,
                               early, wait_done, fold);
}

int launch_barrier_selftest(cudaStream_t s) {
    barrier_selftest_kernel<<<1, 32, 0, s>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "self-test launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

int read_and_clear_master_timeout_flag(unsigned int *value) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_master_timeout_flag, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_master_timeout_flag, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "reading the timeout flag failed: %s", cudaGetErrorString(e));
    *value = v;
    return FP8MP_OK;
}

}  // namespace fp8mp
