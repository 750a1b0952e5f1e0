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
#include <atomic>
#include <mutex>

#include "fp8mp_async.cuh"

namespace fp8mp {

// Raised by a tiled cast whose bounded mbarrier wait ran out; fp8mp_check()
// reads and clears it.
__device__ unsigned int g_cast_timeout_flag = 0;

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

// Row-major cast of a flat array of n elements in chunks of 16 elements (one
// 16-byte store of codes each). Block b owns the kChunksPerThread * 256
// consecutive chunks from b * kChunksPerThread * 256 on; thread t takes
// chunks t, t + 256, ... of them (each load and store instruction of a warp
// is one coalesced 512-byte (bf16) or 1 KB (fp32) access) and issues all of
// its loads before it converts anything, so a resident block keeps 32 KB
// (bf16) in flight. The grid has one block per such run: small, equal
// blocks that the block scheduler deals out to SMs as they free up. The
// n % 16 tail is done element by element by the last block.
constexpr int kChunksPerThread = 4;

//
// EARLY (FP8MP_OVERLAP_PREVIOUS): the caller guarantees that the kernel still
// running before this one on the stream neither writes nor reads x, out or
// *amax, so the blocks start without waiting for it (they use what it leaves
// free of the SMs); block 0 waits for it at its very end, so the grid still
// completes after it and whatever follows on the stream sees both. Like
// every kernel of the library it lets the next kernel start only after its
// own wait has returned (here: block 0's, at the end; the other blocks let
// it by exiting), so a kernel that starts early behind this one still knows
// every kernel before this one complete.
template <int FMT, bool BF16, bool EARLY>
__global__ void __launch_bounds__(kThreads, 4)
cast_rows_kernel(const void *__restrict__ x, int64_t n, const float *__restrict__ scale_p,
                 uint8_t *__restrict__ out, float *__restrict__ amax_p) {
    if constexpr (!EARLY) {
        pdl_wait();
        pdl_launch_dependents();
    }
    const float scale = __ldg(scale_p);
    float am = 0.0f;
    const int64_t nchunk = n >> 4;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * (kChunksPerThread * kThreads) + threadIdx.x;
    if constexpr (BF16) {
        uint4 raw[kChunksPerThread][2];
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            const int64_t c = c0 + u * kThreads;
            if (c < nchunk) {
                const uint4 *p = reinterpret_cast<const uint4 *>(x) + 2 * c;
                raw[u][0] = __ldcs(p);
                raw[u][1] = __ldcs(p + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            const int64_t c = c0 + u * kThreads;
            if (c < nchunk) {
                uint32_t o[4], probe = 0;
                o[0] = cast4_bf16<FMT>(raw[u][0].x, raw[u][0].y, scale, am, probe);
                o[1] = cast4_bf16<FMT>(raw[u][0].z, raw[u][0].w, scale, am, probe);
                o[2] = cast4_bf16<FMT>(raw[u][1].x, raw[u][1].y, scale, am, probe);
                o[3] = cast4_bf16<FMT>(raw[u][1].z, raw[u][1].w, scale, am, probe);
                if (probe & 0x80808080u) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) o[j] = canonical_nan<FMT>(o[j]);
                }
                reinterpret_cast<uint4 *>(out)[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    } else {
        // fp32: two chunks (eight 16-byte loads) at a time
#pragma unroll
        for (int h = 0; h < kChunksPerThread; h += 2) {
            float4 raw[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t c = c0 + (h + u) * kThreads;
                if (c < nchunk) {
                    const float4 *p = reinterpret_cast<const float4 *>(x) + 4 * c;
#pragma unroll
                    for (int j = 0; j < 4; ++j) raw[u][j] = __ldcs(p + j);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t c = c0 + (h + u) * kThreads;
                if (c < nchunk) {
                    uint32_t o[4], probe = 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[j] = cast4<FMT>(raw[u][j].x, raw[u][j].y, raw[u][j].z, raw[u][j].w, scale, am, probe);
                    if (probe & 0x80808080u) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) o[j] = canonical_nan<FMT>(o[j]);
                    }
                    reinterpret_cast<uint4 *>(out)[c] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
    }
    if (blockIdx.x == gridDim.x - 1) {
        for (int64_t i = (nchunk << 4) + threadIdx.x; i < n; i += blockDim.x) {
            const float v = load1<BF16>(x, i);
            out[i] = static_cast<uint8_t>(cvt_pair<FMT>(__fmul_rn(v, scale), 0.0f) & 0xFFu);
            am = fmaxf(am, fabsf(v));
        }
    }
    if (amax_p != nullptr) block_amax_atomic(am, amax_p);
    if constexpr (EARLY) {
        if (blockIdx.x == 0) {
            pdl_wait();
            pdl_launch_dependents();
        }
    }
}

// Blocks of cast_rows_kernel / amax_kernel for n elements: one per run of
// kChunksPerThread * 256 chunks, at least one (the last block also does the
// n % 16 tail).
inline int64_t row_blocks(int64_t n) {
    const int64_t per_block = static_cast<int64_t>(kChunksPerThread) * kThreads;
    const int64_t blocks = ((n >> 4) + per_block - 1) / per_block;
    return blocks < 1 ? 1 : blocks;
}

// Row-major + transposed cast of one 128 x 128 tile per block of 256 threads.
// Thread t covers rows r0 + 4 * (t >> 3) .. + 3 and columns c0 + 16 * (t & 7)
// .. + 15: it issues the loads of its whole 4 x 16 patch first (eight 16-byte
// loads for bf16, sixteen for fp32), converts it, and writes the four 16-byte
// row segments of codes (eight threads write one 128-byte row segment). For
// the transposed copy it turns the 4 x 16 codes into sixteen 4-byte column
// words (4 consecutive rows of one column, by byte permutes) and parks them
// in shared memory, where word (column cc, row group g) sits at index
// cc * 32 + (g ^ 4 * ((cc >> 4) & 7)): one store instruction of a warp then
// touches 32 distinct banks, and the four words of 16 consecutive rows stay
// adjacent, so phase 2 moves 16 rows of one column with one 16-byte shared
// load and one 16-byte store to out_t (eight threads write one 128-byte row
// segment of out_t).
// EARLY: as for cast_rows_kernel.
template <int FMT, bool BF16, bool EARLY>
__global__ void __launch_bounds__(kThreads, BF16 ? 4 : 3)
cast_rows_t_kernel(const void *__restrict__ x, int64_t rows, int64_t cols, const float *__restrict__ scale_p,
                   uint8_t *__restrict__ out, uint8_t *__restrict__ out_t, float *__restrict__ amax_p) {
    if constexpr (!EARLY) {
        pdl_wait();
        pdl_launch_dependents();
    }
    __shared__ __align__(16) uint32_t sT[128 * 32];
    const int64_t tiles_c = (cols + 127) >> 7;
    const int64_t tr = blockIdx.x / tiles_c, tc = blockIdx.x - tr * tiles_c;
    const int64_t r0 = tr * 128, c0 = tc * 128;
    const int tx = threadIdx.x & 7, ty = threadIdx.x >> 3;
    const int64_t r = r0 + 4 * ty, c = c0 + 16 * tx;
    const float scale = __ldg(scale_p);
    float am = 0.0f;
    if (r < rows && c < cols) {
        uint32_t q[4][4];  // codes of row i, word k = columns 4k .. 4k+3
        if constexpr (BF16) {
            uint4 raw[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 *p = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) +
                                                                 (r + i) * cols + c);
                raw[i][0] = __ldcs(p);
                raw[i][1] = __ldcs(p + 1);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w[8] = {raw[i][0].x, raw[i][0].y, raw[i][0].z, raw[i][0].w,
                                       raw[i][1].x, raw[i][1].y, raw[i][1].z, raw[i][1].w};
                uint32_t probe = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) q[i][k] = cast4_bf16<FMT>(w[2 * k], w[2 * k + 1], scale, am, probe);
                if (probe & 0x80808080u) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) q[i][k] = canonical_nan<FMT>(q[i][k]);
                }
            }
        } else {
            float4 raw[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) +
                                                                   (r + i) * cols + c);
#pragma unroll
                for (int k = 0; k < 4; ++k) raw[i][k] = __ldcs(p + k);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t probe = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 v = raw[i][k];
                    q[i][k] = cast4<FMT>(v.x, v.y, v.z, v.w, scale, am, probe);
                }
                if (probe & 0x80808080u) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) q[i][k] = canonical_nan<FMT>(q[i][k]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4 *>(out + (r + i) * cols + c) = make_uint4(q[i][0], q[i][1], q[i][2], q[i][3]);
        if (out_t != nullptr) {
            const int sw = ty ^ (4 * tx);  // row group ty, XOR-swizzled by the column's 16-wide group tx
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // 4 x 4 byte transpose: rows r .. r+3 of columns c + 4k .. c + 4k + 3
                const uint32_t t0 = __byte_perm(q[0][k], q[1][k], 0x5140), t1 = __byte_perm(q[0][k], q[1][k], 0x7362);
                const uint32_t t2 = __byte_perm(q[2][k], q[3][k], 0x5140), t3 = __byte_perm(q[2][k], q[3][k], 0x7362);
                uint32_t *col = &sT[(16 * tx + 4 * k) * 32 + sw];
                col[0] = __byte_perm(t0, t2, 0x5410);
                col[32] = __byte_perm(t0, t2, 0x7632);
                col[64] = __byte_perm(t1, t3, 0x5410);
                col[96] = __byte_perm(t1, t3, 0x7632);
            }
        }
    }
    __syncthreads();
    if (out_t != nullptr) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int id = threadIdx.x + kThreads * i;  // 0 .. 1023
            const int cc = id >> 3, k = id & 7;          // tile column, 16-row chunk
            const int64_t col = c0 + cc, row = r0 + 16 * k;
            if (col < cols && row < rows) {
                const uint4 P = *reinterpret_cast<const uint4 *>(&sT[cc * 32 + 4 * (k ^ ((cc >> 4) & 7))]);
                *reinterpret_cast<uint4 *>(out_t + col * rows + row) = P;
            }
        }
    }
    if (amax_p != nullptr) block_amax_atomic(am, amax_p);
    if constexpr (EARLY) {
        if (blockIdx.x == 0) {
            pdl_wait();
            pdl_launch_dependents();
        }
    }
}

// ---------------------------------------------------------------------------
// The bias-gradient cast: a persistent, TMA-fed version of the tile cast.
//
// The grid has k CTAs per 128-column strip (k = dbias_ctas_per_strip(), a
// function of the shape only: 4 at 8192 x 4096, so 128 CTAs); CTA j of a
// strip converts the strip's tile rows j, j + k, j + 2k, ..., so at any
// moment the grid works on a band of k tile rows across the whole width.
// Warp 8 (one lane) streams those 128 x 128 input tiles into a ring of
// shared-memory stages with TMA (two or four 128-byte-swizzled boxes of 128
// rows per tile) and re-arms a stage when the consumers have used it; warps
// 0-7 read each tile from shared memory (each thread a 4 x 16 patch, as in
// cast_rows_t_kernel), write the 16-byte row segments of codes, optionally
// the transposed copy through sT, and add their rows to column sums they keep
// in registers across all their tiles. The loads of the next tiles are in
// flight while a tile is converted, and the CTA publishes its column sums,
// fences and counts its arrival once, at the end. The arithmetic runs on
// pairs of fp32 lanes (mul/add .f32x2: one instruction per two elements, each
// lane rounded as its own fp32 operation).
//
// Column-sum order (fixed by the shape): each thread adds its 4 rows of each
// of its CTA's tiles, tile after tile, in row order; the four threads of a
// warp that share columns are combined by a butterfly (xor 8, then xor 16);
// the 8 warps in warp order; then the strip's k CTA sums in order of j, by
// the CTA that arrives last on the strip's counter, which writes dbias and
// sets the k sums and the counter back to zero, so a workspace that is zero
// before a call is zero after it.
//
// CL: the strip's k CTAs are one thread-block cluster (k <= 8, launched only
// when the device holds all the strips' clusters at once): blocks
// strip * k .. strip * k + k - 1, CTA j being cluster rank j. Each CTA leaves
// its column sums in its own shared memory, and after a cluster barrier CTA
// 0 reads the others' through distributed shared memory and adds them in
// the same order of j; a second barrier keeps every CTA resident until it
// has. No workspace, counter, fence or global atomic: the same sums, bit for
// bit, without the round trips through L2 at the end of the launch.
constexpr int kTileThreads = 288;       // 8 consumer warps + 1 producer warp
constexpr int kBoxBytes = 128 * 128;    // one box: 128 rows x 128 bytes
constexpr int kDbiasTargetCtas = 152;   // the split aims at this many CTAs

template <bool BF16>
struct TileCfg {
    static constexpr int ESIZE = BF16 ? 2 : 4;
    static constexpr int BOX_COLS = 128 / ESIZE;      // elements per box row
    static constexpr int BOXES = 128 / BOX_COLS;      // boxes per 128-column tile
    static constexpr int STAGE_BYTES = BOXES * kBoxBytes;
    static constexpr int STAGES = BF16 ? 4 : 2;
    static constexpr int ST_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int PART_OFFSET = ST_OFFSET + 128 * 32 * 4;
    static constexpr int BAR_OFFSET = PART_OFFSET + 8 * 128 * 4;
    static constexpr int MISC_OFFSET = BAR_OFFSET + 16 * STAGES;
    static constexpr int SMEM_BYTES = MISC_OFFSET + 64 + 1024;  // + the 1024-byte alignment pad
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Pairs of fp32 values in one 64-bit register (low lane first) and the
// two-lane fp32 arithmetic of sm_100-class GPUs: each lane is one IEEE
// round-to-nearest-even operation, bit-identical to the scalar one.
__device__ __forceinline__ uint64_t f2_from_bits(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void f2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two (lo, hi) pairs -> four codes under scale2 = (scale, scale); the pairs
// join the column sums and their |x| the running amax. NaN inputs give NaN
// codes here; the caller canonicalises them (they also make the column sums
// NaN, which is how it notices).
template <int FMT>
__device__ __forceinline__ uint32_t cast_pairs(uint64_t p0, uint64_t p1, uint64_t scale2, uint64_t &s0, uint64_t &s1,
                                               float &am) {
    float a, b, c, d;
    f2_split(f2_mul(p0, scale2), a, b);
    f2_split(f2_mul(p1, scale2), c, d);
    s0 = f2_add(s0, p0);
    s1 = f2_add(s1, p1);
    float x0, x1, x2, x3;
    f2_split(p0, x0, x1);
    f2_split(p1, x2, x3);
    am = fmaxf(fmaxf(am, fabsf(x0)), fmaxf(fabsf(x1), fmaxf(fabsf(x2), fabsf(x3))));
    return cvt_pair_raw<FMT>(a, b) | (cvt_pair_raw<FMT>(c, d) << 16);
}

template <int FMT, bool BF16, bool CL>
__global__ void __launch_bounds__(kTileThreads, 1)
cast_dbias_kernel(const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, int k_per_strip,
                  const float *__restrict__ scale_p, uint8_t *__restrict__ out, uint8_t *__restrict__ out_t,
                  float *__restrict__ amax_p, float *__restrict__ ws, uint32_t *__restrict__ counters,
                  void *__restrict__ dbias, int dbias_bf16) {
    using C = TileCfg<BF16>;
    extern __shared__ uint8_t smem_raw[];
    uint32_t base = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    base += pad;
    uint32_t *sT = reinterpret_cast<uint32_t *>(smem + C::ST_OFFSET);
    float *s_part = reinterpret_cast<float *>(smem + C::PART_OFFSET);
    const uint32_t bar0 = base + C::BAR_OFFSET;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFFSET);
    int *s_last = reinterpret_cast<int *>(smem + C::MISC_OFFSET + 4);
    float *s_red = reinterpret_cast<float *>(smem + C::MISC_OFFSET + 32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_r = (rows + 127) >> 7, tiles_c = (cols + 127) >> 7;
    const int64_t strip = CL ? blockIdx.x / k_per_strip : blockIdx.x % tiles_c;
    const int64_t j = CL ? blockIdx.x % k_per_strip : blockIdx.x / tiles_c;
    const int64_t c0 = strip * 128;
    const int64_t ntile = j < tiles_r ? (tiles_r - 1 - j) / k_per_strip + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar0 + 8u * s, 1);                  // full: the producer's arrival + the TMA bytes
            mbar_init(bar0 + 8u * (C::STAGES + s), 8);    // empty: one arrival per consumer warp
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap);
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    if (warp == 8) {
        if (lane == 0) {
            // ---------------- TMA producer
            int64_t i = 0;
            for (; i < ntile; ++i) {
                const int s = static_cast<int>(i % C::STAGES);
                const uint32_t ph = static_cast<uint32_t>(i / C::STAGES) & 1u;
                if (!wait_bounded(bar0 + 8u * (C::STAGES + s), ph ^ 1u, abort_flag, &g_cast_timeout_flag)) break;
                mbar_arrive_expect_tx(bar0 + 8u * s, C::STAGE_BYTES);
                const int32_t r0 = static_cast<int32_t>((j + i * k_per_strip) * 128);
#pragma unroll
                for (int bx = 0; bx < C::BOXES; ++bx)
                    tma_load_2d_cta(base + s * C::STAGE_BYTES + bx * kBoxBytes, &tmap, bar0 + 8u * s,
                                    static_cast<int32_t>(c0) + bx * C::BOX_COLS, r0);
            }
            if (i < ntile) {
                // aborted: let the loads already issued land before the CTA goes away
                volatile int never = 0;
                for (int64_t q = i - 1; q >= 0 && q >= i - C::STAGES; --q)
                    wait_bounded(bar0 + 8u * static_cast<uint32_t>(q % C::STAGES),
                                 static_cast<uint32_t>(q / C::STAGES) & 1u, &never, &g_cast_timeout_flag);
            }
        }
        if constexpr (CL) {
            // the producer warp takes part in the cluster's two barriers too
            __syncwarp();
            if (k_per_strip > 1) {
                cluster_sync_all();
                cluster_sync_all();
            }
        }
        return;
    }

    // ---------------- consumers: warps 0-7, thread (tx, ty) = 4 rows x 16 columns
    const int tx = threadIdx.x & 7, ty = threadIdx.x >> 3;
    const int64_t c = c0 + 16 * tx;
    const float scale = __ldg(scale_p);
    const uint64_t scale2 = f2_from_bits(__float_as_uint(scale), __float_as_uint(scale));
    float am = 0.0f;
    uint64_t csum[8];  // column pairs (2q, 2q + 1) of the thread's 16 columns
#pragma unroll
    for (int q = 0; q < 8; ++q) csum[q] = 0ull;
    for (int64_t i = 0; i < ntile; ++i) {
        const int s = static_cast<int>(i % C::STAGES);
        const uint32_t ph = static_cast<uint32_t>(i / C::STAGES) & 1u;
        // lane 0 waits for the stage; the warp follows its result (uniform
        // per warp, so the __syncwarp below is never divergent)
        int okw = 0;
        if (lane == 0) okw = wait_bounded(bar0 + 8u * s, ph, abort_flag, &g_cast_timeout_flag) ? 1 : 0;
        const bool ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
        __syncwarp();
        const int64_t r0 = (j + i * k_per_strip) * 128;
        const int64_t r = r0 + 4 * ty;
        if (ok) {
            const uint8_t *stage = smem + s * C::STAGE_BYTES;
            uint32_t q4[4][4];  // codes of row rr, word w = columns 4w .. 4w+3
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int row = 4 * ty + rr;
                uint64_t p[8];  // the row's 16 values as pairs
                if constexpr (BF16) {
                    const uint8_t *box = stage + (tx >> 2) * kBoxBytes + row * 128;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(box + (((2 * (tx & 3) + h) ^ (row & 7)) << 4));
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) p[4 * h + e] = f2_from_bits(w[e] << 16, w[e] & 0xFFFF0000u);
                    }
                } else {
                    const uint8_t *box = stage + (tx >> 1) * kBoxBytes + row * 128;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(box + (((4 * (tx & 1) + h) ^ (row & 7)) << 4));
                        p[2 * h] = f2_from_bits(v.x, v.y);
                        p[2 * h + 1] = f2_from_bits(v.z, v.w);
                    }
                }
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    q4[rr][w] = cast_pairs<FMT>(p[2 * w], p[2 * w + 1], scale2, csum[2 * w], csum[2 * w + 1], am);
            }
            // Release the stage only now that every loaded value has been used:
            // a shared-memory load whose value is consumed has been performed,
            // so the refill cannot overwrite data the warp has not read yet (a
            // release right after the loads let the next tile's TMA write reach
            // a few 16-byte chunks first, about once in tens of launches).
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8u * (C::STAGES + s));
            // a NaN input makes its column sum NaN (and so, from then on, does
            // nothing else: Inf - Inf also gives NaN, and canonicalising codes
            // that hold no NaN changes nothing)
            bool any_nan = false;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float lo, hi;
                f2_split(csum[q], lo, hi);
                any_nan |= (lo != lo) | (hi != hi);
            }
            if (any_nan) {
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int w = 0; w < 4; ++w) q4[rr][w] = canonical_nan<FMT>(q4[rr][w]);
            }
            if (r < rows && c < cols) {
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
                    *reinterpret_cast<uint4 *>(out + (r + rr) * cols + c) =
                        make_uint4(q4[rr][0], q4[rr][1], q4[rr][2], q4[rr][3]);
                if (out_t != nullptr) {
                    const int sw = ty ^ (4 * tx);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t t0 = __byte_perm(q4[0][w], q4[1][w], 0x5140), t1 = __byte_perm(q4[0][w], q4[1][w], 0x7362);
                        const uint32_t t2 = __byte_perm(q4[2][w], q4[3][w], 0x5140), t3 = __byte_perm(q4[2][w], q4[3][w], 0x7362);
                        uint32_t *col = &sT[(16 * tx + 4 * w) * 32 + sw];
                        col[0] = __byte_perm(t0, t2, 0x5410);
                        col[32] = __byte_perm(t0, t2, 0x7632);
                        col[64] = __byte_perm(t1, t3, 0x5410);
                        col[96] = __byte_perm(t1, t3, 0x7632);
                    }
                }
            }
        }
        if (out_t != nullptr) {
            // every consumer thread passes both barriers on every tile, aborted or not
            consumer_sync();
            if (ok) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int id = threadIdx.x + 256 * q;
                    const int cc = id >> 3, kk = id & 7;
                    const int64_t col = c0 + cc, row = r0 + 16 * kk;
                    if (col < cols && row < rows) {
                        const uint4 P = *reinterpret_cast<const uint4 *>(&sT[cc * 32 + 4 * (kk ^ ((cc >> 4) & 7))]);
                        *reinterpret_cast<uint4 *>(out_t + col * rows + row) = P;
                    }
                }
            }
            consumer_sync();  // sT is free for the next tile
        }
    }
    // ---------------- the CTA's amax and column sums
    float cs[16];
#pragma unroll
    for (int q = 0; q < 8; ++q) f2_split(csum[q], cs[2 * q], cs[2 * q + 1]);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        cs[q] = __fadd_rn(cs[q], __shfl_xor_sync(0xffffffffu, cs[q], 8));
        cs[q] = __fadd_rn(cs[q], __shfl_xor_sync(0xffffffffu, cs[q], 16));
    }
    if (lane < 8) {
        float *dst = &s_part[warp * 128 + 16 * tx];
#pragma unroll
        for (int q = 0; q < 16; q += 4)
            *reinterpret_cast<float4 *>(dst + q) = make_float4(cs[q], cs[q + 1], cs[q + 2], cs[q + 3]);
    }
    am = warp_max(am);
    if (lane == 0) s_red[warp] = am;
    consumer_sync();
    if (threadIdx.x == 0 && amax_p != nullptr) {
        float t = s_red[0];
        for (int w = 1; w < 8; ++w) t = fmaxf(t, s_red[w]);
        atomicMax(reinterpret_cast<int *>(amax_p), __float_as_int(t));
    }
    if constexpr (CL) {
        // the CTA's column sums in its shared memory (the transpose tile is
        // free: every tile's reads of it ended before the last consumer_sync)
        float *s_col = reinterpret_cast<float *>(sT);
        if (threadIdx.x < 128) {
            float t = s_part[threadIdx.x];
#pragma unroll
            for (int w = 1; w < 8; ++w) t = __fadd_rn(t, s_part[w * 128 + threadIdx.x]);
            s_col[threadIdx.x] = t;
        }
        __syncwarp();
        if (k_per_strip > 1) cluster_sync_all();  // every CTA's sums are written
        if (j == 0 && threadIdx.x < 128 && c0 + threadIdx.x < cols) {
            const uint32_t a = smem_u32(s_col + threadIdx.x);
            float v[8];
#pragma unroll
            for (int r = 1; r < 8; ++r) v[r] = r < k_per_strip ? ld_shared_cluster_f32(mapa_shared(a, r)) : 0.0f;
            float t = s_col[threadIdx.x];
#pragma unroll
            for (int r = 1; r < 8; ++r)
                if (r < k_per_strip) t = __fadd_rn(t, v[r]);
            const int64_t col = c0 + threadIdx.x;
            if (dbias_bf16)
                static_cast<__nv_bfloat16 *>(dbias)[col] = __float2bfloat16_rn(t);
            else
                static_cast<float *>(dbias)[col] = t;
        }
        __syncwarp();
        if (k_per_strip > 1) cluster_sync_all();  // CTA 0 has read them: the others may leave
        return;
    }
    if (threadIdx.x < 128) {
        const int64_t col = c0 + threadIdx.x;
        if (col < cols) {
            float t = s_part[threadIdx.x];
#pragma unroll
            for (int w = 1; w < 8; ++w) t = __fadd_rn(t, s_part[w * 128 + threadIdx.x]);
            ws[j * cols + col] = t;
        }
        __threadfence();  // the CTA's column sums are visible before its arrival is
    }
    consumer_sync();
    if (threadIdx.x == 0) *s_last = atomicAdd(&counters[strip], 1u) == static_cast<uint32_t>(k_per_strip - 1);
    consumer_sync();
    if (*s_last) {
        __threadfence();
        if (threadIdx.x < 128 && c0 + threadIdx.x < cols) {
            const int64_t col = c0 + threadIdx.x;
            float t = __ldcg(ws + col);
            for (int jj = 1; jj < k_per_strip; ++jj) t = __fadd_rn(t, __ldcg(ws + jj * cols + col));
            for (int jj = 0; jj < k_per_strip; ++jj) __stcg(ws + jj * cols + col, 0.0f);
            if (dbias_bf16)
                static_cast<__nv_bfloat16 *>(dbias)[col] = __float2bfloat16_rn(t);
            else
                static_cast<float *>(dbias)[col] = t;
        }
        if (threadIdx.x == 0) counters[strip] = 0u;
    }
}

template <int FMT, bool BF16, bool EARLY>
int launch_typed(const void *x, int64_t rows, int64_t cols, const float *scale, uint8_t *out,
                 uint8_t *out_t, float *amax, cudaStream_t s) {
    if (out_t == nullptr) {
        const int64_t n = rows * cols;
        const int64_t blocks = row_blocks(n);
        if (blocks > 0x7FFFFFFF) return fail(FP8MP_ERR_INVALID, "fp8_quantize: tensor too large");
        launch_kernel(cast_rows_kernel<FMT, BF16, EARLY>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s,
                      x, n, scale, out, amax);
    } else {
        const int64_t tiles = ((rows + 127) >> 7) * ((cols + 127) >> 7);
        if (tiles > 0x7FFFFFFF) return fail(FP8MP_ERR_INVALID, "fp8_quantize: tensor too large");
        launch_kernel(cast_rows_t_kernel<FMT, BF16, EARLY>, dim3(static_cast<unsigned>(tiles)), dim3(kThreads), 0, s,
                      x, rows, cols, scale, out, out_t, amax);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

// The bias-gradient cast's launch: tensor map of x (boxes of 128 rows x 128
// bytes, 128-byte swizzle, zero fill outside the tensor), k CTAs per strip.
// The CL kernel runs when k = 1 (nothing to combine) and, without a
// transposed copy, as clusters of k when 2 <= k <= 8 and the device holds
// every strip's cluster at once (asked of the occupancy calculator once per
// device and k); else the workspace kernel. At 8192 x 4096 bf16 the
// clusters took 20.3-20.8 us against 21.3 without the transposed copy, but
// 26.7-27.1 against 25.3-25.6 with it (presumably because a cluster's CTAs
// must share one GPC, so 32 clusters of 4 load some GPCs with more busy SMs
// than the 128 CTAs spread one per SM do, which costs the launch that moves
// 4 B/elem more than the round trips it saves).
template <int FMT, bool BF16>
int launch_dbias_typed(const void *x, int64_t rows, int64_t cols, const float *scale, uint8_t *out,
                       uint8_t *out_t, float *amax, void *dbias, int dbias_bf16, float *ws, cudaStream_t s,
                       const DeviceInfo &dev) {
    using C = TileCfg<BF16>;
    static std::atomic<bool> ready[64];
    static std::atomic<int> max_clusters[64][9];  // 0: not asked yet, else 1 + the answer
    static std::mutex m;
    if (dev.device < 0 || dev.device >= 64) return fail(FP8MP_ERR_DEVICE, "device index %d out of range", dev.device);
    if (!ready[dev.device].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(m);
        if (!ready[dev.device].load(std::memory_order_relaxed)) {
            cudaError_t e = cudaFuncSetAttribute(cast_dbias_kernel<FMT, BF16, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(cast_dbias_kernel<FMT, BF16, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
            if (e != cudaSuccess)
                return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_dbias: shared-memory attribute: %s", cudaGetErrorString(e));
            ready[dev.device].store(true, std::memory_order_release);
        }
    }
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return fail(FP8MP_ERR_LAUNCH, "cuTensorMapEncodeTiled is not available");
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * C::ESIZE};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(C::BOX_COLS), 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&tmap, BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                           const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_dbias: cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    const int k = dbias_ctas_per_strip(rows, cols);
    const int64_t strips = (cols + 127) >> 7;
    const int64_t grid = k * strips;
    if (grid > 0x7FFFFFFF) return fail(FP8MP_ERR_INVALID, "fp8_quantize_dbias: tensor too large");
    bool cl = k == 1;
    if (out_t == nullptr && k >= 2 && k <= 8) {
        int n = max_clusters[dev.device][k].load(std::memory_order_relaxed) - 1;
        if (n < 0) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            cfg.gridDim = dim3(static_cast<unsigned>(k * ((dev.num_sms + k - 1) / k)));
            cfg.blockDim = dim3(kTileThreads);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(k);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, cast_dbias_kernel<FMT, BF16, true>, &cfg) != cudaSuccess) {
                (void)cudaGetLastError();  // an unanswered query only means the workspace kernel
                n = 0;
            }
            max_clusters[dev.device][k].store(n + 1, std::memory_order_relaxed);
        }
        cl = n >= strips;
    }
    cudaError_t e;
    if (cl) {
        e = launch_kernel_cluster(cast_dbias_kernel<FMT, BF16, true>, dim3(static_cast<unsigned>(grid)),
                                  dim3(kTileThreads), C::SMEM_BYTES, s, static_cast<unsigned>(k), tmap, rows, cols,
                                  k, scale, out, out_t, amax, ws, static_cast<uint32_t *>(nullptr), dbias,
                                  dbias_bf16);
    } else {
        uint32_t *counters = reinterpret_cast<uint32_t *>(ws + static_cast<int64_t>(k) * cols);
        e = launch_kernel(cast_dbias_kernel<FMT, BF16, false>, dim3(static_cast<unsigned>(grid)),
                          dim3(kTileThreads), C::SMEM_BYTES, s, tmap, rows, cols, k, scale, out, out_t, amax, ws,
                          counters, dbias, dbias_bf16);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_dbias: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

// amax pass of current scaling: max |x| over a flat array, one atomic max
// per block into *amax (zeroed by the caller's stream just before). Same
// work split as cast_rows_kernel: a block per run of kChunksPerThread * 256
// chunks, all of a thread's loads issued first.
template <bool BF16>
__global__ void __launch_bounds__(kThreads, 4)
amax_kernel(const void *__restrict__ x, int64_t n, float *__restrict__ amax_p) {
    pdl_wait();
    pdl_launch_dependents();
    float am = 0.0f;
    const int64_t nchunk = n >> 4;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * (kChunksPerThread * kThreads) + threadIdx.x;
#pragma unroll
    for (int h = 0; h < kChunksPerThread; h += (BF16 ? kChunksPerThread : 2)) {
        constexpr int U = BF16 ? kChunksPerThread : 2;
        float f[U][16];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + (h + u) * kThreads;
            if (c < nchunk) {
                load16<BF16>(x, c, f[u]);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) f[u][j] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                am = fmaxf(fmaxf(am, fabsf(f[u][j])),
                           fmaxf(fabsf(f[u][j + 1]), fmaxf(fabsf(f[u][j + 2]), fabsf(f[u][j + 3]))));
        }
    }
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t i = (nchunk << 4) + threadIdx.x; i < n; i += blockDim.x) am = fmaxf(am, fabsf(load1<BF16>(x, i)));
    block_amax_atomic(am, amax_p);
}

// Current scaling in one cooperative launch (row-major output): every block
// takes the amax of its grid-stride share of x, loading it with an L2
// evict-last policy; the blocks meet at a grid barrier counted in the
// caller's scale_inv word (the arrival count; zeroed, with *amax, by a
// one-thread kernel just before); every block then derives the same scale
// from the tensor's amax and the old scale it read before arriving, and casts
// the same share again -- now read from L2 when x fits there -- and the last
// block to finish writes scale and scale_inv. The barrier wait is bounded
// (about 2 s); on expiry the block raises the casts' timeout flag and skips
// its cast (the outputs are then undefined; fp8mp_check() reports it).
constexpr long long kGridWaitCycles = 4000000000ll;

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_keep_in_l2(const uint4 *ptr, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr), "l"(pol)
                 : "memory");
    return r;
}

template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads, 4)
current_cast_kernel(const void *__restrict__ x, int64_t n, int margin, float *__restrict__ scale_p,
                    float *__restrict__ scale_inv_p, float *__restrict__ amax_p, uint8_t *__restrict__ out) {
    pdl_wait();
    __shared__ float s_scale;
    __shared__ int s_ok;
    const float old_scale = *scale_p;  // read before this block arrives at the barrier
    const int64_t nchunk = n >> 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    constexpr int V = BF16 ? 2 : 4;  // 16-byte vectors per 16-element chunk
    const uint4 *x4 = reinterpret_cast<const uint4 *>(x);
    const uint64_t pol = l2_evict_last_policy();
    float am = 0.0f;
    // ---- phase 1: amax, four chunks' loads in flight per thread
    for (int64_t c = t0; c < nchunk; c += 4 * stride) {
        uint4 v[4][V];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t cc = c + u * stride;
            if (cc < nchunk) {
#pragma unroll
                for (int k = 0; k < V; ++k) v[u][k] = ld_keep_in_l2(x4 + V * cc + k, pol);
            } else {
#pragma unroll
                for (int k = 0; k < V; ++k) v[u][k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const uint32_t w[4] = {v[u][k].x, v[u][k].y, v[u][k].z, v[u][k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (BF16)
                        am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
                    else
                        am = fmaxf(am, fabsf(__uint_as_float(w[e])));
                }
            }
        }
    }
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t i = (nchunk << 4) + threadIdx.x; i < n; i += blockDim.x) am = fmaxf(am, fabsf(load1<BF16>(x, i)));
    block_amax_atomic(am, amax_p);
    // ---- grid barrier: arrivals counted in the scale_inv word
    uint32_t *counter = reinterpret_cast<uint32_t *>(scale_inv_p);
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        const volatile uint32_t *vc = counter;
        const long long start = clock64();
        int ok = 1;
        while (*vc < gridDim.x) {
            if (clock64() - start > kGridWaitCycles) {
                atomicOr(&g_cast_timeout_flag, 1u);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        s_ok = ok;
        s_scale = scale_from_amax(*reinterpret_cast<volatile float *>(amax_p), old_scale, FMT, margin);
    }
    __syncthreads();
    pdl_launch_dependents();
    const float sc = s_scale;
    // ---- phase 2: the cast of the same share
    if (s_ok) {
        for (int64_t c = t0; c < nchunk; c += stride) {
            uint32_t o[4], probe = 0;
            float dummy = 0.0f;
            if constexpr (BF16) {
                const uint4 a = __ldcs(x4 + 2 * c), b = __ldcs(x4 + 2 * c + 1);
                o[0] = cast4_bf16<FMT>(a.x, a.y, sc, dummy, probe);
                o[1] = cast4_bf16<FMT>(a.z, a.w, sc, dummy, probe);
                o[2] = cast4_bf16<FMT>(b.x, b.y, sc, dummy, probe);
                o[3] = cast4_bf16<FMT>(b.z, b.w, sc, dummy, probe);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 f = __ldcs(reinterpret_cast<const float4 *>(x4 + 4 * c + j));
                    o[j] = cast4<FMT>(f.x, f.y, f.z, f.w, sc, dummy, probe);
                }
            }
            if (probe & 0x80808080u) {
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = canonical_nan<FMT>(o[j]);
            }
            reinterpret_cast<uint4 *>(out)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (blockIdx.x == gridDim.x - 1)
            for (int64_t i = (nchunk << 4) + threadIdx.x; i < n; i += blockDim.x)
                out[i] = static_cast<uint8_t>(cvt_pair<FMT>(__fmul_rn(load1<BF16>(x, i), sc), 0.0f) & 0xFFu);
    }
    // ---- the last block to finish publishes the scale
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(counter, 1u) == 2u * gridDim.x - 1u) {
            *scale_p = sc;
            *scale_inv_p = __fdiv_rn(1.0f, sc);
        }
    }
}

__global__ void zero_two_words_kernel(uint32_t *a, uint32_t *b) {
    pdl_wait();
    *a = 0u;
    *b = 0u;
    pdl_launch_dependents();
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

// The cooperative current-scaling cast: blocks per SM that fit (queried once
// per device and instantiation), times the SMs, at most one per 16-element
// chunk group of 256 threads.
template <int FMT, bool BF16>
int launch_current_fused(const void *x, int64_t n, int margin, float *scale, float *scale_inv, float *amax,
                         uint8_t *out, cudaStream_t s, const DeviceInfo &dev) {
    static std::atomic<int> per_sm_cache[64];
    if (dev.device < 0 || dev.device >= 64) return fail(FP8MP_ERR_DEVICE, "device index %d out of range", dev.device);
    int per_sm = per_sm_cache[dev.device].load(std::memory_order_relaxed);
    if (per_sm < 1) {
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, current_cast_kernel<FMT, BF16>, kThreads, 0);
        if (e != cudaSuccess || per_sm < 1)
            return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_current: occupancy query failed: %s", cudaGetErrorString(e));
        per_sm_cache[dev.device].store(per_sm, std::memory_order_relaxed);
    }
    int64_t blocks = ((n >> 4) + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_kernel(zero_two_words_kernel, dim3(1), dim3(1), 0, s, reinterpret_cast<uint32_t *>(amax),
                                  reinterpret_cast<uint32_t *>(scale_inv));
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_current: launch failed: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // every block resident: the grid barrier cannot wait forever
    attr[0].val.cooperative = 1;
    // and launched like the library's other kernels: its blocks wait in
    // griddepcontrol.wait, before the grid barrier, for the zeroing kernel
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, current_cast_kernel<FMT, BF16>, x, n, margin, scale, scale_inv, amax, out);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();  // not sticky: the grid did not fit at once; the caller takes the three-pass path
        return 1;
    }
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_current: launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

int launch_quantize_current(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, int margin,
                            float *scale, float *scale_inv, float *amax, uint8_t *out, uint8_t *out_t,
                            cudaStream_t s, const DeviceInfo &dev) {
    if (out_t == nullptr && rows * cols > 0) {
        // one cooperative launch; 1 = its grid did not fit at once (nothing
        // read or written yet beyond *amax and *scale_inv, which the
        // three-pass path below sets again)
        const int64_t n = rows * cols;
        const bool bf16 = x_dtype == FP8MP_BF16;
        int rc;
        if (fmt == FP8MP_E4M3)
            rc = bf16 ? launch_current_fused<FP8MP_E4M3, true>(x, n, margin, scale, scale_inv, amax, out, s, dev)
                      : launch_current_fused<FP8MP_E4M3, false>(x, n, margin, scale, scale_inv, amax, out, s, dev);
        else
            rc = bf16 ? launch_current_fused<FP8MP_E5M2, true>(x, n, margin, scale, scale_inv, amax, out, s, dev)
                      : launch_current_fused<FP8MP_E5M2, false>(x, n, margin, scale, scale_inv, amax, out, s, dev);
        if (rc != 1) return rc;
    }
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "fp8_quantize_current: memset failed: %s", cudaGetErrorString(e));
    const int64_t n = rows * cols;
    const int64_t blocks = row_blocks(n);
    if (blocks > 0x7FFFFFFF) return fail(FP8MP_ERR_INVALID, "fp8_quantize_current: tensor too large");
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

int dbias_ctas_per_strip(int64_t rows, int64_t cols) {
    const int64_t tiles_r = (rows + 127) >> 7, tiles_c = (cols + 127) >> 7;
    int64_t k = tiles_c > 0 ? kDbiasTargetCtas / tiles_c : 1;
    if (k > tiles_r) k = tiles_r;
    if (k < 1) k = 1;
    return static_cast<int>(k);
}

int launch_quantize_dbias(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, const float *scale,
                          uint8_t *out, uint8_t *out_t, float *amax, void *dbias, int dbias_dtype, float *ws,
                          cudaStream_t s, const DeviceInfo &dev) {
    const bool bf16 = x_dtype == FP8MP_BF16;
    const int db16 = dbias_dtype == FP8MP_BF16 ? 1 : 0;
    if (fmt == FP8MP_E4M3)
        return bf16 ? launch_dbias_typed<FP8MP_E4M3, true>(x, rows, cols, scale, out, out_t, amax, dbias, db16, ws, s, dev)
                    : launch_dbias_typed<FP8MP_E4M3, false>(x, rows, cols, scale, out, out_t, amax, dbias, db16, ws, s, dev);
    return bf16 ? launch_dbias_typed<FP8MP_E5M2, true>(x, rows, cols, scale, out, out_t, amax, dbias, db16, ws, s, dev)
                : launch_dbias_typed<FP8MP_E5M2, false>(x, rows, cols, scale, out, out_t, amax, dbias, db16, ws, s, dev);
}

int launch_quantize(const void *x, int x_dtype, int64_t rows, int64_t cols, int fmt, const float *scale,
                    uint8_t *out, uint8_t *out_t, float *amax, cudaStream_t s, const DeviceInfo &, bool early) {
    const bool bf16 = x_dtype == FP8MP_BF16;
    if (early) {
        if (fmt == FP8MP_E4M3)
            return bf16 ? launch_typed<FP8MP_E4M3, true, true>(x, rows, cols, scale, out, out_t, amax, s)
                        : launch_typed<FP8MP_E4M3, false, true>(x, rows, cols, scale, out, out_t, amax, s);
        return bf16 ? launch_typed<FP8MP_E5M2, true, true>(x, rows, cols, scale, out, out_t, amax, s)
                    : launch_typed<FP8MP_E5M2, false, true>(x, rows, cols, scale, out, out_t, amax, s);
    }
    if (fmt == FP8MP_E4M3)
        return bf16 ? launch_typed<FP8MP_E4M3, true, false>(x, rows, cols, scale, out, out_t, amax, s)
                    : launch_typed<FP8MP_E4M3, false, false>(x, rows, cols, scale, out, out_t, amax, s);
    return bf16 ? launch_typed<FP8MP_E5M2, true, false>(x, rows, cols, scale, out, out_t, amax, s)
                : launch_typed<FP8MP_E5M2, false, false>(x, rows, cols, scale, out, out_t, amax, s);
}

int read_and_clear_cast_timeout_flag(unsigned int *value) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_cast_timeout_flag, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_cast_timeout_flag, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "reading the timeout flag failed: %s", cudaGetErrorString(e));
    *value = v;
    return FP8MP_OK;
}

}  // namespace fp8mp
