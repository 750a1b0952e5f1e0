// gemm.cu -- FP8 x FP8 -> fp32-accumulated GEMM on the sm_103a tensor cores
// (tcgen05 + TMEM + TMA), the engine of the forward, dgrad and wgrad GEMMs
// of the FP8 linear layer.
//
// Pages: "Các kiểu dữ liệu FP8 gốc của PyTorch ..." (hotroai.com), the
// torch._scaled_mm listing (two FP8 operands with their scales, a bias, the
// output and its amax); "LLM) Mixed-Precision 개념 및 학습 방법 알아보기"
// (data-newbie.tistory.com) "Accumulation into FP32" (products accumulated in
// single precision, converted on the way out); "Как работает FP8
// quantization на H100 (Transformer Engine)?" (aivaro.ru) section 3, step 4
// (the GEMM result is divided by the scaling factors); "Transformer
// Engine으로 FP8 사용하기" (coniverse.tistory.com) "Introduction to FP8" and
// "FP8 사용방안(recipe)" (HYBRID: E5M2 gradients against E4M3 operands).
//
// Computes out[i, j] = (sum_k A[i, k] * B[j, k]) * sinv_a * sinv_b + bias[j]
// with A (rows_a x kc) and B (rows_b x kc) both contiguous along k. One
// launch runs one such GEMM, or two independent ones (the dgrad and wgrad
// GEMMs of a backward pass) whose tiles share the persistent grid.
//
// Two tile engines share this file:
//   PAIR = true  -- a cluster of two CTAs on the two SMs of a TPC computes a
//                   256 x 256 tile with tcgen05.mma.cta_group::2 (M 256,
//                   N 256, K 32): each CTA stages its own 128 rows of A and
//                   its own 128 rows of B (32 KB per 128-byte k-block, a
//                   6-stage ring); the even CTA issues the MMAs, which read
//                   both CTAs' shared memory and write 128 TMEM lanes in each
//                   CTA. Staging half of B per SM cuts the shared-memory
//                   traffic per MMA by a third against a 128 x 256 tile.
//   PAIR = false -- one CTA computes a 128 x 256 tile with
//                   tcgen05.mma.cta_group::1 (4-stage, 48 KB ring); used when
//                   a problem has too few 256 x 256 tiles to fill the GPU.
// In both, one CTA per SM runs persistently over tiles, dealt one per
// cluster per round in serpentine order (longest contraction first):
//   warp 0, one lane  : TMA producer (128-byte-swizzled boxes), waits on the
//                       stage's empty mbarrier, arms / signals its full one;
//   warp 1, one lane  : MMA issuer (even CTA only with PAIR), 4 MMAs per
//                       stage, tcgen05.commit frees the stage (multicast to
//                       both CTAs with PAIR); two TMEM accumulators of 256
//                       columns let the next tile's mainloop overlap the
//                       previous tile's epilogue;
//   warps 2-5         : epilogue -- tcgen05.ld of the warp's 32 TMEM lanes,
//                       y = acc * (sinv_a * sinv_b) + bias, rounding to the
//                       output type into 128-byte-swizzled staging boxes in
//                       shared memory, one TMA bulk store per 32-row box,
//                       running max |y|; one atomic max per warp at the end.
// Every mbarrier wait sleeps in mbarrier.try_wait and is bounded (about 2 s
// of SM clock cycles, read with clock64); on expiry the thread raises a
// device flag that fp8mp_check() reports, tells the other roles of its CTA
// to stop, waits (bounded) for its own copies / MMAs in flight, and the CTA
// frees its TMEM and returns.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fp8mp_async.cuh"

namespace fp8mp {

__device__ unsigned int g_gemm_timeout_flag = 0;

namespace {

constexpr int BK = 128;           // bytes of k per stage = one 128-byte swizzle row
constexpr int UMMA_K = 32;        // k of one kind::f8f6f4 MMA (32 bytes)
constexpr int TILE_N = 256;       // output columns per tile (TMEM columns per accumulator)
constexpr int ROWS_A = 128;       // rows of A each CTA stages (TMEM lanes)
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int GROUP_M = 16;       // tile raster: at most 16 row-blocks per group
constexpr uint32_t TMEM_COLS = 2 * TILE_N;

template <bool PAIR>
struct Cfg {
    static constexpr int TILE_M = PAIR ? 256 : 128;   // output rows per tile
    static constexpr int ROWS_B = PAIR ? 128 : 256;   // rows of B each CTA stages
    static constexpr int STAGES = PAIR ? 6 : 4;
    static constexpr int A_BYTES = ROWS_A * BK;
    static constexpr int B_BYTES = ROWS_B * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TX_BYTES = PAIR ? 2 * STAGE_BYTES : STAGE_BYTES;  // bytes one full phase waits for
    // output staging: per epilogue warp two 32-row x 128-byte boxes (4 KB each)
    static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int EPI_BOX_BYTES = 32 * 128;
    static constexpr int EPI_BYTES = NUM_EPI_WARPS * 2 * EPI_BOX_BYTES;
    static constexpr int BAR_OFFSET = EPI_OFFSET + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tmem_full[2], tmem_empty[2], drain
    static constexpr int SLOT_OFFSET = BAR_OFFSET + NUM_BARS * 8;
    static constexpr int FLAG_OFFSET = SLOT_OFFSET + 8;
    static constexpr int SMEM_USED = FLAG_OFFSET + 8;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
    static constexpr uint32_t TEMPTY_COUNT = PAIR ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS;
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct GemmParams {
    int rows_a, rows_b, num_kb;
    int tiles_m, tiles_n;
    int group_m;              // tile raster: row-blocks per group, or
    int group_n;              //   when group_n > 0, column-blocks per group
    int a_mn, b_mn;           // operand stored MN-major ([kc x rows], contiguous along M / N)
    uint32_t idesc;           // tcgen05 instruction descriptor (operand formats, majors, M, N)
    const float *sinv_a, *sinv_b;
    const void *bias;
    int bias_bf16;
    void *out;
    int out_bf16;
    int out_fp8;              // output as FP8 codes of out_fmt under *out_scale
    int out_fmt;
    const float *out_scale;
    float *out_amax;
    int32_t *out_nonfinite;   // bf16 / fp32 output: |= 1 when a stored element is Inf or NaN
    int signal_parts;         // > 0: stored tile parts to count in *out_nonfinite before kDoneBit
};

// One GEMM of a launch: its operand and output tensor maps and parameters.
struct GemmProblem {
    CUtensorMap ta, tb, to;
    GemmParams p;
};

// Up to two independent GEMMs share one launch (the dgrad and wgrad GEMMs of
// a layer's backward pass). Their tiles form one list, problem 0's first;
// the host puts the problem with the longer contraction first.
constexpr int MAX_PROBLEMS = 2;
struct GemmBatch {
    GemmProblem prob[MAX_PROBLEMS];
    int nprob;
    int tiles0;     // tiles of problem 0; problem 1's follow
    int num_tiles;  // tiles of all problems
};

// ------------------------------------------------------------ PTX wrappers

// Arrive on an mbarrier given by its shared::cluster address (any CTA of the cluster).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// The shared bounded wait, reporting through the GEMM's timeout flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    return fp8mp::wait_bounded(bar, parity, abort_flag, &g_gemm_timeout_flag);
}

// TMA 2-D tile load into this CTA's shared memory; completion is counted on
// the mbarrier at shared::cluster address `bar` (with PAIR it may sit in the
// peer CTA of the pair).
template <bool PAIR>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t c0,
                                            int32_t c1) {
    if constexpr (PAIR)
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
            : "memory");
}
// TMA 2-D tile store from this CTA's shared memory (rows / columns outside
// the tensor are not written), tracked as a bulk async-group of the thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most one bulk group of this thread still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    if constexpr (PAIR)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                     : "memory");
}
template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (PAIR)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <bool PAIR>
__device__ __forceinline__ void umma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    if constexpr (PAIR)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}
// Arrive once on `bar` when all MMAs this thread issued so far complete: in
// this CTA (PAIR = false), or at the same offset in both CTAs of the pair.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_all(uint32_t bar) {
    if constexpr (PAIR) {
        const uint16_t mask = 0x3;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"(mask)
            : "memory");
    } else {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    }
}
// Arrive once on this CTA's `bar` when the MMAs issued so far complete.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
    if constexpr (PAIR)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (lane i of the
// warp gets TMEM lane base+i); the wait is in the same asm so the registers
// are valid when it returns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): 8-row atoms of 1024 bytes stacked along M/N.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address, bits 0-13
    d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused here), bits 16-29
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset: one 8-row atom, bits 32-45
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version for tcgen05, bits 46-47
    d |= static_cast<uint64_t>(2u) << 61;                 // swizzle mode: 128 bytes, bits 61-63
    return d;
}

// Shared-memory matrix descriptor of an MN-major operand tile: one
// 128-byte row of 128 M/N elements per k (the layout TMA writes for a box
// whose inner dimension runs along M/N, with CU_TENSOR_MAP_SWIZZLE_128B),
// 8-row atoms of 1024 bytes stacked along k. The stride byte offset is the
// step between those 8-row groups along k; the leading byte offset is the
// step between 128-element atoms along M/N (a 256-wide tile is staged as
// two 128-wide halves `lbo` bytes apart; a 128-wide tile has one atom).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address, bits 0-13
    d |= static_cast<uint64_t>(lbo >> 4) << 16;           // leading byte offset: next M/N atom, bits 16-29
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset: next 8 k-rows, bits 32-45
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version for tcgen05, bits 46-47
    d |= static_cast<uint64_t>(2u) << 61;                 // swizzle mode: 128 bytes, bits 61-63
    return d;
}

// Tile of round `r` for cluster `c` of `nc`: one tile per cluster per round,
// dealt forwards in even rounds and backwards in odd ones (serpentine). With
// the tiles sorted by contraction length, longest first, the clusters that
// got the last long tiles get the first short ones, which keeps the
// per-cluster sums of k-blocks within one short tile of each other.
__device__ __forceinline__ int serpentine_tile(int r, int c, int nc) {
    return r * nc + ((r & 1) ? nc - 1 - c : c);
}

// The problem a tile of the batch belongs to, and its index within it.
__device__ __forceinline__ int tile_problem(const GemmBatch &b, int t, int &local) {
    if (t < b.tiles0) {
        local = t;
        return 0;
    }
    local = t - b.tiles0;
    return 1;
}

// Tile index -> (row-block of A, row-block of B), grouped so that the CTAs
// working at the same time share group_m A panels and a few B panels in L2
// (row-block fastest within a group); with group_n > 0 the other way round:
// groups of group_n B panels, column-block fastest, every A panel streamed
// past them once per group.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int group_n, int &mb,
                                            int &nb) {
    if (group_n > 0) {
        const int group = group_n * tiles_m;
        const int g = t / group;
        const int first = g * group_n;
        const int gn = min(tiles_n - first, group_n);
        const int local = t - g * group;
        nb = first + local % gn;
        mb = local / gn;
        return;
    }
    const int group = group_m * tiles_n;
    const int g = t / group;
    const int first = g * group_m;
    const int gm = min(tiles_m - first, group_m);
    const int local = t - g * group;
    mb = first + local % gm;
    nb = local / gm;
}

// A bf16 pair with an all-ones exponent field in either half (Inf or NaN).
__device__ __forceinline__ bool has_nonfinite_bf16x2(uint32_t w) {
    const uint32_t t = (w & 0x7F807F80u) ^ 0x7F807F80u;
    return (t & 0xFFFFu) == 0u || (t >> 16) == 0u;
}

// max |v[j]| over 16 values as a pairwise tree (depth 4 instead of a chain
// of 16); fmaxf ignores a NaN operand, so the result is the max of the
// non-NaN |v| (or NaN when all are NaN, which fmaxf(am, .) then ignores).
__device__ __forceinline__ float abs_max16(const float (&v)[16]) {
    float t[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1]));
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = fmaxf(t[2 * j], t[2 * j + 1]);
    return fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// ------------------------------------------------------------------ kernel

template <bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_fp8_kernel(const __grid_constant__ GemmBatch batch) {
    using C = Cfg<PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint32_t base = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    base += pad;

    const uint32_t bar0 = base + C::BAR_OFFSET;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SLOT_OFFSET);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::FLAG_OFFSET);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // 0 = the CTA that issues the MMAs
    const int cluster_id = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int num_clusters = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), C::TEMPTY_COUNT);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int i = 0; i < batch.nprob; ++i) {
            prefetch_tmap(&batch.prob[i].ta);
            prefetch_tmap(&batch.prob[i].tb);
            prefetch_tmap(&batch.prob[i].to);
        }
    }
    if (warp == 1) {
        tmem_alloc<PAIR>(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish<PAIR>();
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync_all();  // the peer's barriers are initialised before anyone signals them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // everything above touched only this CTA's shared memory and TMEM: it
    // overlaps the previous kernel's tail; global memory waits for its end
    pdl_wait();

    const int num_tiles = batch.num_tiles;
    const int rounds = (num_tiles + num_clusters - 1) / num_clusters;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs of a pair)
            // The next kernel on the stream may be scheduled from now on: an
            // ordinary one waits in griddepcontrol.wait for this grid to
            // complete; one whose buffers this launch does not touch (a cast
            // enqueued with FP8MP_OVERLAP_PREVIOUS) runs in the registers and
            // threads this CTA leaves free, during the mainloop.
            pdl_launch_dependents();
            uint32_t it = 0;
            int issued_stages = 0;
            bool ok = true;
            for (int r = 0; ok && r < rounds; ++r) {
                const int tile = serpentine_tile(r, cluster_id, num_clusters);
                if (tile >= num_tiles) continue;
                int local;
                const GemmProblem &P = batch.prob[tile_problem(batch, tile, local)];
                int mb, nb;
                tile_coords(local, P.p.tiles_m, P.p.tiles_n, P.p.group_m, P.p.group_n, mb, nb);
                const int a_row = mb * C::TILE_M + static_cast<int>(rank) * ROWS_A;
                const int b_row = nb * TILE_N + static_cast<int>(rank) * C::ROWS_B;
                const int num_kb = P.p.num_kb;
                const int a_mn = P.p.a_mn, b_mn = P.p.b_mn;
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int s = static_cast<int>(it % C::STAGES);
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * C::STAGE_BYTES;
                    // the full barrier of a pair lives in the MMA-issuing CTA
                    const uint32_t fb = PAIR ? mapa_shared(full_bar(s), 0) : full_bar(s);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(s), C::TX_BYTES);
                    // K-major: box of rows x 128 bytes of k at (k, row); MN-major:
                    // box of 128 k-rows x 128 bytes of M/N at (row, k)
                    if (a_mn)
                        tma_load_2d<PAIR>(sa, &P.ta, fb, a_row, kb * BK);
                    else
                        tma_load_2d<PAIR>(sa, &P.ta, fb, kb * BK, a_row);
                    if (!b_mn) {
                        tma_load_2d<PAIR>(sa + C::A_BYTES, &P.tb, fb, kb * BK, b_row);
                    } else {
#pragma unroll
                        for (int h = 0; h < C::ROWS_B / 128; ++h)
                            tma_load_2d<PAIR>(sa + C::A_BYTES + h * (BK * 128), &P.tb, fb, b_row + 128 * h, kb * BK);
                    }
                    if (issued_stages < C::STAGES) ++issued_stages;
                }
            }
            if (!ok && rank == 0) {
                // let the loads already issued land before the CTA goes away
                for (int j = 1; j <= issued_stages && j <= static_cast<int>(it); ++j) {
                    const uint32_t last = it - static_cast<uint32_t>(j);
                    volatile int never = 0;
                    wait_bounded(full_bar(static_cast<int>(last % C::STAGES)), (last / C::STAGES) & 1u, &never);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer
            uint32_t it = 0;
            int lt = 0;
            bool ok = true;
            for (int r = 0; ok && r < rounds; ++r) {
                const int tile = serpentine_tile(r, cluster_id, num_clusters);
                if (tile >= num_tiles) continue;
                int local;
                const GemmProblem &P = batch.prob[tile_problem(batch, tile, local)];
                const uint32_t idesc = P.p.idesc;
                const int num_kb = P.p.num_kb;
                const int a_mn = P.p.a_mn, b_mn = P.p.b_mn;
                const int acc = lt & 1;
                const uint32_t aph = (static_cast<uint32_t>(lt) >> 1) & 1u;
                ++lt;
                if (!wait_bounded(tempty_bar(acc), aph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * TILE_N);
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int s = static_cast<int>(it % C::STAGES);
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    if (!wait_bounded(full_bar(s), ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * C::STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        // the k-th 32-element slice: 32 bytes into each K-major row,
                        // or 32 rows (4 KB) into an MN-major tile
                        const uint32_t a_addr = sa + (a_mn ? k * UMMA_K * 128 : k * UMMA_K);
                        const uint32_t b_addr = sa + C::A_BYTES + (b_mn ? k * UMMA_K * 128 : k * UMMA_K);
                        const uint64_t a_desc = a_mn ? sw128_mnmajor_desc(a_addr, 1024u) : sw128_kmajor_desc(a_addr);
                        const uint64_t b_desc =
                            b_mn ? sw128_mnmajor_desc(b_addr, C::ROWS_B > 128 ? BK * 128u : 1024u)
                                 : sw128_kmajor_desc(b_addr);
                        umma_f8f6f4<PAIR>(d_tmem, a_desc, b_desc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit_all<PAIR>(empty_bar(s));
                }
                if (!ok) break;
                umma_commit_all<PAIR>(tfull_bar(acc));
            }
            if (!ok) {
                // wait for the MMAs in flight before TMEM is released
                umma_commit_local<PAIR>(drain_bar);
                volatile int never = 0;
                wait_bounded(drain_bar, 0u, &never);
            }
        }
    } else {
        // ---------------- epilogue warps (both CTAs of a pair)
        // Each warp drains its 32 TMEM lanes (32 output rows) in chunks of
        // 128 bytes per row (64 bf16, 32 fp32 or 128 FP8 columns): tcgen05.ld,
        // scale, bias and rounding in registers, the row written into a
        // 128-byte-swizzled 32 x 128 B staging box, then one TMA store per
        // box. Two boxes per warp alternate so the next chunk overlaps the
        // store; they alternate by committed store, not by chunk, because a
        // chunk past a ragged edge stores nothing (and commits no bulk group),
        // and "at most one group still reading" only protects the box the
        // newest group does not read.
        const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
        const int row_in_tile = static_cast<int>(rank) * ROWS_A + q * 32 + lane;
        const uint32_t stage_box = base + C::EPI_OFFSET + static_cast<uint32_t>((warp - 2) * 2 * C::EPI_BOX_BYTES);
        float am0 = 0.0f, am1 = 0.0f;  // max |y| of problem 0 / 1
        bool bad0 = false, bad1 = false;  // a stored element of problem 0 / 1 is Inf or NaN
        int lt = 0;
        uint32_t stored = 0;  // TMA stores this warp has committed
        for (int r = 0; r < rounds; ++r) {
            const int tile = serpentine_tile(r, cluster_id, num_clusters);
            if (tile >= num_tiles) continue;
            int local;
            const int pi = tile_problem(batch, tile, local);
            const GemmProblem &P = batch.prob[pi];
            const int acc = lt & 1;
            const uint32_t aph = (static_cast<uint32_t>(lt) >> 1) & 1u;
            ++lt;
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), aph, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const float scale = __fmul_rn(__ldg(P.p.sinv_a), __ldg(P.p.sinv_b));
            const int out_fp8 = P.p.out_fp8, out_bf16 = P.p.out_bf16, out_fmt = P.p.out_fmt;
            const int box_cols = out_fp8 ? 128 : (out_bf16 ? 64 : 32);  // 128 bytes per row either way
            const int parts = box_cols / 32;                             // tcgen05.ld of 32 columns each
            const float out_scale = out_fp8 ? __ldg(P.p.out_scale) : 1.0f;
            const void *bias = P.p.bias;
            const int bias_bf16 = P.p.bias_bf16;
            const int rows_a = P.p.rows_a, rows_b = P.p.rows_b;
            int mb, nb;
            tile_coords(local, P.p.tiles_m, P.p.tiles_n, P.p.group_m, P.p.group_n, mb, nb);
            const int64_t m = static_cast<int64_t>(mb) * C::TILE_M + row_in_tile;
            const bool row_ok = m < rows_a;
            const int warp_row0 = mb * C::TILE_M + static_cast<int>(rank) * ROWS_A + q * 32;
            const bool scan_out = P.p.out_nonfinite != nullptr && !out_fp8 && row_ok;
            float am = 0.0f;
            bool bad = false;
#pragma unroll 1
            for (int c = 0; c < TILE_N; c += box_cols) {
                uint32_t packed[32];  // this lane's 128-byte row of the box
#pragma unroll
                for (int half = 0; half < 4; ++half) {
                    if (half >= parts) break;
                    uint32_t r32[32];
                    const int c32 = c + 32 * half;
                    tmem_ld32(tmem_base + static_cast<uint32_t>(acc * TILE_N + c32) +
                                  (static_cast<uint32_t>(q * 32) << 16),
                              r32);
#pragma unroll
                    for (int g = 0; g < 2; ++g) {  // 16-column groups
                        const int n = nb * TILE_N + c32 + 16 * g;
                        const bool col_ok = n < rows_b;
                        float y[16];
                        if (bias == nullptr || !col_ok) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) y[j] = __fmul_rn(__uint_as_float(r32[16 * g + j]), scale);
                        } else if (bias_bf16) {
                            const uint4 *bp = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(bias) + n);
                            const uint4 b0 = __ldg(bp), b1 = __ldg(bp + 1);
                            const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                y[2 * j] = __fmaf_rn(__uint_as_float(r32[16 * g + 2 * j]), scale,
                                                     __uint_as_float(bw[j] << 16));
                                y[2 * j + 1] = __fmaf_rn(__uint_as_float(r32[16 * g + 2 * j + 1]), scale,
                                                         __uint_as_float(bw[j] & 0xFFFF0000u));
                            }
                        } else {
                            const float4 *bp = reinterpret_cast<const float4 *>(static_cast<const float *>(bias) + n);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float4 bb = __ldg(bp + j);
                                y[4 * j] = __fmaf_rn(__uint_as_float(r32[16 * g + 4 * j]), scale, bb.x);
                                y[4 * j + 1] = __fmaf_rn(__uint_as_float(r32[16 * g + 4 * j + 1]), scale, bb.y);
                                y[4 * j + 2] = __fmaf_rn(__uint_as_float(r32[16 * g + 4 * j + 2]), scale, bb.z);
                                y[4 * j + 3] = __fmaf_rn(__uint_as_float(r32[16 * g + 4 * j + 3]), scale, bb.w);
                            }
                        }
                        if (row_ok && col_ok) am = fmaxf(am, abs_max16(y));
                        if (out_fp8) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float a0 = __fmul_rn(y[4 * j], out_scale), a1 = __fmul_rn(y[4 * j + 1], out_scale);
                                const float a2 = __fmul_rn(y[4 * j + 2], out_scale), a3 = __fmul_rn(y[4 * j + 3], out_scale);
                                packed[8 * half + 4 * g + j] = out_fmt == FP8MP_E4M3 ? cvt_quad<FP8MP_E4M3>(a0, a1, a2, a3)
                                                                                    : cvt_quad<FP8MP_E5M2>(a0, a1, a2, a3);
                            }
                        } else if (out_bf16) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) packed[16 * half + 8 * g + j] = pack_bf16x2(y[2 * j], y[2 * j + 1]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) packed[16 * g + j] = __float_as_uint(y[j]);
                        }
                    }
                }
                // the overflow check of the values as stored (rows past the output
                // are skipped; columns past it hold zeros from the zero-filled operand)
                if (scan_out) {
                    if (out_bf16) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) bad |= has_nonfinite_bf16x2(packed[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) bad |= (packed[j] & 0x7F800000u) == 0x7F800000u;
                    }
                }
                // boxes that start outside the output (ragged last tiles) are
                // neither staged nor stored
                if (nb * TILE_N + c >= rows_b || warp_row0 >= rows_a) continue;
                // the staging box of the store before last must have been read
                const uint32_t box = stage_box + (stored & 1u) * C::EPI_BOX_BYTES;
                if (lane == 0 && stored >= 2) bulk_wait_read_le1();
                __syncwarp();
                const uint32_t row_addr = box + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                                 packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&P.to, box, nb * TILE_N + c, warp_row0);
                    bulk_commit_group();
                }
                ++stored;
            }
            if (pi == 0) {
                am0 = max_ignore_nan(am0, am);
                bad0 |= bad;
            } else {
                am1 = max_ignore_nan(am1, am);
                bad1 |= bad;
            }
            if (P.p.signal_parts > 0) {
                // this warp's part of the tile is stored: its flag first, then
                // its count, once the stores are complete and visible
                const bool bad_part = __any_sync(0xffffffffu, bad);
                if (lane == 0) {
                    bulk_wait_all();
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __threadfence();
                    if (bad_part) atomicOr(P.p.out_nonfinite, 1);
                    const uint32_t old =
                        atomicAdd(reinterpret_cast<unsigned int *>(P.p.out_nonfinite), 1u << kPartShift);
                    if (((old >> kPartShift) & kPartMask) + 1u == static_cast<uint32_t>(P.p.signal_parts)) {
                        __threadfence();
                        atomicOr(reinterpret_cast<unsigned int *>(P.p.out_nonfinite), kDoneBit);
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));  // the MMA issuer's barrier
                else
                    mbar_arrive(tempty_bar(acc));
            }
        }
        if (lane == 0) bulk_wait_all();  // stores done before the CTA's shared memory goes away
        for (int i = 0; i < batch.nprob; ++i) {
            const GemmParams &pp = batch.prob[i].p;
            // (a signalling problem flagged each part before counting it: the
            // word's consumer may already have reset it by now)
            if (pp.out_nonfinite != nullptr && pp.signal_parts == 0 &&
                __any_sync(0xffffffffu, i == 0 ? bad0 : bad1) && lane == 0)
                atomicOr(pp.out_nonfinite, 1);
            if (pp.out_amax == nullptr) continue;
            float a = warp_max(i == 0 ? am0 : am1);
            if (pp.out_bf16 && !pp.out_fp8) a = __bfloat162float(__float2bfloat16_rn(a));  // max of the stored values
            if (lane == 0) atomicMax(reinterpret_cast<int *>(pp.out_amax), __float_as_int(a));
        }
    }

    __syncwarp();
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync_all();  // no CTA leaves while its peer may still touch its shared memory
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
}

// Diagnostic of the failure path: one thread waits, with the same bounded
// wait the GEMM roles use, on an mbarrier that nothing ever signals. The wait
// gives up after kWaitLimitCycles and raises the device timeout flag; the
// kernel then returns normally.
__global__ void timeout_selftest_kernel() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0u, &abort_flag);
}

// out = bias (or 0) broadcast over rows: the GEMM of an empty contraction.
__global__ void fill_bias_kernel(int64_t rows, int64_t cols, const void *bias, int bias_bf16, void *out,
                                 int out_bf16, float *out_amax, const float *out_scale, int out_fmt) {
    pdl_wait();
    pdl_launch_dependents();
    float am = 0.0f;
    const int64_t n = rows * cols;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = i % cols;
        float y = 0.0f;
        if (bias != nullptr)
            y = bias_bf16 ? bf16_bits_to_f32(static_cast<const uint16_t *>(bias)[j]) : static_cast<const float *>(bias)[j];
        if (out_scale != nullptr) {
            const float a = __fmul_rn(y, *out_scale);
            static_cast<uint8_t *>(out)[i] = static_cast<uint8_t>(
                (out_fmt == FP8MP_E4M3 ? cvt_pair<FP8MP_E4M3>(a, 0.0f) : cvt_pair<FP8MP_E5M2>(a, 0.0f)) & 0xFFu);
        } else if (out_bf16) {
            const __nv_bfloat16 h = __float2bfloat16_rn(y);
            static_cast<__nv_bfloat16 *>(out)[i] = h;
            y = __bfloat162float(h);
        } else {
            static_cast<float *>(out)[i] = y;
        }
        am = max_ignore_nan(am, fabsf(y));
    }
    block_amax_atomic(am, out_amax);
}

// ------------------------------------------------------------- host side

// Output tensor [rows x cols] of bf16, fp32 or FP8 bytes, box 32 rows x 128
// bytes, 128-byte swizzle.
int make_out_tmap(CUtensorMap *map, void *ptr, uint64_t cols, uint64_t rows, bool bf16, bool fp8 = false) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return fail(FP8MP_ERR_LAUNCH, "cuTensorMapEncodeTiled is not available");
    const uint64_t esize = fp8 ? 1 : (bf16 ? 2 : 4);
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map,
                           fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                               : (bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32),
                           2, ptr,
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FP8MP_ERR_LAUNCH, "cuTensorMapEncodeTiled (output) failed (%d)", static_cast<int>(r));
    return FP8MP_OK;
}

// 2-D byte tensor [outer x inner], inner contiguous; box box_outer x 128 bytes.
// A K-major operand has inner = kc, outer = its rows (box: the tile's rows);
// an MN-major one has inner = its rows, outer = kc (box: 128 k-rows).
int make_tmap(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return fail(FP8MP_ERR_LAUNCH, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP8MP_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return FP8MP_OK;
}

// Row-blocks per raster group of a problem with contraction length kc: as
// many A panels (tile_m rows x kc bytes) as fit in 32 MB, at most GROUP_M.
// Long contractions (the MLP's 14336- and 16384-long ones) get groups of 8-9
// row-blocks, the others stay at 16: measured, the MLP-down forward launch
// 560 against 588 us, the other workload shapes within noise.
int raster_group(int64_t kc, int tile_m) {
    const int64_t panel = static_cast<int64_t>(tile_m) * kc;
    int64_t g = (32ll << 20) / (panel > 0 ? panel : 1);
    if (g > GROUP_M) g = GROUP_M;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

// Which way to group the raster of a problem whose operands do not fit in
// L2 together (more than 64 MB): the DRAM bytes each order needs when the
// group's panels stay in L2 and the other operand streams past them are
// about A + ceil(tiles_m / gm) * B (row-block groups, B read once per
// group) and B + ceil(tiles_n / gn) * A (column-block groups); the order
// with fewer is taken. Returns group_n, 0 for row-block groups. The MLP's
// backward GEMMs and its down projection's forward stream their 235 MB
// operand twice instead of re-reading the 59-67 MB one 7-8 times.
int raster_columns(int64_t rows_a, int64_t rows_b, int64_t kc, int tiles_m, int tiles_n, int gm) {
    const int64_t a = rows_a * kc, b = rows_b * kc;
    if (a + b <= (64ll << 20)) return 0;
    const int gn = raster_group(kc, TILE_N);
    const int64_t by_rows = a + ((tiles_m + gm - 1) / gm) * b;
    const int64_t by_cols = b + ((tiles_n + gn - 1) / gn) * a;
    return by_cols < by_rows ? gn : 0;
}

constexpr uint32_t make_idesc(int fmt_a, int fmt_b, int m, int a_mn, int b_mn) {
    return (1u << 4)                                    // accumulator: f32
           | (static_cast<uint32_t>(fmt_a) << 7)        // A: 0 = E4M3, 1 = E5M2
           | (static_cast<uint32_t>(fmt_b) << 10)       // B: 0 = E4M3, 1 = E5M2
           | (static_cast<uint32_t>(a_mn) << 15)        // A: 0 = K-major, 1 = MN-major
           | (static_cast<uint32_t>(b_mn) << 16)        // B: 0 = K-major, 1 = MN-major
           | (static_cast<uint32_t>(TILE_N >> 3) << 17) // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);     // M / 16
}

// Per device: the kernels' shared-memory attribute set and the SM-pair
// engine's resident cluster count, done once; `ready` is published after the
// data (release) and checked before reading it (acquire).
struct PerDevice {
    std::atomic<bool> ready[2];
    int max_pairs = 0;
};
PerDevice g_dev[64];
std::mutex g_dev_mutex;

template <bool PAIR>
int launch_engine(const GemmBatch &batch, int grid, cudaStream_t s) {
    using C = Cfg<PAIR>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = s;
    cfg.attrs = attr;
    if (PAIR) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = 2;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_fp8_kernel<PAIR>, batch);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "GEMM launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

template <bool PAIR>
int prepare_engine(const DeviceInfo &dev) {
    using C = Cfg<PAIR>;
    PerDevice &pd = g_dev[dev.device & 63];
    if (pd.ready[PAIR].load(std::memory_order_acquire)) return FP8MP_OK;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (pd.ready[PAIR].load(std::memory_order_relaxed)) return FP8MP_OK;
    cudaError_t e =
        cudaFuncSetAttribute(gemm_fp8_kernel<PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "GEMM smem attribute failed: %s", cudaGetErrorString(e));
    if (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(static_cast<unsigned>(dev.num_sms & ~1));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = C::SMEM_ALLOC;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_fp8_kernel<true>, &cfg);
        if (e != cudaSuccess || n < 1) n = dev.num_sms / 2;
        pd.max_pairs = n;
    }
    pd.ready[PAIR].store(true, std::memory_order_release);
    return FP8MP_OK;
}

}  // namespace

int gemm_warp_registers(int *warps) {
    static std::atomic<int> cached{0};
    *warps = NUM_THREADS / 32;
    int r = cached.load(std::memory_order_relaxed);
    if (r > 0) return r;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, gemm_fp8_kernel<true>) != cudaSuccess) return 0;
    r = 32 * ((fa.numRegs + 7) & ~7);
    cached.store(r, std::memory_order_relaxed);
    return r;
}

int launch_gemms(const GemmDesc *descs, int n, cudaStream_t s, const DeviceInfo &dev) {
    if (n < 1 || n > MAX_PROBLEMS) return fail(FP8MP_ERR_INVALID, "a GEMM launch takes 1 or 2 problems");
    const GemmDesc *work[MAX_PROBLEMS];
    int nw = 0;
    for (int i = 0; i < n; ++i) {
        const GemmDesc &d = descs[i];
        if (d.rows_a == 0 || d.rows_b == 0) continue;
        if (d.rows_a > (1ll << 30) || d.rows_b > (1ll << 30) || d.kc > (1ll << 30))
            return fail(FP8MP_ERR_INVALID, "GEMM dimension above 2^30");
        if (d.kc == 0) {
            int64_t blocks = (d.rows_a * d.rows_b + 255) / 256;
            if (blocks > dev.num_sms * 8) blocks = dev.num_sms * 8;
            const cudaError_t e = launch_kernel(fill_bias_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                                s, d.rows_a, d.rows_b, d.bias, d.bias_dtype == FP8MP_BF16 ? 1 : 0,
                                                d.out, d.out_dtype == FP8MP_BF16 ? 1 : 0, d.out_amax, d.out_scale,
                                                d.out_fmt);
            if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "GEMM fill launch failed: %s", cudaGetErrorString(e));
            if (d.signal_done && d.out_nonfinite != nullptr) {  // the filled output is complete
                const cudaError_t e2 = launch_signal_done(d.out_nonfinite, s);
                if (e2 != cudaSuccess)
                    return fail(FP8MP_ERR_LAUNCH, "GEMM signal launch failed: %s", cudaGetErrorString(e2));
            }
            continue;
        }
        work[nw++] = &d;
    }
    if (nw == 0) return FP8MP_OK;
    // longest contraction first: the serpentine deal then balances the
    // clusters' k-blocks (see serpentine_tile)
    if (nw == 2 && work[1]->kc > work[0]->kc) {
        const GemmDesc *t = work[0];
        work[0] = work[1];
        work[1] = t;
    }

    // Pairs of SMs on 256 x 256 tiles when there are enough tiles to occupy
    // most SMs; otherwise single-SM 128 x 256 tiles (twice as many tiles).
    // FP8MP_GEMM_ENGINE=pair|single overrides the choice (used by the tests
    // to run both engines on every shape).
    int64_t pair_tiles = 0;
    for (int i = 0; i < nw; ++i) pair_tiles += ((work[i]->rows_a + 255) / 256) * ((work[i]->rows_b + TILE_N - 1) / TILE_N);
    bool pair = pair_tiles * 2 >= dev.num_sms;
    if (const char *force = std::getenv("FP8MP_GEMM_ENGINE")) {
        if (std::strcmp(force, "pair") == 0) pair = true;
        if (std::strcmp(force, "single") == 0) pair = false;
    }
    int rc = pair ? prepare_engine<true>(dev) : prepare_engine<false>(dev);
    if (rc) return rc;

    GemmBatch batch;
    std::memset(&batch, 0, sizeof batch);
    batch.nprob = nw;
    int64_t tiles = 0;
    for (int i = 0; i < nw; ++i) {
        const GemmDesc &d = *work[i];
        GemmProblem &P = batch.prob[i];
        GemmParams &p = P.p;
        p.rows_a = static_cast<int>(d.rows_a);
        p.rows_b = static_cast<int>(d.rows_b);
        p.num_kb = static_cast<int>((d.kc + BK - 1) / BK);
        p.tiles_n = static_cast<int>((d.rows_b + TILE_N - 1) / TILE_N);
        p.tiles_m = static_cast<int>(pair ? (d.rows_a + 255) / 256 : (d.rows_a + 127) / 128);
        p.group_m = raster_group(d.kc, pair ? 256 : 128);
        p.group_n = raster_columns(d.rows_a, d.rows_b, d.kc, p.tiles_m, p.tiles_n, p.group_m);
        p.a_mn = d.a_mn;
        p.b_mn = d.b_mn;
        p.idesc = make_idesc(d.fmt_a, d.fmt_b, pair ? 256 : 128, d.a_mn, d.b_mn);
        p.sinv_a = d.sinv_a;
        p.sinv_b = d.sinv_b;
        p.bias = d.bias;
        p.bias_bf16 = d.bias_dtype == FP8MP_BF16;
        p.out = d.out;
        p.out_bf16 = d.out_dtype == FP8MP_BF16;
        p.out_fp8 = d.out_scale != nullptr;
        p.out_fmt = d.out_fmt;
        p.out_scale = d.out_scale;
        p.out_amax = d.out_amax;
        p.out_nonfinite = d.out_nonfinite;
        p.signal_parts = 0;
        if (d.signal_done && d.out_nonfinite != nullptr) {
            // each tile is stored in parts by the epilogue warps of its CTA(s)
            const int64_t parts = static_cast<int64_t>(p.tiles_m) * p.tiles_n * (pair ? 2 : 1) * NUM_EPI_WARPS;
            if (parts > static_cast<int64_t>(kPartMask))
                return fail(FP8MP_ERR_INVALID, "GEMM: %lld tile parts are too many to signal completion",
                            static_cast<long long>(parts));
            p.signal_parts = static_cast<int>(parts);
        }
        const uint64_t kc = static_cast<uint64_t>(d.kc);
        const uint64_t ra = static_cast<uint64_t>(d.rows_a), rb = static_cast<uint64_t>(d.rows_b);
        rc = d.a_mn ? make_tmap(&P.ta, d.a, ra, kc, BK) : make_tmap(&P.ta, d.a, kc, ra, ROWS_A);
        if (rc) return rc;
        rc = d.b_mn ? make_tmap(&P.tb, d.b, rb, kc, BK)
                    : make_tmap(&P.tb, d.b, kc, rb, pair ? Cfg<true>::ROWS_B : Cfg<false>::ROWS_B);
        if (rc) return rc;
        rc = make_out_tmap(&P.to, d.out, static_cast<uint64_t>(d.rows_b), static_cast<uint64_t>(d.rows_a),
                           p.out_bf16 != 0, p.out_fp8 != 0);
        if (rc) return rc;
        const int64_t t = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
        if (i == 0) batch.tiles0 = static_cast<int>(t < 0x7FFFFFFF ? t : 0x7FFFFFFF);
        tiles += t;
    }
    if (tiles > 0x7FFFFFFF) return fail(FP8MP_ERR_INVALID, "GEMM has too many tiles");
    batch.num_tiles = static_cast<int>(tiles);

    if (pair) {
        const int max_pairs = g_dev[dev.device & 63].max_pairs;
        const int clusters = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
        return launch_engine<true>(batch, 2 * clusters, s);
    }
    const int grid = static_cast<int>(tiles < dev.num_sms ? tiles : dev.num_sms);
    return launch_engine<false>(batch, grid, s);
}

int launch_gemm(const uint8_t *a, int fmt_a, const uint8_t *b, int fmt_b, int64_t rows_a, int64_t rows_b,
                int64_t kc, const float *sinv_a, const float *sinv_b, const void *bias, int bias_dtype, void *out,
                int out_dtype, float *out_amax, cudaStream_t s, const DeviceInfo &dev, const float *out_scale,
                int out_fmt) {
    const GemmDesc d = {a,    fmt_a,      b,   fmt_b,     rows_a,   rows_b,    kc,     sinv_a,
                        sinv_b, bias, bias_dtype, out, out_dtype, out_amax, out_scale, out_fmt, 0, 0};
    return launch_gemms(&d, 1, s, dev);
}

int launch_timeout_selftest(cudaStream_t s) {
    timeout_selftest_kernel<<<1, 32, 0, s>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "self-test launch failed: %s", cudaGetErrorString(e));
    return FP8MP_OK;
}

int read_and_clear_timeout_flag(unsigned int *value) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_timeout_flag, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_gemm_timeout_flag, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(FP8MP_ERR_LAUNCH, "reading the timeout flag failed: %s", cudaGetErrorString(e));
    *value = v;
    return FP8MP_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace fp8mp
