// fp8mp_async.cuh -- mbarrier and TMA (cp.async.bulk.tensor) wrappers in
// inline PTX for sm_103a, shared by the kernels that stage tiles in shared
// memory with the tensor-memory accelerator (the GEMM and the tiled casts),
// and the host lookup of the tensor-map encoder. Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "fp8mp_internal.cuh"

namespace fp8mp {

constexpr long long kWaitLimitCycles = 4000000000ll;  // about 2 s at the SM clock
constexpr uint32_t kSuspendHintNs = 1000000u;          // longest single sleep inside try_wait

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Tests the phase; if it is not complete the thread sleeps in hardware until
// it completes or kSuspendHintNs pass (no spinning on the issue slots).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Waits until the phase of parity `parity` of `bar` has completed. Returns
// false if another role of the CTA has raised `abort_flag`, or if about
// kWaitLimitCycles SM cycles elapse: then it raises `abort_flag` and ORs 1
// into the kernel's device timeout flag, which fp8mp_check() reports.
static __device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                      unsigned int *timeout_flag) {
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicOr(timeout_flag, 1u);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             unsigned int *timeout_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded_slow(bar, parity, abort_flag, timeout_flag);
}

// TMA 2-D box load into this CTA's shared memory at `dst`, coordinates
// (c0 innermost, c1); completion counted in bytes on the mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d_cta(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t c0,
                                                int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Thread-block clusters: this CTA's rank, the shared::cluster address of the
// variable at local shared address `addr` in CTA `rank`, a load through such
// an address (distributed shared memory), and a barrier over every thread of
// every CTA of the cluster (release / acquire: the shared-memory writes made
// before it are seen by the loads made after it, in any CTA of the cluster;
// all threads of a warp execute it together).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (no link against libcuda); NULL when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace fp8mp
