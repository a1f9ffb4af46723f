// Device building blocks of the shared-memory-staged kernels (rmsnorm_staged.cu,
// layernorm_staged.cu): mbarriers with bounded waits, bulk asynchronous copies from global
// into shared memory, st.async stores into a cluster peer's shared memory, 16-byte shared
// memory loads.
#pragma once

#include "common.cuh"
#include "kernels.h"

// Each translation unit that uses these keeps its own device error word (without relocatable
// device code, device variables do not link across translation units) and reports it
// through a host function that camp_device_errors combines.

namespace camp {
namespace staged {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // one second

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_test, but the thread may be suspended in hardware for up to `hint_ns` while the
// phase is incomplete (it resumes as soon as the phase completes): a waiting warp then
// takes no issue slots from the warps that have work.
__device__ __forceinline__ bool mbar_test_suspend(uint32_t bar, uint32_t parity,
                                                  uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

constexpr uint32_t kSuspendHintNs = 20000;   // per try; the bound below is the real limit

// Wait for the phase of `bar` with this parity to complete; false after `limit_ns`
// nanoseconds (kWaitLimitNs in normal calls).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test_suspend(bar, parity, kSuspendHintNs)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Bulk asynchronous copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// The shared::cluster address of this CTA's shared variable at `addr` in cluster rank `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Store v into a (possibly remote) CTA's shared memory; the write is counted, in bytes, on
// that CTA's mbarrier `bar` (both shared::cluster addresses).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(addr), "r"(__float_as_uint(v)), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ Raw<16> ld_smem16(const unsigned char* p) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    Raw<16> r;
    r.w[0] = q.x;
    r.w[1] = q.y;
    r.w[2] = q.z;
    r.w[3] = q.w;
    return r;
}

// The same from a 32-bit shared-memory address (a shared::cta window offset, as smem_u32
// gives), which takes one register where a generic pointer takes two; ordered as a volatile
// access (the compiler keeps it where it is written).
__device__ __forceinline__ Raw<16> ld_smem16_at(uint32_t addr) {
    Raw<16> r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "r"(addr)
                 : "memory");
    return r;
}

}  // namespace staged
}  // namespace camp
