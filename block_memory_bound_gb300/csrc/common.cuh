// Device-side building blocks shared by the RMSNorm and RoPE kernels: raw vector
// accesses with explicit cache policy, bf16/fp32 unpacking and packing, and warp
// reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace camp {

// ------------------------------------------------------------------ storage types

struct bf16_t {};   // tag: 16-bit brain float, stored as the upper half of an fp32
struct f32_t {};    // tag: IEEE binary32

template <typename S> struct Storage;
template <> struct Storage<bf16_t> { static constexpr int kBytes = 2; };
template <> struct Storage<f32_t> { static constexpr int kBytes = 4; };

// A vector access of BYTES bytes, kept as raw 32-bit words (16-bit for BYTES == 2).
template <int BYTES> struct Raw;
template <> struct Raw<16> { uint32_t w[4]; };
template <> struct Raw<8> { uint32_t w[2]; };
template <> struct Raw<4> { uint32_t w[1]; };
template <> struct Raw<2> { uint16_t h; };

// ------------------------------------------------------------------ global loads
// Streaming loads of x: each element is read once per launch, so it is not kept in L1.
// These are ordinary coherent loads (not the read-only path), which keeps in-place
// calls (y == x) well defined.

template <int BYTES> __device__ __forceinline__ Raw<BYTES> ld_stream(const void* p);

template <> __device__ __forceinline__ Raw<16> ld_stream<16>(const void* p) {
    Raw<16> r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<8> ld_stream<8>(const void* p) {
    Raw<8> r;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(r.w[0]), "=r"(r.w[1])
                 : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<4> ld_stream<4>(const void* p) {
    Raw<4> r;
    asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<2> ld_stream<2>(const void* p) {
    Raw<2> r;
    asm volatile("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(r.h) : "l"(p));
    return r;
}

// Read-only loads of data that many rows share (the RMSNorm weight, the RoPE tables):
// through the non-coherent path, cached in L1. Never used on memory the launch writes.
template <int BYTES> __device__ __forceinline__ Raw<BYTES> ld_shared_ro(const void* p);

template <> __device__ __forceinline__ Raw<16> ld_shared_ro<16>(const void* p) {
    Raw<16> r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<8> ld_shared_ro<8>(const void* p) {
    Raw<8> r;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<4> ld_shared_ro<4>(const void* p) {
    Raw<4> r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<2> ld_shared_ro<2>(const void* p) {
    Raw<2> r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r.h) : "l"(p));
    return r;
}

// ------------------------------------------------------------------ global stores

template <int BYTES> __device__ __forceinline__ void st_out(void* p, const Raw<BYTES>& r);

template <> __device__ __forceinline__ void st_out<16>(void* p, const Raw<16>& r) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(r.w[0]), "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3])
                 : "memory");
}
template <> __device__ __forceinline__ void st_out<8>(void* p, const Raw<8>& r) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(r.w[0]), "r"(r.w[1])
                 : "memory");
}
template <> __device__ __forceinline__ void st_out<4>(void* p, const Raw<4>& r) {
    asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(r.w[0]) : "memory");
}
template <> __device__ __forceinline__ void st_out<2>(void* p, const Raw<2>& r) {
    asm volatile("st.global.u16 [%0], %1;" :: "l"(p), "h"(r.h) : "memory");
}

// ------------------------------------------------------------------ unpack / pack
// Elements in a vector access are in memory order; for bf16 the element at the lower
// address is the low half of each 32-bit word (little endian).

template <typename S, int BYTES> struct Codec;

template <int BYTES> struct Codec<bf16_t, BYTES> {
    static constexpr int kElems = BYTES / 2;
    __device__ __forceinline__ static void unpack(const Raw<BYTES>& r, float (&v)[kElems]) {
        if constexpr (BYTES == 2) {
            v[0] = __uint_as_float(static_cast<uint32_t>(r.h) << 16);
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                v[2 * k] = __uint_as_float(r.w[k] << 16);
                v[2 * k + 1] = __uint_as_float(r.w[k] & 0xFFFF0000u);
            }
        }
    }
    // One rounding per element: fp32 -> bf16, round to nearest even.
    __device__ __forceinline__ static Raw<BYTES> pack(const float (&v)[kElems]) {
        Raw<BYTES> r;
        if constexpr (BYTES == 2) {
            r.h = __bfloat16_as_ushort(__float2bfloat16_rn(v[0]));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                r.w[k] = *reinterpret_cast<const uint32_t*>(&p);
            }
        }
        return r;
    }
};

template <int BYTES> struct Codec<f32_t, BYTES> {
    static_assert(BYTES % 4 == 0, "fp32 vector accesses are whole words");
    static constexpr int kElems = BYTES / 4;
    __device__ __forceinline__ static void unpack(const Raw<BYTES>& r, float (&v)[kElems]) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) v[k] = __uint_as_float(r.w[k]);
    }
    __device__ __forceinline__ static Raw<BYTES> pack(const float (&v)[kElems]) {
        Raw<BYTES> r;
#pragma unroll
        for (int k = 0; k < kElems; ++k) r.w[k] = __float_as_uint(v[k]);
        return r;
    }
};

template <int BYTES> __device__ __forceinline__ Raw<BYTES> raw_zero() {
    Raw<BYTES> r;
    if constexpr (BYTES == 2) {
        r.h = 0;
    } else {
#pragma unroll
        for (int k = 0; k < BYTES / 4; ++k) r.w[k] = 0u;
    }
    return r;
}

// ------------------------------------------------------------------ reductions

// Butterfly (xor) sum over a full warp: every lane receives the total.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

}  // namespace camp
