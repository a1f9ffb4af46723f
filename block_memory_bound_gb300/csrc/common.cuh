// Device-side building blocks shared by the RMSNorm and RoPE kernels: raw vector
// accesses with explicit cache policy, bf16/f16/fp32 unpacking and packing, and warp
// reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

namespace camp {

// ------------------------------------------------------------------ storage types

struct bf16_t {};   // tag: 16-bit brain float, stored as the upper half of an fp32
struct f16_t {};    // tag: IEEE binary16
struct f32_t {};    // tag: IEEE binary32

template <typename S> struct Storage;
template <> struct Storage<bf16_t> { static constexpr int kBytes = 2; };
template <> struct Storage<f16_t> { static constexpr int kBytes = 2; };
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

// Loads of data that many rows share (the RMSNorm weight, the RoPE tables): ordinary
// coherent loads kept in L1 with the evict-last priority. (Read-only "nc" loads would let
// the compiler hoist every one of them above the output stores, holding all of them in
// registers at once.) Never used on memory the launch writes.
template <int BYTES> __device__ __forceinline__ Raw<BYTES> ld_shared_ro(const void* p);

template <> __device__ __forceinline__ Raw<16> ld_shared_ro<16>(const void* p) {
    Raw<16> r;
    asm volatile("ld.global.L1::evict_last.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<8> ld_shared_ro<8>(const void* p) {
    Raw<8> r;
    asm volatile("ld.global.L1::evict_last.v2.u32 {%0, %1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<4> ld_shared_ro<4>(const void* p) {
    Raw<4> r;
    asm volatile("ld.global.L1::evict_last.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
    return r;
}
template <> __device__ __forceinline__ Raw<2> ld_shared_ro<2>(const void* p) {
    Raw<2> r;
    asm volatile("ld.global.L1::evict_last.u16 %0, [%1];" : "=h"(r.h) : "l"(p));
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

// ------------------------------------------------------------------ element access
// Elements in a vector access are in memory order; for bf16 the element at the lower
// address is the low half of each 32-bit word (little endian). The helpers below work one
// 32-bit word at a time, so that only a couple of unpacked fp32 values are live at once:
// every output word is packed as soon as its elements are computed.

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The same two conversions through byte permutes. Kernels that read a vector twice (a
// reduction pass, then an output pass) use one form per pass, so that the compiler
// re-derives the values from the raw words instead of keeping every unpacked fp32 value
// alive across the reduction (which would double the registers per vector).
__device__ __forceinline__ float bf16_lo_p(uint32_t w) { return __uint_as_float(__byte_perm(w, 0u, 0x1044u)); }
__device__ __forceinline__ float bf16_hi_p(uint32_t w) { return __uint_as_float(__byte_perm(w, 0u, 0x3244u)); }

// Two fp32 values -> one word of two bf16, each rounded once to nearest even.
__device__ __forceinline__ uint32_t bf16_pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

// ------------------------------------------------------------------ packed fp32 pairs
// sm_100-class SMs execute add, sub, mul and fma on two fp32 values held in a 64-bit
// register pair as one instruction (PTX .f32x2). Each lane is rounded to nearest even,
// exactly as the scalar instruction rounds it, so pairing elements changes the
// instruction count, not the arithmetic.

struct f32x2 { unsigned long long v; };

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f32x2 f2_words(uint32_t lo, uint32_t hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float f2_lo(f32x2 a) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
    return lo;
}
__device__ __forceinline__ float f2_hi(f32x2 a) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
    return hi;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
// a * b + c, each lane fused (one rounding).
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}

template <typename S, int BYTES> struct Codec;

template <int BYTES> struct Codec<bf16_t, BYTES> {
    static constexpr int kElems = BYTES / 2;

    // f(e, v) for every element e in order.
    template <typename F>
    __device__ __forceinline__ static void each(const Raw<BYTES>& r, F f) {
        if constexpr (BYTES == 2) {
            f(0, __uint_as_float(static_cast<uint32_t>(r.h) << 16));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                f(2 * k, bf16_lo(r.w[k]));
                f(2 * k + 1, bf16_hi(r.w[k]));
            }
        }
    }

    // out_e = f(e, in_e); one rounding per element.
    template <typename F>
    __device__ __forceinline__ static Raw<BYTES> map(const Raw<BYTES>& r, F f) {
        Raw<BYTES> o;
        if constexpr (BYTES == 2) {
            o.h = __bfloat16_as_ushort(
                __float2bfloat16_rn(f(0, __uint_as_float(static_cast<uint32_t>(r.h) << 16))));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k)
                o.w[k] = bf16_pack2(f(2 * k, bf16_lo_p(r.w[k])), f(2 * k + 1, bf16_hi_p(r.w[k])));
        }
        return o;
    }

    // o_e = a_e + b_e, formed in fp32 and rounded once to bf16.
    __device__ __forceinline__ static Raw<BYTES> add(const Raw<BYTES>& a, const Raw<BYTES>& b) {
        Raw<BYTES> o;
        if constexpr (BYTES == 2) {
            o.h = __bfloat16_as_ushort(__float2bfloat16_rn(
                __uint_as_float(static_cast<uint32_t>(a.h) << 16) +
                __uint_as_float(static_cast<uint32_t>(b.h) << 16)));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k)
                o.w[k] = bf16_pack2(bf16_lo_p(a.w[k]) + bf16_lo_p(b.w[k]),
                                    bf16_hi_p(a.w[k]) + bf16_hi_p(b.w[k]));
        }
        return o;
    }

    // (oa_e, ob_e) = f(e, a_e, b_e); f returns a float2 {oa, ob}.
    template <typename F>
    __device__ __forceinline__ static void map2(const Raw<BYTES>& a, const Raw<BYTES>& b,
                                                Raw<BYTES>& oa, Raw<BYTES>& ob, F f) {
        if constexpr (BYTES == 2) {
            const float2 v = f(0, __uint_as_float(static_cast<uint32_t>(a.h) << 16),
                               __uint_as_float(static_cast<uint32_t>(b.h) << 16));
            oa.h = __bfloat16_as_ushort(__float2bfloat16_rn(v.x));
            ob.h = __bfloat16_as_ushort(__float2bfloat16_rn(v.y));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                const float2 v0 = f(2 * k, bf16_lo_p(a.w[k]), bf16_lo_p(b.w[k]));
                const float2 v1 = f(2 * k + 1, bf16_hi_p(a.w[k]), bf16_hi_p(b.w[k]));
                oa.w[k] = bf16_pack2(v0.x, v1.x);
                ob.w[k] = bf16_pack2(v0.y, v1.y);
            }
        }
    }

    // Element pairs (2p, 2p + 1) as packed operands: p = 0 .. kPairs - 1 (BYTES >= 4).
    static constexpr int kPairs = BYTES / 4;

    template <typename F>
    __device__ __forceinline__ static void each_pair(const Raw<BYTES>& r, F f) {
#pragma unroll
        for (int k = 0; k < kPairs; ++k) f(k, f2_make(bf16_lo(r.w[k]), bf16_hi(r.w[k])));
    }

    // out pair p = f(p, in pair p), each element rounded once to bf16.
    template <typename F>
    __device__ __forceinline__ static Raw<BYTES> map_pair(const Raw<BYTES>& r, F f) {
        Raw<BYTES> o;
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
            const f32x2 q = f(k, f2_make(bf16_lo_p(r.w[k]), bf16_hi_p(r.w[k])));
            o.w[k] = bf16_pack2(f2_lo(q), f2_hi(q));
        }
        return o;
    }
};

// binary16 <-> fp32. Every binary16 value is exactly an fp32 value; fp32 -> binary16
// rounds to nearest, ties to even (cvt.rn). The "_p" forms issue the same conversion from
// inline assembly, which the compiler does not merge with the intrinsic's: as with the
// byte-permute forms of bf16, a value unpacked for a reduction pass is unpacked again in
// the output pass rather than kept alive across the reduction.
__device__ __forceinline__ float f16_val(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ float f16_lo(uint32_t w) { return f16_val(static_cast<uint16_t>(w & 0xFFFFu)); }
__device__ __forceinline__ float f16_hi(uint32_t w) { return f16_val(static_cast<uint16_t>(w >> 16)); }
__device__ __forceinline__ float f16_val_p(uint16_t h) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}
__device__ __forceinline__ float f16_lo_p(uint32_t w) { return f16_val_p(static_cast<uint16_t>(w & 0xFFFFu)); }
__device__ __forceinline__ float f16_hi_p(uint32_t w) { return f16_val_p(static_cast<uint16_t>(w >> 16)); }
__device__ __forceinline__ uint32_t f16_pack2(float lo, float hi) {
    const __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

template <int BYTES> struct Codec<f16_t, BYTES> {
    static constexpr int kElems = BYTES / 2;
    static constexpr int kPairs = BYTES / 4;

    template <typename F>
    __device__ __forceinline__ static void each(const Raw<BYTES>& r, F f) {
        if constexpr (BYTES == 2) {
            f(0, f16_val(r.h));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                f(2 * k, f16_lo(r.w[k]));
                f(2 * k + 1, f16_hi(r.w[k]));
            }
        }
    }

    template <typename F>
    __device__ __forceinline__ static Raw<BYTES> map(const Raw<BYTES>& r, F f) {
        Raw<BYTES> o;
        if constexpr (BYTES == 2) {
            o.h = __half_as_ushort(__float2half_rn(f(0, f16_val_p(r.h))));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k)
                o.w[k] = f16_pack2(f(2 * k, f16_lo_p(r.w[k])), f(2 * k + 1, f16_hi_p(r.w[k])));
        }
        return o;
    }

    __device__ __forceinline__ static Raw<BYTES> add(const Raw<BYTES>& a, const Raw<BYTES>& b) {
        Raw<BYTES> o;
        if constexpr (BYTES == 2) {
            o.h = __half_as_ushort(__float2half_rn(f16_val(a.h) + f16_val(b.h)));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k)
                o.w[k] = f16_pack2(f16_lo_p(a.w[k]) + f16_lo_p(b.w[k]),
                                   f16_hi_p(a.w[k]) + f16_hi_p(b.w[k]));
        }
        return o;
    }

    template <typename F>
    __device__ __forceinline__ static void map2(const Raw<BYTES>& a, const Raw<BYTES>& b,
                                                Raw<BYTES>& oa, Raw<BYTES>& ob, F f) {
        if constexpr (BYTES == 2) {
            const float2 v = f(0, f16_val_p(a.h), f16_val_p(b.h));
            oa.h = __half_as_ushort(__float2half_rn(v.x));
            ob.h = __half_as_ushort(__float2half_rn(v.y));
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                const float2 v0 = f(2 * k, f16_lo_p(a.w[k]), f16_lo_p(b.w[k]));
                const float2 v1 = f(2 * k + 1, f16_hi_p(a.w[k]), f16_hi_p(b.w[k]));
                oa.w[k] = f16_pack2(v0.x, v1.x);
                ob.w[k] = f16_pack2(v0.y, v1.y);
            }
        }
    }

    template <typename F>
    __device__ __forceinline__ static void each_pair(const Raw<BYTES>& r, F f) {
#pragma unroll
        for (int k = 0; k < kPairs; ++k) f(k, f2_make(f16_lo(r.w[k]), f16_hi(r.w[k])));
    }

    template <typename F>
    __device__ __forceinline__ static Raw<BYTES> map_pair(const Raw<BYTES>& r, F f) {
        Raw<BYTES> o;
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
            const f32x2 q = f(k, f2_make(f16_lo_p(r.w[k]), f16_hi_p(r.w[k])));
            o.w[k] = f16_pack2(f2_lo(q), f2_hi(q));
        }
        return o;
    }
};

template <int BYTES> struct Codec<f32_t, BYTES> {
    static_assert(BYTES % 4 == 0, "fp32 vector accesses are whole words");
    static constexpr int kElems = BYTES / 4;
    static constexpr int kPairs = BYTES / 8;

    template <typename F>
    __device__ __forceinline__ static void each_pair(const Raw<BYTES>& r, F f) {
#pragma unroll
        for (int k = 0; k < kPairs; ++k) f(k, f2_words(r.w[2 * k], r.w[2 * k + 1]));
    }

    template <typename F>
    __device__ __forceinline__ static Raw<BYTES> map_pair(const Raw<BYTES>& r, F f) {
        Raw<BYTES> o;
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
            const f32x2 q = f(k, f2_words(r.w[2 * k], r.w[2 * k + 1]));
            o.w[2 * k] = __float_as_uint(f2_lo(q));
            o.w[2 * k + 1] = __float_as_uint(f2_hi(q));
        }
        return o;
    }

    template <typename F>
    __device__ __forceinline__ static void each(const Raw<BYTES>& r, F f) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) f(k, __uint_as_float(r.w[k]));
    }

    template <typename F>
    __device__ __forceinline__ static Raw<BYTES> map(const Raw<BYTES>& r, F f) {
        Raw<BYTES> o;
#pragma unroll
        for (int k = 0; k < kElems; ++k) o.w[k] = __float_as_uint(f(k, __uint_as_float(r.w[k])));
        return o;
    }

    __device__ __forceinline__ static Raw<BYTES> add(const Raw<BYTES>& a, const Raw<BYTES>& b) {
        Raw<BYTES> o;
#pragma unroll
        for (int k = 0; k < kElems; ++k)
            o.w[k] = __float_as_uint(__uint_as_float(a.w[k]) + __uint_as_float(b.w[k]));
        return o;
    }

    template <typename F>
    __device__ __forceinline__ static void map2(const Raw<BYTES>& a, const Raw<BYTES>& b,
                                                Raw<BYTES>& oa, Raw<BYTES>& ob, F f) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) {
            const float2 v = f(k, __uint_as_float(a.w[k]), __uint_as_float(b.w[k]));
            oa.w[k] = __float_as_uint(v.x);
            ob.w[k] = __float_as_uint(v.y);
        }
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

// ------------------------------------------------------------------ dependent launch
// Programmatic dependent launch: a kernel launched with programmatic stream serialization
// may start while the previous kernel in the stream is still running. griddep_wait()
// blocks until that kernel has completed and its memory is visible, so every kernel here
// calls it before its first global-memory load or store (an L2 prefetch, below, may come
// first); without the launch attribute it returns at once. griddep_launch_dependents()
// lets the next kernel be scheduled early.

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 prefetch of a CTA's first inputs, issued by one thread BEFORE griddep_wait(), so that
// their HBM reads overlap the tail of the previous kernel in the stream instead of
// following it. cp.async.bulk.prefetch.L2 only fills L2 lines: it returns no data,
// completes on its own and needs no barrier. L2 is where the SMs' global accesses meet
// (every store of the previous kernel lands there, in the line a prefetch may already
// have filled), and this kernel's loads of the same bytes are issued after
// griddep_wait(), so they return what the previous kernel wrote whether a prefetch ran
// before, after or during those writes; at worst a prefetch reads a line that is about
// to be overwritten. Only the 16-byte-aligned interior of [p, p + bytes) is fetched, in
// pieces of at most 32 KB, so nothing outside the buffer is touched; bytes <= 0 is a no-op.
// Number of SM identifiers on this device (at least the SM count).
__device__ __forceinline__ uint32_t sm_id_count() {
    uint32_t n;
    asm("mov.u32 %0, %%nsmid;" : "=r"(n));
    return n;
}

__device__ __forceinline__ void prefetch_l2(const void* p, int64_t bytes) {
    if (bytes <= 0) return;
    const uint64_t a = reinterpret_cast<uint64_t>(p);
    uint64_t lo = (a + 15) & ~uint64_t{15};
    const uint64_t hi = (a + static_cast<uint64_t>(bytes)) & ~uint64_t{15};
    while (lo < hi) {
        const uint32_t n = hi - lo < 32768 ? static_cast<uint32_t>(hi - lo) : 32768u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"(n) : "memory");
        lo += n;
    }
}

// ------------------------------------------------------------------ rotation helpers
// Products for rotate-half RoPE, evaluated with Kahan's compensated 2x2 determinant
// (W. Kahan; error analysis in Jeannerod, Louvet and Muller, "Further analysis of Kahan's
// algorithm for the accurate computation of 2x2 determinants", Math. Comp. 2013): with
// p = c*d rounded and e = fma(c, d, -p) its exact error, a*b - c*d = fma(a, b, -p) - e,
// accurate to about 2 ulp relative to the RESULT even when the two products nearly cancel.

// a*b - c*d
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
    const float p = __fmul_rn(c, d);
    const float e = fmaf(c, d, -p);
    const float f = fmaf(a, b, -p);
    return __fsub_rn(f, e);
}

// a*b + c*d
__device__ __forceinline__ float sum_of_products(float a, float b, float c, float d) {
    const float p = __fmul_rn(c, d);
    const float e = fmaf(c, d, -p);
    const float f = fmaf(a, b, p);
    return __fadd_rn(f, e);
}

// N consecutive fp32 table values through the read-only path, in the widest aligned
// accesses (the host guarantees alignment to min(16, 4N) bytes).
template <int N>
__device__ __forceinline__ void load_table(const float* p, float (&out)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
            const Raw<16> r = ld_shared_ro<16>(p + 4 * k);
#pragma unroll
            for (int i = 0; i < 4; ++i) out[4 * k + i] = __uint_as_float(r.w[i]);
        }
    } else if constexpr (N == 2) {
        const Raw<8> r = ld_shared_ro<8>(p);
        out[0] = __uint_as_float(r.w[0]);
        out[1] = __uint_as_float(r.w[1]);
    } else {
        static_assert(N == 1, "table accesses are 1, 2 or a multiple of 4 floats");
        out[0] = __uint_as_float(ld_shared_ro<4>(p).w[0]);
    }
}

// ------------------------------------------------------------------ reductions

// Butterfly (xor) sum over a full warp: every lane receives the total, with the same bits
// in every lane (each step adds the same two values in either order).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

// Sum of the W partials p[0 .. W-1] (W a power of two, at most 32; shared memory), taken by
// the whole warp; every lane gets the same bits. Up to 8 partials: W independent loads
// and a sequential sum (the shortest dependency chain: measured faster than a butterfly
// at W = 4). Beyond: lane l loads p[l mod W] and a butterfly over aligned groups of W
// lanes adds them (one load per lane instead of W, which at W = 32 also keeps 32 values
// out of the registers).
template <int W>
__device__ __forceinline__ float sum_partials(const float* p) {
    static_assert(W >= 1 && W <= 32 && (W & (W - 1)) == 0, "W is a power of two <= 32");
    if constexpr (W <= 8) {
        float v = 0.0f;
#pragma unroll
        for (int i = 0; i < W; ++i) v += p[i];
        return v;
    } else {
        float v = p[threadIdx.x & (W - 1)];
#pragma unroll
        for (int off = W / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        return v;
    }
}

// ------------------------------------------------------------------ integer division
// Division of 32-bit unsigned integers by a divisor fixed for the whole launch, by
// multiplication (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(m, n) + n) >> l for every 32-bit n. The sum is formed in 64 bits.

struct FastDiv {
    uint32_t d;      // divisor, >= 1
    uint32_t m;      // magic multiplier
    uint32_t l;      // shift
};

inline FastDiv make_fast_div(uint32_t d) {
    uint32_t l = 0;
    while (l < 32 && (uint64_t{1} << l) < d) ++l;
    const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
    const uint64_t t = __umulhi(f.m, n);
    return static_cast<uint32_t>((t + n) >> f.l);
}

// ------------------------------------------------------------------ host-side launch

// Grid for `blocks` CTAs: 1-D up to 2^31 - 1 blocks, 2-D beyond (the kernels flatten
// blockIdx and skip blocks past the end).
inline dim3 grid_2d(int64_t blocks) {
    const int64_t kMaxX = 2147483647;
    if (blocks <= kMaxX) return dim3(static_cast<unsigned>(blocks));
    return dim3(static_cast<unsigned>(kMaxX), static_cast<unsigned>((blocks + kMaxX - 1) / kMaxX));
}

// Launch with programmatic stream serialization, so that the kernel may be scheduled
// while its predecessor in the stream drains (the kernel itself waits for the
// predecessor's memory in griddep_wait()). Returns the launch status.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace camp
