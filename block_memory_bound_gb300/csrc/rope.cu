// Rotate-half RoPE kernel for sm_103a.
//
// Operation (gollamago README, "RoPE"): rope(input, sin_table, cos_table) -> output, with
// input [batch, sequence, heads, head_dim] and tables [sequence, head_dim/2]. Both halves
// of a head are rotated in fp32 registers and written once, which removes the separate
// concatenation pass of a framework-level rotate-half. Pair formula (tilelang tutorial
// ch. 02, exercise E13): y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin.
//
// Mapping: one thread owns vector j (E elements) of the first half and the matching
// vector of the second half, for HPT heads of one position. It loads the E sine and
// cosine values of that position once (L1-cached read-only path; every head of the
// position reuses them) and then streams its 2*HPT head vectors: all loads first, then
// the rotations, then the stores. The position's table row s = (b*S + s) mod S is
// derived from the thread index on the device; nothing is uploaded per call.
//
// Each product difference is evaluated with Kahan's compensated 2x2 determinant
// (W. Kahan; error analysis in Jeannerod, Louvet and Muller, "Further analysis of
// Kahan's algorithm for the accurate computation of 2x2 determinants", Math. Comp.
// 2013): with p = c*d rounded and e = fma(c, d, -p) its exact error, a*b - c*d is
// fma(a, b, -p) - e, accurate to about 2 ulp relative to the RESULT even when the two
// products nearly cancel. A plain fma(a, b, -c*d) has an error relative to c*d, which
// on bf16 outputs can exceed one bf16 ulp of a small result.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

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

template <typename S, int VB, int HPT>
__global__ void __launch_bounds__(kRopeBlock)
rope_kernel(const void* x, const float* __restrict__ sin_t,
            const float* __restrict__ cos_t, void* y, int64_t tokens, int64_t seq,
            int64_t heads, int64_t half) {
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;

    const int64_t nvh = half / E;                          // vectors per half-row
    const int64_t hgroups = (heads + HPT - 1) / HPT;
    const int64_t per_token = hgroups * nvh;               // threads per position
    const int64_t total = tokens * per_token;
    const int64_t row_bytes = 2 * half * ES;
    const int64_t half_bytes = half * ES;
    const char* xb = static_cast<const char*>(x);
    char* yb = static_cast<char*>(y);

    for (int64_t id = static_cast<int64_t>(blockIdx.x) * kRopeBlock + threadIdx.x; id < total;
         id += static_cast<int64_t>(gridDim.x) * kRopeBlock) {
        const int64_t token = id / per_token;              // b * S + s
        const int64_t rem = id - token * per_token;
        const int64_t hg = rem / nvh;
        const int64_t j = rem - hg * nvh;
        const int64_t s = token % seq;

        float sn[E], cs[E];
        load_table<E>(sin_t + s * half + j * E, sn);
        load_table<E>(cos_t + s * half + j * E, cs);

        Raw<VB> lo[HPT], hi[HPT];
#pragma unroll
        for (int u = 0; u < HPT; ++u) {
            const int64_t h = hg * HPT + u;
            if (h < heads) {
                const char* p = xb + (token * heads + h) * row_bytes + j * VB;
                lo[u] = ld_stream<VB>(p);
                hi[u] = ld_stream<VB>(p + half_bytes);
            }
        }
#pragma unroll
        for (int u = 0; u < HPT; ++u) {
            const int64_t h = hg * HPT + u;
            if (h < heads) {
                float x1[E], x2[E], y1[E], y2[E];
                C::unpack(lo[u], x1);
                C::unpack(hi[u], x2);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    y1[e] = diff_of_products(x1[e], cs[e], x2[e], sn[e]);
                    y2[e] = sum_of_products(x2[e], cs[e], x1[e], sn[e]);
                }
                char* q = yb + (token * heads + h) * row_bytes + j * VB;
                st_out<VB>(q, C::pack(y1));
                st_out<VB>(q + half_bytes, C::pack(y2));
            }
        }
    }
}

template <typename S, int VB, int HPT>
void launch_rope(const RopeArgs& a, int64_t grid, cudaStream_t s) {
    rope_kernel<S, VB, HPT><<<static_cast<unsigned>(grid), kRopeBlock, 0, s>>>(
        a.x, a.sin_t, a.cos_t, a.y, a.tokens, a.seq, a.heads, a.half);
}

using RopeFn = void (*)(const RopeArgs&, int64_t, cudaStream_t);

struct RopeEntry {
    DType t;
    int vec_bytes, hpt;
    RopeFn fn;
};

#define CAMP_ROPE(S, DT, VB, H) {DType::DT, VB, H, &launch_rope<S, VB, H>}
#define CAMP_ROPE_H(S, DT, VB) CAMP_ROPE(S, DT, VB, 1), CAMP_ROPE(S, DT, VB, 2), \
                               CAMP_ROPE(S, DT, VB, 4), CAMP_ROPE(S, DT, VB, 8)

const RopeEntry kRope[] = {
    CAMP_ROPE_H(bf16_t, BF16, 16), CAMP_ROPE_H(bf16_t, BF16, 8), CAMP_ROPE_H(bf16_t, BF16, 4),
    CAMP_ROPE_H(bf16_t, BF16, 2),
    CAMP_ROPE_H(f32_t, F32, 16), CAMP_ROPE_H(f32_t, F32, 8), CAMP_ROPE_H(f32_t, F32, 4),
};

#undef CAMP_ROPE_H
#undef CAMP_ROPE

const RopeEntry* find_rope(DType t, int vec_bytes, int hpt) {
    for (const RopeEntry& e : kRope) {
        if (e.t == t && e.vec_bytes == vec_bytes && e.hpt == hpt) return &e;
    }
    return nullptr;
}

}  // namespace

bool rope_compiled(DType t, int vec_bytes, int heads_per_thread) {
    return find_rope(t, vec_bytes, heads_per_thread) != nullptr;
}

bool rope_launch(DType t, int vec_bytes, int heads_per_thread, const RopeArgs& a,
                 int64_t grid, cudaStream_t s) {
    const RopeEntry* e = find_rope(t, vec_bytes, heads_per_thread);
    if (e == nullptr) return false;
    e->fn(a, grid, s);
    return true;
}

}  // namespace camp
