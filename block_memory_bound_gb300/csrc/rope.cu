// Rotate-half RoPE kernel for sm_103a.
//
// Operation (gollamago README, "RoPE"): rope(input, sin_table, cos_table) -> output, with
// input [batch, sequence, heads, head_dim] and tables [sequence, head_dim/2]. Both halves
// of a head are rotated in fp32 registers and written once, which removes the separate
// concatenation pass of a framework-level rotate-half. Pair formula (tilelang tutorial
// ch. 02, exercise E13): y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin.
//
// Mapping: one thread owns vector j (E elements) of the first half and the matching
// vector of the second half, for HPT heads of one position. It issues its 2*HPT head
// loads, then loads the E sine and cosine values of the position once (L1-cached
// read-only path; every head group of the position reuses them), then rotates and
// stores. The table row s of the flattened position b*S + s is derived on the device;
// nothing is uploaded per call.
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

// Rotate one head's vector pair (j of each half) and store it.
template <typename S, int VB>
__device__ __forceinline__ void rotate_store(const Raw<VB>& lo, const Raw<VB>& hi,
                                             const float (&sn)[VB / Storage<S>::kBytes],
                                             const float (&cs)[VB / Storage<S>::kBytes],
                                             char* q, int64_t half_bytes) {
    Raw<VB> o1, o2;
    Codec<S, VB>::map2(lo, hi, o1, o2, [&](int e, float x1, float x2) {
        return make_float2(diff_of_products(x1, cs[e], x2, sn[e]),
                           sum_of_products(x2, cs[e], x1, sn[e]));
    });
    st_out<VB>(q, o1);
    st_out<VB>(q + half_bytes, o2);
}

// Tiled mapping. A CTA covers `tpc` consecutive positions; thread (tk, hg, j) =
// (position, head group, vector) rotates vector j of both halves of heads
// hg*HPT .. hg*HPT+HPT-1 of position blockIdx*tpc + tk, in the first tensor for the first
// ceil(H/HPT)*nvh threads of a position and in the second tensor (if any) for the rest.
// The table row s = position mod S comes from a multiply-shift division, and a position's
// table vectors are shared through L1 by all of its heads in both tensors. One position
// block per CTA; the host guarantees fewer than 2^32 positions and at most kRopeBlock
// threads per position.
template <typename S, int VB, int HPT>
__global__ void __launch_bounds__(kRopeBlock, rope_min_blocks(HPT))
rope_tiled_kernel(const void* x, void* y, int heads, const void* x2, void* y2, int heads2,
                  const float* __restrict__ sin_t, const float* __restrict__ cos_t,
                  int64_t tokens, FastDiv seq, int half) {
    constexpr int E = Codec<S, VB>::kElems;
    constexpr int ES = Storage<S>::kBytes;

    const int nvh = half / E;                                  // vectors per half
    const int first = ((heads + HPT - 1) / HPT) * nvh;         // threads for tensor 1
    const int per_pos = first + ((heads2 + HPT - 1) / HPT) * nvh;
    const int tpc = kRopeBlock / per_pos;                      // positions per CTA
    const int tk = static_cast<int>(threadIdx.x) / per_pos;
    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0 && block * tpc < tokens) {   // this CTA's positions and table rows
        const int64_t p0 = block * tpc;
        const int64_t np = tokens - p0 < tpc ? tokens - p0 : tpc;
        const int64_t rb = static_cast<int64_t>(2 * ES) * half;
        prefetch_l2(static_cast<const char*>(x) + p0 * heads * rb, np * heads * rb);
        if (heads2 > 0) prefetch_l2(static_cast<const char*>(x2) + p0 * heads2 * rb, np * heads2 * rb);
        // table rows s0 .. s0 + ns - 1, up to the end of the sequence
        const uint32_t p32 = static_cast<uint32_t>(p0);
        const uint32_t s0 = p32 - fast_div(p32, seq) * seq.d;
        const int64_t ns = np < seq.d - s0 ? np : seq.d - s0;
        prefetch_l2(sin_t + static_cast<int64_t>(s0) * half, ns * half * 4);
        prefetch_l2(cos_t + static_cast<int64_t>(s0) * half, ns * half * 4);
    }
    griddep_wait();
    griddep_launch_dependents();
    const int64_t pos = block * tpc + tk;
    if (tk >= tpc || pos >= tokens) return;                    // no barrier in this kernel
    int r = static_cast<int>(threadIdx.x) - tk * per_pos;
    const bool second = r >= first;
    if (second) {
        r -= first;
        x = x2;
        y = y2;
        heads = heads2;
    }
    const int hg = r / nvh;
    const int j = r - hg * nvh;
    const int h0 = hg * HPT;
    const int nh = heads - h0 < HPT ? heads - h0 : HPT;
    const uint32_t p32 = static_cast<uint32_t>(pos);
    const uint32_t s = p32 - fast_div(p32, seq) * seq.d;

    const int64_t row_bytes = static_cast<int64_t>(2 * ES) * half;
    const int64_t half_bytes = static_cast<int64_t>(ES) * half;
    const int64_t off = (pos * heads + h0) * row_bytes + static_cast<int64_t>(j) * VB;
    const char* p = static_cast<const char*>(x) + off;
    Raw<VB> lo[HPT], hi[HPT];
#pragma unroll
    for (int u = 0; u < HPT; ++u) {
        if (u < nh) {
            lo[u] = ld_stream<VB>(p + u * row_bytes);
            hi[u] = ld_stream<VB>(p + u * row_bytes + half_bytes);
        }
    }
    float sn[E], cs[E];
    const int64_t toff = static_cast<int64_t>(s) * half + static_cast<int64_t>(j) * E;
    load_table<E>(sin_t + toff, sn);
    load_table<E>(cos_t + toff, cs);
    char* q = static_cast<char*>(y) + off;
#pragma unroll
    for (int u = 0; u < HPT; ++u) {
        if (u < nh) rotate_store<S, VB>(lo[u], hi[u], sn, cs, q + u * row_bytes, half_bytes);
    }
}

// Flat mapping, for shapes whose position does not fit one CTA: one work item per
// (position, head group, vector), decoded with 64-bit division.
template <typename S, int VB, int HPT>
__global__ void __launch_bounds__(kRopeBlock)
rope_flat_kernel(const void* x, const float* __restrict__ sin_t,
                 const float* __restrict__ cos_t, void* y, int64_t tokens, int64_t seq,
                 int64_t heads, int64_t half) {
    constexpr int E = Codec<S, VB>::kElems;
    constexpr int ES = Storage<S>::kBytes;

    griddep_wait();
    griddep_launch_dependents();

    const int64_t nvh = half / E;
    const int64_t hgroups = (heads + HPT - 1) / HPT;
    const int64_t per_token = hgroups * nvh;
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
        float sn[E], cs[E];
        load_table<E>(sin_t + s * half + j * E, sn);
        load_table<E>(cos_t + s * half + j * E, cs);
#pragma unroll
        for (int u = 0; u < HPT; ++u) {
            const int64_t h = hg * HPT + u;
            if (h < heads) {
                rotate_store<S, VB>(lo[u], hi[u], sn, cs,
                                    yb + (token * heads + h) * row_bytes + j * VB, half_bytes);
            }
        }
    }
}

template <typename S, int VB, int HPT>
cudaError_t launch_tiled(const RopeArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(rope_tiled_kernel<S, VB, HPT>, grid_2d(grid), dim3(kRopeBlock), s, a.x,
                      a.y, static_cast<int>(a.heads), a.x2, a.y2, static_cast<int>(a.heads2),
                      a.sin_t, a.cos_t, a.tokens, make_fast_div(static_cast<uint32_t>(a.seq)),
                      static_cast<int>(a.half));
}

template <typename S, int VB, int HPT>
cudaError_t launch_flat(const RopeArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(rope_flat_kernel<S, VB, HPT>, dim3(static_cast<unsigned>(grid)),
                      dim3(kRopeBlock), s, a.x, a.sin_t, a.cos_t, a.y, a.tokens, a.seq,
                      a.heads, a.half);
}

using RopeFn = cudaError_t (*)(const RopeArgs&, int64_t, cudaStream_t);

struct RopeEntry {
    DType t;
    int vec_bytes, hpt;
    RopeFn tiled, flat;
};

#define CAMP_ROPE(S, DT, VB, H) {DType::DT, VB, H, &launch_tiled<S, VB, H>, &launch_flat<S, VB, H>}
#define CAMP_ROPE_H(S, DT, VB) CAMP_ROPE(S, DT, VB, 1), CAMP_ROPE(S, DT, VB, 2), \
                               CAMP_ROPE(S, DT, VB, 4), CAMP_ROPE(S, DT, VB, 8)

const RopeEntry kRope[] = {
    CAMP_ROPE_H(bf16_t, BF16, 16), CAMP_ROPE_H(bf16_t, BF16, 8), CAMP_ROPE_H(bf16_t, BF16, 4),
    CAMP_ROPE_H(bf16_t, BF16, 2),
    CAMP_ROPE_H(f16_t, F16, 16), CAMP_ROPE_H(f16_t, F16, 8), CAMP_ROPE_H(f16_t, F16, 4),
    CAMP_ROPE_H(f16_t, F16, 2),
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

cudaError_t rope_tiled_launch(DType t, int vec_bytes, int heads_per_thread, const RopeArgs& a,
                              int64_t grid, cudaStream_t s) {
    const RopeEntry* e = find_rope(t, vec_bytes, heads_per_thread);
    return e == nullptr ? cudaErrorInvalidValue : e->tiled(a, grid, s);
}

cudaError_t rope_flat_launch(DType t, int vec_bytes, int heads_per_thread, const RopeArgs& a,
                             int64_t grid, cudaStream_t s) {
    const RopeEntry* e = find_rope(t, vec_bytes, heads_per_thread);
    return e == nullptr ? cudaErrorInvalidValue : e->flat(a, grid, s);
}

}  // namespace camp
