// LayerNorm forward for sm_103a.
//
// Definition (xserv "phase 4", csrc/normalization/layernorm.cu and the design notes'
// LayerNorm section): y = gamma * (x - mean) / sqrt(var + eps) + beta per row, with the
// population variance (divisor: the row length). The TileLang tutorial (ch. 02, example 2)
// counts it as one read of x and one write of y when fused.
//
// The row is held in registers, as in the RMSNorm rows kernel (one sweep of 16-byte
// loads, a group of G threads per row), so the statistics cost no extra memory traffic
// and are taken in two passes over the registers instead of xserv's single pass
// var = E[x^2] - mean^2, which cancels catastrophically when |mean| >> sigma:
//   1. shift K = x[row, 0] and mu = sum(x - K) / n, so mean = K + mu is kept as the pair
//      (K, mu) and never rounded to one fp32 number: every deviation is formed as
//      d = (x - K) - mu, whose rounding errors are relative to the spread of the row, not
//      to |mean| (an fp32 mean alone is off by up to ulp(mean) / 2);
//   2. var = sum(d^2) / n from the registers; in 16-bit storage (where the kernel is bound
//      by instruction issue) pass 1 also sums (x - K)^2, and when mu^2 <= 4 (that sum / n -
//      mu^2), i.e. K lies within two standard deviations of the mean, that difference is
//      the variance and pass 2 is skipped: its cancellation then costs at most a few times
//      the summation error of the two-pass value, far below a 16-bit output's rounding;
//      a row whose shift lies further out (or whose difference is negative) takes pass 2;
//   3. y = fma(d * rsqrt(var + eps), gamma, beta), rounded once.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

template <int G>
struct LnShape {
    static constexpr int kBlock = rows_block(G);
    static constexpr int kRowsPerCta = kBlock / G;
    static constexpr int kWarpsPerRow = G / 32;
};

// Sum over the row group; for G > 32 through `scratch` (one slot per warp of the group).
// The caller separates two uses of one scratch array with a barrier or uses two arrays.
template <int G>
__device__ __forceinline__ float group_sum(float v, float (&scratch)[LnShape<G>::kRowsPerCta]
                                                             [LnShape<G>::kWarpsPerRow],
                                           int g, int t) {
    v = warp_sum(v);
    if constexpr (LnShape<G>::kWarpsPerRow > 1) {
        if ((threadIdx.x & 31) == 0) scratch[g][t / 32] = v;
        __syncthreads();
        v = sum_partials<LnShape<G>::kWarpsPerRow>(scratch[g]);
    }
    return v;
}

// Sums of a and b over the row group with one barrier (G > 32), as group_sum.
template <int G>
__device__ __forceinline__ void group_sum2(float& a, float& b,
                                           float (&sa)[LnShape<G>::kRowsPerCta][LnShape<G>::kWarpsPerRow],
                                           float (&sb)[LnShape<G>::kRowsPerCta][LnShape<G>::kWarpsPerRow],
                                           int g, int t) {
    a = warp_sum(a);
    b = warp_sum(b);
    if constexpr (LnShape<G>::kWarpsPerRow > 1) {
        if ((threadIdx.x & 31) == 0) {
            sa[g][t / 32] = a;
            sb[g][t / 32] = b;
        }
        __syncthreads();
        a = sum_partials<LnShape<G>::kWarpsPerRow>(sa[g]);
        b = sum_partials<LnShape<G>::kWarpsPerRow>(sb[g]);
    }
}

// Pass 1 of the one-pass path (packed pairs): this thread's sums of (x - K) and (x - K)^2.
template <typename C, int G, int NV, int VB>
__device__ __forceinline__ void shifted_moments(const Raw<VB> (&v)[NV], float shift, int live,
                                                float& s1, float& s2) {
    const f32x2 k2 = f2_make(shift, shift);
    f32x2 a = f2_make(0.0f, 0.0f), q = f2_make(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < NV; ++k)
        if (k * G < live)
            C::each_pair(v[k], [&](int, f32x2 p) {
                const f32x2 d = f2_sub(p, k2);
                a = f2_add(a, d);
                q = f2_fma(d, d, q);
            });
    s1 = f2_lo(a) + f2_hi(a);
    s2 = f2_lo(q) + f2_hi(q);
}

// Pass 1: this thread's sum of (x - K) over its live accesses.
template <typename C, int G, int NV, int VB>
__device__ __forceinline__ float shifted_sum(const Raw<VB> (&v)[NV], float shift, int live) {
    if constexpr (C::kElems >= 2) {
        const f32x2 k2 = f2_make(shift, shift);
        f32x2 acc = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (k * G < live) C::each_pair(v[k], [&](int, f32x2 p) { acc = f2_add(acc, f2_sub(p, k2)); });
        return f2_lo(acc) + f2_hi(acc);
    } else {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (k * G < live) C::each(v[k], [&](int, float f) { s += f - shift; });
        return s;
    }
}

// Pass 2: this thread's sum of d^2, d = (x - K) - mu, over its live accesses.
template <typename C, int G, int NV, int VB>
__device__ __forceinline__ float squared_deviations(const Raw<VB> (&v)[NV], float shift,
                                                    float mu, int live) {
    if constexpr (C::kElems >= 2) {
        const f32x2 k2 = f2_make(shift, shift), m2 = f2_make(mu, mu);
        f32x2 acc = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (k * G < live)
                C::each_pair(v[k], [&](int, f32x2 p) {
                    const f32x2 d = f2_sub(f2_sub(p, k2), m2);
                    acc = f2_fma(d, d, acc);
                });
        return f2_lo(acc) + f2_hi(acc);
    } else {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (k * G < live)
                C::each(v[k], [&](int, float f) {
                    const float d = (f - shift) - mu;
                    s = fmaf(d, d, s);
                });
        return s;
    }
}

// One output access: fma(((x - K) - mu) * rstd, gamma, beta), rounded once.
template <typename C, int VB>
__device__ __forceinline__ Raw<VB> normalize(const Raw<VB>& xv, const Raw<VB>& gv,
                                             const Raw<VB>& bv, float shift, float mu,
                                             float rstd) {
    if constexpr (C::kElems >= 2) {
        f32x2 gp[C::kPairs], bp[C::kPairs];
        C::each_pair(gv, [&](int p, f32x2 q) { gp[p] = q; });
        C::each_pair(bv, [&](int p, f32x2 q) { bp[p] = q; });
        const f32x2 k2 = f2_make(shift, shift), m2 = f2_make(mu, mu), r2 = f2_make(rstd, rstd);
        return C::map_pair(xv, [&](int p, f32x2 xp) {
            return f2_fma(f2_mul(f2_sub(f2_sub(xp, k2), m2), r2), gp[p], bp[p]);
        });
    } else {
        float gf[C::kElems], bf[C::kElems];
        C::each(gv, [&](int e, float f) { gf[e] = f; });
        C::each(bv, [&](int e, float f) { bf[e] = f; });
        return C::map(xv, [&](int e, float xf) {
            return fmaf(((xf - shift) - mu) * rstd, gf[e], bf[e]);
        });
    }
}

template <typename S, int VB, int G, int NV>
__global__ void __launch_bounds__(LnShape<G>::kBlock, ln_min_blocks(Storage<S>::kBytes, VB, G, NV))
layernorm_rows_kernel(const void* x, const void* __restrict__ gamma,
                      const void* __restrict__ beta, void* y, int64_t rows, int64_t cols,
                      float eps) {
    using Sh = LnShape<G>;
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;

    // The one-pass statistics (pass 2 only where the shift is far from the mean): 16-bit
    // storage in packed pairs.
    constexpr bool kOnePass = ES == 2 && E >= 2;
    __shared__ float part_mean[Sh::kRowsPerCta][Sh::kWarpsPerRow];
    __shared__ float part_var[Sh::kRowsPerCta][Sh::kWarpsPerRow];
    __shared__ float part_sq[kOnePass ? Sh::kRowsPerCta : 1][Sh::kWarpsPerRow];

    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0 && block * Sh::kRowsPerCta < rows) {   // this CTA's rows of x
        const int64_t row0 = block * Sh::kRowsPerCta;
        const int64_t n = (rows - row0 < Sh::kRowsPerCta ? rows - row0 : Sh::kRowsPerCta) * cols * ES;
        prefetch_l2(static_cast<const char*>(x) + row0 * cols * ES, n);
    }
    griddep_wait();
    griddep_launch_dependents();

    const int g = threadIdx.x / G;
    const int t = threadIdx.x % G;
    const int64_t row = block * Sh::kRowsPerCta + g;
    const bool active = row < rows;
    const int live = static_cast<int>(cols / E) - t;
    const int64_t row_off = row * cols * ES;
    const int64_t off = row_off + static_cast<int64_t>(t) * VB;

    Raw<VB> v[NV];
    const char* xr = static_cast<const char*>(x) + off;
#pragma unroll
    for (int k = 0; k < NV; ++k)
        v[k] = (active && k * G < live) ? ld_stream<VB>(xr + k * G * VB) : raw_zero<VB>();
    // The shift: the row's first element (read before any of this row's outputs is written:
    // every store below follows a group reduction that every thread of the group reaches).
    float shift = 0.0f;
    if (active) {
        const Raw<ES> k0 = ld_stream<ES>(static_cast<const char*>(x) + row_off);
        Codec<S, ES>::each(k0, [&](int, float f) { shift = f; });
    }

    const float n = static_cast<float>(cols);
    float mu, var;
    if constexpr (kOnePass) {
        float s1, s2;
        shifted_moments<C, G>(v, shift, live, s1, s2);
        group_sum2<G>(s1, s2, part_mean, part_sq, g, t);
        mu = s1 / n;
        var = s2 / n - mu * mu;
        // Every lane of a group holds the same bits, so the choice is uniform per group; with
        // several warps a row it is made CTA-wide, since the reduction has a barrier.
        const bool two_pass = !(mu * mu <= 4.0f * var);
        bool any;
        if constexpr (Sh::kWarpsPerRow > 1) any = __syncthreads_or(two_pass) != 0;
        else any = two_pass;
        if (any) {
            const float d2 = group_sum<G>(
                two_pass ? squared_deviations<C, G>(v, shift, mu, live) : 0.0f, part_var, g, t);
            if (two_pass) var = d2 / n;
        }
    } else {
        mu = group_sum<G>(shifted_sum<C, G>(v, shift, live), part_mean, g, t) / n;
        var = group_sum<G>(squared_deviations<C, G>(v, shift, mu, live), part_var, g, t) / n;
    }
    const float rstd = rsqrtf(var + eps);

    if (!active) return;
    const char* gt = static_cast<const char*>(gamma) + static_cast<int64_t>(t) * VB;
    const char* bt = static_cast<const char*>(beta) + static_cast<int64_t>(t) * VB;
    char* yr = static_cast<char*>(y) + off;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        if (k * G < live)
            st_out<VB>(yr + k * G * VB,
                       normalize<C>(v[k], ld_shared_ro<VB>(gt + k * G * VB),
                                    ld_shared_ro<VB>(bt + k * G * VB), shift, mu, rstd));
    }
}

template <typename S, int VB, int G, int NV>
cudaError_t launch_ln(const LayernormArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(layernorm_rows_kernel<S, VB, G, NV>, grid_2d(grid), dim3(LnShape<G>::kBlock),
                      s, a.x, a.gamma, a.beta, a.y, a.rows, a.cols, a.eps);
}

using LnFn = cudaError_t (*)(const LayernormArgs&, int64_t, cudaStream_t);

struct LnEntry {
    DType t;
    int vec_bytes, group, per_thread;
    LnFn fn;
};

#define CAMP_LN(S, DT, VB, G, NV) {DType::DT, VB, G, NV, &launch_ln<S, VB, G, NV>}
#define CAMP_LN_NV16(S, DT, G)                                                              \
    CAMP_LN(S, DT, 16, G, 1), CAMP_LN(S, DT, 16, G, 2), CAMP_LN(S, DT, 16, G, 3),           \
    CAMP_LN(S, DT, 16, G, 4), CAMP_LN(S, DT, 16, G, 6), CAMP_LN(S, DT, 16, G, 8)
#define CAMP_LN_FAST(S, DT)                                                                 \
    CAMP_LN_NV16(S, DT, 32), CAMP_LN_NV16(S, DT, 64), CAMP_LN_NV16(S, DT, 128),             \
    CAMP_LN_NV16(S, DT, 256), CAMP_LN_NV16(S, DT, 512), CAMP_LN_NV16(S, DT, 1024)
#define CAMP_LN_ELEM_G(S, DT, VB, G)                                                        \
    CAMP_LN(S, DT, VB, G, 1), CAMP_LN(S, DT, VB, G, 2), CAMP_LN(S, DT, VB, G, 4),           \
    CAMP_LN(S, DT, VB, G, 8), CAMP_LN(S, DT, VB, G, 16)
#define CAMP_LN_ELEM(S, DT, VB)                                                             \
    CAMP_LN_ELEM_G(S, DT, VB, 32), CAMP_LN_ELEM_G(S, DT, VB, 256), CAMP_LN_ELEM_G(S, DT, VB, 1024)

const LnEntry kLn[] = {
    CAMP_LN_FAST(bf16_t, BF16),
    CAMP_LN_FAST(f16_t, F16),
    CAMP_LN_FAST(f32_t, F32),
    CAMP_LN_ELEM(bf16_t, BF16, 2),
    CAMP_LN_ELEM(f16_t, F16, 2),
    CAMP_LN_ELEM(f32_t, F32, 4),
};

#undef CAMP_LN_ELEM
#undef CAMP_LN_ELEM_G
#undef CAMP_LN_FAST
#undef CAMP_LN_NV16
#undef CAMP_LN

}  // namespace

cudaError_t layernorm_rows_launch(DType t, int vec_bytes, int group, int per_thread,
                                  const LayernormArgs& a, int64_t grid, cudaStream_t s) {
    for (const LnEntry& e : kLn) {
        if (e.t == t && e.vec_bytes == vec_bytes && e.group == group &&
            e.per_thread == per_thread)
            return e.fn(a, grid, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace camp
