// LayerNorm for rows wider than the staged kernel holds (any width), for sm_103a.
//
// Definition as in layernorm.cu (xserv "phase 4", csrc/normalization/layernorm.cu, whose
// kernel loops over any hidden size with a block-stride loop): y = gamma * (x - mean) /
// sqrt(var + eps) + beta with the population variance, in coordinates shifted by
// K = x[row, 0].
//
// Mapping: one CTA of kWideBlock threads per row (grid-strided over the rows), sweeping the
// row with block-stride loops; thread t touches vectors t, t + kWideBlock, ... in every
// sweep. A row this wide does not fit one CTA's registers or shared memory, so x is read
// more than once (the later sweeps mostly from L2):
//   1. sum(x - K), and in 16-bit storage also sum((x - K)^2), each thread accumulating with
//      Kahan's compensated summation (the per-thread error stays a few units of fp32
//      roundoff whatever the row length), one block reduction;
//   2. where the shift lies more than two standard deviations from the mean (the rows
//      kernel's rule; always in fp32 storage): sum(((x - K) - mu)^2), compensated, one block
//      reduction;
//   3. y = fma(((x - K) - mu) * rsqrt(var + eps), gamma, beta), with the loads of a few
//      vectors of x, gamma and beta issued before their stores.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

// Kahan's compensated summation of one fp32 stream.
struct Kahan {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float v) {
        const float yv = __fsub_rn(v, c);
        const float t = __fadd_rn(s, yv);
        c = __fsub_rn(__fsub_rn(t, s), yv);
        s = t;
    }
};

// Sum over the CTA (kWideBlock threads) through `part`; every thread gets the total.
__device__ __forceinline__ float block_sum(float v, float* part) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x / 32] = v;
    __syncthreads();
    return sum_partials<kWideBlock / 32>(part);
}

template <typename S, int VB>
__global__ void __launch_bounds__(kWideBlock)
layernorm_wide_kernel(const void* x, const void* __restrict__ gamma,
                      const void* __restrict__ beta, void* y, int64_t rows, int64_t cols,
                      float eps) {
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr int kU = VB == 16 ? 4 : 8;    // vector accesses in flight per thread
    constexpr int kUo = VB == 16 ? 2 : 8;   // the same in the output sweep (x, gamma, beta)
    constexpr bool kOnePass = ES == 2;
    // Three slots of warp partials: a reduction's slot is rewritten only after a later
    // reduction's barrier, or after the barrier that closes the row.
    __shared__ float part[3][kWideBlock / 32];

    const int64_t nvec = cols / E;
    const int64_t pitch = cols * ES;
    if (threadIdx.x == 0 && blockIdx.x < rows) {   // the start of this CTA's first row
        const int64_t n = pitch < 65536 ? pitch : 65536;
        prefetch_l2(static_cast<const char*>(x) + blockIdx.x * pitch, n);
    }
    griddep_wait();
    griddep_launch_dependents();

    const float n = static_cast<float>(cols);
    const int t = threadIdx.x;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const char* xr = static_cast<const char*>(x) + row * pitch;
        float shift = 0.0f;
        Codec<S, ES>::each(ld_stream<ES>(xr), [&](int, float f) { shift = f; });

        // 1. The compensated sums of this thread's elements.
        Kahan s1, s2;
        for (int64_t base = t; base < nvec; base += kU * kWideBlock) {
            Raw<VB> v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t idx = base + static_cast<int64_t>(u) * kWideBlock;
                v[u] = idx < nvec ? ld_stream<VB>(xr + idx * VB) : raw_zero<VB>();
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (base + static_cast<int64_t>(u) * kWideBlock < nvec)
                    C::each(v[u], [&](int, float f) {
                        const float d = f - shift;
                        s1.add(d);
                        if constexpr (kOnePass) s2.add(d * d);
                    });
            }
        }
        const float mu = block_sum(s1.s, part[0]) / n;
        float var = 0.0f;
        bool again = true;
        if constexpr (kOnePass) {
            var = block_sum(s2.s, part[1]) / n - mu * mu;
            again = !(mu * mu <= 4.0f * var);   // the same in every thread
        }
        // 2. The second pass, where the one-pass difference could cancel.
        if (again) {
            Kahan s3;
            for (int64_t base = t; base < nvec; base += kU * kWideBlock) {
                Raw<VB> v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int64_t idx = base + static_cast<int64_t>(u) * kWideBlock;
                    v[u] = idx < nvec ? ld_stream<VB>(xr + idx * VB) : raw_zero<VB>();
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if (base + static_cast<int64_t>(u) * kWideBlock < nvec)
                        C::each(v[u], [&](int, float f) {
                            const float d = (f - shift) - mu;
                            s3.add(d * d);
                        });
                }
            }
            var = block_sum(s3.s, part[2]) / n;
        }
        const float rstd = rsqrtf(var + eps);

        // 3. The output sweep.
        const char* gb = static_cast<const char*>(gamma);
        const char* bb = static_cast<const char*>(beta);
        char* yr = static_cast<char*>(y) + row * pitch;
        for (int64_t base = t; base < nvec; base += kUo * kWideBlock) {
            Raw<VB> v[kUo], gv[kUo], bv[kUo];
#pragma unroll
            for (int u = 0; u < kUo; ++u) {
                const int64_t idx = base + static_cast<int64_t>(u) * kWideBlock;
                if (idx < nvec) {
                    v[u] = ld_stream<VB>(xr + idx * VB);
                    gv[u] = ld_shared_ro<VB>(gb + idx * VB);
                    bv[u] = ld_shared_ro<VB>(bb + idx * VB);
                }
            }
#pragma unroll
            for (int u = 0; u < kUo; ++u) {
                const int64_t idx = base + static_cast<int64_t>(u) * kWideBlock;
                if (idx < nvec) {
                    float gf[E], bf[E];
                    C::each(gv[u], [&](int e, float f) { gf[e] = f; });
                    C::each(bv[u], [&](int e, float f) { bf[e] = f; });
                    st_out<VB>(yr + idx * VB, C::map(v[u], [&](int e, float f) {
                                   return fmaf(((f - shift) - mu) * rstd, gf[e], bf[e]);
                               }));
                }
            }
        }
        __syncthreads();   // part[] is reused by the next row
    }
}

template <typename S, int VB>
cudaError_t launch_wide(const LayernormArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(layernorm_wide_kernel<S, VB>, dim3(static_cast<unsigned>(grid)),
                      dim3(kWideBlock), s, a.x, a.gamma, a.beta, a.y, a.rows, a.cols, a.eps);
}

}  // namespace

bool layernorm_wide_compiled(DType t, int vec_bytes) {
    return vec_bytes == 16 || vec_bytes == elem_bytes(t);
}

cudaError_t layernorm_wide_launch(DType t, int vec_bytes, const LayernormArgs& a, int64_t grid,
                                  cudaStream_t s) {
    switch (t) {
        case DType::BF16:
            if (vec_bytes == 16) return launch_wide<bf16_t, 16>(a, grid, s);
            if (vec_bytes == 2) return launch_wide<bf16_t, 2>(a, grid, s);
            break;
        case DType::F16:
            if (vec_bytes == 16) return launch_wide<f16_t, 16>(a, grid, s);
            if (vec_bytes == 2) return launch_wide<f16_t, 2>(a, grid, s);
            break;
        default:
            if (vec_bytes == 16) return launch_wide<f32_t, 16>(a, grid, s);
            if (vec_bytes == 4) return launch_wide<f32_t, 4>(a, grid, s);
            break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace camp
