// Interleaved RoPE with device position ids, and on-device RoPE table generation, for
// sm_103a.
//
// Interleaved RoPE (xserv "phase 4", csrc/embedding/rope.cu): for each pair (x[2i], x[2i+1])
// of a head at position p = positions[token]:
//   y[2i]   = x[2i] cos - x[2i+1] sin,   y[2i+1] = x[2i] sin + x[2i+1] cos,
// with cos/sin = cos_table[p][i] / sin_table[p][i]. x is [tokens, H, D]; the tables are
// [max_pos, D/2]. A position outside [0, max_pos) leaves the token's rows unwritten (and
// reads nothing out of bounds). The products are the compensated 2x2 determinant of the
// rotate-half kernel, rounded once to the storage type.
//
// Mapping: the tiled mapping of the rotate-half kernel. A 16-byte vector holds E/2 whole
// pairs, so thread (position, head group, vector j) needs table values j*E/2 .. j*E/2 +
// E/2 - 1 of its position's row; it loads them once for its HPT heads.
//
// Tables (xserv compute_rope_cache): freq_i = theta^(-2i/D), angle = p * freq_i,
// cos/sin(angle). Here all of it is fp64 (the pow, the product and sin/cos are CUDA's
// double-precision functions) and each value is rounded once to fp32: an fp32 angle, as
// in xserv, is off by about ulp(angle) ~ 4e-3 rad at position 65536.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

template <typename S, int VB, int HPT>
__global__ void __launch_bounds__(kRopeBlock, rope_min_blocks(HPT))
rope_interleaved_kernel(const void* x, const float* __restrict__ sin_t,
                        const float* __restrict__ cos_t, const int32_t* __restrict__ positions,
                        void* y, int64_t tokens, int heads, int dim, int64_t max_pos) {
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int P = E / 2;                       // pairs per vector
    constexpr int ES = Storage<S>::kBytes;
    static_assert(E % 2 == 0, "a vector holds whole pairs");

    const int nv = dim / E;                                    // vectors per head row
    const int per_pos = ((heads + HPT - 1) / HPT) * nv;        // threads per token
    const int tpc = kRopeBlock / per_pos;
    const int tk = static_cast<int>(threadIdx.x) / per_pos;
    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0 && block * tpc < tokens) {   // this CTA's tokens of x (the table
                                                       // rows depend on the positions)
        const int64_t t0 = block * tpc;
        const int64_t nt = tokens - t0 < tpc ? tokens - t0 : tpc;
        const int64_t rb = static_cast<int64_t>(dim) * ES * heads;
        prefetch_l2(static_cast<const char*>(x) + t0 * rb, nt * rb);
    }
    griddep_wait();
    griddep_launch_dependents();
    const int64_t tok = block * tpc + tk;
    if (tk >= tpc || tok >= tokens) return;                    // no barrier in this kernel
    const int64_t p = positions[tok];
    if (p < 0 || p >= max_pos) return;                         // padding: not written
    const int r = static_cast<int>(threadIdx.x) - tk * per_pos;
    const int hg = r / nv;
    const int j = r - hg * nv;
    const int h0 = hg * HPT;
    const int nh = heads - h0 < HPT ? heads - h0 : HPT;

    const int64_t row_bytes = static_cast<int64_t>(dim) * ES;
    const int64_t off = (tok * heads + h0) * row_bytes + static_cast<int64_t>(j) * VB;
    const char* src = static_cast<const char*>(x) + off;
    Raw<VB> v[HPT];
#pragma unroll
    for (int u = 0; u < HPT; ++u)
        if (u < nh) v[u] = ld_stream<VB>(src + u * row_bytes);

    float sn[P], cs[P];
    const int64_t toff = p * (dim / 2) + static_cast<int64_t>(j) * P;
    load_table<P>(sin_t + toff, sn);
    load_table<P>(cos_t + toff, cs);

    char* dst = static_cast<char*>(y) + off;
#pragma unroll
    for (int u = 0; u < HPT; ++u) {
        if (u < nh) {
            float a[E], o[E];
            C::each(v[u], [&](int e, float f) { a[e] = f; });
#pragma unroll
            for (int q = 0; q < P; ++q) {
                o[2 * q] = diff_of_products(a[2 * q], cs[q], a[2 * q + 1], sn[q]);
                o[2 * q + 1] = sum_of_products(a[2 * q], sn[q], a[2 * q + 1], cs[q]);
            }
            st_out<VB>(dst + u * row_bytes, C::map(v[u], [&](int e, float) { return o[e]; }));
        }
    }
}

template <typename S, int VB, int HPT>
cudaError_t launch_interleaved(const RopeInterleavedArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(rope_interleaved_kernel<S, VB, HPT>, grid_2d(grid), dim3(kRopeBlock), s,
                      a.x, a.sin_t, a.cos_t, a.positions, a.y, a.tokens,
                      static_cast<int>(a.heads), static_cast<int>(a.dim), a.max_pos);
}

template <typename S, int VB>
cudaError_t launch_interleaved_hpt(int hpt, const RopeInterleavedArgs& a, int64_t grid,
                                   cudaStream_t s) {
    switch (hpt) {
        case 1: return launch_interleaved<S, VB, 1>(a, grid, s);
        case 2: return launch_interleaved<S, VB, 2>(a, grid, s);
        case 4: return launch_interleaved<S, VB, 4>(a, grid, s);
        case 8: return launch_interleaved<S, VB, 8>(a, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

// One thread per table entry (position p, frequency i), fp64 throughout, one rounding.
__global__ void __launch_bounds__(256)
rope_tables_kernel(float* sin_t, float* cos_t, int64_t max_pos, int half, double theta,
                   double dim) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = max_pos * half;
    for (int64_t id = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; id < n;
         id += static_cast<int64_t>(gridDim.x) * 256) {
        const int64_t p = id / half;
        const int i = static_cast<int>(id - p * half);
        const double freq = pow(theta, (-2.0 * static_cast<double>(i)) / dim);
        const double angle = static_cast<double>(p) * freq;
        double s, c;
        sincos(angle, &s, &c);
        sin_t[id] = static_cast<float>(s);
        cos_t[id] = static_cast<float>(c);
    }
}

}  // namespace

bool rope_interleaved_compiled(DType t, int vec_bytes, int heads_per_thread) {
    const bool hpt = heads_per_thread == 1 || heads_per_thread == 2 || heads_per_thread == 4 ||
                     heads_per_thread == 8;
    if (t != DType::F32) return hpt && (vec_bytes == 16 || vec_bytes == 8 || vec_bytes == 4);
    return hpt && (vec_bytes == 16 || vec_bytes == 8);
}

cudaError_t rope_interleaved_launch(DType t, int vec_bytes, int heads_per_thread,
                                    const RopeInterleavedArgs& a, int64_t grid,
                                    cudaStream_t s) {
    if (t == DType::BF16) {
        if (vec_bytes == 16) return launch_interleaved_hpt<bf16_t, 16>(heads_per_thread, a, grid, s);
        if (vec_bytes == 8) return launch_interleaved_hpt<bf16_t, 8>(heads_per_thread, a, grid, s);
        if (vec_bytes == 4) return launch_interleaved_hpt<bf16_t, 4>(heads_per_thread, a, grid, s);
    } else if (t == DType::F16) {
        if (vec_bytes == 16) return launch_interleaved_hpt<f16_t, 16>(heads_per_thread, a, grid, s);
        if (vec_bytes == 8) return launch_interleaved_hpt<f16_t, 8>(heads_per_thread, a, grid, s);
        if (vec_bytes == 4) return launch_interleaved_hpt<f16_t, 4>(heads_per_thread, a, grid, s);
    } else {
        if (vec_bytes == 16) return launch_interleaved_hpt<f32_t, 16>(heads_per_thread, a, grid, s);
        if (vec_bytes == 8) return launch_interleaved_hpt<f32_t, 8>(heads_per_thread, a, grid, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t rope_tables_launch(float* sin_t, float* cos_t, int64_t max_pos, int64_t dim,
                               double theta, cudaStream_t s) {
    const int64_t n = max_pos * (dim / 2);
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;   // grid-stride beyond
    return launch_pdl(rope_tables_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), s,
                      sin_t, cos_t, max_pos, static_cast<int>(dim / 2), theta,
                      static_cast<double>(dim));
}

}  // namespace camp
