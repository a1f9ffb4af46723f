// RMSNorm forward kernels for sm_103a, plain and with a fused residual add. Included by
// rmsnorm.cu (ADD = false) and rmsnorm_add.cu (ADD = true), one translation unit each.
//
// Definition (xserv "phase 4" design notes, RMSNorm section): per row,
// rms = sqrt(sum(x^2) / hidden + eps) and y = x / rms * gamma. Design constraints from
// the gollamago README ("RMSNorm optimisation (TileLang)"): a bandwidth-bound operator
// must read each row from global memory once (a second read "doubles the read
// traffic") and write it once; the sum of squares and the scaling stay in fp32 and
// the result is rounded once on write-back.
//
// Fused residual add (the "Add before RmsNorm" fusion the TileLang tutorial, ch. 02
// section 4.2, cites from Ascend's AddRmsNorm operators, done to save a round trip
// through memory): h = x + r is formed in fp32, rounded once to the storage type and
// stored, and the row that is normalized is h as stored; so the fused call gives exactly
// what an add followed by an RMSNorm gives, with one read of x and r and no re-read of h.
//
// rmsnorm_rows_kernel: a group of G threads owns one row. Each thread issues all of its
// NV vector loads up front (16-byte accesses on the fast path), keeps the raw vectors in
// registers, reduces its share of sum(x^2) in fp32, combines the group with a butterfly
// warp shuffle (and, for G > 32, a small shared-memory exchange between the group's
// warps), and then writes y from the registers. x is read from HBM exactly once; w is
// an L1-resident load shared by every row on the SM.
//
// rmsnorm_cluster_kernel: a cluster of C CTAs owns one row, each CTA a contiguous chunk
// of 256 * NV vectors held in registers (rows too wide for one CTA's registers). Every
// CTA reduces its chunk and stores the partial sum into a slot of every CTA of the
// cluster (distributed shared memory); after one hardware cluster barrier each CTA sums
// the C slots in rank order, so all get the same sum. x is read from HBM once; there is
// no spinning. (rmsnorm_staged.cu holds the shared-memory-staged alternative.)
//
// rmsnorm_wide_kernel: rows wider than a cluster's registers take two sweeps in one CTA per
// row (the second sweep re-reads x, or h on the add path, mostly from L2).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace rms {

template <int G>
struct RowsShape {
    static constexpr int kBlock = rows_block(G);        // threads per CTA
    static constexpr int kRowsPerCta = kBlock / G;
    static constexpr int kWarpsPerRow = G / 32;
};

// This thread's share of sum(x^2) over its NV raw vectors (zeros where it has none), in
// fp32: two packed accumulators (even and odd elements) where an access holds pairs.
template <typename C, int NV, int VB>
__device__ __forceinline__ float sum_squares(const Raw<VB> (&v)[NV]) {
    if constexpr (C::kElems >= 2) {
        f32x2 acc = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) C::each_pair(v[k], [&](int, f32x2 p) { acc = f2_fma(p, p, acc); });
        return f2_lo(acc) + f2_hi(acc);
    } else {
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) C::each(v[k], [&](int, float f) { ss = fmaf(f, f, ss); });
        return ss;
    }
}

// One output access: (x * rinv) * w per element, in fp32, rounded once.
template <typename C, int VB>
__device__ __forceinline__ Raw<VB> scale_row(const Raw<VB>& xv, const Raw<VB>& wv, float rinv) {
    if constexpr (C::kElems >= 2) {
        f32x2 wp[C::kPairs];
        C::each_pair(wv, [&](int p, f32x2 q) { wp[p] = q; });
        const f32x2 r2 = f2_make(rinv, rinv);
        return C::map_pair(xv, [&](int p, f32x2 xp) { return f2_mul(f2_mul(xp, r2), wp[p]); });
    } else {
        float wf[C::kElems];
        C::each(wv, [&](int e, float f) { wf[e] = f; });
        return C::map(xv, [&](int e, float xf) { return (xf * rinv) * wf[e]; });
    }
}

// Load access k of this thread (x, or h = x + r stored on the way on the add path).
template <typename S, int VB, bool ADD, int NV>
__device__ __forceinline__ void load_row(const char* xr, const char* rr, char* hr, int live,
                                         int stride_bytes, int stride_vecs, Raw<VB> (&v)[NV],
                                         bool active) {
    using C = Codec<S, VB>;
    if constexpr (!ADD) {
#pragma unroll
        for (int k = 0; k < NV; ++k)
            v[k] = (active && k * stride_vecs < live) ? ld_stream<VB>(xr + k * stride_bytes)
                                                      : raw_zero<VB>();
    } else {
        Raw<VB> rv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const bool on = active && k * stride_vecs < live;
            v[k] = on ? ld_stream<VB>(xr + k * stride_bytes) : raw_zero<VB>();
            rv[k] = on ? ld_stream<VB>(rr + k * stride_bytes) : raw_zero<VB>();
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            v[k] = C::add(v[k], rv[k]);
            if (active && k * stride_vecs < live) st_out<VB>(hr + k * stride_bytes, v[k]);
        }
    }
}

template <typename S, int VB, int G, int NV, bool ADD>
__global__ void __launch_bounds__(RowsShape<G>::kBlock, rows_min_blocks(VB, G, ADD ? 2 * NV : NV))
rmsnorm_rows_kernel(const void* x, const void* r, void* h, const void* __restrict__ w, void* y,
                    int64_t rows, int64_t cols, float eps) {
    static_assert(G % 32 == 0 && G <= 1024, "a row group is whole warps");
    using Sh = RowsShape<G>;
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;

    __shared__ float partial[Sh::kRowsPerCta][Sh::kWarpsPerRow];

    // One row block per CTA (the host sizes the grid; a second grid dimension only
    // appears for more than 2^31 - 1 blocks).
    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0 && block * Sh::kRowsPerCta < rows) {   // this CTA's rows of x (and r)
        const int64_t row0 = block * Sh::kRowsPerCta;
        const int64_t n = (rows - row0 < Sh::kRowsPerCta ? rows - row0 : Sh::kRowsPerCta) * cols * ES;
        prefetch_l2(static_cast<const char*>(x) + row0 * cols * ES, n);
        if constexpr (ADD) prefetch_l2(static_cast<const char*>(r) + row0 * cols * ES, n);
        // Without the residual add, and when x is small next to L2 (at most 32 MB), also the
        // rows of the CTA one resident wave later, so that a second wave finds its rows in
        // L2 (bf16 4096 x 3000: 9.47 -> 9.08 us, 8192 x 2048: 11.8 -> 11.2 us; the add path
        // measured no gain).
        if (!ADD && rows * cols * ES <= (int64_t{32} << 20)) {
            const int64_t wave = static_cast<int64_t>(rows_min_blocks(VB, G, NV)) * sm_id_count();
            const int64_t r1 = (block + wave) * Sh::kRowsPerCta;
            if (r1 < rows) {
                const int64_t n1 = (rows - r1 < Sh::kRowsPerCta ? rows - r1 : Sh::kRowsPerCta) * cols * ES;
                prefetch_l2(static_cast<const char*>(x) + r1 * cols * ES, n1);
            }
        }
    }
    griddep_wait();
    griddep_launch_dependents();

    const int g = threadIdx.x / G;       // row slot inside the CTA
    const int t = threadIdx.x % G;       // thread inside the row group
    const int64_t row = block * Sh::kRowsPerCta + g;
    const bool active = row < rows;
    // Access k of this thread is vector k*G + t of the row; it exists iff k*G < live.
    // On this path a row has at most G*NV <= 16384 vectors, so 32 bits suffice.
    const int live = static_cast<int>(cols / E) - t;
    const int64_t off = row * cols * ES + static_cast<int64_t>(t) * VB;

    // One sweep of loads: everything this thread needs is in flight at once.
    Raw<VB> v[NV];
    load_row<S, VB, ADD, NV>(static_cast<const char*>(x) + off,
                             ADD ? static_cast<const char*>(r) + off : nullptr,
                             ADD ? static_cast<char*>(h) + off : nullptr, live, G * VB, G, v,
                             active);

    float ss = sum_squares<C>(v);
    ss = warp_sum(ss);
    if constexpr (Sh::kWarpsPerRow > 1) {
        if ((threadIdx.x & 31) == 0) partial[g][t / 32] = ss;
        __syncthreads();
        ss = sum_partials<Sh::kWarpsPerRow>(partial[g]);
    }
    const float rinv = rsqrtf(ss / static_cast<float>(cols) + eps);

    if (!active) return;
    const char* wt = static_cast<const char*>(w) + static_cast<int64_t>(t) * VB;
    char* yr = static_cast<char*>(y) + off;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        if (k * G < live)
            st_out<VB>(yr + k * G * VB, scale_row<C>(v[k], ld_shared_ro<VB>(wt + k * G * VB), rinv));
    }
}

template <typename S, int NV, bool ADD>
__global__ void __launch_bounds__(kClusterBlock, rows_min_blocks(16, kClusterBlock, ADD ? 2 * NV : NV))
rmsnorm_cluster_kernel(const void* x, const void* r, void* h, const void* __restrict__ w,
                       void* y, int64_t rows, int64_t cols, float eps) {
    namespace cg = cooperative_groups;
    constexpr int VB = 16;
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr int kWarps = kClusterBlock / 32;

    __shared__ float partial[kWarps];
    __shared__ float slot[16];   // slot[r]: the partial sum of cluster rank r

    // First phase of the cluster barrier, split: arrive now, wait just before the remote
    // stores below, so every CTA of the cluster has started (and owns its shared memory)
    // before any CTA writes into it; the wait costs nothing by then.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    cg::cluster_group cluster = cg::this_cluster();
    const unsigned nct = cluster.num_blocks();
    const unsigned rank = cluster.block_rank();
    const int t = threadIdx.x;
    const int64_t row = static_cast<int64_t>(blockIdx.x) / nct;   // the host launches rows * C CTAs
    if (t == 0 && row < rows) {   // this CTA's chunk of the row (and of r)
        const int64_t v0 = static_cast<int64_t>(rank) * NV * kClusterBlock;
        const int64_t left = cols / E - v0;
        const int64_t n = (left < NV * kClusterBlock ? left : NV * kClusterBlock) * VB;
        prefetch_l2(static_cast<const char*>(x) + row * cols * ES + v0 * VB, n);
        if constexpr (ADD) prefetch_l2(static_cast<const char*>(r) + row * cols * ES + v0 * VB, n);
    }

    griddep_wait();
    griddep_launch_dependents();
    // Access k of this thread is vector (rank*NV + k)*256 + t of the row; live iff < nvec.
    const int live = static_cast<int>(cols / E) - static_cast<int>(rank) * NV * kClusterBlock - t;
    const int64_t off = row * cols * ES +
                        (static_cast<int64_t>(rank) * NV * kClusterBlock + t) * VB;

    Raw<VB> v[NV];
    load_row<S, VB, ADD, NV>(static_cast<const char*>(x) + off,
                             ADD ? static_cast<const char*>(r) + off : nullptr,
                             ADD ? static_cast<char*>(h) + off : nullptr, live,
                             kClusterBlock * VB, kClusterBlock, v, true);

    float ss = warp_sum(sum_squares<C>(v));
    if ((t & 31) == 0) partial[t / 32] = ss;
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    // Thread r < C writes this CTA's partial into slot[rank] of cluster rank r: one round of
    // remote stores, then a single cluster barrier (its release/acquire makes the stores
    // visible, and no shared memory of another CTA is touched after it).
    if (t < static_cast<int>(nct)) {
        float c = 0.0f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) c += partial[i];
        *cluster.map_shared_rank(&slot[rank], static_cast<unsigned>(t)) = c;
    }
    cluster.sync();
    ss = 0.0f;
    for (unsigned q = 0; q < nct; ++q) ss += slot[q];          // rank order in every CTA
    const float rinv = rsqrtf(ss / static_cast<float>(cols) + eps);

    (void)rows;
    const char* wt = static_cast<const char*>(w) +
                     (static_cast<int64_t>(rank) * NV * kClusterBlock + t) * VB;
    char* yr = static_cast<char*>(y) + off;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        if (k * kClusterBlock < live)
            st_out<VB>(yr + k * kClusterBlock * VB,
                       scale_row<C>(v[k], ld_shared_ro<VB>(wt + k * kClusterBlock * VB), rinv));
    }
}

template <typename S, int VB, bool ADD>
__global__ void __launch_bounds__(kWideBlock)
rmsnorm_wide_kernel(const void* x, const void* r, void* h, const void* __restrict__ w, void* y,
                    int64_t rows, int64_t cols, float eps) {
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr int kUnroll = 4;
    __shared__ float partial[kWideBlock / 32];

    const int64_t nvec = cols / E;
    const int64_t pitch = cols * ES;
    if (threadIdx.x == 0 && blockIdx.x < rows) {   // the start of this CTA's first row
        const int64_t n = pitch < 65536 ? pitch : 65536;
        prefetch_l2(static_cast<const char*>(x) + blockIdx.x * pitch, n);
        if constexpr (ADD) prefetch_l2(static_cast<const char*>(r) + blockIdx.x * pitch, n);
    }

    griddep_wait();
    griddep_launch_dependents();

    const char* wb = static_cast<const char*>(w);
    const float fcols = static_cast<float>(cols);

    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const char* xr = static_cast<const char*>(x) + row * pitch;
        const char* rr = ADD ? static_cast<const char*>(r) + row * pitch : nullptr;
        char* hr = ADD ? static_cast<char*>(h) + row * pitch : nullptr;
        float ss = 0.0f;
        // Sweep 1: sum of squares (and h = x + r, stored, on the add path). Every index a
        // thread touches is threadIdx.x mod kWideBlock, in both sweeps, so a thread re-reads
        // only what it wrote itself.
        for (int64_t base = threadIdx.x; base < nvec; base += kUnroll * kWideBlock) {
            Raw<VB> v[kUnroll];
            load_row<S, VB, ADD, kUnroll>(xr + base * VB, rr ? rr + base * VB : nullptr,
                                          hr ? hr + base * VB : nullptr,
                                          static_cast<int>(nvec - base < 0x40000000 ? nvec - base : 0x40000000),
                                          kWideBlock * VB, kWideBlock, v, true);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) C::each(v[u], [&](int, float f) { ss = fmaf(f, f, ss); });
        }
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) partial[threadIdx.x / 32] = ss;
        __syncthreads();
        ss = sum_partials<kWideBlock / 32>(partial);
        const float rinv = rsqrtf(ss / fcols + eps);

        // Sweep 2: normalize the row as stored (x, or h on the add path).
        const char* src = ADD ? static_cast<const char*>(hr) : xr;
        char* yr = static_cast<char*>(y) + row * pitch;
        for (int64_t idx = threadIdx.x; idx < nvec; idx += kWideBlock) {
            st_out<VB>(yr + idx * VB,
                       scale_row<C>(ld_stream<VB>(src + idx * VB), ld_shared_ro<VB>(wb + idx * VB), rinv));
        }
        __syncthreads();   // partial[] is reused by the next row
    }
}

// ------------------------------------------------------------------ launchers

template <typename S, int VB, int G, int NV, bool ADD>
cudaError_t launch_rows(const RmsnormArgs& a, int64_t grid, cudaStream_t s) {
    if constexpr (!rows_variant_compiled(ADD, VB, G, NV)) {
        return cudaErrorInvalidValue;   // not built (see rows_variant_compiled)
    } else {
        return launch_pdl(rmsnorm_rows_kernel<S, VB, G, NV, ADD>, grid_2d(grid),
                          dim3(RowsShape<G>::kBlock), s, a.x, a.r, a.h, a.w, a.y, a.rows,
                          a.cols, a.eps);
    }
}

template <typename S, int VB, bool ADD>
cudaError_t launch_wide(const RmsnormArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(rmsnorm_wide_kernel<S, VB, ADD>, dim3(static_cast<unsigned>(grid)),
                      dim3(kWideBlock), s, a.x, a.r, a.h, a.w, a.y, a.rows, a.cols, a.eps);
}

template <typename S, int NV, bool ADD>
cudaError_t launch_cluster(const RmsnormArgs& a, int cluster, cudaStream_t s) {
    auto kernel = rmsnorm_cluster_kernel<S, NV, ADD>;
    if (cluster > 8) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.rows * cluster));
    cfg.blockDim = dim3(kClusterBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, a.x, a.r, a.h, a.w, a.y, a.rows, a.cols, a.eps);
}

// ------------------------------------------------------------------ dispatch tables

using RowsFn = cudaError_t (*)(const RmsnormArgs&, int64_t, cudaStream_t);

struct RowsEntry {
    DType t;
    int vec_bytes, group, per_thread;
    RowsFn fn;
};

#define CAMP_ROWS(S, DT, VB, G, NV, A) {DType::DT, VB, G, NV, &launch_rows<S, VB, G, NV, A>}

#define CAMP_ROWS_NV16(S, DT, G, A)                                                           \
    CAMP_ROWS(S, DT, 16, G, 1, A), CAMP_ROWS(S, DT, 16, G, 2, A), CAMP_ROWS(S, DT, 16, G, 3, A), \
    CAMP_ROWS(S, DT, 16, G, 4, A), CAMP_ROWS(S, DT, 16, G, 6, A), CAMP_ROWS(S, DT, 16, G, 8, A)

#define CAMP_ROWS_FAST(S, DT, A)                                                              \
    CAMP_ROWS_NV16(S, DT, 32, A), CAMP_ROWS_NV16(S, DT, 64, A), CAMP_ROWS_NV16(S, DT, 128, A),  \
    CAMP_ROWS_NV16(S, DT, 256, A), CAMP_ROWS_NV16(S, DT, 512, A), CAMP_ROWS_NV16(S, DT, 1024, A)

#define CAMP_ROWS_ELEM_G(S, DT, VB, G, A)                                                     \
    CAMP_ROWS(S, DT, VB, G, 1, A), CAMP_ROWS(S, DT, VB, G, 2, A), CAMP_ROWS(S, DT, VB, G, 4, A), \
    CAMP_ROWS(S, DT, VB, G, 8, A), CAMP_ROWS(S, DT, VB, G, 16, A)

#define CAMP_ROWS_ELEM(S, DT, VB, A)                                                          \
    CAMP_ROWS_ELEM_G(S, DT, VB, 32, A), CAMP_ROWS_ELEM_G(S, DT, VB, 256, A),                  \
    CAMP_ROWS_ELEM_G(S, DT, VB, 1024, A)

// Every compiled register-resident variant; rmsnorm_rows_compiled() lists the same set.
template <bool ADD>
struct Tables {
    static cudaError_t rows(DType t, int vec_bytes, int group, int per_thread,
                            const RmsnormArgs& a, int64_t grid, cudaStream_t s) {
        static const RowsEntry kRows[] = {
            CAMP_ROWS_FAST(bf16_t, BF16, ADD),
            CAMP_ROWS_FAST(f16_t, F16, ADD),
            CAMP_ROWS_FAST(f32_t, F32, ADD),
            CAMP_ROWS_ELEM(bf16_t, BF16, 2, ADD),
            CAMP_ROWS_ELEM(f16_t, F16, 2, ADD),
            CAMP_ROWS_ELEM(f32_t, F32, 4, ADD),
        };
        for (const RowsEntry& e : kRows) {
            if (e.t == t && e.vec_bytes == vec_bytes && e.group == group &&
                e.per_thread == per_thread)
                return e.fn(a, grid, s);
        }
        return cudaErrorInvalidValue;
    }

    static cudaError_t cluster(DType t, int per_thread, int cl, const RmsnormArgs& a,
                               cudaStream_t s) {
        if (cl < 2 || cl > 16 || (cl & (cl - 1)) != 0) return cudaErrorInvalidValue;
        switch (t) {
            case DType::BF16: return cluster_nv<bf16_t>(per_thread, cl, a, s);
            case DType::F16: return cluster_nv<f16_t>(per_thread, cl, a, s);
            default: return cluster_nv<f32_t>(per_thread, cl, a, s);
        }
    }

    template <typename S>
    static cudaError_t cluster_nv(int per_thread, int cl, const RmsnormArgs& a, cudaStream_t s) {
        switch (per_thread) {
            case 1: return launch_cluster<S, 1, ADD>(a, cl, s);
            case 2: return launch_cluster<S, 2, ADD>(a, cl, s);
            case 3: return launch_cluster<S, 3, ADD>(a, cl, s);
            case 4: return launch_cluster<S, 4, ADD>(a, cl, s);
            case 6: return launch_cluster<S, 6, ADD>(a, cl, s);
            case 8: return launch_cluster<S, 8, ADD>(a, cl, s);
            default: return cudaErrorInvalidValue;
        }
    }

    static cudaError_t wide(DType t, int vec_bytes, const RmsnormArgs& a, int64_t grid,
                            cudaStream_t s) {
        if (t == DType::BF16) {
            if (vec_bytes == 16) return launch_wide<bf16_t, 16, ADD>(a, grid, s);
            if (vec_bytes == 2) return launch_wide<bf16_t, 2, ADD>(a, grid, s);
        } else if (t == DType::F16) {
            if (vec_bytes == 16) return launch_wide<f16_t, 16, ADD>(a, grid, s);
            if (vec_bytes == 2) return launch_wide<f16_t, 2, ADD>(a, grid, s);
        } else {
            if (vec_bytes == 16) return launch_wide<f32_t, 16, ADD>(a, grid, s);
            if (vec_bytes == 4) return launch_wide<f32_t, 4, ADD>(a, grid, s);
        }
        return cudaErrorInvalidValue;
    }
};

#undef CAMP_ROWS_ELEM
#undef CAMP_ROWS_ELEM_G
#undef CAMP_ROWS_FAST
#undef CAMP_ROWS_NV16
#undef CAMP_ROWS

}  // namespace rms
}  // namespace camp
