// Shared-memory-staged LayerNorm for wide rows, for sm_103a.
//
// Definition as in layernorm.cu (xserv "phase 4", csrc/normalization/layernorm.cu and the
// design notes' LayerNorm section): y = gamma * (x - mean) / sqrt(var + eps) + beta with the
// population variance, taken in two passes from the shift K = x[row, 0]:
// mu = sum(x - K) / n, d = (x - K) - mu, var = sum(d^2) / n, y = fma(d * rstd, gamma, beta).
//
// Mapping: the staged RMSNorm kernel's (rmsnorm_staged.cu). Persistent clusters of C CTAs;
// CTA rank k owns a contiguous chunk of 16-byte vectors of every row of its cluster and
// reads its chunks of gamma and beta through L1 in the output pass (the same chunk every
// row, so they stay cached; holding them in shared memory cost a third of the CTAs an SM
// could run). A ring of `stages` row buffers is
// filled by bulk asynchronous copies: each copies the CTA's chunk plus the row's first 16
// bytes (every CTA needs the shift K). Per row, each CTA takes the statistics of its own
// chunk in two passes over its registers, in shifted coordinates: m_k = sum(x - K) / n_k and
// M2_k = sum(((x - K) - m_k)^2); one exchange sends (m_k, M2_k) to every CTA of the cluster
// (st.async stores counted on the receiving CTA's mbarrier; two slot sets alternating by
// row), and every CTA merges the C pairs with Chan, Golub and LeVeque's pairwise formula
// (mu = sum n_k m_k / n, M2 = sum M2_k + sum n_k (m_k - mu)^2; lane k of each warp takes
// pair k and warp butterflies sum, the same bits in every warp and CTA): one
// cluster round trip a row instead of one per statistic, and no value rounded in
// unshifted coordinates. The buffer is refilled as soon as the CTA has moved its vectors
// into registers.
//
// Waits: every mbarrier wait gives up after one second; a CTA whose wait ran out sets a bit
// in this file's device error word (read by camp_device_errors), stops issuing copies and
// storing, keeps sending and receiving partials, and before returning waits (at most a
// second each) for the copies it still has in flight.
#include <cooperative_groups.h>

#include "staged.cuh"

namespace camp {
namespace {

using namespace staged;

__device__ unsigned int g_ln_device_error = 0;

// Sum of (x - K) over one access, as packed pairs.
template <typename C>
__device__ __forceinline__ float shifted16(const Raw<16>& v, f32x2 k2) {
    f32x2 acc = f2_make(0.0f, 0.0f);
    C::each_pair(v, [&](int, f32x2 p) { acc = f2_add(acc, f2_sub(p, k2)); });
    return f2_lo(acc) + f2_hi(acc);
}

// Sum of ((x - K) - mu)^2 over one access.
template <typename C>
__device__ __forceinline__ float deviations16(const Raw<16>& v, f32x2 k2, f32x2 m2) {
    f32x2 acc = f2_make(0.0f, 0.0f);
    C::each_pair(v, [&](int, f32x2 p) {
        const f32x2 d = f2_sub(f2_sub(p, k2), m2);
        acc = f2_fma(d, d, acc);
    });
    return f2_lo(acc) + f2_hi(acc);
}

template <typename C>
__device__ __forceinline__ Raw<16> affine16(const Raw<16>& xv, const Raw<16>& gv,
                                            const Raw<16>& bv, f32x2 k2, f32x2 m2, f32x2 r2) {
    f32x2 gp[C::kPairs], bp[C::kPairs];
    C::each_pair(gv, [&](int p, f32x2 q) { gp[p] = q; });
    C::each_pair(bv, [&](int p, f32x2 q) { bp[p] = q; });
    return C::map_pair(xv, [&](int p, f32x2 xp) {
        return f2_fma(f2_mul(f2_sub(f2_sub(xp, k2), m2), r2), gp[p], bp[p]);
    });
}

// Store v into a (possibly remote) CTA's shared memory as two 4-byte st.async stores.
__device__ __forceinline__ void send_pair(float* slot_m, float* slot_v, unsigned long long* bar,
                                          float m, float v, int rank, int peer) {
    const uint32_t b = map_rank(smem_u32(bar), static_cast<uint32_t>(peer));
    st_async_f32(map_rank(smem_u32(&slot_m[rank]), static_cast<uint32_t>(peer)), m, b);
    st_async_f32(map_rank(smem_u32(&slot_v[rank]), static_cast<uint32_t>(peer)), v, b);
}

template <typename S, int NVT>
__global__ void __launch_bounds__(kStagedBlock, 1)
layernorm_staged_kernel(const void* x, const void* __restrict__ gamma,
                        const void* __restrict__ beta, void* y, int64_t rows, int64_t cols,
                        float eps, int chunk_vecs, int stages) {
    namespace cg = cooperative_groups;
    using C = Codec<S, 16>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr int kWarps = kStagedBlock / 32;

    // Dynamic shared memory: gamma chunk, beta chunk, then `stages` buffers of (the row's
    // first 16 bytes, the CTA's chunk of the row).
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[kStagedMaxStages];
    __shared__ __align__(8) unsigned long long bar_x[2];   // this row's (m_k, M2_k) pairs
    __shared__ float part_a[2][kWarps], part_b[2][kWarps];
    __shared__ float slot_m[2][16], slot_v[2][16];
    __shared__ int timed_out;

    cg::cluster_group cluster = cg::this_cluster();
    const int nct = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t ncl = gridDim.x / nct;
    const int64_t cid = blockIdx.x / nct;
    const int t = threadIdx.x;
    const int64_t nvec = cols / E;
    const int64_t v0 = static_cast<int64_t>(rank) * chunk_vecs;
    const int64_t left = nvec - v0;
    const int my_vecs = left <= 0 ? 0 : (left < chunk_vecs ? static_cast<int>(left) : chunk_vecs);
    const uint32_t my_bytes = static_cast<uint32_t>(my_vecs) * 16u;
    const int64_t pitch = cols * ES;
    const int64_t stage_bytes = 16 + static_cast<int64_t>(chunk_vecs) * 16;
    unsigned char* ring = smem;

    if (t == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&full[s]), 1);
        mbar_init(smem_u32(&bar_x[0]), 1);
        mbar_init(smem_u32(&bar_x[1]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        timed_out = 0;
        // The chunks that the first bulk loads below, and the first output pass, will read
        // (after griddep_wait).
        prefetch_l2(static_cast<const char*>(gamma) + v0 * 16, my_bytes);
        prefetch_l2(static_cast<const char*>(beta) + v0 * 16, my_bytes);
        for (int s = 0; s < stages; ++s) {
            const int64_t row = cid + s * ncl;
            if (row >= rows) break;
            prefetch_l2(static_cast<const char*>(x) + row * pitch, 16);
            prefetch_l2(static_cast<const char*>(x) + row * pitch + v0 * 16, my_bytes);
        }
    }
    // Every CTA of the cluster has started and initialized its barriers before any CTA
    // stores into a peer's shared memory (split cluster barrier).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    __syncthreads();

    griddep_wait();
    griddep_launch_dependents();

    const char* xb = static_cast<const char*>(x);
    auto issue = [&](int s, int64_t row) {   // one thread: the row's head and this chunk
        const uint32_t bar = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(ring + s * stage_bytes);
        mbar_arrive_expect_tx(bar, 16u + my_bytes);
        bulk_load(dst, xb + row * pitch, 16u, bar);
        if (my_bytes > 0) bulk_load(dst + 16, xb + row * pitch + v0 * 16, my_bytes, bar);
    };
    if (t == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t row = cid + s * ncl;
            if (row < rows) issue(s, row);
        }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    const float n = static_cast<float>(cols);
    // Elements of cluster rank `lane` (lanes past the cluster: none), for the merge.
    float n_lane = 0.0f;
    {
        const int lane = t & 31;
        const int64_t lq = nvec - static_cast<int64_t>(lane) * chunk_vecs;
        if (lane < nct && lq > 0) n_lane = static_cast<float>((lq < chunk_vecs ? lq : chunk_vecs) * E);
    }
    int64_t fail_iter = -1;
    int64_t i = 0;
    for (int64_t row = cid; row < rows; row += ncl, ++i) {
        const int s = static_cast<int>(i % stages);
        const int set = static_cast<int>(i & 1);
        const unsigned char* buf = ring + s * stage_bytes;
        if (fail_iter < 0 &&
            !mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>((i / stages) & 1)))
            timed_out = 1;
        __syncthreads();
        if (fail_iter < 0 && timed_out) fail_iter = i;   // the same in every thread
        const bool ok = fail_iter < 0;

        // The shift (the row's first element) and this thread's vectors, into registers.
        float shift = 0.0f;
        Raw<16> v[NVT];
        if (ok) Codec<S, 16>::each(ld_smem16(buf), [&](int e, float f) { if (e == 0) shift = f; });
#pragma unroll
        for (int k = 0; k < NVT; ++k) {
            const int vi = t + k * kStagedBlock;
            v[k] = (ok && vi < my_vecs) ? ld_smem16(buf + 16 + vi * 16) : raw_zero<16>();
        }
        const f32x2 k2 = f2_make(shift, shift);
        // This CTA's chunk: m_k = sum(x - K) / n_k ...
        float a = 0.0f;
#pragma unroll
        for (int k = 0; k < NVT; ++k)
            if (t + k * kStagedBlock < my_vecs) a += shifted16<C>(v[k], k2);
        a = warp_sum(a);
        if ((t & 31) == 0) part_a[set][t / 32] = a;
        __syncthreads();   // the buffer has been read: refill it now
        if (ok && t == 0) {
            const int64_t next = row + stages * ncl;
            if (next < rows) {
                // Order this CTA's generic-proxy reads of the buffer before the async-proxy
                // write that refills it.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(s, next);
            }
        }
        float sa = 0.0f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) sa += part_a[set][k];
        const float m_k = my_vecs > 0 ? sa / static_cast<float>(my_vecs * E) : 0.0f;
        // ... and M2_k = sum(((x - K) - m_k)^2)
        const f32x2 mk2 = f2_make(m_k, m_k);
        float b = 0.0f;
#pragma unroll
        for (int k = 0; k < NVT; ++k)
            if (t + k * kStagedBlock < my_vecs) b += deviations16<C>(v[k], k2, mk2);
        b = warp_sum(b);
        if ((t & 31) == 0) part_b[set][t / 32] = b;
        __syncthreads();
        if (t == 0) mbar_arrive_expect_tx(smem_u32(&bar_x[set]), static_cast<uint32_t>(nct) * 8u);
        if (t < nct) {
            float m2k = 0.0f;
#pragma unroll
            for (int k = 0; k < kWarps; ++k) m2k += part_b[set][k];
            send_pair(slot_m[set], slot_v[set], &bar_x[set], m_k, m2k, rank, t);
        }
        if (!mbar_wait_bounded(smem_u32(&bar_x[set]), static_cast<uint32_t>((i >> 1) & 1)))
            timed_out = 1;
        // Merge the C chunks' statistics: lane q of every warp takes rank q's pair and the
        // butterfly sums give every lane of every warp, in every CTA, the same bits.
        const int lane = t & 31;
        const float mq = lane < nct ? slot_m[set][lane] : 0.0f;
        const float mu = warp_sum(n_lane * mq) / n;
        const float dq = mq - mu;
        const float var = warp_sum(lane < nct ? fmaf(n_lane * dq, dq, slot_v[set][lane]) : 0.0f) / n;
        const float rstd = rsqrtf(var + eps);
        const f32x2 m2v = f2_make(mu, mu);

        if (ok) {
            const f32x2 r2 = f2_make(rstd, rstd);
            char* yr = static_cast<char*>(y) + row * pitch + v0 * 16;
            const char* gb = static_cast<const char*>(gamma) + v0 * 16;
            const char* bb = static_cast<const char*>(beta) + v0 * 16;
#pragma unroll
            for (int k = 0; k < NVT; ++k) {
                const int vi = t + k * kStagedBlock;
                if (vi < my_vecs)
                    st_out<16>(yr + static_cast<int64_t>(vi) * 16,
                               affine16<C>(v[k], ld_shared_ro<16>(gb + vi * 16),
                                           ld_shared_ro<16>(bb + vi * 16), k2, m2v, r2));
            }
        }
    }

    __syncthreads();
    if (timed_out && t == 0) {
        atomicOr(&g_ln_device_error, kDeviceErrorWaitTimeout);
        // Copies that may still be in flight into this CTA's shared memory: those issued for
        // iterations fail_iter .. fail_iter + stages - 1. Wait for each, at most a second.
        const int64_t f = fail_iter < 0 ? i : fail_iter;
        for (int64_t j = f; j < f + stages; ++j) {
            if (cid + j * ncl < rows)
                mbar_wait_bounded(smem_u32(&full[j % stages]), static_cast<uint32_t>((j / stages) & 1));
        }
    }
}

template <typename S, int NVT>
cudaError_t launch_ln_staged(const LayernormArgs& a, int cluster, int stages, int chunk_vecs,
                             cudaStream_t s) {
    auto kernel = layernorm_staged_kernel<S, NVT>;
    const size_t smem = static_cast<size_t>(ln_staged_smem_bytes(chunk_vecs, stages));
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kStagedBlock);
    cfg.dynamicSmemBytes = smem;
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
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    int active = 0;
    e = cudaOccupancyMaxActiveClusters(&active, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (active < 1) return cudaErrorInvalidConfiguration;
    const int64_t ncl = a.rows < active ? a.rows : active;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * cluster));
    return cudaLaunchKernelEx(&cfg, kernel, a.x, a.gamma, a.beta, a.y, a.rows, a.cols, a.eps,
                              chunk_vecs, stages);
}

template <typename S>
cudaError_t launch_ln_staged_nvt(const LayernormArgs& a, int cluster, int stages,
                                 cudaStream_t s) {
    constexpr int E = 16 / Storage<S>::kBytes;
    const int64_t nvec = a.cols / E;
    const int chunk = static_cast<int>((nvec + cluster - 1) / cluster);
    const int need = (chunk + kStagedBlock - 1) / kStagedBlock;
    if (need <= 1) return launch_ln_staged<S, 1>(a, cluster, stages, chunk, s);
    if (need <= 2) return launch_ln_staged<S, 2>(a, cluster, stages, chunk, s);
    if (need <= 4) return launch_ln_staged<S, 4>(a, cluster, stages, chunk, s);
    if (need <= kStagedMaxVecsPerThread) return launch_ln_staged<S, 8>(a, cluster, stages, chunk, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t layernorm_staged_launch(DType t, int cluster, int stages, const LayernormArgs& a,
                                    cudaStream_t s) {
    if (cluster < 1 || cluster > 16 || stages < 2 || stages > kStagedMaxStages)
        return cudaErrorInvalidValue;
    switch (t) {
        case DType::BF16: return launch_ln_staged_nvt<bf16_t>(a, cluster, stages, s);
        case DType::F16: return launch_ln_staged_nvt<f16_t>(a, cluster, stages, s);
        default: return launch_ln_staged_nvt<f32_t>(a, cluster, stages, s);
    }
}

cudaError_t read_layernorm_device_errors(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_ln_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_ln_device_error, &zero, sizeof(unsigned int));
}

}  // namespace camp
