// TMA-staged RMSNorm for wide rows (and the fused residual add), for sm_103a.
//
// Definition and precision rules as in rmsnorm_kernels.cuh (xserv "phase 4" design notes,
// RMSNorm section; gollamago README, "RMSNorm optimisation (TileLang)": one read of x, one
// write of y, fp32 sum of squares and scaling, one rounding). For rows too wide to keep in
// one CTA's registers, the row is staged in shared memory instead.
//
// Mapping: persistent clusters of C CTAs (C = 1..16). Cluster c owns rows c, c + n, c + 2n,
// ... (n clusters); CTA rank k of a cluster owns the contiguous chunk of 16-byte vectors
// [k * chunk, min((k + 1) * chunk, nvec)) of each of its rows (chunk <= 8 * 256 vectors).
// The CTA's chunk of w is copied into shared memory once. Each CTA keeps a ring of
// `stages` shared-memory row buffers: one thread issues one bulk asynchronous copy
// (cp.async.bulk, completion counted in bytes on an mbarrier) per buffer and row, so the
// loads of the next rows stream while the current row is reduced and written. Per row:
// every thread moves its vectors of the buffer into registers and sums their squares; as
// soon as the CTA has read the buffer it is refilled with the row `stages` rows ahead
// (before the cluster exchange, so the copy overlaps it); the CTA combines its warps and
// sends its partial into a slot of every CTA of the cluster with st.async (distributed
// shared memory; each store counted in bytes on the receiving CTA's mbarrier; two slot
// sets and barriers alternate by row). Each CTA waits on its own mbarrier for the C
// partials, sums them in rank order (the same bits everywhere), and writes
// y = x * rinv * w from the registers and the staged w with 16-byte stores. There is no
// cluster-wide barrier per row: a release barrier would make every row wait for the
// previous row's global stores to complete (measured: the top stall, "membar", with it).
// On the add path both x and r are staged; h = x + r is formed in registers and stored,
// and never re-read from HBM.
//
// Waits: every mbarrier wait gives up after one second (the copies complete in
// microseconds; only a broken copy could hold one). A CTA whose wait ran out sets a bit in
// the library's device error word (camp_device_errors), stops issuing copies and storing,
// keeps sending its partials (so no peer waits for them) and receiving its peers' (so none
// lands after it has exited), and before returning waits, again for at most a second
// each, for the copies it still has in flight.
#include <cooperative_groups.h>

#include "staged.cuh"

namespace camp {

// Bits of the device error word, set by kernels whose bounded waits ran out.
__device__ unsigned int g_device_error = 0;

namespace {

using namespace staged;

template <typename C>
__device__ __forceinline__ float sum_squares16(const Raw<16>& v) {
    if constexpr (C::kElems >= 2) {
        f32x2 acc = f2_make(0.0f, 0.0f);
        C::each_pair(v, [&](int, f32x2 p) { acc = f2_fma(p, p, acc); });
        return f2_lo(acc) + f2_hi(acc);
    } else {
        float ss = 0.0f;
        C::each(v, [&](int, float f) { ss = fmaf(f, f, ss); });
        return ss;
    }
}

template <typename C>
__device__ __forceinline__ Raw<16> scale16(const Raw<16>& xv, const Raw<16>& wv, float rinv) {
    f32x2 wp[C::kPairs];
    C::each_pair(wv, [&](int p, f32x2 q) { wp[p] = q; });
    const f32x2 r2 = f2_make(rinv, rinv);
    return C::map_pair(xv, [&](int p, f32x2 xp) { return f2_mul(f2_mul(xp, r2), wp[p]); });
}

// PROBE: the wait diagnostic's variant (plain RMSNorm only): every mbarrier wait bounded by
// `wait_ns` instead of one second, and each CTA's first row copy armed on its barrier but
// never issued, so every CTA's first wait runs out. The normal variants ignore `wait_ns`.
template <typename S, bool ADD, int NVT, bool PROBE>
__global__ void __launch_bounds__(kStagedBlock, 1)
rmsnorm_staged_kernel(const void* x, const void* r, void* h, const void* __restrict__ w,
                      void* y, int64_t rows, int64_t cols, float eps, int chunk_vecs,
                      int stages, unsigned long long wait_ns) {
    namespace cg = cooperative_groups;
    using C = Codec<S, 16>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr int kWarps = kStagedBlock / 32;
    constexpr int NB = ADD ? 2 : 1;   // staged tensors per row: x (and r)
    const unsigned long long limit = PROBE ? wait_ns : kWaitLimitNs;

    // Dynamic shared memory: this CTA's chunk of w, then `stages` row buffers.
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[kStagedMaxStages + 1];   // + w
    __shared__ __align__(8) unsigned long long sum_bar[2];   // partials of rows i, i + 1
    __shared__ float partial[2][kWarps];
    __shared__ float slot[2][16];
    __shared__ int timed_out;

    cg::cluster_group cluster = cg::this_cluster();
    const int nct = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t ncl = gridDim.x / nct;           // clusters in the grid
    const int64_t cid = blockIdx.x / nct;          // this cluster
    const int t = threadIdx.x;
    const int64_t nvec = cols / E;
    const int64_t v0 = static_cast<int64_t>(rank) * chunk_vecs;
    const int64_t left = nvec - v0;
    const int my_vecs = left <= 0 ? 0 : (left < chunk_vecs ? static_cast<int>(left) : chunk_vecs);
    const uint32_t my_bytes = static_cast<uint32_t>(my_vecs) * 16u;
    const int64_t pitch = cols * ES;
    const int64_t stage_bytes = static_cast<int64_t>(NB) * chunk_vecs * 16;
    unsigned char* wbuf = smem;
    unsigned char* ring = smem + static_cast<int64_t>(chunk_vecs) * 16;
    const uint32_t wbar = smem_u32(&full[kStagedMaxStages]);

    if (t == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&full[s]), 1);
        mbar_init(wbar, 1);
        mbar_init(smem_u32(&sum_bar[0]), 1);
        mbar_init(smem_u32(&sum_bar[1]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        timed_out = 0;
        // The chunks that the first bulk loads below will read (after griddep_wait).
        prefetch_l2(static_cast<const char*>(w) + v0 * 16, my_bytes);
        for (int s = 0; s < stages; ++s) {
            const int64_t row = cid + s * ncl;
            if (row >= rows) break;
            prefetch_l2(static_cast<const char*>(x) + row * pitch + v0 * 16, my_bytes);
            if constexpr (ADD) prefetch_l2(static_cast<const char*>(r) + row * pitch + v0 * 16, my_bytes);
        }
    }
    // Every CTA of the cluster has started, and its barriers are initialized, before any
    // CTA stores into a peer's shared memory (split cluster barrier: arrive now, wait
    // before the first exchange).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    __syncthreads();

    griddep_wait();
    griddep_launch_dependents();

    const char* xb = static_cast<const char*>(x) + v0 * 16;
    const char* rb = ADD ? static_cast<const char*>(r) + v0 * 16 : nullptr;
    auto issue = [&](int s, int64_t row) {   // one thread
        const uint32_t bar = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(ring + s * stage_bytes);
        mbar_arrive_expect_tx(bar, my_bytes * NB);
        if (PROBE && row == cid) return;   // diagnostic: the first row's copy is never issued
        bulk_load(dst, xb + row * pitch, my_bytes, bar);
        if constexpr (ADD) bulk_load(dst + chunk_vecs * 16, rb + row * pitch, my_bytes, bar);
    };
    if (t == 0 && my_bytes > 0) {
        mbar_arrive_expect_tx(wbar, my_bytes);
        bulk_load(smem_u32(wbuf), static_cast<const char*>(w) + v0 * 16, my_bytes, wbar);
        for (int s = 0; s < stages; ++s) {
            const int64_t row = cid + s * ncl;
            if (row < rows) issue(s, row);
        }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    bool w_ready = false;
    int64_t fail_iter = -1;
    int64_t i = 0;
    for (int64_t row = cid; row < rows; row += ncl, ++i) {
        const int s = static_cast<int>(i % stages);
        const int set = static_cast<int>(i & 1);
        const unsigned char* buf = ring + s * stage_bytes;
        if (fail_iter < 0 && my_bytes > 0 &&
            !mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>((i / stages) & 1), limit))
            timed_out = 1;
        __syncthreads();
        if (fail_iter < 0 && timed_out) fail_iter = i;   // the same in every thread
        const bool ok = fail_iter < 0;

        // Pass 1: this thread's vectors into registers (h = x + r stored on the add path),
        // and its share of the sum of squares.
        Raw<16> v[NVT];
        float ss = 0.0f;
        char* hr = ADD ? static_cast<char*>(h) + row * pitch + v0 * 16 : nullptr;
#pragma unroll
        for (int k = 0; k < NVT; ++k) {
            const int vi = t + k * kStagedBlock;
            if (ok && vi < my_vecs) {
                v[k] = ld_smem16(buf + vi * 16);
                if constexpr (ADD) {
                    v[k] = C::add(v[k], ld_smem16(buf + chunk_vecs * 16 + vi * 16));
                    st_out<16>(hr + static_cast<int64_t>(vi) * 16, v[k]);
                }
                ss += sum_squares16<C>(v[k]);
            } else {
                v[k] = raw_zero<16>();
            }
        }
        ss = warp_sum(ss);
        if ((t & 31) == 0) partial[set][t / 32] = ss;
        __syncthreads();   // the buffer has been read: refill it now
        if (t == 0) {
            if (ok && my_bytes > 0) {
                const int64_t next = row + stages * ncl;
                if (next < rows) {
                    // Order this CTA's generic-proxy reads of the buffer before the
                    // async-proxy write that refills it.
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(s, next);
                }
            }
            // This row's partials: one 4-byte store from every CTA of the cluster.
            mbar_arrive_expect_tx(smem_u32(&sum_bar[set]), static_cast<uint32_t>(nct) * 4u);
        }
        // Thread q < C sends this CTA's partial (zero if its data never came) into slot
        // [set][rank] of cluster rank q, counted on that CTA's sum_bar[set]: no cluster-wide
        // barrier, so nothing waits for this CTA's global stores to complete.
        if (t < nct) {
            float c = 0.0f;
#pragma unroll
            for (int k = 0; k < kWarps; ++k) c += partial[set][k];
            st_async_f32(map_rank(smem_u32(&slot[set][rank]), static_cast<uint32_t>(t)), c,
                         map_rank(smem_u32(&sum_bar[set]), static_cast<uint32_t>(t)));
        }
        // Every CTA waits for all partials of every row, even after a failure: a peer's
        // stores must have landed before this CTA's shared memory is released.
        if (!mbar_wait_bounded(smem_u32(&sum_bar[set]), static_cast<uint32_t>((i >> 1) & 1), limit))
            timed_out = 1;
        float tot = 0.0f;
        for (int q = 0; q < nct; ++q) tot += slot[set][q];   // rank order in every CTA
        const float rinv = rsqrtf(tot / static_cast<float>(cols) + eps);

        // Pass 2: y = x * rinv * w from the registers and the staged w.
        if (ok && my_bytes > 0 && !w_ready) {
            if (!mbar_wait_bounded(wbar, 0, limit)) timed_out = 1;
            w_ready = true;
        }
        if (ok) {
            char* yr = static_cast<char*>(y) + row * pitch + v0 * 16;
#pragma unroll
            for (int k = 0; k < NVT; ++k) {
                const int vi = t + k * kStagedBlock;
                if (vi < my_vecs)
                    st_out<16>(yr + static_cast<int64_t>(vi) * 16,
                               scale16<C>(v[k], ld_smem16(wbuf + vi * 16), rinv));
            }
        }
    }

    __syncthreads();
    if (timed_out && t == 0) {
        atomicOr(&g_device_error, kDeviceErrorWaitTimeout);
        // Copies that may still be in flight into this CTA's shared memory: w, and those
        // issued for iterations fail_iter .. fail_iter + stages - 1. Wait for each, bounded.
        if (my_bytes > 0) mbar_wait_bounded(wbar, 0, limit);
        const int64_t f = fail_iter < 0 ? i : fail_iter;
        for (int64_t j = f; j < f + stages; ++j) {
            if (my_bytes > 0 && cid + j * ncl < rows)
                mbar_wait_bounded(smem_u32(&full[j % stages]),
                                  static_cast<uint32_t>((j / stages) & 1), limit);
        }
    }
}

template <typename S, bool ADD, int NVT, bool PROBE>
cudaError_t launch_staged_kernel(const RmsnormArgs& a, int cluster, int stages, int chunk_vecs,
                                 unsigned long long wait_ns, cudaStream_t s) {
    auto kernel = rmsnorm_staged_kernel<S, ADD, NVT, PROBE>;
    const size_t smem = static_cast<size_t>(staged_smem_bytes(ADD, chunk_vecs, stages));
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
    // As many clusters as fit on the device at once (each then loops over its rows), at
    // most one per row.
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    int active = 0;
    e = cudaOccupancyMaxActiveClusters(&active, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (active < 1) return cudaErrorInvalidConfiguration;
    const int64_t ncl = a.rows < active ? a.rows : active;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * cluster));
    return cudaLaunchKernelEx(&cfg, kernel, a.x, a.r, a.h, a.w, a.y, a.rows, a.cols, a.eps,
                              chunk_vecs, stages, wait_ns);
}

template <typename S, bool ADD, int NVT>
cudaError_t launch_staged(const RmsnormArgs& a, int cluster, int stages, int chunk_vecs,
                          unsigned long long wait_ns, int probe, cudaStream_t s) {
    if constexpr (!ADD) {
        if (probe)
            return launch_staged_kernel<S, false, NVT, true>(a, cluster, stages, chunk_vecs,
                                                             wait_ns, s);
    }
    if (probe) return cudaErrorInvalidValue;   // the probe has no add-path variant
    return launch_staged_kernel<S, ADD, NVT, false>(a, cluster, stages, chunk_vecs, wait_ns, s);
}

template <typename S, bool ADD>
cudaError_t launch_staged_nvt(const RmsnormArgs& a, int cluster, int stages,
                              unsigned long long wait_ns, int probe, cudaStream_t s) {
    constexpr int E = 16 / Storage<S>::kBytes;
    const int64_t nvec = a.cols / E;
    const int chunk = static_cast<int>((nvec + cluster - 1) / cluster);
    const int need = (chunk + kStagedBlock - 1) / kStagedBlock;
    if (need <= 1) return launch_staged<S, ADD, 1>(a, cluster, stages, chunk, wait_ns, probe, s);
    if (need <= 2) return launch_staged<S, ADD, 2>(a, cluster, stages, chunk, wait_ns, probe, s);
    if (need <= 4) return launch_staged<S, ADD, 4>(a, cluster, stages, chunk, wait_ns, probe, s);
    if (need <= kStagedMaxVecsPerThread)
        return launch_staged<S, ADD, 8>(a, cluster, stages, chunk, wait_ns, probe, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t rmsnorm_staged_launch(bool add, DType t, int cluster, int stages,
                                  const RmsnormArgs& a, cudaStream_t s,
                                  unsigned long long wait_ns, int probe) {
    if (cluster < 1 || cluster > 16 || stages < 2 || stages > kStagedMaxStages)
        return cudaErrorInvalidValue;
    if (t == DType::BF16)
        return add ? launch_staged_nvt<bf16_t, true>(a, cluster, stages, wait_ns, probe, s)
                   : launch_staged_nvt<bf16_t, false>(a, cluster, stages, wait_ns, probe, s);
    if (t == DType::F16)
        return add ? launch_staged_nvt<f16_t, true>(a, cluster, stages, wait_ns, probe, s)
                   : launch_staged_nvt<f16_t, false>(a, cluster, stages, wait_ns, probe, s);
    return add ? launch_staged_nvt<f32_t, true>(a, cluster, stages, wait_ns, probe, s)
               : launch_staged_nvt<f32_t, false>(a, cluster, stages, wait_ns, probe, s);
}

cudaError_t read_device_errors(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace camp
