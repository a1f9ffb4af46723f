// RMSNorm and LayerNorm for rows wider than the staged kernels hold, for sm_103a.
//
// Definitions as in rmsnorm_kernels.cuh (xserv "phase 4" design notes, RMSNorm section;
// gollamago README, "RMSNorm optimisation (TileLang)": one read of x, one write of y, fp32
// sums, one rounding) and layernorm.cu (xserv "phase 4", csrc/normalization/layernorm.cu:
// population variance, in coordinates shifted by K = x[row, 0]).
//
// The staged kernels (rmsnorm_staged.cu, layernorm_staged.cu) hold a CTA's chunk of a row in
// registers, which caps a row at 16 CTAs x 2048 16-byte vectors. Past that, this kernel
// spreads each row over a cluster of C CTAs (up to 16) and keeps each CTA's whole chunk in
// shared memory instead: a chunk of up to about 13,000 vectors (200 KB) with one buffer,
// half that with two, so x is still read from HBM once for rows of up to about 1.7 M bf16
// columns. (16-bit LayerNorm rows past the register kernel, and fp32 LayerNorm rows that
// the staged kernel would hold in ragged chunks, come here too.) Per row:
//   1. each copy group (a warp, or the whole CTA for 16-bit LayerNorm) owns a contiguous
//      segment of the CTA's chunk, which lands in a ring buffer by the group's own bulk
//      asynchronous copy on its own mbarrier (with a copy of the row's first 16 bytes, for
//      the LayerNorm shift);
//   2. every thread sums over its vectors of the segment (one every group-size vectors),
//      in kAcc independent packed accumulators: sum(x^2) for RMSNorm; sum(x - K) and, in
//      16-bit storage, sum((x - K)^2) for LayerNorm; one block reduction;
//   3. the CTA's sums go to every CTA of the cluster by st.async (counted on the receiver's
//      mbarrier; two slot sets alternating by row) and every CTA adds the C of them in rank
//      order (the same bits everywhere);
//   4. LayerNorm rows whose shift lies more than two standard deviations from the mean
//      (the rows kernel's rule; every row in fp32 storage) take a second pass over the
//      buffer, sum(((x - K) - mu)^2), with one more reduction and exchange;
//   5. the output pass re-reads the segment and writes y with 16-byte stores (the weight,
//      or gamma and beta, read through L1, two vectors ahead of their stores);
//   6. as soon as its threads have read the segment, the group refills it with the row
//      `stages` rows on: a group's next copy waits for its own output, not for the CTA's.
//
// Waits: every mbarrier wait gives up after `wait_ns` nanoseconds (one second in normal
// calls); a CTA whose wait ran out sets a bit in this file's device error word
// (camp_device_errors), stops issuing copies and storing, keeps sending and receiving
// partials so that no peer waits for it, and before returning waits (bounded) for the
// copies it still has in flight. With `probe` set (a diagnostic of that path) each CTA's
// first row copy is armed on its barrier but never issued, so every CTA's first wait runs
// out.
#include <climits>

#include <cooperative_groups.h>

#include "staged.cuh"

namespace camp {
namespace {

using namespace staged;

__device__ unsigned int g_spread_device_error = 0;

constexpr int kWarps = kSpreadBlock / 32;
// The copy groups of a CTA: each group of kSpreadBlock / groups threads owns a contiguous
// segment of the chunk, fills it with its own bulk copy on its own barrier and refills it as
// soon as its own threads have written it out. A warp a group in general; the whole CTA for
// 16-bit LayerNorm, whose 40 registers a thread do not hold the per-warp bookkeeping
// without spilling. Measured on GB300 (graphs of back-to-back launches, L2-cold, of the
// measured HBM peak), a group a warp against one a CTA: RMSNorm bf16 1024 x 262152 0.88 ->
// 0.90, 256 x 300000 0.84 -> 0.85, fp32 128 x 262144 0.81 -> 0.86, LayerNorm fp32 128 x
// 262144 0.55 -> 0.60; 16-bit LayerNorm lost (bf16 1024 x 262152 0.69 -> 0.64).
__host__ __device__ constexpr int spread_copy_groups(bool layernorm, int elem_bytes) {
    return layernorm && elem_bytes == 2 ? 1 : kSpreadBlock / 32;
}

// Several CTAs an SM by registers (40 a thread, 64 for fp32 LayerNorm), so that one CTA's
// row can compute while another's lands even with a single buffer each.
// ADD (RMSNorm only): h = x + r, rounded once to the storage type, is stored and normalized,
// as camp_add_rmsnorm defines it; x and r are both staged, and h is formed again from them
// for the output sweep (the same rounding, so the same bits) instead of being re-read.
template <typename S, bool LN, bool ADD>
__global__ void __launch_bounds__(kSpreadBlock, spread_ctas_per_sm(LN, Storage<S>::kBytes, ADD))
norm_spread_kernel(const void* x, const void* r, void* h, const void* __restrict__ w,
                   const void* __restrict__ beta, void* y, int64_t rows, int64_t cols,
                   float eps, int chunk_vecs, int stages, unsigned long long wait_ns,
                   int probe) {
    namespace cg = cooperative_groups;
    using C = Codec<S, 16>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr bool kOnePass = ES == 2;   // LayerNorm: one-pass statistics where they hold
    static_assert(!(LN && ADD), "the residual add is an RMSNorm path");
    constexpr int NB = ADD ? 2 : 1;   // staged tensors: x (and r)
    constexpr int kGroups = spread_copy_groups(LN, ES);
    constexpr int GS = kSpreadBlock / kGroups;   // threads a copy group
    // Independent packed accumulators a thread: two for 16-bit LayerNorm (two sums a pair
    // within 40 registers; 1024 x 262152 bf16 0.708 -> 0.715 of the measured peak against
    // four), four otherwise.
    constexpr int kAcc = (LN && ES == 2) ? 2 : 4;

    // Dynamic shared memory: `stages` buffers, each kSpreadHeadBytes of row heads (a copy of
    // the row's first 16 bytes a group, for the LayerNorm shift) and then the chunk (of x,
    // then of r on the add path).
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[kSpreadMaxStages][kGroups];
    __shared__ __align__(8) unsigned long long bar_x[2], bar_z[2];
    __shared__ float part_a[2][kWarps], part_b[2][kWarps];
    // The second pass's partials: written after this row's exchange, which not every warp
    // has finished reading part_a from; rewritten only after a later row's first barrier.
    __shared__ float part_c[kWarps];
    __shared__ float slot_a[2][16], slot_b[2][16], slot_z[2][16];
    __shared__ int timed_out;

    cg::cluster_group cluster = cg::this_cluster();
    const int nct = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t ncl = gridDim.x / nct;
    const int64_t cid = blockIdx.x / nct;
    const int t = threadIdx.x;
    const int wid = t >> 5;
    const int lane = t & 31;
    static_assert(GS == 32 || GS == kSpreadBlock, "a copy group is a warp or the CTA");
    const int g = kGroups == 1 ? 0 : wid;    // this thread's copy group ...
    const int gt = kGroups == 1 ? t : lane;  // ... and its index in it
    const int64_t nvec = cols / E;
    const int64_t v0 = static_cast<int64_t>(rank) * chunk_vecs;
    const int64_t left = nvec - v0;
    const int my_vecs = left <= 0 ? 0 : (left < chunk_vecs ? static_cast<int>(left) : chunk_vecs);
    const uint32_t my_bytes = static_cast<uint32_t>(my_vecs) * 16u;
    // The group's segment of the chunk: vectors [g_lo, g_lo + g_len).
    const int seg = (my_vecs + kGroups - 1) / kGroups;
    const int g_lo = g * seg < my_vecs ? g * seg : my_vecs;
    const int g_len = my_vecs - g_lo < seg ? my_vecs - g_lo : seg;
    const int64_t pitch = cols * ES;
    const uint32_t stage_bytes =
        kSpreadHeadBytes + static_cast<uint32_t>(NB) * static_cast<uint32_t>(chunk_vecs) * 16u;
    const uint32_t r_off = static_cast<uint32_t>(chunk_vecs) * 16u;   // r's chunk after x's
    // The launcher refuses grids that would give a cluster more than INT_MAX rows.
    const int my_rows = cid < rows ? static_cast<int>((rows - cid + ncl - 1) / ncl) : 0;

    if (t == 0) {
        for (int s = 0; s < stages; ++s)
            for (int q = 0; q < kGroups; ++q) mbar_init(smem_u32(&full[s][q]), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bar_x[s]), 1);
            mbar_init(smem_u32(&bar_z[s]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        timed_out = 0;
        // The inputs the first bulk loads and output pass will read (after griddep_wait).
        prefetch_l2(static_cast<const char*>(w) + v0 * 16, my_bytes);
        if constexpr (LN) prefetch_l2(static_cast<const char*>(beta) + v0 * 16, my_bytes);
        for (int s = 0; s < stages && s < my_rows; ++s) {
            prefetch_l2(static_cast<const char*>(x) + (cid + s * ncl) * pitch + v0 * 16, my_bytes);
            if constexpr (ADD)
                prefetch_l2(static_cast<const char*>(r) + (cid + s * ncl) * pitch + v0 * 16,
                            my_bytes);
        }
    }
    // Every CTA of the cluster has started and initialized its barriers before any CTA
    // stores into a peer's shared memory (split cluster barrier).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    __syncthreads();

    griddep_wait();
    griddep_launch_dependents();

    const char* xb = static_cast<const char*>(x);
    const char* rb = ADD ? static_cast<const char*>(r) : nullptr;
    // The group's first thread: its segment of row j (of x, and of r on the add path; for
    // LayerNorm also the row's first 16 bytes) into ring slot s, counted on the group's own
    // barrier.
    auto issue = [&](int j, int s) {
        const int64_t off = (cid + static_cast<int64_t>(j) * ncl) * pitch;
        const uint32_t bar = smem_u32(&full[s][g]);
        const uint32_t base = smem_u32(smem) + static_cast<uint32_t>(s) * stage_bytes;
        const uint32_t g_bytes = static_cast<uint32_t>(g_len) * 16u;
        mbar_arrive_expect_tx(bar, (LN ? 16u : 0u) + NB * g_bytes);
        if (probe && j == 0) return;   // diagnostic: this copy is never issued
        if constexpr (LN) bulk_load(base + g * 16, xb + off, 16u, bar);
        if (g_bytes > 0) {
            const uint32_t dst = base + kSpreadHeadBytes + g_lo * 16;
            bulk_load(dst, xb + off + (v0 + g_lo) * 16, g_bytes, bar);
            if constexpr (ADD) bulk_load(dst + r_off, rb + off + (v0 + g_lo) * 16, g_bytes, bar);
        }
    };
    if (gt == 0) {
        for (int j = 0; j < stages && j < my_rows; ++j) issue(j, j);
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    // Shared-memory loads of the ring: for the one-group CTA plain loads through pointers
    // into smem, which the compiler can schedule; for warp groups loads at 32-bit shared
    // addresses, since their extra bookkeeping would otherwise spill fp32 RMSNorm out of 40
    // registers.
    const uint32_t smem_at = smem_u32(smem);
    const float n = static_cast<float>(cols);
    const char* wb = static_cast<const char*>(w) + (v0 + g_lo) * 16;
    const char* bb = LN ? static_cast<const char*>(beta) + (v0 + g_lo) * 16 : nullptr;
    int nz = 0;       // second-pass exchanges so far (the same count in every CTA)
    int fail = -1;
    int s = 0;        // ring slot of row j (j mod stages) ...
    uint32_t par = 0; // ... and its phase parity, advanced by counters
    for (int j = 0; j < my_rows; ++j) {
        const int set = static_cast<int>(j & 1);
        // 1. The group's segment of the row has landed (each group waits for its own copy).
        if (fail < 0 && !mbar_wait_bounded(smem_u32(&full[s][g]), par, wait_ns)) timed_out = 1;
        const uint32_t slot = static_cast<uint32_t>(s) * stage_bytes;
        const unsigned char* segp = smem + slot + kSpreadHeadBytes + g_lo * 16;
        const uint32_t sega = smem_at + slot + kSpreadHeadBytes + g_lo * 16;
        auto ld1 = [&](int v, uint32_t o) -> Raw<16> {   // vector v of a staged segment
            if constexpr (kGroups == 1) return ld_smem16(segp + o + v * 16);
            else return ld_smem16_at(sega + o + v * 16);
        };
        // Vector v of the row the operator normalizes: x, or h = x + r on the add path.
        auto ldv = [&](int v) -> Raw<16> {
            if constexpr (ADD) return C::add(ld1(v, 0), ld1(v, r_off));
            else return ld1(v, 0);
        };
        char* hr = ADD ? static_cast<char*>(h) + (cid + static_cast<int64_t>(j) * ncl) * pitch +
                             (v0 + g_lo) * 16
                       : nullptr;

        // 2. This thread's sums over its vectors of the segment.
        float shift = 0.0f;
        if (LN && fail < 0) {
            const Raw<16> h =
                kGroups == 1 ? ld_smem16(smem + slot) : ld_smem16_at(smem_at + slot + g * 16);
            C::each(h, [&](int e, float f) { if (e == 0) shift = f; });
        }
        const f32x2 k2 = f2_make(shift, shift);
        f32x2 acc1[kAcc], acc2[kAcc];
#pragma unroll
        for (int a = 0; a < kAcc; ++a) {
            acc1[a] = f2_make(0.0f, 0.0f);
            acc2[a] = f2_make(0.0f, 0.0f);
        }
        if (fail < 0) {
            for (int vi = gt; vi < g_len; vi += kAcc * GS) {
#pragma unroll
                for (int a = 0; a < kAcc; ++a) {
                    const int vj = vi + a * GS;
                    if (vj < g_len) {
                        const Raw<16> v = ldv(vj);
                        if constexpr (ADD) st_out<16>(hr + static_cast<int64_t>(vj) * 16, v);
                        C::each_pair(v, [&](int, f32x2 p) {
                            if constexpr (!LN) {
                                acc1[a] = f2_fma(p, p, acc1[a]);
                            } else {
                                const f32x2 d = f2_sub(p, k2);
                                acc1[a] = f2_add(acc1[a], d);
                                if constexpr (kOnePass) acc2[a] = f2_fma(d, d, acc2[a]);
                            }
                        });
                    }
                }
            }
        }
        float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
        for (int a = 0; a < kAcc; ++a) {
            s1 += f2_lo(acc1[a]) + f2_hi(acc1[a]);
            s2 += f2_lo(acc2[a]) + f2_hi(acc2[a]);
        }
        s1 = warp_sum(s1);
        if constexpr (LN && kOnePass) s2 = warp_sum(s2);
        if (lane == 0) {
            part_a[set][wid] = s1;
            part_b[set][wid] = s2;
        }
        __syncthreads();
        if (fail < 0 && timed_out) fail = j;   // the same in every thread
        const bool ok = fail < 0;

        // 3. The exchange: this CTA's sums to every CTA of the cluster.
        if (t == 0) mbar_arrive_expect_tx(smem_u32(&bar_x[set]), static_cast<uint32_t>(nct) * 8u);
        if (t < nct) {
            float ca = 0.0f, cb = 0.0f;
            for (int q = 0; q < kWarps; ++q) {
                ca += part_a[set][q];
                cb += part_b[set][q];
            }
            const uint32_t b = map_rank(smem_u32(&bar_x[set]), static_cast<uint32_t>(t));
            st_async_f32(map_rank(smem_u32(&slot_a[set][rank]), static_cast<uint32_t>(t)), ca, b);
            st_async_f32(map_rank(smem_u32(&slot_b[set][rank]), static_cast<uint32_t>(t)), cb, b);
        }
        // Every CTA waits for all sums of every row, even after a failure: a peer's
        // stores must have landed before this CTA's shared memory is released.
        if (!mbar_wait_bounded(smem_u32(&bar_x[set]), static_cast<uint32_t>((j >> 1) & 1), wait_ns))
            timed_out = 1;
        float ta = 0.0f, tb = 0.0f;
        for (int q = 0; q < nct; ++q) {   // rank order in every CTA
            ta += slot_a[set][q];
            tb += slot_b[set][q];
        }
        float scale, mu = 0.0f;
        if constexpr (!LN) {
            scale = rsqrtf(ta / n + eps);
        } else {
            mu = ta / n;
            float var = tb / n - mu * mu;
            // 4. The second pass, where the one-pass difference could cancel.
            if (!kOnePass || !(mu * mu <= 4.0f * var)) {
                const f32x2 m2 = f2_make(mu, mu);
                f32x2 acc[kAcc];
#pragma unroll
                for (int a = 0; a < kAcc; ++a) acc[a] = f2_make(0.0f, 0.0f);
                if (ok) {
                    for (int vi = gt; vi < g_len; vi += kAcc * GS) {
#pragma unroll
                        for (int a = 0; a < kAcc; ++a) {
                            const int vj = vi + a * GS;
                            if (vj < g_len)
                                C::each_pair(ldv(vj), [&](int, f32x2 p) {
                                    const f32x2 d = f2_sub(f2_sub(p, k2), m2);
                                    acc[a] = f2_fma(d, d, acc[a]);
                                });
                        }
                    }
                }
                float s3 = 0.0f;
#pragma unroll
                for (int a = 0; a < kAcc; ++a) s3 += f2_lo(acc[a]) + f2_hi(acc[a]);
                s3 = warp_sum(s3);
                if (lane == 0) part_c[wid] = s3;
                __syncthreads();
                const int zs = nz & 1;
                if (t == 0)
                    mbar_arrive_expect_tx(smem_u32(&bar_z[zs]), static_cast<uint32_t>(nct) * 4u);
                if (t < nct) {
                    float cz = 0.0f;
                    for (int q = 0; q < kWarps; ++q) cz += part_c[q];
                    st_async_f32(map_rank(smem_u32(&slot_z[zs][rank]), static_cast<uint32_t>(t)), cz,
                                 map_rank(smem_u32(&bar_z[zs]), static_cast<uint32_t>(t)));
                }
                if (!mbar_wait_bounded(smem_u32(&bar_z[zs]), static_cast<uint32_t>((nz >> 1) & 1), wait_ns))
                    timed_out = 1;
                float tz = 0.0f;
                for (int q = 0; q < nct; ++q) tz += slot_z[zs][q];
                var = tz / n;
                ++nz;
            }
            scale = rsqrtf(var + eps);
        }

        // 5. The output pass over the group's segment, two vectors an iteration (both
        //    weights loaded ahead of the first store).
        if (ok) {
            char* yr = static_cast<char*>(y) + (cid + static_cast<int64_t>(j) * ncl) * pitch +
                       (v0 + g_lo) * 16;
            const f32x2 r2 = f2_make(scale, scale);
            const f32x2 m2 = f2_make(mu, mu);
            for (int vi = gt; vi < g_len; vi += 2 * GS) {
                const int vj = vi + GS;
                const bool two = vj < g_len;
                const Raw<16> w0 = ld_shared_ro<16>(wb + vi * 16);
                const Raw<16> w1 = two ? ld_shared_ro<16>(wb + vj * 16) : raw_zero<16>();
                Raw<16> b0 = raw_zero<16>(), b1 = raw_zero<16>();
                if constexpr (LN) {
                    b0 = ld_shared_ro<16>(bb + vi * 16);
                    if (two) b1 = ld_shared_ro<16>(bb + vj * 16);
                }
                auto out = [&](int v, const Raw<16>& wv, const Raw<16>& bv) {
                    const Raw<16> xv = ldv(v);
                    f32x2 wp[C::kPairs], bp[C::kPairs];
                    C::each_pair(wv, [&](int p, f32x2 q) { wp[p] = q; });
                    if constexpr (LN) C::each_pair(bv, [&](int p, f32x2 q) { bp[p] = q; });
                    st_out<16>(yr + static_cast<int64_t>(v) * 16, C::map_pair(xv, [&](int p, f32x2 xp) {
                                   if constexpr (!LN)
                                       return f2_mul(f2_mul(xp, r2), wp[p]);
                                   else
                                       return f2_fma(f2_mul(f2_sub(f2_sub(xp, k2), m2), r2), wp[p], bp[p]);
                               }));
                };
                out(vi, w0, b0);
                if (two) out(vj, w1, b1);
            }
        }

        // 6. Every thread of the group has read its segment: refill it with the row `stages`
        //    rows on, without waiting for the other groups.
        if constexpr (kGroups == 1) __syncthreads(); else __syncwarp();
        if (ok && gt == 0 && j + stages < my_rows) {
            // Order the group's generic-proxy reads of the segment before the async-proxy
            // write that refills it.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(j + stages, s);
        }
        if (++s == stages) {
            s = 0;
            par ^= 1u;
        }
    }

    __syncthreads();
    if (timed_out) {
        if (t == 0) atomicOr(&g_spread_device_error, kDeviceErrorWaitTimeout);
        // Copies that may still be in flight into this group's segment: the rows from the
        // failed one up to `stages` rows on. Wait for each, bounded.
        if (gt == 0) {
            const int f = fail < 0 ? my_rows : fail;
            for (int jj = f; jj < f + stages && jj < my_rows; ++jj)
                mbar_wait_bounded(smem_u32(&full[jj % stages][g]),
                                  static_cast<uint32_t>((jj / stages) & 1), wait_ns);
        }
    }
}

template <typename S, bool LN, bool ADD>
cudaError_t launch_spread(const void* x, const void* r, void* h, const void* w, const void* beta,
                          void* y, int64_t rows, int64_t cols, float eps, int cluster,
                          int stages, unsigned long long wait_ns, int probe, cudaStream_t s) {
    auto kernel = norm_spread_kernel<S, LN, ADD>;
    constexpr int E = 16 / Storage<S>::kBytes;
    const int64_t nvec = cols / E;
    const int chunk = static_cast<int>((nvec + cluster - 1) / cluster);
    const size_t smem = static_cast<size_t>(spread_smem_bytes(chunk, stages, ADD ? 2 : 1));
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSpreadBlock);
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
    const int64_t ncl = rows < active ? rows : active;
    if ((rows + ncl - 1) / ncl > INT_MAX) return cudaErrorInvalidValue;   // 32-bit row counters
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * cluster));
    return cudaLaunchKernelEx(&cfg, kernel, x, r, h, w, beta, y, rows, cols, eps, chunk, stages,
                              wait_ns, probe);
}

template <bool LN, bool ADD>
cudaError_t spread_dtype(DType t, const void* x, const void* r, void* h, const void* w,
                         const void* beta, void* y, int64_t rows, int64_t cols, float eps,
                         int cluster, int stages, unsigned long long wait_ns, int probe,
                         cudaStream_t s) {
    switch (t) {
        case DType::BF16:
            return launch_spread<bf16_t, LN, ADD>(x, r, h, w, beta, y, rows, cols, eps, cluster,
                                                  stages, wait_ns, probe, s);
        case DType::F16:
            return launch_spread<f16_t, LN, ADD>(x, r, h, w, beta, y, rows, cols, eps, cluster,
                                                 stages, wait_ns, probe, s);
        default:
            return launch_spread<f32_t, LN, ADD>(x, r, h, w, beta, y, rows, cols, eps, cluster,
                                                 stages, wait_ns, probe, s);
    }
}

}  // namespace

cudaError_t rmsnorm_spread_launch(bool add, DType t, int cluster, int stages,
                                  const RmsnormArgs& a, cudaStream_t s,
                                  unsigned long long wait_ns, int probe) {
    if (cluster < 1 || cluster > 16 || stages < 1 || stages > kSpreadMaxStages)
        return cudaErrorInvalidValue;
    if (add)
        return spread_dtype<false, true>(t, a.x, a.r, a.h, a.w, nullptr, a.y, a.rows, a.cols,
                                         a.eps, cluster, stages, wait_ns, probe, s);
    return spread_dtype<false, false>(t, a.x, nullptr, nullptr, a.w, nullptr, a.y, a.rows,
                                      a.cols, a.eps, cluster, stages, wait_ns, probe, s);
}

cudaError_t layernorm_spread_launch(DType t, int cluster, int stages, const LayernormArgs& a,
                                    cudaStream_t s, unsigned long long wait_ns, int probe) {
    if (cluster < 1 || cluster > 16 || stages < 1 || stages > kSpreadMaxStages)
        return cudaErrorInvalidValue;
    return spread_dtype<true, false>(t, a.x, nullptr, nullptr, a.gamma, a.beta, a.y, a.rows,
                                     a.cols, a.eps, cluster, stages, wait_ns, probe, s);
}

cudaError_t read_spread_device_errors(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_spread_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_spread_device_error, &zero, sizeof(unsigned int));
}

}  // namespace camp
