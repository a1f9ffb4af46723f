// Shared-memory-staged LayerNorm for wide rows, for sm_103a.
//
// Definition as in layernorm.cu (xserv "phase 4", csrc/normalization/layernorm.cu and the
// design notes' LayerNorm section): y = gamma * (x - mean) / sqrt(var + eps) + beta with the
// population variance, in coordinates shifted by K = x[row, 0] so that no deviation is
// formed from a rounded fp32 mean.
//
// Mapping: persistent clusters of C CTAs (the staged RMSNorm kernel's, rmsnorm_staged.cu).
// CTA rank k owns a contiguous chunk of 16-byte vectors of every row of its cluster and
// reads its chunks of gamma and beta through L1 (the same chunk every row, so they stay
// cached where the SM's shared memory leaves room; holding them in shared memory cost the
// CTAs an SM could run). A ring of `stages` row buffers is filled by bulk asynchronous
// copies: each copies the CTA's chunk plus the row's first 16 bytes (every CTA needs the
// shift K).
//
// A step takes RP rows (RP = 1 or 2) of the cluster at once, so that the per-row chain of
// two block reductions and a cluster round trip is paid once for RP rows and each vector
// of gamma and beta is loaded once for RP rows. Per step:
//   1. every thread moves its vectors of the RP rows into registers;
//   2. the CTA's chunk statistics in two passes over the registers, in shifted
//      coordinates: m_k = sum(x - K) / n_k (first block reduction; the buffers are
//      refilled right after it, so the copies overlap everything below), then
//      M2_k = sum(((x - K) - m_k)^2) (second);
//   3. one exchange sends (m_k, M2_k) of the RP rows to every CTA of the cluster (st.async
//      stores counted on the receiver's mbarrier; two slot sets alternating by step), and
//      every CTA merges the C pairs with Chan, Golub and LeVeque's formula (mu =
//      sum n_q m_q / n, M2 = sum M2_q + sum n_q (m_q - mu)^2; lane q of each warp takes rank
//      q and warp butterflies sum, the same bits in every warp and CTA): no value is rounded
//      in unshifted coordinates;
//   4. y = fma(((x - K) - mu) * rsqrt(M2 / n + eps), gamma, beta) from the registers,
//      16-byte stores.
//
// Waits: every mbarrier wait gives up after `wait_ns` nanoseconds (one second in normal
// calls; copies land in microseconds). A CTA whose wait ran out sets a bit in this file's
// device error word (read by camp_device_errors), stops issuing copies and storing, keeps
// sending and receiving partials so that no peer waits for it, and before returning waits
// (again bounded) for the copies it still has in flight. With `probe` set (a diagnostic
// entry point only) no CTA issues the copies of its first row, so every CTA takes that path.
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

constexpr int kLnMaxRp = 2;
constexpr int kLnGammaBatch = 2;
// CTAs an SM by registers: 4 (at most 64 registers a thread) up to 4 vectors a thread in
// flight (vectors per row x rows per step), else 3 (80), the occupancy the shared memory of
// the common rings (2 buffers of 2048 vectors, 4 of 1024) allows; none spills.
constexpr int ln_staged_min_blocks(int nvt, int rp) { return nvt * rp <= 4 ? 4 : 3; }

template <typename S, int NVT, int RP, bool GBS>
__global__ void __launch_bounds__(kStagedBlock, ln_staged_min_blocks(NVT, RP))
layernorm_staged_kernel(const void* x, const void* __restrict__ gamma,
                        const void* __restrict__ beta, void* y, int64_t rows, int64_t cols,
                        float eps, int chunk_vecs, int stages, unsigned long long wait_ns,
                        int probe) {
    namespace cg = cooperative_groups;
    using C = Codec<S, 16>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;
    constexpr int kWarps = kStagedBlock / 32;
    // 16-bit storage takes the one-pass statistics where the shift is near the mean (the
    // rows kernel's rule, layernorm.cu); fp32 storage always takes two passes.
    constexpr bool kOnePass = ES == 2;
    // gamma and beta vectors in flight at once in the output pass.
    constexpr int kGb = NVT < kLnGammaBatch ? NVT : kLnGammaBatch;

    // Dynamic shared memory: with GBS the CTA's chunks of gamma and beta, then `stages`
    // buffers of (the row's first 16 bytes, the CTA's chunk of the row).
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[kStagedMaxStages];
    __shared__ __align__(8) unsigned long long gb_bar;      // GBS: gamma and beta landed
    __shared__ __align__(8) unsigned long long bar_x[2];    // this step's pairs
    __shared__ __align__(8) unsigned long long bar_z[2];    // second-pass sums (16-bit only)
    __shared__ float part_a[2][RP][kWarps], part_b[2][RP][kWarps];
    // Second-pass partials: written after this step's exchange, which not every warp of the
    // CTA has finished reading part_a from; the next write comes after a later step's
    // opening barrier.
    __shared__ float part_c[RP][kWarps];
    __shared__ float slot_m[2][RP][16], slot_v[2][RP][16], slot_z[2][RP][16];
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
    unsigned char* gsm = smem;
    unsigned char* bsm = smem + static_cast<int64_t>(chunk_vecs) * 16;
    unsigned char* ring = GBS ? smem + static_cast<int64_t>(chunk_vecs) * 32 : smem;
    // Rows of this cluster: cid, cid + ncl, ...; the j-th uses ring slot j mod stages.
    const int64_t my_rows = cid < rows ? (rows - cid + ncl - 1) / ncl : 0;

    if (t == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&full[s]), 1);
        mbar_init(smem_u32(&bar_x[0]), 1);
        mbar_init(smem_u32(&bar_x[1]), 1);
        mbar_init(smem_u32(&bar_z[0]), 1);
        mbar_init(smem_u32(&bar_z[1]), 1);
        mbar_init(smem_u32(&gb_bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        timed_out = 0;
        // The chunks that the first bulk loads below, and the first output pass, will read
        // (after griddep_wait).
        prefetch_l2(static_cast<const char*>(gamma) + v0 * 16, my_bytes);
        prefetch_l2(static_cast<const char*>(beta) + v0 * 16, my_bytes);
        for (int s = 0; s < stages && s < my_rows; ++s) {
            const int64_t row = cid + s * ncl;
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
    // One thread: the head of row j and this CTA's chunk, into ring slot s (j mod stages).
    auto issue = [&](int64_t j, int s) {
        const int64_t row = cid + j * ncl;
        const uint32_t bar = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(ring + s * stage_bytes);
        mbar_arrive_expect_tx(bar, 16u + my_bytes);
        if (probe && j == 0) return;   // diagnostic: this copy is never issued
        bulk_load(dst, xb + row * pitch, 16u, bar);
        if (my_bytes > 0) bulk_load(dst + 16, xb + row * pitch + v0 * 16, my_bytes, bar);
    };
    if (t == 0) {
        if (GBS && my_bytes > 0) {
            mbar_arrive_expect_tx(smem_u32(&gb_bar), 2u * my_bytes);
            bulk_load(smem_u32(gsm), static_cast<const char*>(gamma) + v0 * 16, my_bytes,
                      smem_u32(&gb_bar));
            bulk_load(smem_u32(bsm), static_cast<const char*>(beta) + v0 * 16, my_bytes,
                      smem_u32(&gb_bar));
        }
        for (int j = 0; j < stages && j < my_rows; ++j) issue(j, j);
    }
    bool gb_ready = !GBS || my_bytes == 0;
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    const float n = static_cast<float>(cols);
    // Elements of cluster rank `lane` (lanes past the cluster: none), for the merge.
    float n_lane = 0.0f;
    {
        const int lane = t & 31;
        const int64_t lq = nvec - static_cast<int64_t>(lane) * chunk_vecs;
        if (lane < nct && lq > 0) n_lane = static_cast<float>((lq < chunk_vecs ? lq : chunk_vecs) * E);
    }
    const float n_k = static_cast<float>(my_vecs * E);
    int64_t nz = 0;   // second-pass exchanges so far (the same count in every CTA)
    int64_t fail_step = -1;
    int64_t i = 0;
    // Ring slot and phase parity of the step's first row (row j0 uses slot j0 mod stages,
    // phase (j0 / stages) mod 2), advanced without dividing.
    int slot0 = 0;
    uint32_t par0 = 0;
    for (int64_t j0 = 0; j0 < my_rows; j0 += RP, ++i) {
        const int set = static_cast<int>(i & 1);
        int slot[RP];
        uint32_t par[RP];
#pragma unroll
        for (int u = 0; u < RP; ++u) {
            slot[u] = slot0 + u;
            par[u] = par0;
            if (slot[u] >= stages) {
                slot[u] -= stages;
                par[u] ^= 1u;
            }
        }
        slot0 += RP;
        if (slot0 >= stages) {
            slot0 -= stages;
            par0 ^= 1u;
        }
        if (fail_step < 0) {
#pragma unroll
            for (int u = 0; u < RP; ++u) {
                if (j0 + u < my_rows &&
                    !mbar_wait_bounded(smem_u32(&full[slot[u]]), par[u], wait_ns))
                    timed_out = 1;
            }
        }
        __syncthreads();
        if (fail_step < 0 && timed_out) fail_step = i;   // the same in every thread
        const bool ok = fail_step < 0;

        // 1. The shifts and this thread's vectors of the step's rows, into registers.
        float shift[RP];
        Raw<16> v[RP][NVT];
#pragma unroll
        for (int u = 0; u < RP; ++u) {
            const unsigned char* buf = ring + slot[u] * stage_bytes;
            const bool on = ok && j0 + u < my_rows;
            shift[u] = 0.0f;
            if (on) C::each(ld_smem16(buf), [&](int e, float f) { if (e == 0) shift[u] = f; });
#pragma unroll
            for (int k = 0; k < NVT; ++k) {
                const int vi = t + k * kStagedBlock;
                v[u][k] = (on && vi < my_vecs) ? ld_smem16(buf + 16 + vi * 16) : raw_zero<16>();
            }
        }
        // 2. The chunk's sums: sum(x - K), and in 16-bit storage also sum((x - K)^2).
#pragma unroll
        for (int u = 0; u < RP; ++u) {
            const f32x2 k2 = f2_make(shift[u], shift[u]);
            float a = 0.0f, q = 0.0f;
            if constexpr (kOnePass) {
                f32x2 a2 = f2_make(0.0f, 0.0f), q2 = f2_make(0.0f, 0.0f);
#pragma unroll
                for (int k = 0; k < NVT; ++k)
                    if (t + k * kStagedBlock < my_vecs)
                        C::each_pair(v[u][k], [&](int, f32x2 p) {
                            const f32x2 d = f2_sub(p, k2);
                            a2 = f2_add(a2, d);
                            q2 = f2_fma(d, d, q2);
                        });
                a = f2_lo(a2) + f2_hi(a2);
                q = f2_lo(q2) + f2_hi(q2);
                q = warp_sum(q);
                if ((t & 31) == 0) part_b[set][u][t / 32] = q;
            } else {
#pragma unroll
                for (int k = 0; k < NVT; ++k)
                    if (t + k * kStagedBlock < my_vecs) a += shifted16<C>(v[u][k], k2);
            }
            a = warp_sum(a);
            if ((t & 31) == 0) part_a[set][u][t / 32] = a;
        }
        __syncthreads();   // the buffers have been read: refill them now
        if (ok && t == 0) {
            // Order this CTA's generic-proxy reads of the buffers before the async-proxy
            // writes that refill them.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
            for (int u = 0; u < RP; ++u) {
                const int64_t j = j0 + u + stages;   // the same slot as row j0 + u
                if (j < my_rows) issue(j, slot[u]);
            }
        }
        // Two-pass form (fp32 storage): m_k = sum(x - K) / n_k, then M2_k = sum(((x - K) -
        // m_k)^2) in a second reduction; the pair is merged with Chan's formula. One-pass form
        // (16-bit storage): the sums themselves are exchanged.
        float ex_a[RP], ex_b[RP];
#pragma unroll
        for (int u = 0; u < RP; ++u) {
            float sa = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sa += part_a[set][u][w];
            if constexpr (kOnePass) {
                ex_a[u] = sa;
            } else {
                ex_a[u] = my_vecs > 0 ? sa / n_k : 0.0f;
                const f32x2 k2 = f2_make(shift[u], shift[u]);
                const f32x2 mk2 = f2_make(ex_a[u], ex_a[u]);
                float b = 0.0f;
#pragma unroll
                for (int k = 0; k < NVT; ++k)
                    if (t + k * kStagedBlock < my_vecs) b += deviations16<C>(v[u][k], k2, mk2);
                b = warp_sum(b);
                if ((t & 31) == 0) part_b[set][u][t / 32] = b;
            }
        }
        if constexpr (!kOnePass) __syncthreads();
        // 3. The exchange: this CTA's pair of every row of the step to every CTA of the
        // cluster.
        if (t == 0) {
            mbar_arrive_expect_tx(smem_u32(&bar_x[set]), static_cast<uint32_t>(nct) * RP * 8u);
        }
        if (t < nct) {
            const uint32_t b = map_rank(smem_u32(&bar_x[set]), static_cast<uint32_t>(t));
#pragma unroll
            for (int u = 0; u < RP; ++u) {
                float sb = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sb += part_b[set][u][w];
                ex_b[u] = sb;
                st_async_f32(map_rank(smem_u32(&slot_m[set][u][rank]), static_cast<uint32_t>(t)),
                             ex_a[u], b);
                st_async_f32(map_rank(smem_u32(&slot_v[set][u][rank]), static_cast<uint32_t>(t)),
                             ex_b[u], b);
            }
        }
        // Every CTA waits for all pairs of every step, even after a failure: a peer's
        // stores must have landed before this CTA's shared memory is released.
        if (!mbar_wait_bounded(smem_u32(&bar_x[set]), static_cast<uint32_t>((i >> 1) & 1), wait_ns))
            timed_out = 1;
        // Merge the C chunks' statistics: lane q of every warp takes rank q's pair and the
        // butterfly sums give every lane of every warp, in every CTA, the same bits.
        const int lane = t & 31;
        float mu[RP], var[RP];
        bool again = false;   // a row of the step needs the second pass (the same everywhere)
#pragma unroll
        for (int u = 0; u < RP; ++u) {
            if constexpr (kOnePass) {
                mu[u] = warp_sum(lane < nct ? slot_m[set][u][lane] : 0.0f) / n;
                const float s2 = warp_sum(lane < nct ? slot_v[set][u][lane] : 0.0f) / n;
                var[u] = s2 - mu[u] * mu[u];
                // The shift within two standard deviations of the mean: the difference
                // cancels at most about 5 var against its inputs and is kept; otherwise
                // the row takes the second pass below.
                if (!(mu[u] * mu[u] <= 4.0f * var[u])) again = true;
            } else {
                const float mq = lane < nct ? slot_m[set][u][lane] : 0.0f;
                mu[u] = warp_sum(n_lane * mq) / n;
                const float dq = mq - mu[u];
                var[u] = warp_sum(lane < nct ? fmaf(n_lane * dq, dq, slot_v[set][u][lane]) : 0.0f) / n;
            }
        }
        if constexpr (kOnePass) {
            if (again) {
                // Second pass for the rows whose shift lies far from the mean (or whose
                // difference rounded below 0): sum(((x - K) - mu)^2) over the chunk, one
                // more block reduction and exchange (uniform across the cluster: every CTA
                // merged the same bits).
                const int zs = static_cast<int>(nz & 1);
#pragma unroll
                for (int u = 0; u < RP; ++u) {
                    const f32x2 k2 = f2_make(shift[u], shift[u]);
                    const f32x2 m2v = f2_make(mu[u], mu[u]);
                    float b = 0.0f;
#pragma unroll
                    for (int k = 0; k < NVT; ++k)
                        if (t + k * kStagedBlock < my_vecs) b += deviations16<C>(v[u][k], k2, m2v);
                    b = warp_sum(b);
                    if ((t & 31) == 0) part_c[u][t / 32] = b;
                }
                __syncthreads();
                if (t == 0) {
                    mbar_arrive_expect_tx(smem_u32(&bar_z[zs]), static_cast<uint32_t>(nct) * RP * 4u);
                }
                if (t < nct) {
                    const uint32_t b = map_rank(smem_u32(&bar_z[zs]), static_cast<uint32_t>(t));
#pragma unroll
                    for (int u = 0; u < RP; ++u) {
                        float sb = 0.0f;
#pragma unroll
                        for (int w = 0; w < kWarps; ++w) sb += part_c[u][w];
                        st_async_f32(map_rank(smem_u32(&slot_z[zs][u][rank]), static_cast<uint32_t>(t)),
                                     sb, b);
                    }
                }
                if (!mbar_wait_bounded(smem_u32(&bar_z[zs]), static_cast<uint32_t>((nz >> 1) & 1), wait_ns))
                    timed_out = 1;
#pragma unroll
                for (int u = 0; u < RP; ++u) {
                    if (!(mu[u] * mu[u] <= 4.0f * var[u]))
                        var[u] = warp_sum(lane < nct ? slot_z[zs][u][lane] : 0.0f) / n;
                }
                ++nz;
            }
        }
        f32x2 kk[RP], mm[RP], rr[RP];
#pragma unroll
        for (int u = 0; u < RP; ++u) {
            const float rstd = rsqrtf(var[u] + eps);
            kk[u] = f2_make(shift[u], shift[u]);
            mm[u] = f2_make(mu[u], mu[u]);
            rr[u] = f2_make(rstd, rstd);
        }
        // 4. The output pass: each vector of gamma and beta loaded once for the step's rows,
        // in batches of kGb vectors whose loads are all issued before the batch's stores (the
        // loads and stores are ordered asm statements, so loads interleaved with stores would
        // wait out one L2 round trip per vector).
        if (ok && !gb_ready) {
            if (!mbar_wait_bounded(smem_u32(&gb_bar), 0u, wait_ns)) timed_out = 1;
            gb_ready = true;
        }
        if (ok) {
            const char* gb = static_cast<const char*>(gamma) + v0 * 16;
            const char* bb = static_cast<const char*>(beta) + v0 * 16;
#pragma unroll
            for (int k0 = 0; k0 < NVT; k0 += kGb) {
                Raw<16> gv[kGb], bv[kGb];
#pragma unroll
                for (int q = 0; q < kGb; ++q) {
                    const int vi = t + (k0 + q) * kStagedBlock;
                    if (vi < my_vecs) {
                        if constexpr (GBS) {
                            gv[q] = ld_smem16(gsm + vi * 16);
                            bv[q] = ld_smem16(bsm + vi * 16);
                        } else {
                            gv[q] = ld_shared_ro<16>(gb + vi * 16);
                            bv[q] = ld_shared_ro<16>(bb + vi * 16);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < kGb; ++q) {
                    const int vi = t + (k0 + q) * kStagedBlock;
                    if (vi < my_vecs) {
#pragma unroll
                        for (int u = 0; u < RP; ++u) {
                            if (j0 + u < my_rows) {
                                const int64_t row = cid + (j0 + u) * ncl;
                                st_out<16>(static_cast<char*>(y) + row * pitch + (v0 + vi) * 16,
                                           affine16<C>(v[u][k0 + q], gv[q], bv[q], kk[u], mm[u],
                                                       rr[u]));
                            }
                        }
                    }
                }
            }
        }
    }

    __syncthreads();
    if (timed_out && t == 0) {
        atomicOr(&g_ln_device_error, kDeviceErrorWaitTimeout);
        // Copies that may still be in flight into this CTA's shared memory: gamma and beta
        // (GBS), and the rows from the failed step's first up to `stages` rows on. Wait for
        // each, bounded.
        if (!gb_ready) mbar_wait_bounded(smem_u32(&gb_bar), 0u, wait_ns);
        const int64_t f = (fail_step < 0 ? i : fail_step) * RP;
        for (int64_t j = f; j < f + stages && j < my_rows; ++j)
            mbar_wait_bounded(smem_u32(&full[j % stages]), static_cast<uint32_t>((j / stages) & 1),
                              wait_ns);
    }
}

template <typename S, int NVT, int RP, bool GBS>
cudaError_t launch_ln_staged_gbs(const LayernormArgs& a, int cluster, int stages,
                                 int chunk_vecs, unsigned long long wait_ns, int probe,
                                 cudaStream_t s) {
    auto kernel = layernorm_staged_kernel<S, NVT, RP, GBS>;
    const size_t smem = static_cast<size_t>(ln_staged_smem_bytes(chunk_vecs, stages, GBS));
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
                              chunk_vecs, stages, wait_ns, probe);
}

// gamma and beta go to shared memory when they fit beside the ring without costing
// occupancy (ln_staged_gamma_in_smem), which happens only for chunks of up to 4 vectors a
// thread.
template <typename S, int NVT, int RP>
cudaError_t launch_ln_staged(const LayernormArgs& a, int cluster, int stages, int chunk_vecs,
                             unsigned long long wait_ns, int probe, cudaStream_t s) {
    if constexpr (NVT <= 4) {
        if (ln_staged_gamma_in_smem(chunk_vecs, stages))
            return launch_ln_staged_gbs<S, NVT, RP, true>(a, cluster, stages, chunk_vecs,
                                                          wait_ns, probe, s);
    }
    return launch_ln_staged_gbs<S, NVT, RP, false>(a, cluster, stages, chunk_vecs, wait_ns,
                                                   probe, s);
}

template <typename S, int RP>
cudaError_t launch_ln_staged_nvt(const LayernormArgs& a, int cluster, int stages,
                                 unsigned long long wait_ns, int probe, cudaStream_t s) {
    constexpr int E = 16 / Storage<S>::kBytes;
    const int64_t nvec = a.cols / E;
    const int chunk = static_cast<int>((nvec + cluster - 1) / cluster);
    const int need = (chunk + kStagedBlock - 1) / kStagedBlock;
    if (need <= 1) return launch_ln_staged<S, 1, RP>(a, cluster, stages, chunk, wait_ns, probe, s);
    if (need <= 2) return launch_ln_staged<S, 2, RP>(a, cluster, stages, chunk, wait_ns, probe, s);
    if (need <= 4) return launch_ln_staged<S, 4, RP>(a, cluster, stages, chunk, wait_ns, probe, s);
    if constexpr (RP == 1) {
        if (need <= kStagedMaxVecsPerThread)
            return launch_ln_staged<S, 8, 1>(a, cluster, stages, chunk, wait_ns, probe, s);
    }
    return cudaErrorInvalidValue;
}

template <typename S>
cudaError_t launch_ln_staged_rp(const LayernormArgs& a, int cluster, int stages, int rp,
                                unsigned long long wait_ns, int probe, cudaStream_t s) {
    return rp == 2 ? launch_ln_staged_nvt<S, 2>(a, cluster, stages, wait_ns, probe, s)
                   : launch_ln_staged_nvt<S, 1>(a, cluster, stages, wait_ns, probe, s);
}

}  // namespace

cudaError_t layernorm_staged_launch(DType t, int cluster, int stages, int rows_per_step,
                                    const LayernormArgs& a, cudaStream_t s,
                                    unsigned long long wait_ns, int probe) {
    if (cluster < 1 || cluster > 16 || stages < 2 || stages > kStagedMaxStages ||
        rows_per_step < 1 || rows_per_step > kLnMaxRp || stages < rows_per_step)
        return cudaErrorInvalidValue;
    switch (t) {
        case DType::BF16: return launch_ln_staged_rp<bf16_t>(a, cluster, stages, rows_per_step, wait_ns, probe, s);
        case DType::F16: return launch_ln_staged_rp<f16_t>(a, cluster, stages, rows_per_step, wait_ns, probe, s);
        default: return launch_ln_staged_rp<f32_t>(a, cluster, stages, rows_per_step, wait_ns, probe, s);
    }
}

cudaError_t read_layernorm_device_errors(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_ln_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_ln_device_error, &zero, sizeof(unsigned int));
}

}  // namespace camp
