// Fused KV RMSNorm + RoPE + cache scatter for sm_103a.
//
// Operation (TileLang tutorial ch. 02, section 1.2, describing Ascend's KvRmsNormRopeCache
// operator): the last axis of the kv tensor is split, the left part goes through RMSNorm
// and the right part through RoPE, and the two results are scattered into two caches.
// Here kv is [B, S, Dn + Dr] (one KV head, as in multi-head latent attention), the norm
// part is RMSNorm with weight gamma[Dn] (the same arithmetic as camp_rmsnorm), the rope
// part is rotate-half RoPE with the tables' row s (the same arithmetic as camp_rope), and
// token t = b*S + s is written to row slots[t] of cache_n[num_slots, Dn] and of
// cache_r[num_slots, Dr]; a slot outside [0, num_slots) is not written (padding).
//
// Mapping: one warp per token, 8 tokens per CTA. Lane l loads norm accesses l, l+32, ...
// (NVN of them) and, for l < (Dr/2)/E, vector l of both rope halves; all loads are issued
// before any arithmetic. The sum of squares is a butterfly warp shuffle (no barrier), the
// table row is s = t mod S, and both outputs are written once to the cache rows.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

template <typename S, int VB, int NVN>
__global__ void __launch_bounds__(kKvBlock, 4)
kv_rmsnorm_rope_cache_kernel(const void* kv, const void* __restrict__ gamma,
                             const float* __restrict__ sin_t, const float* __restrict__ cos_t,
                             const int64_t* __restrict__ slots, void* cache_n, void* cache_r,
                             int64_t tokens, int64_t seq, int dn, int dr, int64_t num_slots,
                             float eps) {
    using C = Codec<S, VB>;
    constexpr int E = C::kElems;
    constexpr int ES = Storage<S>::kBytes;

    griddep_wait();
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31;
    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    const int64_t token = block * kKvTokensPerCta + threadIdx.x / 32;
    if (token >= tokens) return;                       // whole warps only; no barrier below
    const int64_t slot = slots[token];
    if (slot < 0 || slot >= num_slots) return;         // padding: nothing is written

    const int half = dr / 2;
    const int nvh = half / E;                          // rope vectors per half
    const int live = dn / E - lane;                    // norm access k exists iff k*32 < live
    const char* row = static_cast<const char*>(kv) + token * static_cast<int64_t>(dn + dr) * ES;
    const char* xn = row + static_cast<int64_t>(lane) * VB;
    const char* xr = row + static_cast<int64_t>(dn) * ES + static_cast<int64_t>(lane) * VB;

    Raw<VB> v[NVN];
#pragma unroll
    for (int k = 0; k < NVN; ++k)
        v[k] = (k * 32 < live) ? ld_stream<VB>(xn + k * 32 * VB) : raw_zero<VB>();
    const bool roper = lane < nvh;
    Raw<VB> lo = raw_zero<VB>(), hi = raw_zero<VB>();
    if (roper) {
        lo = ld_stream<VB>(xr);
        hi = ld_stream<VB>(xr + static_cast<int64_t>(half) * ES);
    }

    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < NVN; ++k) C::each(v[k], [&](int, float f) { ss = fmaf(f, f, ss); });
    ss = warp_sum(ss);
    const float rinv = rsqrtf(ss / static_cast<float>(dn) + eps);

    char* yn = static_cast<char*>(cache_n) + slot * static_cast<int64_t>(dn) * ES +
               static_cast<int64_t>(lane) * VB;
    const char* gt = static_cast<const char*>(gamma) + static_cast<int64_t>(lane) * VB;
#pragma unroll
    for (int k = 0; k < NVN; ++k) {
        if (k * 32 < live) {
            float gf[E];
            C::each(ld_shared_ro<VB>(gt + k * 32 * VB), [&](int e, float f) { gf[e] = f; });
            st_out<VB>(yn + k * 32 * VB,
                       C::map(v[k], [&](int e, float xf) { return (xf * rinv) * gf[e]; }));
        }
    }

    if (roper) {
        const int64_t s = token % seq;
        float sn[E], cs[E];
        const int64_t toff = s * half + static_cast<int64_t>(lane) * E;
        load_table<E>(sin_t + toff, sn);
        load_table<E>(cos_t + toff, cs);
        Raw<VB> o1, o2;
        C::map2(lo, hi, o1, o2, [&](int e, float x1, float x2) {
            return make_float2(diff_of_products(x1, cs[e], x2, sn[e]),
                               sum_of_products(x2, cs[e], x1, sn[e]));
        });
        char* yr = static_cast<char*>(cache_r) + slot * static_cast<int64_t>(dr) * ES +
                   static_cast<int64_t>(lane) * VB;
        st_out<VB>(yr, o1);
        st_out<VB>(yr + static_cast<int64_t>(half) * ES, o2);
    }
}

template <typename S, int VB, int NVN>
cudaError_t launch_kv(const KvCacheArgs& a, cudaStream_t s) {
    const int64_t blocks = (a.tokens + kKvTokensPerCta - 1) / kKvTokensPerCta;
    return launch_pdl(kv_rmsnorm_rope_cache_kernel<S, VB, NVN>, grid_2d(blocks), dim3(kKvBlock),
                      s, a.kv, a.gamma, a.sin_t, a.cos_t, a.slots, a.cache_n, a.cache_r,
                      a.tokens, a.seq, static_cast<int>(a.dn), static_cast<int>(a.dr),
                      a.num_slots, a.eps);
}

template <typename S, int VB>
cudaError_t launch_kv_nvn(int nvn, const KvCacheArgs& a, cudaStream_t s) {
    switch (nvn) {
        case 1: return launch_kv<S, VB, 1>(a, s);
        case 2: return launch_kv<S, VB, 2>(a, s);
        case 4: return launch_kv<S, VB, 4>(a, s);
        case 8: return launch_kv<S, VB, 8>(a, s);
        case 16:
            if constexpr (VB == 16) return cudaErrorInvalidValue;   // not built: would spill
            else return launch_kv<S, VB, 16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t kv_cache_launch(DType t, int vec_bytes, int nvn, const KvCacheArgs& a,
                            cudaStream_t s) {
    if (t == DType::BF16) {
        if (vec_bytes == 16) return launch_kv_nvn<bf16_t, 16>(nvn, a, s);
        if (vec_bytes == 2) return launch_kv_nvn<bf16_t, 2>(nvn, a, s);
    } else {
        if (vec_bytes == 16) return launch_kv_nvn<f32_t, 16>(nvn, a, s);
        if (vec_bytes == 4) return launch_kv_nvn<f32_t, 4>(nvn, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace camp
