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
// (NVN accesses of VB bytes) and, for l < (Dr/2) / RE, elements l*RE .. l*RE + RE - 1 of
// both rope halves (RB bytes each, RE = RB / element size) with their RE sine and cosine
// values; all loads are issued before any arithmetic. The rope width is spread over as
// many lanes as it fills (RB is the narrowest access that holds a pair and keeps it within
// one warp), so that no lane holds much more than another: at the common widths the
// kernel fits 32 registers and a full SM of warps keeps enough bytes in flight. The sum of squares is a butterfly warp shuffle
// (no barrier); the table row s = t mod S is a multiply-shift division when there are
// fewer than 2^32 tokens, else a 64-bit remainder; both outputs are written once.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

template <typename S, int VB, int NVN, int RB>
__global__ void __launch_bounds__(kKvBlock, kv_min_blocks(Storage<S>::kBytes, VB, NVN, RB))
kv_rmsnorm_rope_cache_kernel(const void* kv, const void* __restrict__ gamma,
                             const float* __restrict__ sin_t, const float* __restrict__ cos_t,
                             const int64_t* __restrict__ slots, void* cache_n, void* cache_r,
                             int64_t tokens, int64_t seq, FastDiv seq_div, bool fast_seq,
                             int dn, int dr, int64_t num_slots, float eps) {
    using C = Codec<S, VB>;
    using CR = Codec<S, RB>;
    constexpr int E = C::kElems;
    constexpr int RE = CR::kElems;
    constexpr int ES = Storage<S>::kBytes;

    const int lane = threadIdx.x & 31;
    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0 && block * kKvTokensPerCta < tokens) {   // this CTA's kv rows, their
        const int64_t t0 = block * kKvTokensPerCta;               // slots and table rows
        const int64_t nt = tokens - t0 < kKvTokensPerCta ? tokens - t0 : kKvTokensPerCta;
        const int64_t rb = static_cast<int64_t>(dn + dr) * ES;
        prefetch_l2(static_cast<const char*>(kv) + t0 * rb, nt * rb);
        prefetch_l2(slots + t0, nt * 8);
        const int64_t s0 = t0 % seq;
        const int64_t ns = nt < seq - s0 ? nt : seq - s0;
        prefetch_l2(sin_t + s0 * (dr / 2), ns * (dr / 2) * 4);
        prefetch_l2(cos_t + s0 * (dr / 2), ns * (dr / 2) * 4);
    }
    griddep_wait();
    griddep_launch_dependents();

    const int64_t token = block * kKvTokensPerCta + threadIdx.x / 32;
    if (token >= tokens) return;                       // whole warps only; no barrier below

    const int half = dr / 2;
    const int live = dn / E - lane;                    // norm access k exists iff k*32 < live
    const char* row = static_cast<const char*>(kv) + token * static_cast<int64_t>(dn + dr) * ES;
    const char* xn = row + static_cast<int64_t>(lane) * VB;
    const char* xr = row + static_cast<int64_t>(dn) * ES + static_cast<int64_t>(lane) * RB;

    Raw<VB> v[NVN];
#pragma unroll
    for (int k = 0; k < NVN; ++k)
        v[k] = (k * 32 < live) ? ld_stream<VB>(xn + k * 32 * VB) : raw_zero<VB>();
    const bool roper = lane < half / RE;
    Raw<RB> lo = raw_zero<RB>(), hi = raw_zero<RB>();
    float sn[RE], cs[RE];
    if (roper) {
        lo = ld_stream<RB>(xr);
        hi = ld_stream<RB>(xr + static_cast<int64_t>(half) * ES);
        const int64_t s = fast_seq ? static_cast<int64_t>(
                                         static_cast<uint32_t>(token) -
                                         fast_div(static_cast<uint32_t>(token), seq_div) *
                                             static_cast<uint32_t>(seq))
                                   : token % seq;
        const int64_t toff = s * half + static_cast<int64_t>(lane) * RE;
        load_table<RE>(sin_t + toff, sn);
        load_table<RE>(cos_t + toff, cs);
    }
    const int64_t slot = slots[token];

    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < NVN; ++k) C::each(v[k], [&](int, float f) { ss = fmaf(f, f, ss); });
    ss = warp_sum(ss);
    if (slot < 0 || slot >= num_slots) return;         // padding: nothing is written
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
        Raw<RB> o1, o2;
        CR::map2(lo, hi, o1, o2, [&](int e, float x1, float x2) {
            return make_float2(diff_of_products(x1, cs[e], x2, sn[e]),
                               sum_of_products(x2, cs[e], x1, sn[e]));
        });
        char* yr = static_cast<char*>(cache_r) + slot * static_cast<int64_t>(dr) * ES +
                   static_cast<int64_t>(lane) * RB;
        st_out<RB>(yr, o1);
        st_out<RB>(yr + static_cast<int64_t>(half) * ES, o2);
    }
}

template <typename S, int VB, int NVN, int RB>
cudaError_t launch_kv(const KvCacheArgs& a, cudaStream_t s) {
    const int64_t blocks = (a.tokens + kKvTokensPerCta - 1) / kKvTokensPerCta;
    const bool fast = a.tokens <= 0xFFFFFFFFll;
    const FastDiv d = make_fast_div(static_cast<uint32_t>(fast ? a.seq : 1));
    return launch_pdl(kv_rmsnorm_rope_cache_kernel<S, VB, NVN, RB>, grid_2d(blocks),
                      dim3(kKvBlock), s, a.kv, a.gamma, a.sin_t, a.cos_t, a.slots, a.cache_n,
                      a.cache_r, a.tokens, a.seq, d, fast, static_cast<int>(a.dn),
                      static_cast<int>(a.dr), a.num_slots, a.eps);
}

// 16-byte norm accesses: the rope part takes 4- (16-bit types only), 8- or 16-byte accesses.
template <typename S, int NVN>
cudaError_t launch_kv_rb(int rb, const KvCacheArgs& a, cudaStream_t s) {
    switch (rb) {
        case 4:
            if constexpr (Storage<S>::kBytes == 2) return launch_kv<S, 16, NVN, 4>(a, s);
            else return cudaErrorInvalidValue;
        case 8: return launch_kv<S, 16, NVN, 8>(a, s);
        case 16: return launch_kv<S, 16, NVN, 16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename S>
cudaError_t launch_kv_vec(int nvn, int rb, const KvCacheArgs& a, cudaStream_t s) {
    switch (nvn) {
        case 1: return launch_kv_rb<S, 1>(rb, a, s);
        case 2: return launch_kv_rb<S, 2>(rb, a, s);
        case 4: return launch_kv_rb<S, 4>(rb, a, s);
        case 8: return launch_kv_rb<S, 8>(rb, a, s);
        default: return cudaErrorInvalidValue;   // 16 is not built here: it would spill
    }
}

// Element accesses for both parts.
template <typename S>
cudaError_t launch_kv_elem(int nvn, const KvCacheArgs& a, cudaStream_t s) {
    constexpr int ES = Storage<S>::kBytes;
    switch (nvn) {
        case 1: return launch_kv<S, ES, 1, ES>(a, s);
        case 2: return launch_kv<S, ES, 2, ES>(a, s);
        case 4: return launch_kv<S, ES, 4, ES>(a, s);
        case 8: return launch_kv<S, ES, 8, ES>(a, s);
        case 16: return launch_kv<S, ES, 16, ES>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool kv_cache_compiled(DType t, int vec_bytes, int nvn, int rope_bytes) {
    const int es = elem_bytes(t);
    if (vec_bytes == 16)
        return (nvn == 1 || nvn == 2 || nvn == 4 || nvn == 8) &&
               ((rope_bytes == 4 && es == 2) || rope_bytes == 8 || rope_bytes == 16);
    if (vec_bytes == es)
        return (nvn == 1 || nvn == 2 || nvn == 4 || nvn == 8 || nvn == 16) && rope_bytes == es;
    return false;
}

cudaError_t kv_cache_launch(DType t, int vec_bytes, int nvn, int rope_bytes,
                            const KvCacheArgs& a, cudaStream_t s) {
    if (!kv_cache_compiled(t, vec_bytes, nvn, rope_bytes)) return cudaErrorInvalidValue;
    if (t == DType::BF16)
        return vec_bytes == 16 ? launch_kv_vec<bf16_t>(nvn, rope_bytes, a, s)
                               : launch_kv_elem<bf16_t>(nvn, a, s);
    if (t == DType::F16)
        return vec_bytes == 16 ? launch_kv_vec<f16_t>(nvn, rope_bytes, a, s)
                               : launch_kv_elem<f16_t>(nvn, a, s);
    return vec_bytes == 16 ? launch_kv_vec<f32_t>(nvn, rope_bytes, a, s)
                           : launch_kv_elem<f32_t>(nvn, a, s);
}

}  // namespace camp
