// Concatenation of cached and new keys along the sequence with the grouped-query head
// repeat, in one pass, for sm_103a.
//
// Operation (gollamago README, "RoPE 与 RMSNorm 实现说明", list of what is not handled:
// attention's repeat_interleave stays on the PyTorch path, after the torch.cat of the
// cached keys with the new ones):
//   out[b, t, h*n_rep + r, :]   = past[b, t, h, :]                              t < P
//   out[b, P+s, h*n_rep + r, :] = rope(fresh[b, s, h, :]) at table row P + s      s < S
// for every r < n_rep. The rotation is camp_rope's rotate-half arithmetic (compensated
// products, one rounding); without tables the new rows are copied. A copied value is
// bit-exact.
//
// Mapping: camp_rope's tiled mapping over the (b, t) rows of the output. A CTA covers `tpc`
// consecutive rows; thread (row, head group, vector j) loads vector j of both halves of HPT
// source heads, once, then (new rows with tables only) the row's E sine and cosine values,
// and stores each head n_rep times: output heads h*n_rep .. h*n_rep + n_rep - 1 are
// adjacent rows, so the copies of one vector are n_rep stores one head row apart. Every
// source byte is read from HBM once and every output byte written once.
#include "common.cuh"
#include "kernels.h"

namespace camp {
namespace {

template <typename S, int VB, int HPT>
__global__ void __launch_bounds__(kRopeBlock, kv_cat_min_blocks(HPT, std::is_same_v<S, f16_t>))
kv_cat_repeat_kernel(const void* past, const void* fresh, const float* __restrict__ sin_t,
                     const float* __restrict__ cos_t, void* out, int64_t rows, FastDiv seq,
                     uint32_t past_len, int heads, int n_rep, int half) {
    constexpr int E = Codec<S, VB>::kElems;
    constexpr int ES = Storage<S>::kBytes;

    const int nvh = half / E;                                  // vectors per half
    const int per_row = ((heads + HPT - 1) / HPT) * nvh;       // threads per (b, t) row
    const int tpc = kRopeBlock / per_row;
    const int tk = static_cast<int>(threadIdx.x) / per_row;
    const int64_t block = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0) {
        // The source rows of this CTA's output rows, as runs that are contiguous in past or
        // in fresh (at most a few per batch entry the CTA spans), and the table rows of
        // the rotated ones.
        const int64_t T = seq.d, P = past_len, S = T - P;
        const int64_t hb = static_cast<int64_t>(heads) * 2 * ES * half;   // one (b, t) row
        int64_t g = block * tpc;
        const int64_t g1 = rows - g < tpc ? rows : g + tpc;
        while (g < g1) {
            const int64_t b = g / T, t = g - b * T;
            const bool old = t < P;
            const int64_t end = old ? (b * T + P < g1 ? b * T + P : g1) : (b * T + T < g1 ? b * T + T : g1);
            if (old) {
                prefetch_l2(static_cast<const char*>(past) + (b * P + t) * hb, (end - g) * hb);
            } else {
                prefetch_l2(static_cast<const char*>(fresh) + (b * S + t - P) * hb, (end - g) * hb);
                if (sin_t != nullptr) {
                    prefetch_l2(sin_t + t * half, (end - g) * half * 4);
                    prefetch_l2(cos_t + t * half, (end - g) * half * 4);
                }
            }
            g = end;
        }
    }
    griddep_wait();
    griddep_launch_dependents();
    const int64_t g = block * tpc + tk;                        // b * (P + S) + t
    if (tk >= tpc || g >= rows) return;                        // no barrier in this kernel
    const int r = static_cast<int>(threadIdx.x) - tk * per_row;
    const int hg = r / nvh;
    const int j = r - hg * nvh;
    const int h0 = hg * HPT;
    const int nh = heads - h0 < HPT ? heads - h0 : HPT;

    const uint32_t g32 = static_cast<uint32_t>(g);
    const uint32_t b = fast_div(g32, seq);
    const uint32_t t = g32 - b * seq.d;
    const bool old_row = t < past_len;
    const int64_t src_row = old_row
        ? static_cast<int64_t>(b) * past_len + t
        : static_cast<int64_t>(b) * (seq.d - past_len) + (t - past_len);

    const int64_t row_bytes = static_cast<int64_t>(2 * ES) * half;
    const int64_t half_bytes = static_cast<int64_t>(ES) * half;
    const char* p = static_cast<const char*>(old_row ? past : fresh) +
                    (src_row * heads + h0) * row_bytes + static_cast<int64_t>(j) * VB;
    Raw<VB> lo[HPT], hi[HPT];
#pragma unroll
    for (int u = 0; u < HPT; ++u) {
        if (u < nh) {
            lo[u] = ld_stream<VB>(p + u * row_bytes);
            hi[u] = ld_stream<VB>(p + u * row_bytes + half_bytes);
        }
    }

    if (!old_row && sin_t != nullptr) {
        float sn[E], cs[E];
        const int64_t toff = static_cast<int64_t>(t) * half + static_cast<int64_t>(j) * E;
        load_table<E>(sin_t + toff, sn);
        load_table<E>(cos_t + toff, cs);
#pragma unroll
        for (int u = 0; u < HPT; ++u) {
            if (u < nh) {
                Raw<VB> o1, o2;
                Codec<S, VB>::map2(lo[u], hi[u], o1, o2, [&](int e, float x1, float x2) {
                    return make_float2(diff_of_products(x1, cs[e], x2, sn[e]),
                                       sum_of_products(x2, cs[e], x1, sn[e]));
                });
                lo[u] = o1;
                hi[u] = o2;
            }
        }
    }

    const int64_t hout = static_cast<int64_t>(heads) * n_rep;
    char* q = static_cast<char*>(out) + (g * hout + static_cast<int64_t>(h0) * n_rep) * row_bytes +
              static_cast<int64_t>(j) * VB;
#pragma unroll
    for (int u = 0; u < HPT; ++u) {
        if (u < nh) {
            char* qu = q + static_cast<int64_t>(u) * n_rep * row_bytes;
            for (int k = 0; k < n_rep; ++k) {
                st_out<VB>(qu + k * row_bytes, lo[u]);
                st_out<VB>(qu + k * row_bytes + half_bytes, hi[u]);
            }
        }
    }
}

template <typename S, int VB, int HPT>
cudaError_t launch_kv_cat(const KvCatArgs& a, int64_t grid, cudaStream_t s) {
    return launch_pdl(kv_cat_repeat_kernel<S, VB, HPT>, grid_2d(grid), dim3(kRopeBlock), s,
                      a.past, a.fresh, a.sin_t, a.cos_t, a.out, a.batch * (a.past_len + a.new_len),
                      make_fast_div(static_cast<uint32_t>(a.past_len + a.new_len)),
                      static_cast<uint32_t>(a.past_len), static_cast<int>(a.heads),
                      static_cast<int>(a.n_rep), static_cast<int>(a.half));
}

template <typename S, int VB>
cudaError_t launch_kv_cat_hpt(int hpt, const KvCatArgs& a, int64_t grid, cudaStream_t s) {
    switch (hpt) {
        case 1: return launch_kv_cat<S, VB, 1>(a, grid, s);
        case 2: return launch_kv_cat<S, VB, 2>(a, grid, s);
        case 4: return launch_kv_cat<S, VB, 4>(a, grid, s);
        case 8: return launch_kv_cat<S, VB, 8>(a, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool kv_cat_compiled(DType t, int vec_bytes, int heads_per_thread) {
    const bool hpt = heads_per_thread == 1 || heads_per_thread == 2 || heads_per_thread == 4 ||
                     heads_per_thread == 8;
    if (t != DType::F32)
        return hpt && (vec_bytes == 16 || vec_bytes == 8 || vec_bytes == 4 || vec_bytes == 2);
    return hpt && (vec_bytes == 16 || vec_bytes == 8 || vec_bytes == 4);
}

cudaError_t kv_cat_launch(DType t, int vec_bytes, int heads_per_thread, const KvCatArgs& a,
                          int64_t grid, cudaStream_t s) {
    if (t == DType::BF16) {
        switch (vec_bytes) {
            case 16: return launch_kv_cat_hpt<bf16_t, 16>(heads_per_thread, a, grid, s);
            case 8: return launch_kv_cat_hpt<bf16_t, 8>(heads_per_thread, a, grid, s);
            case 4: return launch_kv_cat_hpt<bf16_t, 4>(heads_per_thread, a, grid, s);
            case 2: return launch_kv_cat_hpt<bf16_t, 2>(heads_per_thread, a, grid, s);
            default: break;
        }
    } else if (t == DType::F16) {
        switch (vec_bytes) {
            case 16: return launch_kv_cat_hpt<f16_t, 16>(heads_per_thread, a, grid, s);
            case 8: return launch_kv_cat_hpt<f16_t, 8>(heads_per_thread, a, grid, s);
            case 4: return launch_kv_cat_hpt<f16_t, 4>(heads_per_thread, a, grid, s);
            case 2: return launch_kv_cat_hpt<f16_t, 2>(heads_per_thread, a, grid, s);
            default: break;
        }
    } else {
        switch (vec_bytes) {
            case 16: return launch_kv_cat_hpt<f32_t, 16>(heads_per_thread, a, grid, s);
            case 8: return launch_kv_cat_hpt<f32_t, 8>(heads_per_thread, a, grid, s);
            case 4: return launch_kv_cat_hpt<f32_t, 4>(heads_per_thread, a, grid, s);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace camp
