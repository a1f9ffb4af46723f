// CPU oracle for RMSNorm forward and rotate-half RoPE: plain, slow, fp64.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link, load or
// call this file. Its callers are the tests, the smoke check of the package entry
// point and the CPU-baseline leg of the benchmark. It shares no header, helper,
// table or constant with the CUDA library: the only thing the two sides share is
// the seeded input data.
//
// What it computes (the plain definitions, in fp64, rounded once at the end):
//
//   RMSNorm  (xserv "phase 4" design notes, RMSNorm section: rms = sqrt(sum(x^2)/hidden
//            + eps), y = x / rms * gamma; gollamago README, "RMSNorm optimisation":
//            accumulate and scale in fp32 or wider, round once on write-back)
//       ss_r  = sum_j x[r,j]^2                  (Neumaier-compensated fp64 sum)
//       rms_r = sqrt(ss_r / cols + eps)
//       y[r,j] = x[r,j] / rms_r * w[j]          then one rounding to the storage type
//
//   Residual add + RMSNorm  (TileLang tutorial ch. 02, section 4.2: the "Add before
//            RmsNorm" fused into it; the pages give no formula beyond the two operations)
//       h[r,j] = round(x[r,j] + r[r,j])         (the exact sum, one rounding)
//       y      = RMSNorm(h as stored) * w       (as above)
//
//   KV RMSNorm + RoPE + cache scatter  (TileLang tutorial ch. 02, section 1.2, describing
//            Ascend's KvRmsNormRopeCache: split the kv tail axis, RMSNorm the left part,
//            RoPE the right part, scatter both into two caches)
//       for token t = b*S + s with 0 <= slots[t] < num_slots:
//       cache_n[slots[t], :] = RMSNorm(kv[t, :Dn]) * gamma      (as above)
//       cache_r[slots[t], :] = rotate-half RoPE of kv[t, Dn:] with table row s (below)
//       other cache rows are left as they are.
//
//   RoPE, rotate-half  (gollamago README, "RoPE": rope(input, sin_table, cos_table),
//            input [batch, sequence, heads, head_dim], tables [sequence, head_dim/2],
//            each head split into two halves and rotated; tilelang tutorial ch. 02,
//            exercise E13: y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin)
//       for every (b, s, h) and i < D/2, with c = cos[s,i], sn = sin[s,i]:
//       y[b,s,h,i]       = x[b,s,h,i] * c - x[b,s,h,i+D/2] * sn
//       y[b,s,h,i+D/2]   = x[b,s,h,i+D/2] * c + x[b,s,h,i] * sn
//       then one rounding to the storage type.
//
// Storage types: fp32 (IEEE binary32), bf16 (the upper 16 bits of a binary32: 1 sign,
// 8 exponent, 7 fraction bits) and fp16 (IEEE binary16: 1 sign, 5 exponent, 10 fraction
// bits; the Intro-ops runtime's F16, code 0). Decoding any of them to fp64 is exact.
// Encoding rounds to nearest, ties to even (the pages are silent; this is the IEEE
// default).
//
//   LayerNorm  (xserv "phase 4", csrc/normalization/layernorm.cu: y = gamma * (x - mean) /
//            sqrt(var + eps) + beta, population variance)
//       mean = sum_j x_j / n,  var = sum_j (x_j - mean)^2 / n   (Neumaier sums, fp64)
//       y_j  = (x_j - mean) / sqrt(var + eps) * gamma_j + beta_j, one rounding.
//
//   KV concatenation + GQA head repeat (gollamago README, "not handled" list: attention's
//   repeat_interleave is left on the PyTorch path; the torch.cat of cached and new keys
//   along the sequence): out [B, P+S, Hk*n_rep, D] with
//       out[b, t, h*n_rep + r, :] = past[b, t, h, :]                      t < P
//       out[b, P+s, h*n_rep + r, :] = rope(new[b, s, h, :], table row P+s)  s < S
//   (rotate-half, as above; without tables the new rows are copied unrotated).
//
//   Interleaved RoPE with position ids  (xserv "phase 4" rope kernel: pairs (x[2i], x[2i+1]),
//            y0 = x0 cos - x1 sin, y1 = x0 sin + x1 cos, table row positions[token])
//       tokens whose position is outside [0, max_pos) are left unwritten.
//
//   RoPE tables  (xserv compute_rope_cache: freq_i = theta^(-2i/D), angle = p * freq_i)
//       sin[p, i] = round_fp32(sin(p * theta^(-2i/D))), cos likewise, all in fp64.
//
// Build flags matter: no -ffast-math, and -ffp-contract=off so that no multiply-add
// is fused (results must be identical on x86-64 and aarch64).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include <sched.h>

namespace {

constexpr int kOracleF16 = 0;
constexpr int kOracleF32 = 1;
constexpr int kOracleBF16 = 3;

bool storage_ok(int dtype) {
    return dtype == kOracleF16 || dtype == kOracleF32 || dtype == kOracleBF16;
}

// ---------------------------------------------------------------- storage formats

double bf16_to_double(uint16_t bits) {
    uint32_t u = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

// Round an fp64 value to the nearest bf16, ties to even, directly (no detour through
// fp32, which would round twice). Finite bf16 magnitudes are m * 2^(E-7) with integer
// m in [128, 255] for E in [-126, 127], plus the subnormals m * 2^-133, m in [0, 127].
uint16_t double_to_bf16(double v) {
    const uint16_t sign = std::signbit(v) ? 0x8000u : 0x0000u;
    if (std::isnan(v)) return static_cast<uint16_t>(sign | 0x7FC0u);
    const double a = std::fabs(v);
    if (std::isinf(a)) return static_cast<uint16_t>(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e2 = 0;
    std::frexp(a, &e2);               // a = f * 2^e2, f in [0.5, 1)
    int E = e2 - 1;                   // a in [2^E, 2^(E+1))
    if (E < -126) E = -126;           // below the normal range the spacing stays 2^-133
    const double q = std::ldexp(1.0, E - 7);   // spacing of bf16 values near a
    const double n = a / q;                    // exact: division by a power of two
    const double fl = std::floor(n);
    const double frac = n - fl;                // exact
    double m = fl;
    if (frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0)) m = fl + 1.0;
    const double r = m * q;                    // exact: m <= 256
    if (r >= std::ldexp(1.0, 128)) return static_cast<uint16_t>(sign | 0x7F80u);
    const float f = static_cast<float>(r);     // exact: every bf16 value is an fp32 value
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>(sign | (u >> 16));
}

// IEEE binary16: sign, 5 exponent bits (bias 15), 10 fraction bits. Normal values are
// (1024 + f) * 2^(e - 25) for exponent field e in [1, 30]; subnormals f * 2^-24.
double f16_to_double(uint16_t bits) {
    const double sign = (bits & 0x8000u) ? -1.0 : 1.0;
    const int e = (bits >> 10) & 0x1F;
    const int f = bits & 0x3FF;
    if (e == 31) return f ? std::nan("") : sign * INFINITY;
    if (e == 0) return sign * std::ldexp(static_cast<double>(f), -24);
    return sign * std::ldexp(static_cast<double>(1024 + f), e - 25);
}

// Round an fp64 value to the nearest binary16, ties to even, in one rounding. Finite
// magnitudes are m * 2^(E-10) with integer m in [1024, 2047] for E in [-14, 15], plus the
// subnormals m * 2^-24, m in [0, 1023]; from 65520 (the tie above 65504) on: infinity.
uint16_t double_to_f16(double v) {
    const uint16_t sign = std::signbit(v) ? 0x8000u : 0x0000u;
    if (std::isnan(v)) return static_cast<uint16_t>(sign | 0x7E00u);
    const double a = std::fabs(v);
    if (std::isinf(a)) return static_cast<uint16_t>(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int e2 = 0;
    std::frexp(a, &e2);               // a = f * 2^e2, f in [0.5, 1)
    int E = e2 - 1;                   // a in [2^E, 2^(E+1))
    if (E < -14) E = -14;             // below the normal range the spacing stays 2^-24
    const double q = std::ldexp(1.0, E - 10);   // spacing of binary16 values near a
    const double n = a / q;                     // exact: division by a power of two
    const double fl = std::floor(n);
    const double frac = n - fl;                 // exact
    double m = fl;
    if (frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0)) m = fl + 1.0;
    const double r = m * q;                     // exact: m <= 2048
    if (r >= 65536.0) return static_cast<uint16_t>(sign | 0x7C00u);
    if (r < std::ldexp(1.0, -14))               // subnormal (m <= 1024; 1024 encodes 2^-14)
        return static_cast<uint16_t>(sign | static_cast<uint16_t>(std::ldexp(r, 24)));
    std::frexp(r, &e2);
    const int Er = e2 - 1;
    const int mant = static_cast<int>(std::ldexp(r, 10 - Er)) - 1024;
    return static_cast<uint16_t>(sign | ((Er + 15) << 10) | mant);
}

double load_elem(const void* base, int64_t i, int dtype) {
    if (dtype == kOracleBF16) return bf16_to_double(static_cast<const uint16_t*>(base)[i]);
    if (dtype == kOracleF16) return f16_to_double(static_cast<const uint16_t*>(base)[i]);
    return static_cast<double>(static_cast<const float*>(base)[i]);
}

// One rounding from fp64 to the storage type. The C++ conversion double -> float rounds
// to nearest, ties to even, under the default floating-point environment.
void store_elem(void* base, int64_t i, double v, int dtype) {
    if (dtype == kOracleBF16) {
        static_cast<uint16_t*>(base)[i] = double_to_bf16(v);
    } else if (dtype == kOracleF16) {
        static_cast<uint16_t*>(base)[i] = double_to_f16(v);
    } else {
        static_cast<float*>(base)[i] = static_cast<float>(v);
    }
}

// ---------------------------------------------------------------- RMSNorm, fp64

// Sum of squares with Neumaier's compensation (improved Kahan summation). Each square of
// a bf16 or fp32 value is exact in fp64, so the only error is in the additions.
double sum_of_squares(const double* x, int64_t n) {
    double sum = 0.0;
    double comp = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double t = x[j] * x[j];
        const double s = sum + t;
        if (std::fabs(sum) >= std::fabs(t)) {
            comp += (sum - s) + t;
        } else {
            comp += (t - s) + sum;
        }
        sum = s;
    }
    return sum + comp;
}

void rmsnorm_row(const double* x, const double* w, double* y, int64_t cols, double eps) {
    const double ss = sum_of_squares(x, cols);
    const double mean_sq = ss / static_cast<double>(cols);
    const double rms = std::sqrt(mean_sq + eps);
    for (int64_t j = 0; j < cols; ++j) {
        y[j] = x[j] / rms * w[j];
    }
}

// ---------------------------------------------------------------- LayerNorm, fp64

double neumaier_sum(const double* v, int64_t n) {
    double sum = 0.0;
    double comp = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double t = v[j];
        const double s = sum + t;
        if (std::fabs(sum) >= std::fabs(t)) {
            comp += (sum - s) + t;
        } else {
            comp += (t - s) + sum;
        }
        sum = s;
    }
    return sum + comp;
}

// y = normalized row * gamma + beta; `scale` (may be null) receives |xhat * gamma| + |beta|,
// the magnitude the fp32 arithmetic of a kernel is relative to.
void layernorm_row(const double* x, const double* g, const double* b, double* y, double* scale,
                   int64_t n, double eps) {
    const double mean = neumaier_sum(x, n) / static_cast<double>(n);
    std::vector<double> d2(static_cast<size_t>(n));
    for (int64_t j = 0; j < n; ++j) d2[j] = (x[j] - mean) * (x[j] - mean);
    const double var = neumaier_sum(d2.data(), n) / static_cast<double>(n);
    const double den = std::sqrt(var + eps);
    for (int64_t j = 0; j < n; ++j) {
        const double xhat = (x[j] - mean) / den;
        y[j] = xhat * g[j] + b[j];
        if (scale) scale[j] = std::fabs(xhat * g[j]) + std::fabs(b[j]);
    }
}

// ---------------------------------------------------------------- RoPE, fp64

// Rotate one head row of D = 2*half values by the table row (c[i], sn[i]).
void rope_head(const double* x, const double* sn, const double* c, double* y, int64_t half) {
    for (int64_t i = 0; i < half; ++i) {
        const double x1 = x[i];
        const double x2 = x[i + half];
        y[i] = x1 * c[i] - x2 * sn[i];
        y[i + half] = x2 * c[i] + x1 * sn[i];
    }
}

// ---------------------------------------------------------------- threading

int affinity_threads() {
    cpu_set_t set;
    CPU_ZERO(&set);
    if (sched_getaffinity(0, sizeof set, &set) == 0) {
        const int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    const unsigned hc = std::thread::hardware_concurrency();
    return hc > 0 ? static_cast<int>(hc) : 1;
}

// Run body(begin, end) over [0, n) split into contiguous blocks, one per thread. The split
// only decides which thread computes which rows; every row is computed the same way.
template <typename Body>
void parallel_blocks(int64_t n, int nthreads, Body body) {
    if (nthreads <= 0) nthreads = affinity_threads();
    if (n <= 0) return;
    if (nthreads > n) nthreads = static_cast<int>(n);
    if (nthreads <= 1) {
        body(int64_t{0}, n);
        return;
    }
    std::vector<std::thread> pool;
    pool.reserve(static_cast<size_t>(nthreads));
    for (int t = 0; t < nthreads; ++t) {
        const int64_t b = n * t / nthreads;
        const int64_t e = n * (t + 1) / nthreads;
        pool.emplace_back([=] { body(b, e); });
    }
    for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Status: 0 on success, 1 on an invalid argument, 2 on an unknown storage type.

uint16_t oracle_bf16_round(double v) { return double_to_bf16(v); }

double oracle_bf16_value(uint16_t bits) { return bf16_to_double(bits); }

uint16_t oracle_f16_round(double v) { return double_to_f16(v); }

double oracle_f16_value(uint16_t bits) { return f16_to_double(bits); }

int oracle_threads_available(void) { return affinity_threads(); }

// RMSNorm over fp64 inputs, fp64 output, no rounding: x[rows, cols], w[cols], y[rows, cols].
int oracle_rmsnorm_f64(const double* x, const double* w, double* y, int64_t rows, int64_t cols,
                       double eps) {
    if (rows < 0 || cols <= 0 || !(eps >= 0.0)) return 1;
    if (rows == 0) return 0;
    if (!x || !w || !y) return 1;
    for (int64_t r = 0; r < rows; ++r) {
        rmsnorm_row(x + r * cols, w, y + r * cols, cols, eps);
    }
    return 0;
}

// RMSNorm over storage-typed inputs: decode exactly, compute in fp64, round once.
// x, y: [rows, cols]; w: [cols]; all of storage type `dtype` (1 = fp32, 3 = bf16).
// nthreads <= 0 uses every core this process may run on.
int oracle_rmsnorm(const void* x, const void* w, void* y, int64_t rows, int64_t cols, double eps,
                   int dtype, int nthreads) {
    if (!storage_ok(dtype)) return 2;
    if (rows < 0 || cols <= 0 || !(eps >= 0.0)) return 1;
    if (rows == 0) return 0;
    if (!x || !w || !y) return 1;
    std::vector<double> wd(static_cast<size_t>(cols));
    for (int64_t j = 0; j < cols; ++j) wd[j] = load_elem(w, j, dtype);
    parallel_blocks(rows, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<double> xr(static_cast<size_t>(cols)), yr(static_cast<size_t>(cols));
        for (int64_t r = r0; r < r1; ++r) {
            for (int64_t j = 0; j < cols; ++j) xr[j] = load_elem(x, r * cols + j, dtype);
            rmsnorm_row(xr.data(), wd.data(), yr.data(), cols, eps);
            for (int64_t j = 0; j < cols; ++j) store_elem(y, r * cols + j, yr[j], dtype);
        }
    });
    return 0;
}

// Residual add then RMSNorm over storage-typed x, r (summands), w; outputs h = x + r rounded
// once (the sum of two bf16 or two fp32 values is exact in fp64) and y = RMSNorm(h) * w
// computed from h as stored, rounded once. nthreads as for oracle_rmsnorm.
int oracle_add_rmsnorm(const void* x, const void* r, const void* w, void* h, void* y,
                       int64_t rows, int64_t cols, double eps, int dtype, int nthreads) {
    if (!storage_ok(dtype)) return 2;
    if (rows < 0 || cols <= 0 || !(eps >= 0.0)) return 1;
    if (rows == 0) return 0;
    if (!x || !r || !w || !h || !y) return 1;
    std::vector<double> wd(static_cast<size_t>(cols));
    for (int64_t j = 0; j < cols; ++j) wd[j] = load_elem(w, j, dtype);
    parallel_blocks(rows, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<double> hr(static_cast<size_t>(cols)), yr(static_cast<size_t>(cols));
        for (int64_t row = r0; row < r1; ++row) {
            for (int64_t j = 0; j < cols; ++j) {
                const int64_t i = row * cols + j;
                store_elem(h, i, load_elem(x, i, dtype) + load_elem(r, i, dtype), dtype);
                hr[j] = load_elem(h, i, dtype);
            }
            rmsnorm_row(hr.data(), wd.data(), yr.data(), cols, eps);
            for (int64_t j = 0; j < cols; ++j) store_elem(y, row * cols + j, yr[j], dtype);
        }
    });
    return 0;
}

// KV RMSNorm + RoPE + cache scatter over storage-typed kv [B, S, Dn + Dr], gamma [Dn] and
// caches [num_slots, Dn] / [num_slots, Dr] (updated in place), fp32 tables [S, Dr/2] and
// int64 slots [B*S]. Tokens whose slot is outside [0, num_slots) are skipped.
int oracle_kv_rmsnorm_rope_cache(const void* kv, const void* gamma, const float* sin_t,
                                 const float* cos_t, const int64_t* slots, void* cache_n,
                                 void* cache_r, int64_t B, int64_t S, int64_t Dn, int64_t Dr,
                                 int64_t num_slots, double eps, int dtype) {
    if (!storage_ok(dtype)) return 2;
    if (B < 0 || S < 0 || Dn < 1 || Dr < 2 || Dr % 2 != 0 || num_slots < 0 || !(eps >= 0.0))
        return 1;
    if (B * S == 0) return 0;
    if (!kv || !gamma || !sin_t || !cos_t || !slots || !cache_n || !cache_r) return 1;
    const int64_t half = Dr / 2;
    std::vector<double> g(static_cast<size_t>(Dn)), xn(static_cast<size_t>(Dn)),
        yn(static_cast<size_t>(Dn)), xr(static_cast<size_t>(Dr)), yr(static_cast<size_t>(Dr)),
        sn(static_cast<size_t>(half)), c(static_cast<size_t>(half));
    for (int64_t j = 0; j < Dn; ++j) g[j] = load_elem(gamma, j, dtype);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t s = 0; s < S; ++s) {
            const int64_t t = b * S + s;
            const int64_t slot = slots[t];
            if (slot < 0 || slot >= num_slots) continue;
            const int64_t base = t * (Dn + Dr);
            for (int64_t j = 0; j < Dn; ++j) xn[j] = load_elem(kv, base + j, dtype);
            for (int64_t j = 0; j < Dr; ++j) xr[j] = load_elem(kv, base + Dn + j, dtype);
            for (int64_t i = 0; i < half; ++i) {
                sn[i] = static_cast<double>(sin_t[s * half + i]);
                c[i] = static_cast<double>(cos_t[s * half + i]);
            }
            rmsnorm_row(xn.data(), g.data(), yn.data(), Dn, eps);
            rope_head(xr.data(), sn.data(), c.data(), yr.data(), half);
            for (int64_t j = 0; j < Dn; ++j) store_elem(cache_n, slot * Dn + j, yn[j], dtype);
            for (int64_t j = 0; j < Dr; ++j) store_elem(cache_r, slot * Dr + j, yr[j], dtype);
        }
    }
    return 0;
}

// LayerNorm over fp64 x [rows, cols], gamma, beta [cols]: unrounded y and the error scale.
int oracle_layernorm_f64(const double* x, const double* g, const double* b, double* y,
                         double* scale, int64_t rows, int64_t cols, double eps) {
    if (rows < 0 || cols <= 0 || !(eps >= 0.0)) return 1;
    if (rows == 0) return 0;
    if (!x || !g || !b || !y || !scale) return 1;
    for (int64_t r = 0; r < rows; ++r)
        layernorm_row(x + r * cols, g, b, y + r * cols, scale + r * cols, cols, eps);
    return 0;
}

// LayerNorm over storage-typed x, gamma, beta: decode, fp64, one rounding of y.
int oracle_layernorm(const void* x, const void* gamma, const void* beta, void* y, int64_t rows,
                     int64_t cols, double eps, int dtype, int nthreads) {
    if (!storage_ok(dtype)) return 2;
    if (rows < 0 || cols <= 0 || !(eps >= 0.0)) return 1;
    if (rows == 0) return 0;
    if (!x || !gamma || !beta || !y) return 1;
    std::vector<double> g(static_cast<size_t>(cols)), b(static_cast<size_t>(cols));
    for (int64_t j = 0; j < cols; ++j) {
        g[j] = load_elem(gamma, j, dtype);
        b[j] = load_elem(beta, j, dtype);
    }
    parallel_blocks(rows, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<double> xr(static_cast<size_t>(cols)), yr(static_cast<size_t>(cols));
        for (int64_t r = r0; r < r1; ++r) {
            for (int64_t j = 0; j < cols; ++j) xr[j] = load_elem(x, r * cols + j, dtype);
            layernorm_row(xr.data(), g.data(), b.data(), yr.data(), nullptr, cols, eps);
            for (int64_t j = 0; j < cols; ++j) store_elem(y, r * cols + j, yr[j], dtype);
        }
    });
    return 0;
}

// Concatenation of past [B, P, Hk, D] and new [B, S, Hk, D] along the sequence, with each
// head repeated n_rep times in place (head h -> heads h*n_rep .. h*n_rep + n_rep - 1) and
// the new rows rotated at their absolute positions P + s (tables [P + S, D/2]; sin_t and
// cos_t both null: no rotation). Storage-typed; a copied value is exact, a rotated one is
// the fp64 pair formula rounded once.
int oracle_kv_cat_repeat(const void* past, const void* fresh, const float* sin_t,
                         const float* cos_t, void* out, int64_t B, int64_t P, int64_t S,
                         int64_t Hk, int64_t D, int64_t n_rep, int dtype) {
    if (!storage_ok(dtype)) return 2;
    if (B < 0 || P < 0 || S < 0 || Hk < 0 || D <= 0 || D % 2 != 0 || n_rep < 1) return 1;
    if ((sin_t == nullptr) != (cos_t == nullptr)) return 1;
    const int64_t T = P + S;
    if (B * T * Hk == 0) return 0;
    if (!out || (P > 0 && !past) || (S > 0 && !fresh)) return 1;
    const int64_t half = D / 2;
    const int64_t Hout = Hk * n_rep;
    std::vector<double> xr(static_cast<size_t>(D)), yr(static_cast<size_t>(D));
    std::vector<double> sn(static_cast<size_t>(half)), c(static_cast<size_t>(half));
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            const bool old_row = t < P;
            const bool rotate = !old_row && sin_t != nullptr;
            if (rotate) {
                for (int64_t i = 0; i < half; ++i) {
                    sn[i] = static_cast<double>(sin_t[t * half + i]);
                    c[i] = static_cast<double>(cos_t[t * half + i]);
                }
            }
            for (int64_t h = 0; h < Hk; ++h) {
                const void* src = old_row ? past : fresh;
                const int64_t src_row = old_row ? (b * P + t) * Hk + h : (b * S + (t - P)) * Hk + h;
                for (int64_t j = 0; j < D; ++j) xr[j] = load_elem(src, src_row * D + j, dtype);
                if (rotate) {
                    rope_head(xr.data(), sn.data(), c.data(), yr.data(), half);
                } else {
                    yr = xr;
                }
                for (int64_t r = 0; r < n_rep; ++r) {
                    const int64_t dst_row = (b * T + t) * Hout + h * n_rep + r;
                    for (int64_t j = 0; j < D; ++j) store_elem(out, dst_row * D + j, yr[j], dtype);
                }
            }
        }
    }
    return 0;
}

// Interleaved RoPE over storage-typed x [tokens, H, D], fp32 tables [max_pos, D/2] and int32
// positions [tokens]; y (same layout) is updated only for tokens with a valid position.
int oracle_rope_interleaved(const void* x, const float* sin_t, const float* cos_t,
                            const int32_t* positions, void* y, int64_t tokens, int64_t H,
                            int64_t D, int64_t max_pos, int dtype) {
    if (!storage_ok(dtype)) return 2;
    if (tokens < 0 || H < 0 || D < 2 || D % 2 != 0 || max_pos < 0) return 1;
    if (tokens * H == 0) return 0;
    if (!x || !sin_t || !cos_t || !positions || !y) return 1;
    const int64_t half = D / 2;
    for (int64_t t = 0; t < tokens; ++t) {
        const int64_t p = positions[t];
        if (p < 0 || p >= max_pos) continue;
        for (int64_t h = 0; h < H; ++h) {
            const int64_t base = (t * H + h) * D;
            for (int64_t i = 0; i < half; ++i) {
                const double x0 = load_elem(x, base + 2 * i, dtype);
                const double x1 = load_elem(x, base + 2 * i + 1, dtype);
                const double c = static_cast<double>(cos_t[p * half + i]);
                const double sn = static_cast<double>(sin_t[p * half + i]);
                store_elem(y, base + 2 * i, x0 * c - x1 * sn, dtype);
                store_elem(y, base + 2 * i + 1, x0 * sn + x1 * c, dtype);
            }
        }
    }
    return 0;
}

// RoPE tables [max_pos, D/2]: angle = p * theta^(-2i/D) in fp64, sin and cos rounded once.
int oracle_rope_tables(float* sin_t, float* cos_t, int64_t max_pos, int64_t D, double theta) {
    if (max_pos < 0 || D < 2 || D % 2 != 0 || !(theta > 0.0)) return 1;
    if (max_pos == 0) return 0;
    if (!sin_t || !cos_t) return 1;
    const int64_t half = D / 2;
    for (int64_t p = 0; p < max_pos; ++p) {
        for (int64_t i = 0; i < half; ++i) {
            const double freq = std::pow(theta, (-2.0 * static_cast<double>(i)) /
                                                    static_cast<double>(D));
            const double angle = static_cast<double>(p) * freq;
            sin_t[p * half + i] = static_cast<float>(std::sin(angle));
            cos_t[p * half + i] = static_cast<float>(std::cos(angle));
        }
    }
    return 0;
}

// Rotate-half RoPE over fp64 inputs, fp64 output, no rounding.
// x, y: [B, S, H, D]; sin_t, cos_t: [S, D/2].
int oracle_rope_f64(const double* x, const double* sin_t, const double* cos_t, double* y,
                    int64_t B, int64_t S, int64_t H, int64_t D) {
    if (B < 0 || S < 0 || H < 0 || D <= 0 || D % 2 != 0) return 1;
    if (B * S * H == 0) return 0;
    if (!x || !sin_t || !cos_t || !y) return 1;
    const int64_t half = D / 2;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t s = 0; s < S; ++s) {
            for (int64_t h = 0; h < H; ++h) {
                const int64_t off = ((b * S + s) * H + h) * D;
                rope_head(x + off, sin_t + s * half, cos_t + s * half, y + off, half);
            }
        }
    }
    return 0;
}

// Rotate-half RoPE over storage-typed x/y (1 = fp32, 3 = bf16) and fp32 tables:
// decode exactly, rotate in fp64, round once. Threads split the (b, s) positions.
int oracle_rope(const void* x, const float* sin_t, const float* cos_t, void* y, int64_t B,
                int64_t S, int64_t H, int64_t D, int dtype, int nthreads) {
    if (!storage_ok(dtype)) return 2;
    if (B < 0 || S < 0 || H < 0 || D <= 0 || D % 2 != 0) return 1;
    if (B * S * H == 0) return 0;
    if (!x || !sin_t || !cos_t || !y) return 1;
    const int64_t half = D / 2;
    parallel_blocks(B * S, nthreads, [&](int64_t t0, int64_t t1) {
        std::vector<double> xr(static_cast<size_t>(D)), yr(static_cast<size_t>(D));
        std::vector<double> sn(static_cast<size_t>(half)), c(static_cast<size_t>(half));
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t b = t / S;
            const int64_t s = t - b * S;
            for (int64_t i = 0; i < half; ++i) {
                sn[i] = static_cast<double>(sin_t[s * half + i]);
                c[i] = static_cast<double>(cos_t[s * half + i]);
            }
            for (int64_t h = 0; h < H; ++h) {
                const int64_t off = ((b * S + s) * H + h) * D;
                for (int64_t k = 0; k < D; ++k) xr[k] = load_elem(x, off + k, dtype);
                rope_head(xr.data(), sn.data(), c.data(), yr.data(), half);
                for (int64_t k = 0; k < D; ++k) store_elem(y, off + k, yr[k], dtype);
            }
        }
    });
    return 0;
}

}  // extern "C"
