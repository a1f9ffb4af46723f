// C ABI of libcamp: host-side argument validation, kernel planning and launch.
//
// Every argument error is found here, on the host, before any CUDA call; the kernels
// assume validated, in-bounds arguments. Nothing here synchronizes the device or
// allocates memory. Status codes follow the Intro-ops operator runtime
// (include/operator_runtime/api.h), minus the workspace code: this library has no
// workspace.
#include <cmath>
#include <cstdint>
#include <limits>

#include "camp.h"
#include "kernels.h"

namespace {

using camp::DType;

thread_local int g_last_cuda_error = 0;

constexpr int64_t kMaxGrid = 2147483647;   // gridDim.x limit; kernels loop past it

bool dtype_ok(camp_dtype_t d) { return d == CAMP_DTYPE_F32 || d == CAMP_DTYPE_BF16; }

DType to_dtype(camp_dtype_t d) { return d == CAMP_DTYPE_BF16 ? DType::BF16 : DType::F32; }

bool aligned(const void* p, int64_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

// n = a * b * c without int64 overflow (all factors >= 0); false on overflow.
bool mul_ok(int64_t a, int64_t b, int64_t c, int64_t* n) {
    const int64_t kMax = std::numeric_limits<int64_t>::max();
    if (a != 0 && b > kMax / a) return false;
    const int64_t ab = a * b;
    if (ab != 0 && c > kMax / ab) return false;
    *n = ab * c;
    return true;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

camp_status_t runtime_status() {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return CAMP_SUCCESS;
    g_last_cuda_error = static_cast<int>(e);
    return CAMP_ERR_RUNTIME;
}

// ------------------------------------------------------------------ RMSNorm

struct RmsCall {
    camp::RmsnormArgs a;
    DType t;
    int64_t bytes;   // bytes of x (and of y)
};

// Checks shared by camp_rmsnorm, camp_rmsnorm_plan and camp_rmsnorm_with_plan.
// Sets *empty for rows == 0 (a successful no-op).
camp_status_t rms_validate(const void* x, const void* w, const void* y, int64_t rows,
                           int64_t cols, camp_dtype_t dtype, RmsCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || cols < 1) return CAMP_ERR_INVALID_ARG;
    if (rows == 0) { *empty = true; return CAMP_SUCCESS; }
    if (x == nullptr || w == nullptr || y == nullptr) return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t bytes = 0;
    if (!mul_ok(rows, cols, es, &bytes)) return CAMP_ERR_INVALID_ARG;
    if (!aligned(x, es) || !aligned(w, es) || !aligned(y, es)) return CAMP_ERR_INVALID_ARG;
    if (y != x && overlaps(y, bytes, x, bytes)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(y, bytes, w, cols * es)) return CAMP_ERR_INVALID_ARG;
    c->a.x = x;
    c->a.w = w;
    c->a.y = const_cast<void*>(y);
    c->a.rows = rows;
    c->a.cols = cols;
    c->a.eps = 0.0f;
    c->t = t;
    c->bytes = bytes;
    return CAMP_SUCCESS;
}

// The widest vector access that every row start and every pointer allows.
int rms_vec_bytes(const RmsCall& c) {
    const int es = camp::elem_bytes(c.t);
    const int64_t pitch = c.a.cols * es;
    if (pitch % 16 == 0 && aligned(c.a.x, 16) && aligned(c.a.w, 16) && aligned(c.a.y, 16))
        return 16;
    return es;
}

int round_up_in(int v, const int* set, int n) {
    for (int i = 0; i < n; ++i)
        if (set[i] >= v) return set[i];
    return -1;
}

// Fill the kernel choice for the rows kernel; falls back to the two-sweep kernel when no
// register-resident variant can hold the row.
void rms_plan(const RmsCall& c, camp_plan_t* p) {
    const int vb = rms_vec_bytes(c);
    const int es = camp::elem_bytes(c.t);
    const int64_t nvec = c.a.cols * es / vb;
    *p = camp_plan_t{};
    p->vec_bytes = vb;
    if (vb == 16) {
        // Smallest group that needs at most 4 accesses per thread: short rows stay on one
        // warp (no CTA barrier), long rows spread over more warps to keep the register
        // footprint, and hence occupancy and bytes in flight, high.
        static const int kGroups[] = {32, 64, 128, 256, 512, 1024};
        static const int kPer[] = {1, 2, 3, 4, 6, 8};
        for (int g : kGroups) {
            const int64_t nv = ceil_div(nvec, g);
            if (nv <= 4 || (g == 1024 && nv <= 8)) {
                p->kernel = CAMP_KERNEL_RMSNORM_ROWS;
                p->group = g;
                p->per_thread = round_up_in(static_cast<int>(nv), kPer, 6);
                break;
            }
        }
    } else {
        static const int kGroups[] = {32, 256, 1024};
        static const int kPer[] = {1, 2, 4, 8, 16};
        for (int g : kGroups) {
            const int64_t nv = ceil_div(nvec, g);
            if (nv <= 16) {
                p->kernel = CAMP_KERNEL_RMSNORM_ROWS;
                p->group = g;
                p->per_thread = round_up_in(static_cast<int>(nv), kPer, 5);
                break;
            }
        }
    }
    if (p->kernel == CAMP_KERNEL_RMSNORM_ROWS) {
        p->block = camp::rmsnorm_rows_block(p->group);
        const int64_t rows_per_cta = p->block / p->group;
        const int64_t blocks = ceil_div(c.a.rows, rows_per_cta);
        p->grid = blocks < kMaxGrid ? blocks : kMaxGrid;
    } else {
        p->kernel = CAMP_KERNEL_RMSNORM_WIDE;
        p->group = camp::kWideBlock;
        p->per_thread = 0;
        p->block = camp::kWideBlock;
        p->grid = c.a.rows < kMaxGrid ? c.a.rows : kMaxGrid;
    }
}

// Check that an explicit plan fits these arguments and fill in block and grid.
camp_status_t rms_accept_plan(const RmsCall& c, const camp_plan_t& in, camp_plan_t* p) {
    const int es = camp::elem_bytes(c.t);
    const int vb = in.vec_bytes;
    if (vb != 16 && vb != 8 && vb != 4 && vb != 2) return CAMP_ERR_NOT_SUPPORTED;
    if (vb < es || vb > rms_vec_bytes(c) || (c.a.cols * es) % vb != 0) return CAMP_ERR_NOT_SUPPORTED;
    *p = in;
    if (in.kernel == CAMP_KERNEL_RMSNORM_ROWS) {
        if (!camp::rmsnorm_rows_compiled(c.t, vb, in.group, in.per_thread))
            return CAMP_ERR_NOT_SUPPORTED;
        const int64_t nvec = c.a.cols * es / vb;
        if (static_cast<int64_t>(in.group) * in.per_thread < nvec) return CAMP_ERR_NOT_SUPPORTED;
        p->block = camp::rmsnorm_rows_block(in.group);
        const int64_t blocks = ceil_div(c.a.rows, p->block / in.group);
        p->grid = blocks < kMaxGrid ? blocks : kMaxGrid;
        return CAMP_SUCCESS;
    }
    if (in.kernel == CAMP_KERNEL_RMSNORM_WIDE) {
        if (!camp::rmsnorm_wide_compiled(c.t, vb)) return CAMP_ERR_NOT_SUPPORTED;
        p->group = camp::kWideBlock;
        p->per_thread = 0;
        p->block = camp::kWideBlock;
        p->grid = c.a.rows < kMaxGrid ? c.a.rows : kMaxGrid;
        return CAMP_SUCCESS;
    }
    return CAMP_ERR_NOT_SUPPORTED;
}

camp_status_t rms_launch(const RmsCall& c, const camp_plan_t& p, cudaStream_t s) {
    bool ok = false;
    if (p.kernel == CAMP_KERNEL_RMSNORM_ROWS) {
        ok = camp::rmsnorm_rows_launch(c.t, p.vec_bytes, p.group, p.per_thread, c.a, p.grid,
                                       p.block, s);
    } else if (p.kernel == CAMP_KERNEL_RMSNORM_WIDE) {
        ok = camp::rmsnorm_wide_launch(c.t, p.vec_bytes, c.a, p.grid, s);
    }
    if (!ok) return CAMP_ERR_NOT_SUPPORTED;
    return runtime_status();
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.0f; }

// ------------------------------------------------------------------ RoPE

struct RopeCall {
    camp::RopeArgs a;
    DType t;
};

camp_status_t rope_validate(const void* x, const float* sin_t, const float* cos_t,
                            const void* y, int64_t B, int64_t S, int64_t H, int64_t D,
                            camp_dtype_t dtype, RopeCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || S < 0 || H < 0 || D < 2 || D % 2 != 0) return CAMP_ERR_INVALID_ARG;
    if (B == 0 || S == 0 || H == 0) { *empty = true; return CAMP_SUCCESS; }
    if (x == nullptr || sin_t == nullptr || cos_t == nullptr || y == nullptr)
        return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t tokens = 0, rows = 0, bytes = 0, table_bytes = 0;
    if (!mul_ok(B, S, 1, &tokens) || !mul_ok(tokens, H, 1, &rows) || !mul_ok(rows, D, es, &bytes))
        return CAMP_ERR_INVALID_ARG;
    if (!mul_ok(S, D / 2, 4, &table_bytes)) return CAMP_ERR_INVALID_ARG;
    if (!aligned(x, es) || !aligned(y, es) || !aligned(sin_t, 4) || !aligned(cos_t, 4))
        return CAMP_ERR_INVALID_ARG;
    if (y != x && overlaps(y, bytes, x, bytes)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(y, bytes, sin_t, table_bytes) || overlaps(y, bytes, cos_t, table_bytes))
        return CAMP_ERR_INVALID_ARG;
    c->a.x = x;
    c->a.sin_t = sin_t;
    c->a.cos_t = cos_t;
    c->a.y = const_cast<void*>(y);
    c->a.tokens = tokens;
    c->a.seq = S;
    c->a.heads = H;
    c->a.half = D / 2;
    c->t = t;
    return CAMP_SUCCESS;
}

// Is a vector access of vb bytes legal for every pointer and every half-row start?
bool rope_vec_ok(const RopeCall& c, int vb) {
    const int es = camp::elem_bytes(c.t);
    if (vb < es) return false;
    if ((c.a.half * es) % vb != 0) return false;
    const int elems = vb / es;
    const int table_align = elems * 4 < 16 ? elems * 4 : 16;
    return aligned(c.a.x, vb) && aligned(c.a.y, vb) && aligned(c.a.sin_t, table_align) &&
           aligned(c.a.cos_t, table_align);
}

int64_t rope_grid(const RopeCall& c, int vb, int hpt) {
    const int es = camp::elem_bytes(c.t);
    const int64_t nvh = c.a.half * es / vb;
    const int64_t work = c.a.tokens * ceil_div(c.a.heads, hpt) * nvh;
    const int64_t blocks = ceil_div(work, camp::kRopeBlock);
    return blocks < kMaxGrid ? blocks : kMaxGrid;
}

void rope_plan(const RopeCall& c, camp_plan_t* p) {
    *p = camp_plan_t{};
    p->kernel = CAMP_KERNEL_ROPE;
    static const int kVec[] = {16, 8, 4, 2};
    for (int vb : kVec) {
        if (rope_vec_ok(c, vb)) { p->vec_bytes = vb; break; }
    }
    // Heads per thread: the largest of 4, 2, 1 that divides H, so that no thread idles.
    p->group = (c.a.heads % 4 == 0) ? 4 : (c.a.heads % 2 == 0) ? 2 : 1;
    p->per_thread = 0;
    p->block = camp::kRopeBlock;
    p->grid = rope_grid(c, p->vec_bytes, p->group);
}

camp_status_t rope_accept_plan(const RopeCall& c, const camp_plan_t& in, camp_plan_t* p) {
    if (in.kernel != CAMP_KERNEL_ROPE) return CAMP_ERR_NOT_SUPPORTED;
    if (!rope_vec_ok(c, in.vec_bytes)) return CAMP_ERR_NOT_SUPPORTED;
    if (!camp::rope_compiled(c.t, in.vec_bytes, in.group)) return CAMP_ERR_NOT_SUPPORTED;
    *p = in;
    p->per_thread = 0;
    p->block = camp::kRopeBlock;
    p->grid = rope_grid(c, in.vec_bytes, in.group);
    return CAMP_SUCCESS;
}

camp_status_t rope_launch(const RopeCall& c, const camp_plan_t& p, cudaStream_t s) {
    if (!camp::rope_launch(c.t, p.vec_bytes, p.group, c.a, p.grid, s)) return CAMP_ERR_NOT_SUPPORTED;
    return runtime_status();
}

}  // namespace

extern "C" {

CAMP_API const char* camp_status_string(camp_status_t status) {
    switch (status) {
        case CAMP_SUCCESS: return "success";
        case CAMP_ERR_INVALID_ARG: return "invalid argument";
        case CAMP_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case CAMP_ERR_RUNTIME: return "CUDA runtime error";
        case CAMP_ERR_NOT_SUPPORTED: return "not supported";
    }
    return "unknown status";
}

CAMP_API int camp_last_cuda_error(void) { return g_last_cuda_error; }

CAMP_API camp_status_t camp_rmsnorm(const void* x, const void* w, void* y, int64_t rows,
                                    int64_t cols, float eps, camp_dtype_t dtype,
                                    void* stream) {
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_validate(x, w, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps)) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    c.a.eps = eps;
    camp_plan_t p;
    rms_plan(c, &p);
    return rms_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_rmsnorm_plan(const void* x, const void* w, const void* y,
                                         int64_t rows, int64_t cols, camp_dtype_t dtype,
                                         camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_validate(x, w, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    rms_plan(c, plan);
    return CAMP_SUCCESS;
}

CAMP_API camp_status_t camp_rmsnorm_with_plan(const void* x, const void* w, void* y,
                                              int64_t rows, int64_t cols, float eps,
                                              camp_dtype_t dtype, const camp_plan_t* plan,
                                              void* stream) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_validate(x, w, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps)) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    c.a.eps = eps;
    camp_plan_t p;
    st = rms_accept_plan(c, *plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return rms_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_rope(const void* x, const float* sin, const float* cos, void* y,
                                 int64_t B, int64_t S, int64_t H, int64_t D,
                                 camp_dtype_t dtype, void* stream) {
    RopeCall c;
    bool empty = false;
    camp_status_t st = rope_validate(x, sin, cos, y, B, S, H, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    rope_plan(c, &p);
    return rope_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_rope_plan(const void* x, const float* sin, const float* cos,
                                      const void* y, int64_t B, int64_t S, int64_t H,
                                      int64_t D, camp_dtype_t dtype, camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RopeCall c;
    bool empty = false;
    camp_status_t st = rope_validate(x, sin, cos, y, B, S, H, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    rope_plan(c, plan);
    return CAMP_SUCCESS;
}

CAMP_API camp_status_t camp_rope_with_plan(const void* x, const float* sin, const float* cos,
                                           void* y, int64_t B, int64_t S, int64_t H, int64_t D,
                                           camp_dtype_t dtype, const camp_plan_t* plan,
                                           void* stream) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RopeCall c;
    bool empty = false;
    camp_status_t st = rope_validate(x, sin, cos, y, B, S, H, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    st = rope_accept_plan(c, *plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return rope_launch(c, p, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
