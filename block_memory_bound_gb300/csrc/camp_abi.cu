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

constexpr int64_t kMaxGrid = 2147483647;   // gridDim.x limit for the looping kernels

bool dtype_ok(camp_dtype_t d) {
    return d == CAMP_DTYPE_F16 || d == CAMP_DTYPE_F32 || d == CAMP_DTYPE_BF16;
}

DType to_dtype(camp_dtype_t d) {
    return d == CAMP_DTYPE_BF16 ? DType::BF16 : d == CAMP_DTYPE_F16 ? DType::F16 : DType::F32;
}

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

// Map a launch result (and any error the runtime recorded with it) to a status.
camp_status_t runtime_status(cudaError_t launched) {
    const cudaError_t recorded = cudaGetLastError();   // also clears the recorded error
    const cudaError_t e = launched != cudaSuccess ? launched : recorded;
    if (e == cudaSuccess) return CAMP_SUCCESS;
    g_last_cuda_error = static_cast<int>(e);
    return CAMP_ERR_RUNTIME;
}

// ------------------------------------------------------------------ RMSNorm

struct RmsCall {
    camp::RmsnormArgs a;
    DType t;
    int64_t bytes;     // bytes of x (and of y)
    bool add = false;  // fused residual add: h = x + r is stored and normalized
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
    c->a = camp::RmsnormArgs{};
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

// Checks of camp_add_rmsnorm: as rms_validate, but every output (h and y) either equals
// one input (x or r) exactly, in place, or is disjoint from both; h and y are disjoint from
// each other and from w. Each element of x and r is read by the thread that writes h and y
// at that index, before it writes them, so an exact alias is safe.
camp_status_t rms_add_validate(const void* x, const void* r, const void* w, const void* h,
                               const void* y, int64_t rows, int64_t cols, camp_dtype_t dtype,
                               RmsCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || cols < 1) return CAMP_ERR_INVALID_ARG;
    if (rows == 0) { *empty = true; return CAMP_SUCCESS; }
    if (x == nullptr || r == nullptr || w == nullptr || h == nullptr || y == nullptr)
        return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t bytes = 0;
    if (!mul_ok(rows, cols, es, &bytes)) return CAMP_ERR_INVALID_ARG;
    for (const void* p : {x, r, w, h, y})
        if (!aligned(p, es)) return CAMP_ERR_INVALID_ARG;
    for (const void* out : {h, y})
        for (const void* in : {x, r})
            if (out != in && overlaps(out, bytes, in, bytes)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(h, bytes, y, bytes)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(h, bytes, w, cols * es) || overlaps(y, bytes, w, cols * es))
        return CAMP_ERR_INVALID_ARG;
    c->a = camp::RmsnormArgs{};
    c->a.x = x;
    c->a.w = w;
    c->a.y = const_cast<void*>(y);
    c->a.r = r;
    c->a.h = const_cast<void*>(h);
    c->a.rows = rows;
    c->a.cols = cols;
    c->t = t;
    c->bytes = bytes;
    c->add = true;
    return CAMP_SUCCESS;
}

// The widest vector access that every row start and every pointer allows.
int rms_vec_bytes(const RmsCall& c) {
    const int es = camp::elem_bytes(c.t);
    const int64_t pitch = c.a.cols * es;
    bool ok = pitch % 16 == 0 && aligned(c.a.x, 16) && aligned(c.a.w, 16) && aligned(c.a.y, 16);
    if (c.add) ok = ok && aligned(c.a.r, 16) && aligned(c.a.h, 16);
    return ok ? 16 : es;
}

int round_up_in(int v, const int* set, int n) {
    for (int i = 0; i < n; ++i)
        if (set[i] >= v) return set[i];
    return -1;
}

struct RowsCandidate {
    int group, per_thread;
    int64_t ctas, idle;
    bool one_wave;     // every CTA resident at once (CTAs <= SMs x CTAs per SM)
    bool many_waves;   // at least 2 waves of CTAs
    bool add16;        // residual-add path on 16-byte vectors (may take 1024-thread groups)
};

// Is candidate a preferred over b? Measured on GB300 (L2-cold, back-to-back launches):
//  1. cover as many SMs as there are (min(CTAs, SM count)); this only decides tiny row
//     counts (decode), where one row per CTA spreads the rows over the most SMs;
//  2. 2 to 4 accesses per thread with at most 256 threads per row: below that there is
//     too little in flight per thread, above it the row group's barrier and the
//     1024-thread CTAs cost more than they save;
//  3. fewest idle vector slots (a ragged last access per thread wastes issue slots);
//  4. a grid that is resident in one wave: then every load is issued at the start instead
//     of when a CTA of the first wave retires (4096 x 2048 bf16: 64 x 4 in one wave
//     6.98 us, 128 x 2 in 1.7 waves 7.25 us);
//  5. within 2., fewer accesses per thread (more threads, shorter serial work per thread);
//     outside it (rows of more than 1024 vectors), at most 4 accesses in groups of at
//     most 512 threads, then the smaller group. With each CTA's rows prefetched into L2
//     before it waits on the previous kernel, 512 x 3 / 512 x 4 beat 256 x 6 / 256 x 8
//     (bf16, 4096 rows of 12288 / 16384 columns: RMSNorm 0.97 / 0.98 of the measured peak
//     against 0.94 / 0.94, with the residual add 1.00 / 1.00 against 0.97 / 0.97), and
//     1024-thread CTAs lose where the rule would otherwise reach them (1024 x 4 at 32768
//     columns: 0.75 against 512 x 8's 0.92).
// For bf16 this picks 64 x 4 at 4096 x 2048, 128 x 2 at 8192 x 2048 and more rows,
// 128 x 3 at 3000 columns, 256 x 4 at 8192, and 512 x 3 / 512 x 4 at 12288 / 16384
// columns: the fastest of the compiled variants at each, or within 2-5% of it.
// LayerNorm (`layernorm`) differs in 5.: its per-thread cost (two reductions) is higher,
// so outside the band it keeps the smaller group (4096 x 12288: 256 x 6 0.86, 512 x 3
// 0.82), and when both candidates run at least 2 waves the one with more accesses per
// thread wins (bf16, 64 x 4 against 128 x 2: 65536 x 2048 80.5 / 90.9 us, 8192 x 2048 14.3 /
// 14.5 us; 8192 x 4096: 128 x 4 24.2 us, 256 x 2 24.6 us); closer to one wave the RMSNorm
// order holds (4096 x 2048: 128 x 2 9.0 us, 64 x 4 in 1.1 waves 10.2 us).
// At decode sizes (no more rows than SMs) a launch is latency-bound, not bandwidth-bound,
// and after 1. the rule is: groups of at most 512 threads, the fewest accesses per thread
// (the shortest serial chain of loads and arithmetic), the fewest idle slots, the smaller
// group. Measured on GB300 (bf16, graphs of back-to-back launches): 1 x 8192 512 x 2
// 1.97 us against 256 x 4 2.22 us, 1 x 3000 512 x 1 1.70 against 128 x 3 1.94, 8 x 8192
// 512 x 2 2.05 against 2.21, 64 x 8192 2.07 against 2.32; 1 x 2048 256 x 1 1.52.
// Rows of RMSNorm and LayerNorm up to kRowsFewRows rows take the 2..4-accesses band with
// groups of up to 512 threads, and the residual-add path takes 2 accesses a thread in groups of up to 512
// at every row count: a sweep of every rows variant at 256..8192 rows of 2048, 3000 and
// 8192 bf16 columns (36 shapes, both paths) changed 15 plans, each 0.5-21% faster (512 x
// 8192: 512 x 2 3.62 us against 256 x 4 4.41; with the add, 256 x 8192 3.56 against 4.53,
// 1024 x 3000 4.45 against 4.97) and none slower. With few rows a launch is short of
// threads in flight, and the add path holds twice the data a thread. The same band for
// LayerNorm (18 bf16 and 6 fp16 shapes at 256..8192 rows of 2048..8192 columns): 3 plans
// changed, 7-12% faster (512 x 8192: 512 x 2 4.75 us against 256 x 4 5.40), none slower.
// The residual-add path on 16-byte vectors lifts the 512-thread cap to 1024 wherever a
// 1024-thread group gives every thread at least 2 accesses, that is past 1024 vectors a row
// (the band's 2 accesses, otherwise at most 4; at decode sizes the fewest accesses): each
// thread holds x and r, and halving a thread's work pays more than the wider barrier costs.
// Measured at 1..8192 rows of 1536, 2048, 3072 and 4096 vectors (bf16 and fp32, 64 shapes):
// the 1024-thread group is 0.1-32% faster in 55 of them (152 x 12288 fp32: 1024 x 3 6.29 us
// against 512 x 6 8.32; 512 x 32768 bf16: 1024 x 4 25.9 against 29.2; 2048 x 16384 bf16:
// 1024 x 2 40.3 against 41.2), at most 5% slower in the others (fp32 at 3072 vectors and
// 512..4096 rows, 1536 vectors at 1..8 rows). Plain RMSNorm keeps 512: there the
// 1024-thread group loses at 768 rows and more (2048 x 32768 bf16: 1024 x 4 51.0 us against
// 512 x 8 43.3).
constexpr int64_t kRowsFewRows = 2048;

bool rows_better(const RowsCandidate& a, const RowsCandidate& b, bool layernorm,
                 bool latency, bool add = false, int64_t rows = 0) {
    const int64_t sa = a.ctas < camp::kSmCount ? a.ctas : camp::kSmCount;
    const int64_t sb = b.ctas < camp::kSmCount ? b.ctas : camp::kSmCount;
    if (sa != sb) return sa > sb;
    const int add_gmax = a.add16 ? 1024 : 512;
    if (latency) {
        const bool la = a.group <= 512 || (a.group <= add_gmax && a.per_thread >= 2);
        const bool lb = b.group <= 512 || (b.group <= add_gmax && b.per_thread >= 2);
        if (la != lb) return la;
        if (a.per_thread != b.per_thread) return a.per_thread < b.per_thread;
        if (a.idle != b.idle) return a.idle < b.idle;
        return a.group < b.group;
    }
    auto in_band = [&](const RowsCandidate& k) {
        if (!layernorm && add) return k.per_thread == 2 && k.group <= add_gmax;
        const int gmax = rows <= kRowsFewRows ? 512 : 256;
        return k.per_thread >= 2 && k.per_thread <= 4 && k.group <= gmax;
    };
    const bool ma = in_band(a);
    const bool mb = in_band(b);
    if (ma != mb) return ma;
    if (a.idle != b.idle) return a.idle < b.idle;
    if (a.one_wave != b.one_wave) return a.one_wave;
    if (ma && layernorm && a.many_waves && b.many_waves) return a.per_thread > b.per_thread;
    if (ma) return a.per_thread < b.per_thread;
    if (!layernorm) {
        const bool na = a.per_thread <= 4 && a.group <= add_gmax;
        const bool nb = b.per_thread <= 4 && b.group <= add_gmax;
        if (na != nb) return na;
    }
    return a.group < b.group;
}

// Choose the register-resident variant; false if no compiled variant holds the row.
// `layernorm` selects the LayerNorm kernel's occupancy for the one-wave test.
bool rms_choose_rows(const RmsCall& c, int vb, int* group, int* per_thread,
                     bool layernorm = false) {
    const int es = camp::elem_bytes(c.t);
    const int64_t nvec = c.a.cols * es / vb;
    static const int kGroupsVec[] = {32, 64, 128, 256, 512, 1024};
    static const int kPerVec[] = {1, 2, 3, 4, 6, 8};
    static const int kGroupsElem[] = {32, 256, 1024};
    static const int kPerElem[] = {1, 2, 4, 8, 16};
    const bool vec = vb == 16;
    const int* groups = vec ? kGroupsVec : kGroupsElem;
    const int ngroups = vec ? 6 : 3;
    const int* pers = vec ? kPerVec : kPerElem;
    const int npers = vec ? 6 : 5;
    const int max_per = pers[npers - 1];

    bool found = false;
    RowsCandidate best{};
    for (int i = 0; i < ngroups; ++i) {
        const int g = groups[i];
        const int64_t need = ceil_div(nvec, g);
        if (need > max_per) continue;
        RowsCandidate k;
        k.group = g;
        k.per_thread = round_up_in(static_cast<int>(need), pers, npers);
        if (!camp::rows_variant_compiled(c.add, vb, g, k.per_thread)) continue;
        k.ctas = ceil_div(c.a.rows, camp::rows_block(g) / g);
        k.idle = static_cast<int64_t>(g) * k.per_thread - nvec;
        const int per_sm =
            layernorm ? camp::ln_min_blocks(es, vb, g, k.per_thread)
                      : camp::rows_min_blocks(vb, g, c.add ? 2 * k.per_thread : k.per_thread);
        k.one_wave = k.ctas <= static_cast<int64_t>(camp::kSmCount) * per_sm;
        k.many_waves = k.ctas >= 2 * static_cast<int64_t>(camp::kSmCount) * per_sm;
        k.add16 = c.add && vec && !layernorm;
        if (!found || rows_better(k, best, layernorm, c.a.rows <= camp::kSmCount, c.add, c.a.rows))
            best = k;
        found = true;
    }
    if (!found) return false;
    *group = best.group;
    *per_thread = best.per_thread;
    return true;
}

// Cluster split of one row (register cluster kernel): the smallest power-of-two cluster
// (2..16 CTAs of 256 threads) whose CTAs hold the row with at most 8 accesses per thread
// (measured: 256 rows of 131072 bf16 run 29.6 us as 8 x 8 and 31.3 us as 16 x 4). The
// planner reaches it only for rows past kClusterFrom vectors that the staged kernel cannot
// hold; with today's limits (both 16 x 2048 vectors) that never happens, so it runs through
// explicit plans (the staged kernel replaced it: 0.67 -> 0.76 at 256 x 131072). False if
// even 16 x 256 x 8 vectors cannot hold the row (the two-sweep kernel takes it).
constexpr int64_t kClusterFrom = 8192;

bool rms_choose_cluster(const RmsCall& c, int64_t nvec, int* cluster, int* per_thread) {
    static const int kPer[] = {1, 2, 3, 4, 6, 8};
    if (c.a.rows > kMaxGrid / 16) return false;   // the grid is rows * cluster CTAs
    for (int cl : {2, 4, 8, 16}) {
        const int64_t need = ceil_div(nvec, static_cast<int64_t>(cl) * camp::kClusterBlock);
        if (need <= 8) {
            *cluster = cl;
            *per_thread = round_up_in(static_cast<int>(need), kPer, 6);
            return true;
        }
    }
    return false;
}

// Staged (shared-memory) split of a row: chunk vectors per CTA for `cluster` CTAs, and
// the resulting dynamic shared memory; false if the variant cannot hold the row.
bool rms_staged_fits(const RmsCall& c, int64_t nvec, int cluster, int stages,
                     int64_t* chunk) {
    if (cluster < 1 || cluster > 16 || (cluster & (cluster - 1)) != 0) return false;
    if (stages < 2 || stages > camp::kStagedMaxStages) return false;
    *chunk = ceil_div(nvec, cluster);
    return *chunk <= static_cast<int64_t>(camp::kStagedMaxVecsPerThread) * camp::kStagedBlock &&
           camp::staged_smem_bytes(c.add, *chunk, stages) <= camp::kStagedSmemMax;
}

// Fill the plan fields of a staged launch: group = vectors per CTA chunk, per_thread =
// stages, grid = an estimate of the CTAs launched (the launch sizes the grid to the
// clusters the device holds at once, at most one per row).
void rms_staged_plan_fields(const RmsCall& c, int cluster, int stages, int64_t chunk,
                            camp_plan_t* p) {
    p->kernel = CAMP_KERNEL_RMSNORM_STAGED;
    p->vec_bytes = 16;
    p->group = static_cast<int32_t>(chunk);
    p->per_thread = stages;
    p->block = camp::kStagedBlock;
    p->cluster = cluster;
    const int64_t per_sm = camp::kSmSmemBytes / (camp::staged_smem_bytes(c.add, chunk, stages) + 1024);
    int64_t clusters = (camp::kSmCount * (per_sm < 1 ? 1 : per_sm)) / cluster;
    if (clusters < 1) clusters = 1;
    if (clusters > c.a.rows) clusters = c.a.rows;
    p->grid = clusters * cluster;
}

// Rows of more than kStagedFrom 16-byte vectors go to the shared-memory-staged kernel:
// C = the power of two (at most 16) that makes a CTA's chunk about 1024 vectors (16 KB),
// 3 buffers deep, 2 at C = 16. Measured on GB300 (bf16, L2-cold, graphs of back-to-back
// launches), against the register kernels' default plans: 1024 x 65536 0.90 / 0.80 of the
// measured HBM peak, 512 x 131072 0.84 / 0.75, 256 x 131072 0.76 / 0.67, 64 x 262144
// 0.63 / 0.50; with the residual add 1024 x 65536 0.92 / 0.80, 512 x 131072 0.98 / 0.77;
// fp32 256 x 65536 0.83 / 0.68. At 4096 vectors and below the register kernels are as
// fast (2048 x 32768: 0.87 / 0.88) and keep those rows.
constexpr int64_t kStagedFrom = 4096;

// With the residual add (x and r both staged) the measured best split differs (bf16,
// graph-timed, two passes agreeing, fraction of the measured peak against the plain rule's
// 8 CTAs of about 1024 vectors): up to 6144 vectors 4 CTAs with 3 buffers (2048 and 4096
// rows of 40000 columns: 0.94 / 0.95 against 0.85 / 0.85); at 6144..8192 vectors 16 CTAs
// with 3 buffers from 1024 rows on (1024 and 2048 rows of 65536: 0.94 / 0.95 against 0.86 /
// 0.88) and 4 CTAs below (512 rows: 0.95 against 0.89).
constexpr int64_t kStagedAddFew = 6144;
constexpr int64_t kStagedAddManyRows = 1024;

bool rms_choose_staged(const RmsCall& c, int64_t nvec, int* cluster, int* stages,
                       int64_t* chunk) {
    int cl = 1, st = 3;
    if (c.add && nvec <= 8192) {
        cl = (nvec <= kStagedAddFew || c.a.rows < kStagedAddManyRows) ? 4 : 16;
    } else {
        while (cl < 16 && ceil_div(nvec, cl) > 1024) cl *= 2;
        st = cl == 16 ? 2 : 3;
    }
    if (!rms_staged_fits(c, nvec, cl, st, chunk)) return false;
    *cluster = cl;
    *stages = st;
    return true;
}

// Rows past the staged kernel (more than 16 x 2048 16-byte vectors) that still fit a
// cluster's shared memory take the spread kernel: one buffer a CTA and the smallest
// power-of-two cluster whose chunks hold at most spread_chunk_max vectors, else 16 CTAs
// (rows of up to about 1.7 M bf16 columns). The limit is the chunk at which shared memory
// (228 KB an SM, 1 KB of it reserved a CTA, and under 1 KB of static arrays) still holds
// as many CTAs an SM as the registers allow: 3 (73 KB chunks), or 2 for fp32 LayerNorm
// (109 KB). The plan's grid counts no more resident CTAs than that. On RMSNorm's residual-
// add path (`staged` = 2: x and r in shared memory) the limit is halved.
constexpr int64_t spread_chunk_max(int per_sm) { return per_sm >= 3 ? 4700 : 7000; }

bool spread_fits(int64_t nvec, int cluster, int stages, int64_t* chunk, int staged = 1) {
    if (cluster < 1 || cluster > 16 || (cluster & (cluster - 1)) != 0) return false;
    if (stages < 1 || stages > camp::kSpreadMaxStages) return false;
    *chunk = ceil_div(nvec, cluster);
    return camp::spread_smem_bytes(*chunk, stages, staged) <= camp::kStagedSmemMax;
}

bool spread_choose(int64_t nvec, int64_t rows, int per_sm, int* cluster, int* stages,
                   int64_t* chunk, int staged = 1) {
    for (int cl = 1; cl <= 16; cl *= 2) {
        if ((ceil_div(nvec, cl) <= spread_chunk_max(per_sm) / staged || cl == 16) &&
            spread_fits(nvec, cl, 1, chunk, staged)) {
            // So few rows that their CTAs would leave half the SMs idle: split each row
            // further (GB300, bf16: 5 x 40000 0.03 -> 0.05, fp32 3 x 131080 0.11 -> 0.14;
            // splitting while the rows' CTAs fill fewer than all resident slots lost at
            // 32 x 131072, 0.36 -> 0.25, and 100 x 100000, 0.51 -> 0.44).
            while (cl < 16 && rows * cl < camp::kSmCount / 2) cl *= 2;
            spread_fits(nvec, cl, 1, chunk, staged);
            *cluster = cl;
            *stages = 1;
            return true;
        }
    }
    return false;
}

void spread_plan_fields(int64_t rows, int kernel, int per_sm_regs, int cluster, int stages,
                        int64_t chunk, camp_plan_t* p, int staged = 1) {
    p->kernel = kernel;
    p->vec_bytes = 16;
    p->group = static_cast<int32_t>(chunk);
    p->per_thread = stages;
    p->block = camp::kSpreadBlock;
    p->cluster = cluster;
    int64_t per_sm = camp::kSmSmemBytes / (camp::spread_smem_bytes(chunk, stages, staged) + 2048);
    if (per_sm > per_sm_regs) per_sm = per_sm_regs;
    int64_t clusters = (camp::kSmCount * (per_sm < 1 ? 1 : per_sm)) / cluster;
    if (clusters < 1) clusters = 1;
    if (clusters > rows) clusters = rows;
    p->grid = clusters * cluster;
}

// CTAs an SM the spread kernel's registers allow for this call (fewer with the residual add).
int rms_spread_per_sm(const RmsCall& c) {
    return camp::spread_ctas_per_sm(false, camp::elem_bytes(c.t), c.add);
}

void rms_plan(const RmsCall& c, camp_plan_t* p) {
    *p = camp_plan_t{};
    p->vec_bytes = rms_vec_bytes(c);
    p->cluster = 1;
    const int64_t nvec = c.a.cols * camp::elem_bytes(c.t) / p->vec_bytes;
    int g = 0, nv = 0, cl = 0, st = 0;
    int64_t chunk = 0;
    const int64_t cluster_from = c.add ? kClusterFrom / 2 : kClusterFrom;
    if (p->vec_bytes == 16 && nvec > kStagedFrom && rms_choose_staged(c, nvec, &cl, &st, &chunk)) {
        rms_staged_plan_fields(c, cl, st, chunk, p);
    } else if (p->vec_bytes == 16 && nvec > kStagedFrom &&
               spread_choose(nvec, c.a.rows, rms_spread_per_sm(c), &cl, &st, &chunk,
                             c.add ? 2 : 1)) {
        spread_plan_fields(c.a.rows, CAMP_KERNEL_RMSNORM_SPREAD, rms_spread_per_sm(c), cl, st,
                           chunk, p, c.add ? 2 : 1);
    } else if (p->vec_bytes == 16 && nvec > cluster_from && rms_choose_cluster(c, nvec, &cl, &nv)) {
        p->kernel = CAMP_KERNEL_RMSNORM_CLUSTER;
        p->group = cl * camp::kClusterBlock;
        p->per_thread = nv;
        p->block = camp::kClusterBlock;
        p->cluster = cl;
        p->grid = c.a.rows * cl;
    } else if (rms_choose_rows(c, p->vec_bytes, &g, &nv)) {
        p->kernel = CAMP_KERNEL_RMSNORM_ROWS;
        p->group = g;
        p->per_thread = nv;
        p->block = camp::rows_block(g);
        p->grid = ceil_div(c.a.rows, p->block / g);   // one row block per CTA
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
    const int64_t nvec = c.a.cols * es / vb;
    *p = in;
    p->cluster = 1;
    if (in.kernel == CAMP_KERNEL_RMSNORM_ROWS) {
        if (!camp::rmsnorm_rows_compiled(c.add, c.t, vb, in.group, in.per_thread))
            return CAMP_ERR_NOT_SUPPORTED;
        if (static_cast<int64_t>(in.group) * in.per_thread < nvec) return CAMP_ERR_NOT_SUPPORTED;
        p->block = camp::rows_block(in.group);
        p->grid = ceil_div(c.a.rows, p->block / in.group);
        return CAMP_SUCCESS;
    }
    if (in.kernel == CAMP_KERNEL_RMSNORM_CLUSTER) {
        const int cl = in.cluster;
        if (vb != 16 || (cl != 2 && cl != 4 && cl != 8 && cl != 16)) return CAMP_ERR_NOT_SUPPORTED;
        if (!camp::rmsnorm_cluster_compiled(c.t, in.per_thread)) return CAMP_ERR_NOT_SUPPORTED;
        if (static_cast<int64_t>(cl) * camp::kClusterBlock * in.per_thread < nvec)
            return CAMP_ERR_NOT_SUPPORTED;
        if (c.a.rows > kMaxGrid / cl) return CAMP_ERR_NOT_SUPPORTED;
        p->group = cl * camp::kClusterBlock;
        p->block = camp::kClusterBlock;
        p->cluster = cl;
        p->grid = c.a.rows * cl;
        return CAMP_SUCCESS;
    }
    if (in.kernel == CAMP_KERNEL_RMSNORM_STAGED) {
        int64_t chunk = 0;
        if (vb != 16 || !rms_staged_fits(c, nvec, in.cluster, in.per_thread, &chunk))
            return CAMP_ERR_NOT_SUPPORTED;
        rms_staged_plan_fields(c, in.cluster, in.per_thread, chunk, p);
        return CAMP_SUCCESS;
    }
    if (in.kernel == CAMP_KERNEL_RMSNORM_SPREAD) {
        int64_t chunk = 0;
        if (vb != 16 || !spread_fits(nvec, in.cluster, in.per_thread, &chunk, c.add ? 2 : 1))
            return CAMP_ERR_NOT_SUPPORTED;
        spread_plan_fields(c.a.rows, CAMP_KERNEL_RMSNORM_SPREAD, rms_spread_per_sm(c),
                           in.cluster, in.per_thread, chunk, p, c.add ? 2 : 1);
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
    cudaError_t e = cudaErrorInvalidValue;
    if (p.kernel == CAMP_KERNEL_RMSNORM_ROWS) {
        e = camp::rmsnorm_rows_launch(c.add, c.t, p.vec_bytes, p.group, p.per_thread, c.a,
                                      p.grid, s);
    } else if (p.kernel == CAMP_KERNEL_RMSNORM_CLUSTER) {
        e = camp::rmsnorm_cluster_launch(c.add, c.t, p.per_thread, p.cluster, c.a, s);
    } else if (p.kernel == CAMP_KERNEL_RMSNORM_WIDE) {
        e = camp::rmsnorm_wide_launch(c.add, c.t, p.vec_bytes, c.a, p.grid, s);
    } else if (p.kernel == CAMP_KERNEL_RMSNORM_STAGED) {
        e = camp::rmsnorm_staged_launch(c.add, c.t, p.cluster, p.per_thread, c.a, s);
    } else if (p.kernel == CAMP_KERNEL_RMSNORM_SPREAD) {
        e = camp::rmsnorm_spread_launch(c.add, c.t, p.cluster, p.per_thread, c.a, s);
    }
    return runtime_status(e);
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.0f; }

// ------------------------------------------------------------------ RoPE

struct RopeCall {
    camp::RopeArgs a;
    DType t;
};

// Checks for one tensor (H2 == 0, x2/y2 ignored) or two tensors of the same [B, S, *, D]
// layout sharing the tables. Every output must be disjoint from every input except its
// own input (in place), from the other output and from the tables. A single remaining
// tensor is always put in the first slot.
camp_status_t rope_validate(const void* x, const void* x2, const float* sin_t,
                            const float* cos_t, const void* y, const void* y2, int64_t B,
                            int64_t S, int64_t H, int64_t H2, int64_t D, camp_dtype_t dtype,
                            RopeCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || S < 0 || H < 0 || H2 < 0 || D < 2 || D % 2 != 0) return CAMP_ERR_INVALID_ARG;
    if (B == 0 || S == 0 || (H == 0 && H2 == 0)) { *empty = true; return CAMP_SUCCESS; }
    if (sin_t == nullptr || cos_t == nullptr) return CAMP_ERR_INVALID_ARG;
    if (H > 0 && (x == nullptr || y == nullptr)) return CAMP_ERR_INVALID_ARG;
    if (H2 > 0 && (x2 == nullptr || y2 == nullptr)) return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t tokens = 0, rows = 0, rows2 = 0, bytes = 0, bytes2 = 0, table_bytes = 0;
    if (!mul_ok(B, S, 1, &tokens) || !mul_ok(tokens, H, 1, &rows) ||
        !mul_ok(tokens, H2, 1, &rows2) || !mul_ok(rows, D, es, &bytes) ||
        !mul_ok(rows2, D, es, &bytes2) || !mul_ok(S, D / 2, 4, &table_bytes))
        return CAMP_ERR_INVALID_ARG;
    if (!aligned(sin_t, 4) || !aligned(cos_t, 4)) return CAMP_ERR_INVALID_ARG;
    if (H > 0) {
        if (!aligned(x, es) || !aligned(y, es)) return CAMP_ERR_INVALID_ARG;
        if (y != x && overlaps(y, bytes, x, bytes)) return CAMP_ERR_INVALID_ARG;
        if (overlaps(y, bytes, sin_t, table_bytes) || overlaps(y, bytes, cos_t, table_bytes))
            return CAMP_ERR_INVALID_ARG;
    }
    if (H2 > 0) {
        if (!aligned(x2, es) || !aligned(y2, es)) return CAMP_ERR_INVALID_ARG;
        if (y2 != x2 && overlaps(y2, bytes2, x2, bytes2)) return CAMP_ERR_INVALID_ARG;
        if (overlaps(y2, bytes2, sin_t, table_bytes) || overlaps(y2, bytes2, cos_t, table_bytes))
            return CAMP_ERR_INVALID_ARG;
    }
    if (H > 0 && H2 > 0) {
        if (overlaps(y, bytes, x2, bytes2) || overlaps(y2, bytes2, x, bytes) ||
            overlaps(y, bytes, y2, bytes2))
            return CAMP_ERR_INVALID_ARG;
    }
    c->a = camp::RopeArgs{};
    c->a.sin_t = sin_t;
    c->a.cos_t = cos_t;
    c->a.tokens = tokens;
    c->a.seq = S;
    c->a.half = D / 2;
    if (H > 0) {
        c->a.x = x;
        c->a.y = const_cast<void*>(y);
        c->a.heads = H;
        if (H2 > 0) {
            c->a.x2 = x2;
            c->a.y2 = const_cast<void*>(y2);
            c->a.heads2 = H2;
        }
    } else {
        c->a.x = x2;
        c->a.y = const_cast<void*>(y2);
        c->a.heads = H2;
    }
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
    if (c.a.heads2 > 0 && (!aligned(c.a.x2, vb) || !aligned(c.a.y2, vb))) return false;
    return aligned(c.a.x, vb) && aligned(c.a.y, vb) && aligned(c.a.sin_t, table_align) &&
           aligned(c.a.cos_t, table_align);
}

int rope_widest_vec(const RopeCall& c) {
    static const int kVec[] = {16, 8, 4, 2};
    for (int vb : kVec)
        if (rope_vec_ok(c, vb)) return vb;
    return camp::elem_bytes(c.t);   // not reached: element accesses are always legal
}

// Positions one CTA of the tiled kernel covers, or 0 if the tiled kernel cannot run
// this shape (a position needs more than one CTA, or the sizes exceed its 32-bit math).
int64_t rope_positions_per_cta(const RopeCall& c, int vb, int hpt) {
    const int es = camp::elem_bytes(c.t);
    if (c.a.tokens > 0xFFFFFFFFll || c.a.heads > 0x7FFFFFFFll || c.a.heads2 > 0x7FFFFFFFll ||
        c.a.half > 0x7FFFFFFFll)
        return 0;
    const int64_t per_pos =
        (ceil_div(c.a.heads, hpt) + ceil_div(c.a.heads2, hpt)) * (c.a.half * es / vb);
    return per_pos <= camp::kRopeBlock ? camp::kRopeBlock / per_pos : 0;
}

// CTAs launched: the tiled kernel runs one position block per CTA (any count; the launch
// uses a second grid dimension past 2^31 - 1); the flat kernel loops, so its grid is capped.
int64_t rope_grid(const RopeCall& c, int kernel, int vb, int hpt) {
    if (kernel == CAMP_KERNEL_ROPE) return ceil_div(c.a.tokens, rope_positions_per_cta(c, vb, hpt));
    const int es = camp::elem_bytes(c.t);
    const int64_t work = c.a.tokens * ceil_div(c.a.heads, hpt) * (c.a.half * es / vb);
    const int64_t blocks = ceil_div(work, camp::kRopeBlock);
    return blocks < kMaxGrid ? blocks : kMaxGrid;
}

// The second tensor of a call as a single-tensor call of its own.
RopeCall rope_second(const RopeCall& c) {
    RopeCall d = c;
    d.a.x = c.a.x2;
    d.a.y = c.a.y2;
    d.a.heads = c.a.heads2;
    d.a.x2 = nullptr;
    d.a.y2 = nullptr;
    d.a.heads2 = 0;
    return d;
}

RopeCall rope_first(const RopeCall& c) {
    RopeCall d = c;
    d.a.x2 = nullptr;
    d.a.y2 = nullptr;
    d.a.heads2 = 0;
    return d;
}

// Choose the RoPE variant: the widest legal vector, then the heads per thread, then the
// kernel. Measured on GB300 (L2-cold, back-to-back launches): with many positions (16384
// and up, many waves) 4 heads per thread is fastest (Q+K of 32+8 heads of 128 at 65536
// positions: 196 us against 208 us with 2); with fewer positions 2 heads per thread is
// fastest or within 1% (4096 positions: Q+K 8.37 us, Q 6.87 us, K 3.16 us). A ragged head
// count takes the largest of 4, 2, 1 that divides every head count. The tiled kernel runs
// when a position fits one CTA; otherwise one tensor takes the flat kernel and two
// tensors are split into two single-tensor launches.
// Decode sizes (no more positions than SMs) are latency-bound: the tiled variant with the
// most threads per position (up to one CTA), then the widest access, then the fewest heads
// per thread. Measured on GB300 (bf16, graphs of back-to-back launches), against the
// bandwidth choice (16-byte accesses, 2 heads per thread): 8 positions x 32 heads x 64
// 1.41 / 1.81 us, 64 x 8 x 64 1.39 / 1.81, 8 x 8 x 128 1.29 / 1.79, Q+K 8 x (32 + 8) x 64
// 1.53 / 1.80; from 512 positions on the bandwidth choice is as fast or faster.
bool rope_plan_latency(const RopeCall& c, camp_plan_t* p) {
    const int es = camp::elem_bytes(c.t);
    int64_t best = 0;
    for (int vb : {16, 8, 4}) {
        if (vb < 2 * es || !rope_vec_ok(c, vb)) continue;
        for (int hpt : {1, 2, 4, 8}) {
            if (!camp::rope_compiled(c.t, vb, hpt) || rope_positions_per_cta(c, vb, hpt) == 0)
                continue;
            const int64_t per_pos =
                (ceil_div(c.a.heads, hpt) + ceil_div(c.a.heads2, hpt)) * (c.a.half * es / vb);
            if (per_pos > best) {   // ties keep the wider access / fewer heads seen first
                best = per_pos;
                p->vec_bytes = vb;
                p->group = hpt;
            }
        }
    }
    return best > 0;
}

// Between the decode sizes and a grid of kRopeFillCtas CTAs, the bandwidth choice leaves
// most SMs idle: there the planner takes the tiled variant whose grid is the smallest one
// of at least kRopeFillCtas CTAs (then the widest access, then the fewest heads per
// thread). Measured on GB300 (bf16, graphs of back-to-back launches, every tiled variant
// of Q, and of Q+K, at 256..8192 positions of 8 and 32 heads of 64 and 128): it changes the
// plan of 7 of those 36 shapes, each 5-24% faster (256 x 8 x 64: 1.25 us against 1.61,
// 512 x 8 x 64: 1.30 against 1.69, 1024 x 8 x 64: 1.62 against 1.75) and none slower;
// reaching for 152 CTAs or more instead made 4 shapes 15-21% slower.
constexpr int64_t kRopeFillCtas = 128;

bool rope_plan_fill(const RopeCall& c, camp_plan_t* p) {
    const int es = camp::elem_bytes(c.t);
    int64_t best = 0;
    for (int vb : {16, 8, 4}) {
        if (vb < 2 * es || !rope_vec_ok(c, vb)) continue;
        for (int hpt : {1, 2, 4, 8}) {
            if (!camp::rope_compiled(c.t, vb, hpt) || rope_positions_per_cta(c, vb, hpt) == 0)
                continue;
            const int64_t g = rope_grid(c, CAMP_KERNEL_ROPE, vb, hpt);
            if (g >= kRopeFillCtas && (best == 0 || g < best)) {   // ties keep the first seen
                best = g;
                p->vec_bytes = vb;
                p->group = hpt;
            }
        }
    }
    return best > 0;
}

void rope_plan(const RopeCall& c, camp_plan_t* p) {
    *p = camp_plan_t{};
    p->cluster = 1;
    if (c.a.tokens <= camp::kSmCount && rope_plan_latency(c, p)) {
        p->kernel = CAMP_KERNEL_ROPE;
        p->per_thread = 0;
        p->block = camp::kRopeBlock;
        p->grid = rope_grid(c, CAMP_KERNEL_ROPE, p->vec_bytes, p->group);
        return;
    }
    p->vec_bytes = rope_widest_vec(c);
    const bool by4 = c.a.heads % 4 == 0 && c.a.heads2 % 4 == 0;
    const bool by2 = c.a.heads % 2 == 0 && c.a.heads2 % 2 == 0;
    p->group = (by4 && c.a.tokens >= 16384 && rope_positions_per_cta(c, p->vec_bytes, 4) > 0)
                   ? 4 : by2 ? 2 : 1;
    p->per_thread = 0;
    p->block = camp::kRopeBlock;
    if (rope_positions_per_cta(c, p->vec_bytes, p->group) > 0) {
        p->kernel = CAMP_KERNEL_ROPE;
        p->grid = rope_grid(c, CAMP_KERNEL_ROPE, p->vec_bytes, p->group);
        if (p->grid < kRopeFillCtas && rope_plan_fill(c, p))
            p->grid = rope_grid(c, CAMP_KERNEL_ROPE, p->vec_bytes, p->group);
    } else if (c.a.heads2 == 0) {
        p->kernel = CAMP_KERNEL_ROPE_FLAT;
        p->grid = rope_grid(c, CAMP_KERNEL_ROPE_FLAT, p->vec_bytes, p->group);
    } else {
        camp_plan_t p1, p2;
        rope_plan(rope_first(c), &p1);
        rope_plan(rope_second(c), &p2);
        p->kernel = CAMP_KERNEL_ROPE_SPLIT;
        p->grid = p1.grid + p2.grid;
    }
}

camp_status_t rope_accept_plan(const RopeCall& c, const camp_plan_t& in, camp_plan_t* p) {
    if (in.kernel != CAMP_KERNEL_ROPE && in.kernel != CAMP_KERNEL_ROPE_FLAT)
        return CAMP_ERR_NOT_SUPPORTED;
    if (in.kernel == CAMP_KERNEL_ROPE_FLAT && c.a.heads2 > 0) return CAMP_ERR_NOT_SUPPORTED;
    if (!rope_vec_ok(c, in.vec_bytes)) return CAMP_ERR_NOT_SUPPORTED;
    if (!camp::rope_compiled(c.t, in.vec_bytes, in.group)) return CAMP_ERR_NOT_SUPPORTED;
    if (in.kernel == CAMP_KERNEL_ROPE && rope_positions_per_cta(c, in.vec_bytes, in.group) == 0)
        return CAMP_ERR_NOT_SUPPORTED;
    *p = in;
    p->per_thread = 0;
    p->cluster = 1;
    p->block = camp::kRopeBlock;
    p->grid = rope_grid(c, in.kernel, in.vec_bytes, in.group);
    return CAMP_SUCCESS;
}

camp_status_t rope_launch(const RopeCall& c, const camp_plan_t& p, cudaStream_t s) {
    if (p.kernel == CAMP_KERNEL_ROPE_SPLIT) {
        const RopeCall parts[2] = {rope_first(c), rope_second(c)};
        for (const RopeCall& part : parts) {
            camp_plan_t q;
            rope_plan(part, &q);
            const camp_status_t st = rope_launch(part, q, s);
            if (st != CAMP_SUCCESS) return st;
        }
        return CAMP_SUCCESS;
    }
    const cudaError_t e =
        p.kernel == CAMP_KERNEL_ROPE
            ? camp::rope_tiled_launch(c.t, p.vec_bytes, p.group, c.a, p.grid, s)
            : camp::rope_flat_launch(c.t, p.vec_bytes, p.group, c.a, p.grid, s);
    return runtime_status(e);
}

// ------------------------------------------------------------------ KV RMSNorm + RoPE + cache

struct KvCall {
    camp::KvCacheArgs a;
    DType t;
};

camp_status_t kv_validate(const void* kv, const void* gamma, const float* sin_t,
                          const float* cos_t, const int64_t* slots, const void* cache_n,
                          const void* cache_r, int64_t B, int64_t S, int64_t dn, int64_t dr,
                          int64_t num_slots, camp_dtype_t dtype, KvCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || S < 0 || dn < 1 || dr < 2 || dr % 2 != 0 || num_slots < 0)
        return CAMP_ERR_INVALID_ARG;
    if (dn > 0x7FFFFFFF || dr > 0x7FFFFFFF) return CAMP_ERR_INVALID_ARG;
    if (B == 0 || S == 0) { *empty = true; return CAMP_SUCCESS; }
    if (!kv || !gamma || !sin_t || !cos_t || !slots || !cache_n || !cache_r)
        return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t tokens = 0, kv_bytes = 0, cn_bytes = 0, cr_bytes = 0, table_bytes = 0, slot_bytes = 0;
    if (!mul_ok(B, S, 1, &tokens) || !mul_ok(tokens, dn + dr, es, &kv_bytes) ||
        !mul_ok(num_slots, dn, es, &cn_bytes) || !mul_ok(num_slots, dr, es, &cr_bytes) ||
        !mul_ok(S, dr / 2, 4, &table_bytes) || !mul_ok(tokens, 8, 1, &slot_bytes))
        return CAMP_ERR_INVALID_ARG;
    for (const void* p : {kv, gamma, cache_n, cache_r})
        if (!aligned(p, es)) return CAMP_ERR_INVALID_ARG;
    if (!aligned(sin_t, 4) || !aligned(cos_t, 4) || !aligned(slots, 8)) return CAMP_ERR_INVALID_ARG;
    // The caches are outputs: disjoint from every input and from each other.
    const void* ins[] = {kv, gamma, sin_t, cos_t, slots};
    const int64_t in_bytes[] = {kv_bytes, dn * es, table_bytes, table_bytes, slot_bytes};
    for (int i = 0; i < 5; ++i) {
        if (overlaps(cache_n, cn_bytes, ins[i], in_bytes[i]) ||
            overlaps(cache_r, cr_bytes, ins[i], in_bytes[i]))
            return CAMP_ERR_INVALID_ARG;
    }
    if (overlaps(cache_n, cn_bytes, cache_r, cr_bytes)) return CAMP_ERR_INVALID_ARG;
    c->a = camp::KvCacheArgs{kv, gamma, sin_t, cos_t, slots, const_cast<void*>(cache_n),
                             const_cast<void*>(cache_r), tokens, S, dn, dr, num_slots, 0.0f};
    c->t = t;
    return CAMP_SUCCESS;
}

bool kv_rope_ok(const KvCall& c, int rb);

// 16-byte norm accesses when the norm part of every row starts on a 16-byte boundary, the
// pointers allow them and the rope part can take 4-, 8- or 16-byte accesses; else element
// accesses for both parts.
int kv_vec_bytes(const KvCall& c) {
    const int es = camp::elem_bytes(c.t);
    const bool ok = (c.a.dn * es) % 16 == 0 && ((c.a.dn + c.a.dr) * es) % 16 == 0 &&
                    aligned(c.a.kv, 16) && aligned(c.a.gamma, 16) && aligned(c.a.cache_n, 16) &&
                    ((es == 2 && kv_rope_ok(c, 4)) || kv_rope_ok(c, 8) || kv_rope_ok(c, 16));
    return ok ? 16 : es;
}

// Can the rope part use rb-byte accesses per half and lane (rb/es elements of each half
// and as many sine and cosine values) within one warp?
bool kv_rope_ok(const KvCall& c, int rb) {
    const int es = camp::elem_bytes(c.t);
    const int64_t half_bytes = (c.a.dr / 2) * es;
    const int re = rb / es;
    const int table_align = 4 * re < 16 ? 4 * re : 16;
    return half_bytes % rb == 0 && half_bytes / rb <= 32 && (c.a.dn * es) % rb == 0 &&
           aligned(c.a.kv, rb) && aligned(c.a.cache_r, rb) && aligned(c.a.sin_t, table_align) &&
           aligned(c.a.cos_t, table_align);
}

// The rope access width for a norm access width: the element size on the element path;
// with 16-byte norm accesses the narrowest of 4, 8 and 16 bytes that holds a pair and
// fits (the rope part spread over the most lanes); 0 if none does.
int kv_rope_bytes(const KvCall& c, int vb) {
    const int es = camp::elem_bytes(c.t);
    if (vb != 16) return kv_rope_ok(c, es) ? es : 0;
    for (int rb : {4, 8, 16})
        if (rb >= 2 * es && kv_rope_ok(c, rb)) return rb;
    return 0;
}

// Norm accesses per lane for a vector width, or 0 if the norm part does not fit one warp
// (at most 8 16-byte or 16 element accesses per lane).
int kv_nvn(const KvCall& c, int vb) {
    const int es = camp::elem_bytes(c.t);
    const int64_t nvec = c.a.dn * es / vb;
    const int64_t need = ceil_div(nvec, 32);
    const int max_nvn = vb == 16 ? 8 : 16;
    if (need > max_nvn) return 0;
    static const int kNvn[] = {1, 2, 4, 8, 16};
    return round_up_in(static_cast<int>(need), kNvn, 5);
}

// Plan fields: vec_bytes = norm access width, per_thread = norm accesses per lane,
// group = rope access width per half and lane (0 in a forced plan: the default for its
// vec_bytes).
camp_status_t kv_plan(const KvCall& c, const camp_plan_t* forced, camp_plan_t* p) {
    if (forced && forced->kernel != CAMP_KERNEL_KV_CACHE) return CAMP_ERR_NOT_SUPPORTED;
    *p = camp_plan_t{};
    p->kernel = CAMP_KERNEL_KV_CACHE;
    const int es = camp::elem_bytes(c.t);
    p->vec_bytes = forced ? forced->vec_bytes : kv_vec_bytes(c);
    if (p->vec_bytes != 16 && p->vec_bytes != es) return CAMP_ERR_NOT_SUPPORTED;
    if (p->vec_bytes > kv_vec_bytes(c)) return CAMP_ERR_NOT_SUPPORTED;
    const int need = kv_nvn(c, p->vec_bytes);
    if (need == 0) return CAMP_ERR_NOT_SUPPORTED;
    p->per_thread = forced ? forced->per_thread : need;
    if (p->per_thread < need) return CAMP_ERR_NOT_SUPPORTED;
    p->group = forced && forced->group != 0 ? forced->group : kv_rope_bytes(c, p->vec_bytes);
    if (p->group == 0 || !kv_rope_ok(c, p->group)) return CAMP_ERR_NOT_SUPPORTED;
    if (!camp::kv_cache_compiled(c.t, p->vec_bytes, p->per_thread, p->group))
        return CAMP_ERR_NOT_SUPPORTED;
    p->block = camp::kKvBlock;
    p->cluster = 1;
    p->grid = ceil_div(c.a.tokens, camp::kKvTokensPerCta);
    return CAMP_SUCCESS;
}

// ------------------------------------------------------------------ interleaved RoPE

struct RopeIlCall {
    camp::RopeInterleavedArgs a;
    DType t;
};

camp_status_t rope_il_validate(const void* x, const float* sin_t, const float* cos_t,
                               const int32_t* positions, const void* y, int64_t tokens,
                               int64_t H, int64_t D, int64_t max_pos, camp_dtype_t dtype,
                               RopeIlCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (tokens < 0 || H < 0 || D < 2 || D % 2 != 0 || max_pos < 0) return CAMP_ERR_INVALID_ARG;
    if (H > 0x7FFFFFFF || D > 0x7FFFFFFF) return CAMP_ERR_INVALID_ARG;
    if (tokens == 0 || H == 0) { *empty = true; return CAMP_SUCCESS; }
    if (!x || !sin_t || !cos_t || !positions || !y) return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t rows = 0, bytes = 0, table_bytes = 0, pos_bytes = 0;
    if (!mul_ok(tokens, H, 1, &rows) || !mul_ok(rows, D, es, &bytes) ||
        !mul_ok(max_pos, D / 2, 4, &table_bytes) || !mul_ok(tokens, 4, 1, &pos_bytes))
        return CAMP_ERR_INVALID_ARG;
    if (!aligned(x, es) || !aligned(y, es) || !aligned(sin_t, 4) || !aligned(cos_t, 4) ||
        !aligned(positions, 4))
        return CAMP_ERR_INVALID_ARG;
    if (y != x && overlaps(y, bytes, x, bytes)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(y, bytes, sin_t, table_bytes) || overlaps(y, bytes, cos_t, table_bytes) ||
        overlaps(y, bytes, positions, pos_bytes))
        return CAMP_ERR_INVALID_ARG;
    c->a = camp::RopeInterleavedArgs{x, sin_t, cos_t, positions, const_cast<void*>(y), tokens,
                                     H, D, max_pos};
    c->t = t;
    return CAMP_SUCCESS;
}

bool rope_il_vec_ok(const RopeIlCall& c, int vb) {
    const int es = camp::elem_bytes(c.t);
    if (vb < 2 * es) return false;                           // a vector holds whole pairs
    if ((c.a.dim * es) % vb != 0) return false;
    const int pairs = vb / es / 2;
    const int table_align = pairs * 4 < 16 ? pairs * 4 : 16;
    return aligned(c.a.x, vb) && aligned(c.a.y, vb) && aligned(c.a.sin_t, table_align) &&
           aligned(c.a.cos_t, table_align);
}

int64_t rope_il_tpc(const RopeIlCall& c, int vb, int hpt) {
    const int es = camp::elem_bytes(c.t);
    const int64_t per_pos = ceil_div(c.a.heads, hpt) * (c.a.dim * es / vb);
    return per_pos <= camp::kRopeBlock ? camp::kRopeBlock / per_pos : 0;
}

// Widest legal vector; 4 heads per thread when the head count is a multiple of 4, else 2
// (1 for odd head counts), more when a token's heads would not fit one CTA;
// CAMP_ERR_NOT_SUPPORTED when even 8 do not. Measured on GB300 (bf16, random positions,
// L2-cold): 4 heads per thread against 2 run 65536 x 32 x 128 in 160.9 / 185.0 us,
// 4096 x 32 x 128 in 12.3 / 13.6 us, 65536 x 8 x 64 in 23.7 / 26.7 us (each token's
// table row is loaded once per head group, so more heads per thread load it fewer times).
camp_status_t rope_il_plan(const RopeIlCall& c, const camp_plan_t* forced, camp_plan_t* p) {
    if (forced && forced->kernel != CAMP_KERNEL_ROPE_INTERLEAVED) return CAMP_ERR_NOT_SUPPORTED;
    *p = camp_plan_t{};
    p->kernel = CAMP_KERNEL_ROPE_INTERLEAVED;
    p->cluster = 1;
    p->block = camp::kRopeBlock;
    if (forced) {
        p->vec_bytes = forced->vec_bytes;
        p->group = forced->group;
        if (!rope_il_vec_ok(c, p->vec_bytes)) return CAMP_ERR_NOT_SUPPORTED;
    } else if (c.a.tokens <= camp::kSmCount) {
        // Decode sizes: the most threads per token within one CTA, then the widest access,
        // then the fewest heads per thread (the rotate-half planner's latency rule).
        int64_t best = 0;
        const int es = camp::elem_bytes(c.t);
        for (int vb : {16, 8, 4}) {
            if (!rope_il_vec_ok(c, vb)) continue;
            for (int hpt : {1, 2, 4, 8}) {
                if (!camp::rope_interleaved_compiled(c.t, vb, hpt) || rope_il_tpc(c, vb, hpt) == 0)
                    continue;
                const int64_t per_tok = ceil_div(c.a.heads, hpt) * (c.a.dim * es / vb);
                if (per_tok > best) {
                    best = per_tok;
                    p->vec_bytes = vb;
                    p->group = hpt;
                }
            }
        }
        if (best == 0) return CAMP_ERR_NOT_SUPPORTED;
    } else {
        for (int vb : {16, 8, 4}) {
            if (rope_il_vec_ok(c, vb)) { p->vec_bytes = vb; break; }
        }
        if (p->vec_bytes == 0) return CAMP_ERR_NOT_SUPPORTED;   // pointers not pair-aligned
        p->group = c.a.heads % 4 == 0 ? 4 : c.a.heads % 2 == 0 ? 2 : 1;
        while (p->group < 8 && rope_il_tpc(c, p->vec_bytes, p->group) == 0) p->group *= 2;
        // The rotate-half planner's fill rule: fewer than kRopeFillCtas CTAs leave most SMs
        // idle, so take the variant with the smallest grid of at least that many.
        const int64_t t0 = rope_il_tpc(c, p->vec_bytes, p->group);
        if (t0 > 0 && ceil_div(c.a.tokens, t0) < kRopeFillCtas) {
            int64_t best = 0;
            for (int vb : {16, 8, 4}) {
                if (!rope_il_vec_ok(c, vb)) continue;
                for (int hpt : {1, 2, 4, 8}) {
                    const int64_t tpc = camp::rope_interleaved_compiled(c.t, vb, hpt)
                                            ? rope_il_tpc(c, vb, hpt) : 0;
                    if (tpc == 0) continue;
                    const int64_t g = ceil_div(c.a.tokens, tpc);
                    if (g >= kRopeFillCtas && (best == 0 || g < best)) {
                        best = g;
                        p->vec_bytes = vb;
                        p->group = hpt;
                    }
                }
            }
        }
    }
    if (!camp::rope_interleaved_compiled(c.t, p->vec_bytes, p->group)) return CAMP_ERR_NOT_SUPPORTED;
    const int64_t tpc = rope_il_tpc(c, p->vec_bytes, p->group);
    if (tpc == 0 || c.a.tokens > 0xFFFFFFFFll) return CAMP_ERR_NOT_SUPPORTED;
    p->grid = ceil_div(c.a.tokens, tpc);
    return CAMP_SUCCESS;
}

// ------------------------------------------------------------------ KV concat + head repeat

struct KvCatCall {
    camp::KvCatArgs a;
    DType t;
    int64_t rows;      // B * (P + S)
};

camp_status_t kv_cat_validate(const void* past, const void* fresh, const float* sin_t,
                              const float* cos_t, const void* out, int64_t B, int64_t P,
                              int64_t S, int64_t Hk, int64_t D, int64_t n_rep,
                              camp_dtype_t dtype, KvCatCall* c, bool* empty) {
    *empty = false;
    if (!dtype_ok(dtype)) return CAMP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || P < 0 || S < 0 || Hk < 0 || D < 2 || D % 2 != 0 || n_rep < 1)
        return CAMP_ERR_INVALID_ARG;
    if ((sin_t == nullptr) != (cos_t == nullptr)) return CAMP_ERR_INVALID_ARG;
    if (Hk > 0x7FFFFFFF || D > 0x7FFFFFFF || n_rep > 0x7FFFFFFF) return CAMP_ERR_INVALID_ARG;
    const int64_t kMax = std::numeric_limits<int64_t>::max();
    if (P > kMax - S) return CAMP_ERR_INVALID_ARG;
    const int64_t T = P + S;
    if (B == 0 || T == 0 || Hk == 0) { *empty = true; return CAMP_SUCCESS; }
    if (out == nullptr || (P > 0 && past == nullptr) || (S > 0 && fresh == nullptr))
        return CAMP_ERR_INVALID_ARG;
    const DType t = to_dtype(dtype);
    const int64_t es = camp::elem_bytes(t);
    int64_t rows = 0, hout = 0, out_bytes = 0, past_bytes = 0, new_bytes = 0, table_bytes = 0;
    int64_t past_rows = 0, new_rows = 0;
    if (!mul_ok(B, T, 1, &rows) || !mul_ok(Hk, n_rep, 1, &hout) ||
        !mul_ok(rows, hout, 1, &out_bytes) || !mul_ok(out_bytes, D, es, &out_bytes) ||
        !mul_ok(B, P, Hk, &past_rows) || !mul_ok(past_rows, D, es, &past_bytes) ||
        !mul_ok(B, S, Hk, &new_rows) || !mul_ok(new_rows, D, es, &new_bytes) ||
        !mul_ok(T, D / 2, 4, &table_bytes))
        return CAMP_ERR_INVALID_ARG;
    if (!aligned(out, es) || (P > 0 && !aligned(past, es)) || (S > 0 && !aligned(fresh, es)))
        return CAMP_ERR_INVALID_ARG;
    // The output is disjoint from every input (its shape differs, so in place is impossible).
    if (P > 0 && overlaps(out, out_bytes, past, past_bytes)) return CAMP_ERR_INVALID_ARG;
    if (S > 0 && overlaps(out, out_bytes, fresh, new_bytes)) return CAMP_ERR_INVALID_ARG;
    if (sin_t != nullptr) {
        if (!aligned(sin_t, 4) || !aligned(cos_t, 4)) return CAMP_ERR_INVALID_ARG;
        if (overlaps(out, out_bytes, sin_t, table_bytes) ||
            overlaps(out, out_bytes, cos_t, table_bytes))
            return CAMP_ERR_INVALID_ARG;
    }
    c->a = camp::KvCatArgs{P > 0 ? past : nullptr, S > 0 ? fresh : nullptr,
                           S > 0 ? sin_t : nullptr, S > 0 ? cos_t : nullptr,
                           const_cast<void*>(out), B, P, S, Hk, D / 2, n_rep};
    c->t = t;
    c->rows = rows;
    return CAMP_SUCCESS;
}

// Is an access of vb bytes per half legal for every pointer and every half-row start?
bool kv_cat_vec_ok(const KvCatCall& c, int vb) {
    const int es = camp::elem_bytes(c.t);
    if (vb < es || (c.a.half * es) % vb != 0) return false;
    const int table_align = (vb / es) * 4 < 16 ? (vb / es) * 4 : 16;
    if (c.a.past != nullptr && !aligned(c.a.past, vb)) return false;
    if (c.a.fresh != nullptr && !aligned(c.a.fresh, vb)) return false;
    if (c.a.sin_t != nullptr && (!aligned(c.a.sin_t, table_align) || !aligned(c.a.cos_t, table_align)))
        return false;
    return aligned(c.a.out, vb);
}

// Rows per CTA, or 0 if a row's heads need more than one CTA or the row count exceeds the
// kernel's 32-bit row arithmetic.
int64_t kv_cat_tpc(const KvCatCall& c, int vb, int hpt) {
    if (c.rows > 0xFFFFFFFFll) return 0;
    const int es = camp::elem_bytes(c.t);
    const int64_t per_row = ceil_div(c.a.heads, hpt) * (c.a.half * es / vb);
    return per_row <= camp::kRopeBlock ? camp::kRopeBlock / per_row : 0;
}

// Widest legal access; 2 heads per thread when the head count is even (each thread then
// issues 4 loads and 4 * n_rep stores), 1 for odd counts, more when a row's heads would not
// fit one CTA; CAMP_ERR_NOT_SUPPORTED when even 8 do not.
camp_status_t kv_cat_plan(const KvCatCall& c, const camp_plan_t* forced, camp_plan_t* p) {
    if (forced && forced->kernel != CAMP_KERNEL_KV_CAT) return CAMP_ERR_NOT_SUPPORTED;
    *p = camp_plan_t{};
    p->kernel = CAMP_KERNEL_KV_CAT;
    p->cluster = 1;
    p->block = camp::kRopeBlock;
    if (forced) {
        p->vec_bytes = forced->vec_bytes;
        p->group = forced->group;
        if (!kv_cat_vec_ok(c, p->vec_bytes)) return CAMP_ERR_NOT_SUPPORTED;
    } else {
        for (int vb : {16, 8, 4, 2}) {
            if (kv_cat_vec_ok(c, vb)) { p->vec_bytes = vb; break; }
        }
        p->group = c.a.heads % 2 == 0 ? 2 : 1;
        while (p->group < 8 && kv_cat_tpc(c, p->vec_bytes, p->group) == 0) p->group *= 2;
        // The rotate-half planner's fill rule (fewer than kRopeFillCtas CTAs: the variant
        // with the smallest grid of at least that many).
        const int64_t t0 = kv_cat_tpc(c, p->vec_bytes, p->group);
        if (t0 > 0 && ceil_div(c.rows, t0) < kRopeFillCtas) {
            int64_t best = 0;
            for (int vb : {16, 8, 4, 2}) {
                if (!kv_cat_vec_ok(c, vb)) continue;
                for (int hpt : {1, 2, 4, 8}) {
                    const int64_t tpc =
                        camp::kv_cat_compiled(c.t, vb, hpt) ? kv_cat_tpc(c, vb, hpt) : 0;
                    if (tpc == 0) continue;
                    const int64_t g = ceil_div(c.rows, tpc);
                    if (g >= kRopeFillCtas && (best == 0 || g < best)) {
                        best = g;
                        p->vec_bytes = vb;
                        p->group = hpt;
                    }
                }
            }
        }
    }
    if (!camp::kv_cat_compiled(c.t, p->vec_bytes, p->group)) return CAMP_ERR_NOT_SUPPORTED;
    const int64_t tpc = kv_cat_tpc(c, p->vec_bytes, p->group);
    if (tpc == 0) return CAMP_ERR_NOT_SUPPORTED;
    p->grid = ceil_div(c.rows, tpc);
    return CAMP_SUCCESS;
}

// ------------------------------------------------------------------ LayerNorm

struct LnCall {
    RmsCall rc;          // x, w = gamma, y, sizes: planned like the RMSNorm rows kernel
    const void* beta;
};

camp_status_t ln_validate(const void* x, const void* gamma, const void* beta, const void* y,
                          int64_t rows, int64_t cols, camp_dtype_t dtype, LnCall* c,
                          bool* empty) {
    camp_status_t st = rms_validate(x, gamma, y, rows, cols, dtype, &c->rc, empty);
    if (st != CAMP_SUCCESS || *empty) return st;
    if (beta == nullptr) return CAMP_ERR_INVALID_ARG;
    const int64_t es = camp::elem_bytes(c->rc.t);
    if (!aligned(beta, es)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(y, c->rc.bytes, beta, cols * es)) return CAMP_ERR_INVALID_ARG;
    c->beta = beta;
    return CAMP_SUCCESS;
}

// Staged LayerNorm: chunk vectors per CTA and whether gamma, beta and the ring fit shared
// memory, for `rps` rows a step (chunks of at most 8 vectors a thread with one row a step,
// 4 with two).
bool ln_staged_fits(int64_t nvec, int cluster, int stages, int rps, int64_t* chunk) {
    if (cluster < 1 || cluster > 16 || (cluster & (cluster - 1)) != 0) return false;
    if (rps < 1 || rps > camp::kLnStagedMaxRowsPerStep) return false;
    if (stages < rps || stages < 2 || stages > camp::kStagedMaxStages) return false;
    *chunk = ceil_div(nvec, cluster);
    const int64_t max_chunk =
        static_cast<int64_t>(camp::kStagedMaxVecsPerThread / rps) * camp::kStagedBlock;
    return *chunk <= max_chunk &&
           camp::ln_staged_smem_bytes(*chunk, stages) <= camp::kStagedSmemMax;
}

void ln_staged_plan_fields(const LnCall& c, int cluster, int stages, int rps, int64_t chunk,
                           camp_plan_t* p) {
    p->kernel = CAMP_KERNEL_LAYERNORM_STAGED;
    p->vec_bytes = 16;
    p->group = static_cast<int32_t>(chunk);
    p->per_thread = stages;
    p->rows_per_step = rps;
    p->block = camp::kStagedBlock;
    p->cluster = cluster;
    const int64_t per_sm = camp::kSmSmemBytes / (camp::ln_staged_smem_bytes(chunk, stages) + 1024);
    int64_t clusters = (camp::kSmCount * (per_sm < 1 ? 1 : per_sm)) / cluster;
    if (clusters < 1) clusters = 1;
    if (clusters > c.rc.a.rows) clusters = c.rc.a.rows;
    p->grid = clusters * cluster;
}

// Rows of more than kLnStagedFrom 16-byte vectors, and rows of more than kLnStagedFewFrom
// vectors when there are at most kLnFewRows of them, take the staged kernel. In fp32 storage,
// where a cluster of at most kLnPairsMaxCluster CTAs gives chunks of at most kLnStagedChunk2
// vectors (4 a thread), it takes two rows a step with 2 buffers; otherwise (and always in
// 16-bit storage) one row a step, 2 buffers, and the smallest power-of-two cluster whose
// chunks hold at most kLnStagedChunk vectors (8 a thread). Measured on GB300 (L2-cold, graphs
// of back-to-back launches, of the measured HBM peak), fp32, two rows a step against the
// one-row rule: 1024 x 32768 0.745 / 0.661, 2048 x 32768 0.794 / 0.729, 512 x 32768 0.682 /
// 0.646, 1024 x 16384 0.754 / 0.709; with a cluster of 16 it loses (256 x 65536: 0.621 /
// 0.645), and in 16-bit storage it loses everywhere measured (bf16 1024 x 65536: 0.58 /
// 0.63 at its best cluster). The one-row rule with 2048-vector chunks is the measured best
// of every cluster and buffer count at bf16 1024 x 65536 (0.63), 2048 x 65536 (0.70),
// 256 x 131072 (0.59), 512 x 131072 (0.64), 64 x 262144 (0.50), 1024 x 32768 (0.63), 2048
// x 32768 (0.77), 2048 x 16384 (0.83), fp16 1024 x 65536 (0.65) or within 0.02 of it.
constexpr int64_t kLnStagedFrom = 4096;
constexpr int64_t kLnStagedFewFrom = 2048;
constexpr int64_t kLnFewRows = 1024;
constexpr int64_t kLnStagedChunk = 2048;
constexpr int64_t kLnStagedChunk2 = 1024;
constexpr int kLnPairsMaxCluster = 8;

bool ln_choose_staged(int64_t nvec, int es, int* cluster, int* stages, int* rps,
                      int64_t* chunk) {
    for (int cl = 1; cl <= kLnPairsMaxCluster && es == 4; cl *= 2) {
        if (ceil_div(nvec, cl) <= kLnStagedChunk2 && ln_staged_fits(nvec, cl, 2, 2, chunk)) {
            *cluster = cl;
            *stages = 2;
            *rps = 2;
            return true;
        }
    }
    for (int cl = 1; cl <= 16; cl *= 2) {
        if (ceil_div(nvec, cl) <= kLnStagedChunk && ln_staged_fits(nvec, cl, 2, 1, chunk)) {
            *cluster = cl;
            *stages = 2;
            *rps = 1;
            return true;
        }
    }
    return false;
}

// The share of the staged kernel's per-thread vector slots a chunk fills: its launcher gives
// each thread 1, 2, 4 or 8 vectors, the fewest that hold the chunk. In fp32 storage (16-bit
// rows take the spread kernel in any case, see ln_plan), below kLnStagedMinFill the spread
// kernel takes the row, if its own chunks hold at least kLnSpreadMinChunk vectors (its
// per-row cost of two cluster exchanges and three sweeps over shared memory pays off only
// over long chunks). Measured on GB300 (L2-cold, graphs of back-to-back launches, of the
// measured HBM peak), fp32, staged against spread: 512 x 70000 (chunks of 1094 vectors, 8 a
// thread: 0.53 full) 0.54 / 0.60, 1024 x 40000 (0.61) 0.71 / 0.73; with a short spread chunk
// the staged kernel keeps the row (1024 x 12288: 768 of 1024 slots against one CTA of 3072,
// 0.70 / 0.53), and at full chunks it wins (1024 x 32768 0.85 / 0.72).
constexpr double kLnStagedMinFill = 0.8;
constexpr int64_t kLnSpreadMinChunk = 4096;

double ln_staged_fill(int64_t chunk) {
    const int64_t need = ceil_div(chunk, camp::kStagedBlock);
    const int64_t nvt = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
    return static_cast<double>(chunk) / static_cast<double>(nvt * camp::kStagedBlock);
}

// The wide kernel: one CTA of kWideBlock threads per row (at most kMaxGrid CTAs, each then
// taking every grid-th row).
void ln_wide_plan_fields(const LnCall& c, int vec_bytes, camp_plan_t* p) {
    p->kernel = CAMP_KERNEL_LAYERNORM_WIDE;
    p->vec_bytes = vec_bytes;
    p->group = camp::kWideBlock;
    p->per_thread = 0;
    p->block = camp::kWideBlock;
    p->cluster = 1;
    p->grid = c.rc.a.rows < kMaxGrid ? c.rc.a.rows : kMaxGrid;
}

// The staged kernel's plan for these arguments, whichever kernel camp_layernorm takes:
// 16-byte pitches and pointers, rows past kLnStagedFrom vectors (kLnStagedFewFrom with at
// most kLnFewRows rows) that a cluster of 16 holds. False if the staged kernel cannot.
bool ln_staged_plan_for(const LnCall& c, camp_plan_t* p) {
    const RmsCall& rc = c.rc;
    const int es = camp::elem_bytes(rc.t);
    if (rms_vec_bytes(rc) != 16 || !aligned(c.beta, 16)) return false;
    const int64_t nvec16 = rc.a.cols * es / 16;
    if (!(nvec16 > kLnStagedFrom || (nvec16 > kLnStagedFewFrom && rc.a.rows <= kLnFewRows)))
        return false;
    int cl = 0, st = 0, rps = 0;
    int64_t chunk = 0;
    if (!ln_choose_staged(nvec16, es, &cl, &st, &rps, &chunk)) return false;
    *p = camp_plan_t{};
    ln_staged_plan_fields(c, cl, st, rps, chunk, p);
    return true;
}

camp_status_t ln_plan(const LnCall& c, const camp_plan_t* forced, camp_plan_t* p) {
    if (forced && forced->kernel != CAMP_KERNEL_LAYERNORM_ROWS &&
        forced->kernel != CAMP_KERNEL_LAYERNORM_STAGED &&
        forced->kernel != CAMP_KERNEL_LAYERNORM_WIDE &&
        forced->kernel != CAMP_KERNEL_LAYERNORM_SPREAD)
        return CAMP_ERR_NOT_SUPPORTED;
    const RmsCall& rc = c.rc;
    const int es = camp::elem_bytes(rc.t);
    const int widest = (rms_vec_bytes(rc) == 16 && aligned(c.beta, 16)) ? 16 : es;
    *p = camp_plan_t{};
    p->kernel = CAMP_KERNEL_LAYERNORM_ROWS;
    p->cluster = 1;
    const int64_t nvec16 = rc.a.cols * es / 16;
    const int ln_per_sm = camp::spread_ctas_per_sm(true, es);
    if (forced && forced->kernel == CAMP_KERNEL_LAYERNORM_SPREAD) {
        int64_t chunk = 0;
        if (widest != 16 || !spread_fits(nvec16, forced->cluster, forced->per_thread, &chunk))
            return CAMP_ERR_NOT_SUPPORTED;
        spread_plan_fields(rc.a.rows, CAMP_KERNEL_LAYERNORM_SPREAD, ln_per_sm, forced->cluster,
                           forced->per_thread, chunk, p);
        return CAMP_SUCCESS;
    }
    if (forced && forced->kernel == CAMP_KERNEL_LAYERNORM_WIDE) {
        const int vb = forced->vec_bytes;
        if ((vb != 16 && vb != es) || vb > widest || !camp::layernorm_wide_compiled(rc.t, vb))
            return CAMP_ERR_NOT_SUPPORTED;
        ln_wide_plan_fields(c, vb, p);
        return CAMP_SUCCESS;
    }
    if (forced && forced->kernel == CAMP_KERNEL_LAYERNORM_STAGED) {
        int64_t chunk = 0;
        const int rps = forced->rows_per_step == 0 ? 1 : forced->rows_per_step;
        if (widest != 16 ||
            !ln_staged_fits(nvec16, forced->cluster, forced->per_thread, rps, &chunk))
            return CAMP_ERR_NOT_SUPPORTED;
        ln_staged_plan_fields(c, forced->cluster, forced->per_thread, rps, chunk, p);
        return CAMP_SUCCESS;
    }
    if (forced) {
        p->vec_bytes = forced->vec_bytes;
        p->group = forced->group;
        p->per_thread = forced->per_thread;
        if (p->vec_bytes != 16 && p->vec_bytes != es) return CAMP_ERR_NOT_SUPPORTED;
        if (p->vec_bytes > widest) return CAMP_ERR_NOT_SUPPORTED;
        if (!camp::rmsnorm_rows_compiled(false, rc.t, p->vec_bytes, p->group, p->per_thread))
            return CAMP_ERR_NOT_SUPPORTED;   // the same variant set
        const int64_t nvec = rc.a.cols * es / p->vec_bytes;
        if (static_cast<int64_t>(p->group) * p->per_thread < nvec) return CAMP_ERR_NOT_SUPPORTED;
    } else {
        if (widest == 16 && (nvec16 > kLnStagedFrom ||
                             (nvec16 > kLnStagedFewFrom && rc.a.rows <= kLnFewRows))) {
            int cl = 0, st = 0, rps = 0;
            int64_t chunk = 0;
            // 16-bit storage: the spread kernel, three CTAs an SM with whole chunks in shared
            // memory. Against the staged kernel (GB300, graphs of back-to-back launches,
            // L2-cold, of the measured HBM peak) it was as fast within 0.01 or faster at 20
            // of 22 shapes: bf16 1024 x 65536 0.75 / 0.66, 2048 x 65536 0.80 / 0.71, 4096 x
            // 36864 0.80 / 0.65, 512 x 140000 0.67 / 0.46, fp16 1024 x 65536 0.72 / 0.68;
            // slower only at 16 and 64 rows of 262144 (0.33 / 0.35, 0.49 / 0.51).
            if (es == 2 && spread_choose(nvec16, rc.a.rows, ln_per_sm, &cl, &st, &chunk)) {
                spread_plan_fields(rc.a.rows, CAMP_KERNEL_LAYERNORM_SPREAD, ln_per_sm, cl, st,
                                   chunk, p);
                return CAMP_SUCCESS;
            }
            if (ln_choose_staged(nvec16, es, &cl, &st, &rps, &chunk)) {
                int scl = 0, sst = 0;
                int64_t schunk = 0;
                if (ln_staged_fill(chunk) < kLnStagedMinFill &&
                    spread_choose(nvec16, rc.a.rows, ln_per_sm, &scl, &sst, &schunk) &&
                    schunk >= kLnSpreadMinChunk) {
                    spread_plan_fields(rc.a.rows, CAMP_KERNEL_LAYERNORM_SPREAD, ln_per_sm, scl, sst, schunk,
                                       p);
                    return CAMP_SUCCESS;
                }
                ln_staged_plan_fields(c, cl, st, rps, chunk, p);
                return CAMP_SUCCESS;
            }
            if (spread_choose(nvec16, rc.a.rows, ln_per_sm, &cl, &st, &chunk)) {   // past the staged kernel
                spread_plan_fields(rc.a.rows, CAMP_KERNEL_LAYERNORM_SPREAD, ln_per_sm, cl, st,
                                   chunk, p);
                return CAMP_SUCCESS;
            }
        }
        p->vec_bytes = widest;
        int g = 0, nv = 0;
        if (!rms_choose_rows(rc, widest, &g, &nv, true)) {
            ln_wide_plan_fields(c, widest, p);   // no register or staged kernel holds the row
            return CAMP_SUCCESS;
        }
        p->group = g;
        p->per_thread = nv;
    }
    p->block = camp::rows_block(p->group);
    p->grid = ceil_div(rc.a.rows, p->block / p->group);
    return CAMP_SUCCESS;
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

CAMP_API camp_status_t camp_device_errors(uint32_t* flags, int clear) {
    if (flags == nullptr) return CAMP_ERR_INVALID_ARG;
    unsigned int a = 0, b = 0, d = 0;
    camp_status_t st = runtime_status(camp::read_device_errors(&a, clear != 0));
    if (st == CAMP_SUCCESS) st = runtime_status(camp::read_layernorm_device_errors(&b, clear != 0));
    if (st == CAMP_SUCCESS) st = runtime_status(camp::read_spread_device_errors(&d, clear != 0));
    *flags = st == CAMP_SUCCESS ? (a | b | d) : 0u;
    return st;
}

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

CAMP_API camp_status_t camp_add_rmsnorm(const void* x, const void* r, const void* w, void* h,
                                        void* y, int64_t rows, int64_t cols, float eps,
                                        camp_dtype_t dtype, void* stream) {
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_add_validate(x, r, w, h, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps)) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    c.a.eps = eps;
    camp_plan_t p;
    rms_plan(c, &p);
    return rms_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_add_rmsnorm_plan(const void* x, const void* r, const void* w,
                                             const void* h, const void* y, int64_t rows,
                                             int64_t cols, camp_dtype_t dtype,
                                             camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_add_validate(x, r, w, h, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    rms_plan(c, plan);
    return CAMP_SUCCESS;
}

CAMP_API camp_status_t camp_add_rmsnorm_with_plan(const void* x, const void* r, const void* w,
                                                  void* h, void* y, int64_t rows, int64_t cols,
                                                  float eps, camp_dtype_t dtype,
                                                  const camp_plan_t* plan, void* stream) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_add_validate(x, r, w, h, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps)) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    c.a.eps = eps;
    camp_plan_t p;
    st = rms_accept_plan(c, *plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return rms_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_kv_rmsnorm_rope_cache_plan(
    const void* kv, const void* gamma, const float* sin, const float* cos, const int64_t* slots,
    const void* cache_n, const void* cache_r, int64_t B, int64_t S, int64_t Dn, int64_t Dr,
    int64_t num_slots, camp_dtype_t dtype, camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    KvCall c;
    bool empty = false;
    camp_status_t st = kv_validate(kv, gamma, sin, cos, slots, cache_n, cache_r, B, S, Dn, Dr,
                                   num_slots, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    return kv_plan(c, nullptr, plan);
}

CAMP_API camp_status_t camp_kv_rmsnorm_rope_cache_with_plan(
    const void* kv, const void* gamma, const float* sin, const float* cos, const int64_t* slots,
    void* cache_n, void* cache_r, int64_t B, int64_t S, int64_t Dn, int64_t Dr,
    int64_t num_slots, float eps, camp_dtype_t dtype, const camp_plan_t* plan, void* stream) {
    KvCall c;
    bool empty = false;
    camp_status_t st = kv_validate(kv, gamma, sin, cos, slots, cache_n, cache_r, B, S, Dn, Dr,
                                   num_slots, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps)) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    c.a.eps = eps;
    camp_plan_t p;
    st = kv_plan(c, plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return runtime_status(camp::kv_cache_launch(c.t, p.vec_bytes, p.per_thread, p.group, c.a,
                                                static_cast<cudaStream_t>(stream)));
}

CAMP_API camp_status_t camp_kv_rmsnorm_rope_cache(
    const void* kv, const void* gamma, const float* sin, const float* cos, const int64_t* slots,
    void* cache_n, void* cache_r, int64_t B, int64_t S, int64_t Dn, int64_t Dr,
    int64_t num_slots, float eps, camp_dtype_t dtype, void* stream) {
    return camp_kv_rmsnorm_rope_cache_with_plan(kv, gamma, sin, cos, slots, cache_n, cache_r,
                                                B, S, Dn, Dr, num_slots, eps, dtype, nullptr,
                                                stream);
}

CAMP_API camp_status_t camp_rope_interleaved_plan(const void* x, const float* sin,
                                                  const float* cos, const int32_t* positions,
                                                  const void* y, int64_t tokens, int64_t H,
                                                  int64_t D, int64_t max_pos, camp_dtype_t dtype,
                                                  camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RopeIlCall c;
    bool empty = false;
    camp_status_t st = rope_il_validate(x, sin, cos, positions, y, tokens, H, D, max_pos, dtype,
                                        &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    return rope_il_plan(c, nullptr, plan);
}

CAMP_API camp_status_t camp_rope_interleaved_with_plan(const void* x, const float* sin,
                                                       const float* cos,
                                                       const int32_t* positions, void* y,
                                                       int64_t tokens, int64_t H, int64_t D,
                                                       int64_t max_pos, camp_dtype_t dtype,
                                                       const camp_plan_t* plan, void* stream) {
    RopeIlCall c;
    bool empty = false;
    camp_status_t st = rope_il_validate(x, sin, cos, positions, y, tokens, H, D, max_pos, dtype,
                                        &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    st = rope_il_plan(c, plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return runtime_status(camp::rope_interleaved_launch(c.t, p.vec_bytes, p.group, c.a, p.grid,
                                                        static_cast<cudaStream_t>(stream)));
}

CAMP_API camp_status_t camp_rope_interleaved(const void* x, const float* sin, const float* cos,
                                             const int32_t* positions, void* y, int64_t tokens,
                                             int64_t H, int64_t D, int64_t max_pos,
                                             camp_dtype_t dtype, void* stream) {
    return camp_rope_interleaved_with_plan(x, sin, cos, positions, y, tokens, H, D, max_pos,
                                           dtype, nullptr, stream);
}

CAMP_API camp_status_t camp_kv_cat_repeat_plan(const void* past, const void* fresh,
                                               const float* sin, const float* cos,
                                               const void* out, int64_t B, int64_t P, int64_t S,
                                               int64_t Hk, int64_t D, int64_t n_rep,
                                               camp_dtype_t dtype, camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    KvCatCall c;
    bool empty = false;
    camp_status_t st = kv_cat_validate(past, fresh, sin, cos, out, B, P, S, Hk, D, n_rep, dtype,
                                       &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    return kv_cat_plan(c, nullptr, plan);
}

CAMP_API camp_status_t camp_kv_cat_repeat_with_plan(const void* past, const void* fresh,
                                                    const float* sin, const float* cos,
                                                    void* out, int64_t B, int64_t P, int64_t S,
                                                    int64_t Hk, int64_t D, int64_t n_rep,
                                                    camp_dtype_t dtype, const camp_plan_t* plan,
                                                    void* stream) {
    KvCatCall c;
    bool empty = false;
    camp_status_t st = kv_cat_validate(past, fresh, sin, cos, out, B, P, S, Hk, D, n_rep, dtype,
                                       &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    st = kv_cat_plan(c, plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return runtime_status(camp::kv_cat_launch(c.t, p.vec_bytes, p.group, c.a, p.grid,
                                              static_cast<cudaStream_t>(stream)));
}

CAMP_API camp_status_t camp_kv_cat_repeat(const void* past, const void* fresh, const float* sin,
                                          const float* cos, void* out, int64_t B, int64_t P,
                                          int64_t S, int64_t Hk, int64_t D, int64_t n_rep,
                                          camp_dtype_t dtype, void* stream) {
    return camp_kv_cat_repeat_with_plan(past, fresh, sin, cos, out, B, P, S, Hk, D, n_rep, dtype,
                                        nullptr, stream);
}

CAMP_API camp_status_t camp_rope_tables(float* sin, float* cos, int64_t max_pos, int64_t D,
                                        double theta, void* stream) {
    if (max_pos < 0 || D < 2 || D % 2 != 0 || !std::isfinite(theta) || !(theta > 0.0))
        return CAMP_ERR_INVALID_ARG;
    if (max_pos == 0) return CAMP_SUCCESS;
    if (sin == nullptr || cos == nullptr || !aligned(sin, 4) || !aligned(cos, 4))
        return CAMP_ERR_INVALID_ARG;
    int64_t table_bytes = 0;
    if (!mul_ok(max_pos, D / 2, 4, &table_bytes)) return CAMP_ERR_INVALID_ARG;
    if (overlaps(sin, table_bytes, cos, table_bytes)) return CAMP_ERR_INVALID_ARG;
    return runtime_status(camp::rope_tables_launch(sin, cos, max_pos, D, theta,
                                                   static_cast<cudaStream_t>(stream)));
}

CAMP_API camp_status_t camp_layernorm_plan(const void* x, const void* gamma, const void* beta,
                                           const void* y, int64_t rows, int64_t cols,
                                           camp_dtype_t dtype, camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    LnCall c;
    bool empty = false;
    camp_status_t st = ln_validate(x, gamma, beta, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    return ln_plan(c, nullptr, plan);
}

CAMP_API camp_status_t camp_layernorm_with_plan(const void* x, const void* gamma,
                                                const void* beta, void* y, int64_t rows,
                                                int64_t cols, float eps, camp_dtype_t dtype,
                                                const camp_plan_t* plan, void* stream) {
    LnCall c;
    bool empty = false;
    camp_status_t st = ln_validate(x, gamma, beta, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps)) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    camp_plan_t p;
    st = ln_plan(c, plan, &p);
    if (st != CAMP_SUCCESS) return st;
    const camp::LayernormArgs a{x, gamma, c.beta, y, rows, cols, eps};
    if (p.kernel == CAMP_KERNEL_LAYERNORM_STAGED)
        return runtime_status(camp::layernorm_staged_launch(c.rc.t, p.cluster, p.per_thread,
                                                            p.rows_per_step, a,
                                                            static_cast<cudaStream_t>(stream)));
    if (p.kernel == CAMP_KERNEL_LAYERNORM_WIDE)
        return runtime_status(camp::layernorm_wide_launch(c.rc.t, p.vec_bytes, a, p.grid,
                                                          static_cast<cudaStream_t>(stream)));
    if (p.kernel == CAMP_KERNEL_LAYERNORM_SPREAD)
        return runtime_status(camp::layernorm_spread_launch(c.rc.t, p.cluster, p.per_thread, a,
                                                            static_cast<cudaStream_t>(stream)));
    return runtime_status(camp::layernorm_rows_launch(c.rc.t, p.vec_bytes, p.group,
                                                      p.per_thread, a, p.grid,
                                                      static_cast<cudaStream_t>(stream)));
}

CAMP_API camp_status_t camp_layernorm(const void* x, const void* gamma, const void* beta,
                                      void* y, int64_t rows, int64_t cols, float eps,
                                      camp_dtype_t dtype, void* stream) {
    return camp_layernorm_with_plan(x, gamma, beta, y, rows, cols, eps, dtype, nullptr, stream);
}

CAMP_API camp_status_t camp_rmsnorm_wait_probe(const void* x, const void* w, void* y,
                                               int64_t rows, int64_t cols, float eps,
                                               camp_dtype_t dtype, const camp_plan_t* plan,
                                               uint64_t wait_ns, void* stream) {
    RmsCall c;
    bool empty = false;
    camp_status_t st = rms_validate(x, w, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps) || wait_ns < 1000 || wait_ns > 1000000000ull) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    c.a.eps = eps;
    camp_plan_t p;
    if (plan != nullptr) {
        if (plan->kernel != CAMP_KERNEL_RMSNORM_STAGED &&
            plan->kernel != CAMP_KERNEL_RMSNORM_SPREAD)
            return CAMP_ERR_NOT_SUPPORTED;
        st = rms_accept_plan(c, *plan, &p);
        if (st != CAMP_SUCCESS) return st;
    } else {
        // The staged kernel's plan for these arguments, whichever kernel camp_rmsnorm takes.
        const int64_t nvec = cols * camp::elem_bytes(c.t) / 16;
        int cl = 0, stg = 0;
        int64_t chunk = 0;
        if (rms_vec_bytes(c) != 16 || nvec <= kStagedFrom ||
            !rms_choose_staged(c, nvec, &cl, &stg, &chunk))
            return CAMP_ERR_NOT_SUPPORTED;
        p = camp_plan_t{};
        rms_staged_plan_fields(c, cl, stg, chunk, &p);
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.kernel == CAMP_KERNEL_RMSNORM_SPREAD)
        return runtime_status(
            camp::rmsnorm_spread_launch(false, c.t, p.cluster, p.per_thread, c.a, s, wait_ns, 1));
    return runtime_status(
        camp::rmsnorm_staged_launch(false, c.t, p.cluster, p.per_thread, c.a, s, wait_ns, 1));
}

CAMP_API camp_status_t camp_layernorm_wait_probe(const void* x, const void* gamma,
                                                 const void* beta, void* y, int64_t rows,
                                                 int64_t cols, float eps, camp_dtype_t dtype,
                                                 const camp_plan_t* plan, uint64_t wait_ns,
                                                 void* stream) {
    LnCall c;
    bool empty = false;
    camp_status_t st = ln_validate(x, gamma, beta, y, rows, cols, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (!eps_ok(eps) || wait_ns < 1000 || wait_ns > 1000000000ull) return CAMP_ERR_INVALID_ARG;
    if (empty) return CAMP_SUCCESS;
    camp_plan_t p;
    if (plan != nullptr) {
        if (plan->kernel != CAMP_KERNEL_LAYERNORM_STAGED &&
            plan->kernel != CAMP_KERNEL_LAYERNORM_SPREAD)
            return CAMP_ERR_NOT_SUPPORTED;
        st = ln_plan(c, plan, &p);
        if (st != CAMP_SUCCESS) return st;
    } else if (!ln_staged_plan_for(c, &p)) {
        return CAMP_ERR_NOT_SUPPORTED;
    }
    const camp::LayernormArgs a{x, gamma, c.beta, y, rows, cols, eps};
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.kernel == CAMP_KERNEL_LAYERNORM_SPREAD)
        return runtime_status(
            camp::layernorm_spread_launch(c.rc.t, p.cluster, p.per_thread, a, s, wait_ns, 1));
    return runtime_status(camp::layernorm_staged_launch(c.rc.t, p.cluster, p.per_thread,
                                                        p.rows_per_step, a, s, wait_ns, 1));
}

CAMP_API camp_status_t camp_rope(const void* x, const float* sin, const float* cos, void* y,
                                 int64_t B, int64_t S, int64_t H, int64_t D,
                                 camp_dtype_t dtype, void* stream) {
    RopeCall c;
    bool empty = false;
    camp_status_t st =
        rope_validate(x, nullptr, sin, cos, y, nullptr, B, S, H, 0, D, dtype, &c, &empty);
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
    camp_status_t st =
        rope_validate(x, nullptr, sin, cos, y, nullptr, B, S, H, 0, D, dtype, &c, &empty);
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
    camp_status_t st =
        rope_validate(x, nullptr, sin, cos, y, nullptr, B, S, H, 0, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    st = rope_accept_plan(c, *plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return rope_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_rope_qk(const void* q, const void* k, const float* sin,
                                    const float* cos, void* yq, void* yk, int64_t B, int64_t S,
                                    int64_t Hq, int64_t Hk, int64_t D, camp_dtype_t dtype,
                                    void* stream) {
    RopeCall c;
    bool empty = false;
    camp_status_t st = rope_validate(q, k, sin, cos, yq, yk, B, S, Hq, Hk, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    rope_plan(c, &p);
    return rope_launch(c, p, static_cast<cudaStream_t>(stream));
}

CAMP_API camp_status_t camp_rope_qk_plan(const void* q, const void* k, const float* sin,
                                         const float* cos, const void* yq, const void* yk,
                                         int64_t B, int64_t S, int64_t Hq, int64_t Hk,
                                         int64_t D, camp_dtype_t dtype, camp_plan_t* plan) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RopeCall c;
    bool empty = false;
    camp_status_t st = rope_validate(q, k, sin, cos, yq, yk, B, S, Hq, Hk, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS) return st;
    if (empty) { *plan = camp_plan_t{}; return CAMP_SUCCESS; }
    rope_plan(c, plan);
    return CAMP_SUCCESS;
}

CAMP_API camp_status_t camp_rope_qk_with_plan(const void* q, const void* k, const float* sin,
                                              const float* cos, void* yq, void* yk, int64_t B,
                                              int64_t S, int64_t Hq, int64_t Hk, int64_t D,
                                              camp_dtype_t dtype, const camp_plan_t* plan,
                                              void* stream) {
    if (plan == nullptr) return CAMP_ERR_INVALID_ARG;
    RopeCall c;
    bool empty = false;
    camp_status_t st = rope_validate(q, k, sin, cos, yq, yk, B, S, Hq, Hk, D, dtype, &c, &empty);
    if (st != CAMP_SUCCESS || empty) return st;
    camp_plan_t p;
    st = rope_accept_plan(c, *plan, &p);
    if (st != CAMP_SUCCESS) return st;
    return rope_launch(c, p, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
