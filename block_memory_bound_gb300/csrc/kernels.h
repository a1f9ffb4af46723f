// Internal interface between the C ABI (camp_abi.cu) and the kernel translation units.
// Host-only declarations; no CUDA types beyond cudaStream_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace camp {

enum class DType : int { F32 = 1, BF16 = 3 };

inline int elem_bytes(DType t) { return t == DType::BF16 ? 2 : 4; }

struct RmsnormArgs {
    const void* x;
    const void* w;
    void* y;
    int64_t rows;
    int64_t cols;
    float eps;
};

struct RopeArgs {
    const void* x;
    const float* sin_t;
    const float* cos_t;
    void* y;
    int64_t tokens;   // B * S
    int64_t seq;      // S
    int64_t heads;    // H
    int64_t half;     // D / 2
};

// Register-resident RMSNorm: `group` threads per row, `per_thread` vector accesses of
// `vec_bytes` each. Returns false (launching nothing) if that variant is not compiled.
bool rmsnorm_rows_compiled(DType t, int vec_bytes, int group, int per_thread);
bool rmsnorm_rows_launch(DType t, int vec_bytes, int group, int per_thread,
                         const RmsnormArgs& a, int64_t grid, int block, cudaStream_t s);
int rmsnorm_rows_block(int group);   // threads per CTA of a group size

// Two-sweep RMSNorm for rows too wide for registers: one CTA of kWideBlock threads per row.
constexpr int kWideBlock = 1024;
bool rmsnorm_wide_compiled(DType t, int vec_bytes);
bool rmsnorm_wide_launch(DType t, int vec_bytes, const RmsnormArgs& a, int64_t grid,
                         cudaStream_t s);

// Rotate-half RoPE: one thread per (position, head group, vector of the half-row).
constexpr int kRopeBlock = 256;
bool rope_compiled(DType t, int vec_bytes, int heads_per_thread);
bool rope_launch(DType t, int vec_bytes, int heads_per_thread, const RopeArgs& a,
                 int64_t grid, cudaStream_t s);

}  // namespace camp
