// Internal interface between the C ABI (camp_abi.cu) and the kernel translation units,
// and the compile-time occupancy rules that both the kernels' launch bounds and the
// host-side planner use. Host-only declarations; no CUDA types beyond cudaStream_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace camp {

enum class DType : int { F16 = 0, F32 = 1, BF16 = 3 };

inline int elem_bytes(DType t) { return t == DType::F32 ? 4 : 2; }

// The planner sizes grids for GB300's 152 SMs; any other SM count only changes how well
// the last wave is filled, never the result.
constexpr int kSmCount = 152;

// RMSNorm of x, or (add path) of h = x + r, which is also stored.
struct RmsnormArgs {
    const void* x;
    const void* w;
    void* y;
    int64_t rows;
    int64_t cols;
    float eps;
    const void* r = nullptr;   // add path: the residual
    void* h = nullptr;         // add path: h = x + r, rounded once to the storage type
};

// One or two tensors of the same [B, S, *, D] layout rotated by the same tables: the
// first with `heads` heads, the second (Q and K of one layer, say) with `heads2` heads;
// heads2 == 0 means a single tensor.
struct RopeArgs {
    const void* x;
    const float* sin_t;
    const float* cos_t;
    void* y;
    int64_t tokens;   // B * S
    int64_t seq;      // S
    int64_t heads;    // H of the first tensor
    int64_t half;     // D / 2
    const void* x2 = nullptr;
    void* y2 = nullptr;
    int64_t heads2 = 0;
};

// ------------------------------------------------------------------ RMSNorm, registers
// A group of `group` threads owns a row; each thread holds `per_thread` vector accesses
// of `vec_bytes`. Each variant is compiled (via __launch_bounds__) to keep a fixed number
// of threads resident per SM, chosen from its data registers: the planner relies on it.

constexpr int rows_block(int group) { return group < 256 ? 256 : group; }

// `loads` raw accesses are live per thread at the peak: per_thread, or twice that on the
// add path (x and r are both in flight before h is formed). Threads per SM by the 32-bit
// registers of raw row data per thread: up to 8, a full SM (32 registers a thread); up to
// 16, a full SM as well for groups of at most 128 threads (checked with -Xptxas -v: those
// variants fit 32 registers without spilling; at 4096 x 2048 bf16 the 64 x 4 variant then
// runs in one wave and measured 4% faster than 128 x 2), else 1536; then 1024 and 512.
constexpr int rows_threads_per_sm(int vec_bytes, int loads, int group) {
    return (loads * (vec_bytes < 4 ? 1 : vec_bytes / 4)) <= 8 ? 2048
         : (loads * (vec_bytes < 4 ? 1 : vec_bytes / 4)) <= 16 ? (group <= 128 ? 2048 : 1536)
         : (loads * (vec_bytes < 4 ? 1 : vec_bytes / 4)) <= 32 ? 1024
         : 512;
}

constexpr int rows_min_blocks(int vec_bytes, int group, int loads) {
    return rows_threads_per_sm(vec_bytes, loads, group) / rows_block(group) < 1
               ? 1
               : rows_threads_per_sm(vec_bytes, loads, group) / rows_block(group);
}

// LayerNorm rows kernel occupancy (CTAs per SM). The LayerNorm passes keep the shift and
// the mean live beside the data, so the row kernels' 2048-thread budget for 16 words does
// not apply (those variants spill); threads per SM by 32-bit data registers are 2048 up to
// 8, 1536 up to 16, 1024 up to 32, else 512. For fp32 the deviations of the variance pass
// stay live into the output pass (the raw words are the values themselves), so the data
// counts twice. The one bf16 variant that does not fit 32 registers at two 1024-thread
// CTAs per SM (1024 x 2 accesses; the planner prefers 256 x 8 for the same rows) runs one
// CTA per SM instead of spilling.
constexpr int ln_min_blocks(int elem_bytes, int vec_bytes, int group, int per_thread) {
    const int per_load = vec_bytes < 4 ? 1 : vec_bytes / 4;
    int words = (elem_bytes == 4 ? 2 : 1) * per_thread * per_load;
    if (elem_bytes == 2 && group == 1024 && per_thread == 2) words += per_load;
    const int threads = words <= 8 ? 2048 : words <= 16 ? 1536 : words <= 32 ? 1024 : 512;
    return threads / rows_block(group) < 1 ? 1 : threads / rows_block(group);
}

// The add path keeps x and r in flight together; with 1024 threads (64 registers each) and
// 8 16-byte accesses that is 64 raw registers, which would spill, so that one variant is not built
// (the planner sends such rows to the cluster kernel).
constexpr bool rows_variant_compiled(bool add, int vec_bytes, int group, int per_thread) {
    return !(add && vec_bytes == 16 && group == 1024 && per_thread == 8);
}

// `add` selects the fused residual-add variants throughout.
bool rmsnorm_rows_compiled(bool add, DType t, int vec_bytes, int group, int per_thread);
cudaError_t rmsnorm_rows_launch(bool add, DType t, int vec_bytes, int group, int per_thread,
                                const RmsnormArgs& a, int64_t grid, cudaStream_t s);

// Cluster-per-row RMSNorm: a cluster of `cluster` CTAs (2..16) of kClusterBlock threads owns
// a row; each thread holds `per_thread` 16-byte accesses of the CTA's contiguous chunk.
constexpr int kClusterBlock = 256;
bool rmsnorm_cluster_compiled(DType t, int per_thread);
cudaError_t rmsnorm_cluster_launch(bool add, DType t, int per_thread, int cluster,
                                   const RmsnormArgs& a, cudaStream_t s);

// Two-sweep RMSNorm for rows too wide for registers: one CTA of kWideBlock threads per row.
constexpr int kWideBlock = 1024;
bool rmsnorm_wide_compiled(DType t, int vec_bytes);
cudaError_t rmsnorm_wide_launch(bool add, DType t, int vec_bytes, const RmsnormArgs& a,
                                int64_t grid, cudaStream_t s);

// TMA-staged RMSNorm (rows staged in shared memory by bulk asynchronous copies): persistent
// clusters of `cluster` (1..16) CTAs of kStagedBlock threads; each CTA owns a contiguous
// chunk of ceil(nvec / cluster) <= 8 * 256 16-byte vectors of every row of its cluster,
// holds its chunk of w, and keeps `stages` (2..kStagedMaxStages) row chunks in flight (x,
// and r on the add path). Needs 16-byte accesses (row pitch and pointers) and
// staged_smem_bytes(add, chunk, stages) <= kStagedSmemMax.
constexpr int kStagedBlock = 256;
constexpr int kStagedMaxStages = 4;
constexpr int kStagedMaxVecsPerThread = 8;   // a CTA chunk holds at most 8 * 256 vectors
constexpr int64_t kStagedSmemMax = 224 * 1024;   // dynamic shared memory per CTA
constexpr int64_t kSmSmemBytes = 228 * 1024;     // shared memory per SM
inline int64_t staged_smem_bytes(bool add, int64_t chunk_vecs, int stages) {
    return chunk_vecs * 16 * (1 + (add ? 2 : 1) * stages);   // w, then the row buffers
}
// `wait_ns` and `probe` as for layernorm_staged_launch (the probe: plain RMSNorm only).
cudaError_t rmsnorm_staged_launch(bool add, DType t, int cluster, int stages,
                                  const RmsnormArgs& a, cudaStream_t s,
                                  unsigned long long wait_ns = 1000000000ull, int probe = 0);

// Rows past the staged kernels' registers (spread.cu): clusters of `cluster` (1..16) CTAs of
// kSpreadBlock threads; each CTA keeps its whole chunk of ceil(nvec / cluster) 16-byte
// vectors of a row in shared memory (`stages` buffers of it, 1..kSpreadMaxStages), so x is
// read from HBM once. RMSNorm without the residual add, and LayerNorm; 16-byte accesses.
constexpr int kSpreadBlock = 512;
constexpr int kSpreadMaxStages = 3;
constexpr int kSpreadHeadBytes = 16 * (kSpreadBlock / 32);   // a row head copy a copy group
// CTAs an SM the launch bounds guarantee by registers (fp32 LayerNorm keeps more live than
// 40 registers hold without spilling); the plan's grid estimate counts no more resident
// CTAs than this.
constexpr int spread_ctas_per_sm(bool layernorm, int elem_bytes, bool add = false) {
    return (layernorm && elem_bytes == 4) || add ? 2 : 3;
}
// `staged`: tensors staged a row, 1 (x), or 2 (x and r) on RMSNorm's residual-add path.
inline int64_t spread_smem_bytes(int64_t chunk_vecs, int stages, int staged = 1) {
    return stages * (kSpreadHeadBytes + staged * chunk_vecs * 16);
}
cudaError_t rmsnorm_spread_launch(bool add, DType t, int cluster, int stages,
                                  const RmsnormArgs& a, cudaStream_t s,
                                  unsigned long long wait_ns = 1000000000ull, int probe = 0);
struct LayernormArgs;
// `wait_ns` bounds every mbarrier wait (one second in normal calls); `probe` != 0 leaves each
// CTA's first row copy unissued (the wait diagnostic), as for layernorm_staged_launch.
cudaError_t layernorm_spread_launch(DType t, int cluster, int stages, const LayernormArgs& a,
                                    cudaStream_t s, unsigned long long wait_ns = 1000000000ull,
                                    int probe = 0);

// The library's device error words (one per translation unit with bounded waits): kernels
// whose bounded waits ran out set bits in them; camp_device_errors reports their union.
constexpr unsigned int kDeviceErrorWaitTimeout = 1u;
cudaError_t read_device_errors(unsigned int* flags, bool clear);            // staged RMSNorm
cudaError_t read_layernorm_device_errors(unsigned int* flags, bool clear);  // staged LayerNorm
cudaError_t read_spread_device_errors(unsigned int* flags, bool clear);     // spread kernels

// The add-path tables live in their own translation unit (compiled in parallel).
namespace add_path {
cudaError_t rows_launch(DType t, int vec_bytes, int group, int per_thread, const RmsnormArgs& a,
                        int64_t grid, cudaStream_t s);
cudaError_t cluster_launch(DType t, int per_thread, int cluster, const RmsnormArgs& a,
                           cudaStream_t s);
cudaError_t wide_launch(DType t, int vec_bytes, const RmsnormArgs& a, int64_t grid,
                        cudaStream_t s);
}  // namespace add_path

// ------------------------------------------------------------------ RoPE
// Tiled: a CTA of kRopeBlock threads covers kRopeBlock / (threads per position)
// positions; thread (position, head group, vector j) rotates vector j of both halves for
// `heads_per_thread` heads, of the first or the second tensor. Needs
// (ceil(H / hpt) + ceil(H2 / hpt)) * (half / elems) <= kRopeBlock, fewer than 2^32
// positions, and H, H2, D/2 below 2^31.
// Flat: one work item per (position, head group, vector), one tensor, any shape.
constexpr int kRopeBlock = 256;

// CTAs per SM of the tiled RoPE kernel by heads per thread (each head holds two vectors
// and the thread the E sine and cosine values of its position). Two heads per thread fit
// 48 registers at 5 CTAs per SM without spilling (6 would spill); at 4096 positions of
// Q[32 heads] + K[8 heads] x 64 that measured 8.19 us against 8.34 us at 4 CTAs per SM.
constexpr int rope_min_blocks(int heads_per_thread) {
    return heads_per_thread <= 1 ? 6 : heads_per_thread <= 2 ? 5 : heads_per_thread <= 4 ? 3 : 2;
}

bool rope_compiled(DType t, int vec_bytes, int heads_per_thread);
cudaError_t rope_tiled_launch(DType t, int vec_bytes, int heads_per_thread, const RopeArgs& a,
                              int64_t grid, cudaStream_t s);
cudaError_t rope_flat_launch(DType t, int vec_bytes, int heads_per_thread, const RopeArgs& a,
                             int64_t grid, cudaStream_t s);

// ------------------------------------------------------------------ LayerNorm
// Register-resident rows kernel, the same (vec_bytes, group, per_thread) variants as the
// RMSNorm rows kernel; no cluster or two-sweep path.
struct LayernormArgs {
    const void* x;
    const void* gamma;
    const void* beta;
    void* y;
    int64_t rows;
    int64_t cols;
    float eps;
};

cudaError_t layernorm_rows_launch(DType t, int vec_bytes, int group, int per_thread,
                                  const LayernormArgs& a, int64_t grid, cudaStream_t s);

// Staged LayerNorm (layernorm_staged.cu): the staged RMSNorm kernel's persistent clusters,
// each row buffer carrying the row's first 16 bytes (the shift) ahead of the CTA's chunk;
// the CTA's chunks of gamma and beta are staged in shared memory too where that leaves
// three CTAs an SM (ln_staged_gamma_in_smem), else read through L1. A step takes
// `rows_per_step` (1 or 2) rows at once: one pair of block reductions and one cluster
// exchange for all of them. Chunks of at most kStagedMaxVecsPerThread * kStagedBlock
// vectors with one row a step, half that with two; `stages` >= rows_per_step buffers.
inline int64_t ln_staged_smem_bytes(int64_t chunk_vecs, int stages, bool gamma_in_smem) {
    return stages * (16 + chunk_vecs * 16) + (gamma_in_smem ? chunk_vecs * 32 : 0);
}
constexpr int64_t kLnGammaSmemMax = 75 * 1024;   // 3 CTAs an SM, with the static part
inline bool ln_staged_gamma_in_smem(int64_t chunk_vecs, int stages) {
    return chunk_vecs <= 4 * 256 && ln_staged_smem_bytes(chunk_vecs, stages, true) <= kLnGammaSmemMax;
}
inline int64_t ln_staged_smem_bytes(int64_t chunk_vecs, int stages) {
    return ln_staged_smem_bytes(chunk_vecs, stages, ln_staged_gamma_in_smem(chunk_vecs, stages));
}
constexpr int kLnStagedMaxRowsPerStep = 2;
// `wait_ns` bounds every mbarrier wait (kLnWaitNs in normal calls); `probe` != 0 leaves
// every CTA's first row copy unissued (a diagnostic of the bounded waits, see camp.h).
constexpr unsigned long long kLnWaitNs = 1000000000ull;
cudaError_t layernorm_staged_launch(DType t, int cluster, int stages, int rows_per_step,
                                    const LayernormArgs& a, cudaStream_t s,
                                    unsigned long long wait_ns = kLnWaitNs, int probe = 0);

// Wide LayerNorm (layernorm_wide.cu): rows no other LayerNorm kernel holds, any width; one
// CTA of kWideBlock threads per row, block-stride sweeps over x (16-byte or element accesses).
bool layernorm_wide_compiled(DType t, int vec_bytes);
cudaError_t layernorm_wide_launch(DType t, int vec_bytes, const LayernormArgs& a, int64_t grid,
                                  cudaStream_t s);

// ------------------------------------------------------------------ interleaved RoPE
// x [tokens, heads, dim], pairs (2i, 2i+1); table row positions[token] of [max_pos, dim/2].
struct RopeInterleavedArgs {
    const void* x;
    const float* sin_t;
    const float* cos_t;
    const int32_t* positions;
    void* y;
    int64_t tokens;
    int64_t heads;
    int64_t dim;
    int64_t max_pos;
};

// Tiled like rope_tiled: kRopeBlock threads, positions per CTA = 256 / (ceil(H/hpt) *
// dim/elems); vec_bytes 16, 8 or 4 (bf16, fp16) / 16 or 8 (fp32): a vector holds whole pairs.
bool rope_interleaved_compiled(DType t, int vec_bytes, int heads_per_thread);
cudaError_t rope_interleaved_launch(DType t, int vec_bytes, int heads_per_thread,
                                    const RopeInterleavedArgs& a, int64_t grid, cudaStream_t s);
// sin/cos [max_pos, dim/2] with angle = p * theta^(-2i/dim), fp64, rounded once to fp32.
cudaError_t rope_tables_launch(float* sin_t, float* cos_t, int64_t max_pos, int64_t dim,
                               double theta, cudaStream_t s);

// ------------------------------------------------------------------ KV RMSNorm + RoPE + cache
// One warp per token of kv[tokens, dn + dr]: RMSNorm of the first dn elements into row
// slots[t] of cache_n[num_slots, dn], rotate-half RoPE of the last dr into cache_r.
struct KvCacheArgs {
    const void* kv;
    const void* gamma;
    const float* sin_t;
    const float* cos_t;
    const int64_t* slots;
    void* cache_n;
    void* cache_r;
    int64_t tokens;     // B * S
    int64_t seq;        // S
    int64_t dn;         // norm width
    int64_t dr;         // rope width (even)
    int64_t num_slots;
    float eps;
};

constexpr int kKvBlock = 256;
constexpr int kKvTokensPerCta = kKvBlock / 32;   // one warp per token

// CTAs per SM of the KV kernel by the 32-bit registers of data a lane holds: its norm
// accesses, both rope halves and as many sine and cosine values as rope elements (element
// accesses counted twice: each takes a whole register and its own address). Up to 16
// words: 8 CTAs (2048 threads, 32 registers); 22: 6; 40: 4; beyond: 2 (checked with
// -Xptxas -v: no variant spills).
constexpr int kv_min_blocks(int elem_bytes, int vec_bytes, int nvn, int rope_bytes) {
    const int norm = vec_bytes == 16 ? 4 * nvn : 2 * nvn;
    const int rope_words = rope_bytes < 4 ? 1 : rope_bytes / 4;
    const int words = norm + 2 * rope_words + 2 * (rope_bytes / elem_bytes);
    return words <= 16 ? 8 : words <= 22 ? 6 : words <= 40 ? 4 : 2;
}

// `vec_bytes`: norm access width (16, or the element size); `nvn`: norm accesses per lane
// (1, 2, 4, 8; 16 on the element path only); `rope_bytes`: rope access width per half and
// lane (with 16-byte norm accesses, 4, 8 or 16 bytes holding at least one pair; the
// element size on the element path).
bool kv_cache_compiled(DType t, int vec_bytes, int nvn, int rope_bytes);
cudaError_t kv_cache_launch(DType t, int vec_bytes, int nvn, int rope_bytes,
                            const KvCacheArgs& a, cudaStream_t s);

// ------------------------------------------------------------------ KV concat + head repeat
// out[b, t, h*n_rep + r, :] from past[b, t, h, :] (t < P) or from fresh[b, t - P, h, :],
// rotated at table row t when sin_t is not null. Tiled like rope_tiled over the B*(P+S)
// rows: kRopeBlock threads, rows per CTA = 256 / (ceil(heads / hpt) * (half / elems)).
// Needs B*(P+S) < 2^32.
struct KvCatArgs {
    const void* past;      // [batch, past_len, heads, 2*half]; null when past_len == 0
    const void* fresh;     // [batch, new_len, heads, 2*half]; null when new_len == 0
    const float* sin_t;    // [past_len + new_len, half] or null (copy the new rows)
    const float* cos_t;
    void* out;             // [batch, past_len + new_len, heads * n_rep, 2*half]
    int64_t batch;
    int64_t past_len;
    int64_t new_len;
    int64_t heads;
    int64_t half;
    int64_t n_rep;
};

// CTAs per SM by heads per thread: camp_rope's budget, except that one head per thread also
// runs 5 CTAs (48 registers): at 6 the 16-byte bf16 variant (8 sine and 8 cosine values
// beside its data) spilled. The fp16 unpack is a conversion, not a shift, and the 16-byte
// fp16 variant with two heads per thread spilled at 5: it runs 4 (checked with -Xptxas -v).
constexpr int kv_cat_min_blocks(int heads_per_thread, bool f16) {
    return heads_per_thread == 1 ? 5 : heads_per_thread == 2 ? (f16 ? 4 : 5)
                                     : heads_per_thread <= 4 ? 3 : 2;
}

// vec_bytes 16, 8, 4, 2 (bf16, fp16) / 16, 8, 4 (fp32): bytes per access of each half.
bool kv_cat_compiled(DType t, int vec_bytes, int heads_per_thread);
cudaError_t kv_cat_launch(DType t, int vec_bytes, int heads_per_thread, const KvCatArgs& a,
                          int64_t grid, cudaStream_t s);

}  // namespace camp
