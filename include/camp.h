/*
 * camp.h: C ABI of libcamp, GB300 (sm_103a) kernels for two bandwidth-bound per-row
 * operators of a Llama-style transformer block.
 *
 *   camp_rmsnorm  RMSNorm forward, y = x / sqrt(mean(x^2) + eps) * w.
 *                 Definition: xserv "phase 4" design notes, RMSNorm section
 *                 (rms = sqrt(sum(x^2)/hidden + eps); y = x / rms * gamma). Precision:
 *                 gollamago README, "RMSNorm optimisation (TileLang)": each row is read
 *                 from global memory once and written once, the sum of squares and the
 *                 scaling stay in fp32, and the result is rounded once on write-back.
 *
 *   camp_rope     Rotate-half rotary position embedding with the signature
 *                 rope(input, sin_table, cos_table) -> output of the gollamago README,
 *                 section "RoPE": input [batch, sequence, heads, head_dim], tables
 *                 [sequence, head_dim/2]; each head is split into two halves that are
 *                 rotated in fp32 registers and written once. Pair formula: tilelang
 *                 tutorial ch. 02, exercise E13 (y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin).
 *
 * Conventions shared by every entry point
 *   - The caller owns every buffer. The library allocates no memory, keeps no per-call
 *     state and has no workspace; its only device state is one static status word that a
 *     kernel sets if a bounded wait ever runs out (camp_device_errors).
 *   - Tensor pointers are DEVICE pointers (or managed memory) to contiguous row-major
 *     data. A pointer need only be aligned to its element size; better-aligned pointers
 *     (16 bytes) and row pitches that are multiples of 16 bytes take the vector path.
 *   - `stream` is a cudaStream_t passed as void*. NULL is the legacy default stream.
 *   - Calls are asynchronous: nothing synchronizes the device. The return value reports
 *     argument errors and launch errors. A fault during execution surfaces later on the
 *     stream, as with any CUDA kernel.
 *   - Status codes follow the Intro-ops operator runtime (include/operator_runtime/api.h:
 *     success 0, invalid argument 1, unsupported dtype 2, runtime 3, not supported 5).
 *   - Argument errors are detected on the host before any CUDA call, so they are
 *     reported even on a machine without a GPU.
 */
#ifndef CAMP_H_
#define CAMP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define CAMP_API __declspec(dllexport)
#else
#define CAMP_API __attribute__((visibility("default")))
#endif

typedef enum {
    CAMP_SUCCESS = 0,
    CAMP_ERR_INVALID_ARG = 1,      /* a null pointer, a bad size, eps, alignment or overlap */
    CAMP_ERR_UNSUPPORTED_DTYPE = 2,
    CAMP_ERR_RUNTIME = 3,          /* a CUDA call failed; see camp_last_cuda_error() */
    CAMP_ERR_NOT_SUPPORTED = 5     /* a valid request that no compiled kernel can run */
} camp_status_t;

/* Storage types. Arithmetic is fp32 for all three: bf16 is the upper half of an fp32,
 * f16 is IEEE binary16 (every value exact in fp32); results are rounded once to the
 * storage type, to nearest, ties to even. */
typedef enum {
    CAMP_DTYPE_F16 = 0,
    CAMP_DTYPE_F32 = 1,
    CAMP_DTYPE_BF16 = 3
} camp_dtype_t;

/*
 * RMSNorm forward over `rows` independent rows of `cols` elements.
 *
 *   x     [rows, cols]  input, storage type `dtype`.
 *   w     [cols]        per-column weight (gamma), storage type `dtype`.
 *   y     [rows, cols]  output, storage type `dtype`. y == x (in place) is allowed;
 *                       any other overlap of y with x, and any overlap of y with w, is
 *                       rejected.
 *   rows  >= 0. rows == 0 is a no-op that returns CAMP_SUCCESS without touching memory.
 *   cols  >= 1.
 *   eps   finite and >= 0; added to mean(x^2) inside the square root.
 *
 * For each row r: ss = sum_j x[r,j]^2 accumulated in fp32; rinv = rsqrt(ss / cols + eps);
 * y[r,j] = round(x[r,j] * rinv * w[j]), where the products are fp32 and round() is the
 * single conversion to the storage type (round to nearest even).
 *
 * Errors: CAMP_ERR_UNSUPPORTED_DTYPE for an unknown dtype; CAMP_ERR_INVALID_ARG for a
 * null pointer (when rows > 0), rows < 0, cols < 1, a negative or non-finite eps, a
 * pointer not aligned to the element size, a size whose byte count overflows int64,
 * or a forbidden overlap; CAMP_ERR_RUNTIME if the launch fails.
 */
CAMP_API camp_status_t camp_rmsnorm(const void* x, const void* w, void* y, int64_t rows,
                                    int64_t cols, float eps, camp_dtype_t dtype,
                                    void* stream);

/*
 * Fused residual add + RMSNorm: h = x + r, y = RMSNorm(h) * w, in one pass over the rows.
 * The TileLang tutorial (ch. 02, section 4.2) cites the fusion of "the Add before RmsNorm"
 * with the RMSNorm (Ascend's AddRmsNorm operators) as a way to save moving data in and
 * out; the pages define no more than that. Here h is formed in fp32, rounded once to the
 * storage type and stored (the residual stream of the next block), and the row that is
 * normalized is h as stored, exactly as camp_rmsnorm does it; so the result is bit for bit
 * that of an add followed by camp_rmsnorm, while x and r are read once and h is never
 * re-read from memory.
 *
 *   x, r  [rows, cols]  the two addends (block output and residual), storage type `dtype`.
 *   w     [cols]        weight.
 *   h     [rows, cols]  output: x + r, rounded once.
 *   y     [rows, cols]  output: RMSNorm(h) * w.
 *   Each output may equal x or r exactly (in place; for example h == r updates the
 *   residual where it is); otherwise it must be disjoint from both. h and y must be
 *   disjoint from each other and from w. Sizes, eps and errors as for camp_rmsnorm.
 */
CAMP_API camp_status_t camp_add_rmsnorm(const void* x, const void* r, const void* w, void* h,
                                        void* y, int64_t rows, int64_t cols, float eps,
                                        camp_dtype_t dtype, void* stream);

/*
 * Rotate-half RoPE of x[B, S, H, D] with fp32 tables sin[S, D/2] and cos[S, D/2].
 *
 *   x     [B, S, H, D]  input, storage type `dtype`.
 *   sin   [S, D/2]      fp32 sine table, row s used by every (b, s, h).
 *   cos   [S, D/2]      fp32 cosine table, same layout (note the order: sin before cos).
 *   y     [B, S, H, D]  output, storage type `dtype`. y == x (in place) is allowed; any
 *                       other overlap of y with x, or any overlap of y with a table, is
 *                       rejected.
 *   B, S, H >= 0; B*S*H == 0 is a no-op returning CAMP_SUCCESS.
 *   D     even, >= 2.
 *
 * For every (b, s, h) and i < D/2, with c = cos[s, i] and sn = sin[s, i]:
 *   y[.., i]       = round(x[.., i] * c - x[.., i + D/2] * sn)
 *   y[.., i + D/2] = round(x[.., i + D/2] * c + x[.., i] * sn)
 * evaluated in fp32 with a compensated product (the error stays relative to the
 * result even under cancellation) and rounded once to the storage type. The table row
 * s is derived on the device from the row index.
 *
 * Errors: CAMP_ERR_UNSUPPORTED_DTYPE for an unknown dtype; CAMP_ERR_INVALID_ARG for a
 * null pointer (when B*S*H > 0), a negative size, D odd or < 2, a misaligned pointer,
 * a byte count that overflows int64, or a forbidden overlap; CAMP_ERR_RUNTIME if the
 * launch fails.
 */
CAMP_API camp_status_t camp_rope(const void* x, const float* sin, const float* cos, void* y,
                                 int64_t B, int64_t S, int64_t H, int64_t D,
                                 camp_dtype_t dtype, void* stream);

/*
 * Rotate-half RoPE of the query and key tensors of one attention layer in one launch:
 * yq = rope(q), yk = rope(k), both with the same tables (the gollamago README's
 * rope(input, sin_table, cos_table) applied to Q and to K; in Llama both are rotated
 * right after the QKV projection). Sharing one launch saves a launch and lets every
 * position's table vectors be read once, through L1, by the heads of both tensors.
 *
 *   q, yq  [B, S, Hq, D]  query input and output, storage type `dtype`.
 *   k, yk  [B, S, Hk, D]  key input and output, storage type `dtype`.
 *   sin, cos [S, D/2]     fp32 tables, as for camp_rope.
 *   Hq, Hk >= 0. Hq == 0 (or Hk == 0) makes this camp_rope of the other tensor; pointers
 *          of a tensor with no heads are not inspected.
 *
 * Each output may equal its own input (in place); otherwise every output must be
 * disjoint from both inputs, from the other output and from both tables. The arithmetic
 * of each element is exactly camp_rope's. One launch when a position's heads of both
 * tensors fit one CTA (the plan reports CAMP_KERNEL_ROPE); otherwise Q and K are rotated
 * by two camp_rope launches (CAMP_KERNEL_ROPE_SPLIT).
 *
 * Errors: as for camp_rope, for either tensor, plus the overlap rules above.
 */
CAMP_API camp_status_t camp_rope_qk(const void* q, const void* k, const float* sin,
                                    const float* cos, void* yq, void* yk, int64_t B, int64_t S,
                                    int64_t Hq, int64_t Hk, int64_t D, camp_dtype_t dtype,
                                    void* stream);

/*
 * Fused KV RMSNorm + RoPE + cache scatter. The TileLang tutorial (ch. 02, section 1.2)
 * describes Ascend's KvRmsNormRopeCache operator: the last axis of the kv tensor is split,
 * the left part goes through RMSNorm, the right part through RoPE, and the two results are
 * scattered into two caches (paged caches are addressed by block tables). Here:
 *
 *   kv       [B, S, Dn + Dr]  one KV head per token (as in multi-head latent attention),
 *                             storage type `dtype`.
 *   gamma    [Dn]             RMSNorm weight, storage type `dtype`.
 *   sin, cos [S, Dr/2]        fp32 RoPE tables; token (b, s) uses row s.
 *   slots    [B*S] int64      destination row of token t = b*S + s in both caches (a paged
 *                             cache is addressed as block * block_size + offset). A slot
 *                             outside [0, num_slots) means "do not write" (padding); two
 *                             tokens with the same slot race, so slots must be distinct.
 *   cache_n  [num_slots, Dn]  receives RMSNorm(kv[t, :Dn]) * gamma (camp_rmsnorm's
 *                             arithmetic, one rounding).
 *   cache_r  [num_slots, Dr]  receives rotate-half RoPE of kv[t, Dn:] (camp_rope's
 *                             arithmetic, one rounding).
 *   Dn >= 1; Dr even, >= 2; eps as for camp_rmsnorm. B*S == 0 is a no-op.
 *
 * One read of kv, one write of each cache row; a padding token's kv row is read (with the
 * rest of the warp's loads, before its slot is known) but nothing is written for it.
 * Supported widths: up to 256 16-byte vectors for the norm part and 32 lanes of at most
 * 16 bytes per rope half (bf16/f16: Dn <= 2048, Dr <= 512; fp32: Dn <= 1024, Dr <= 256); when
 * the norm rows or the pointers are not 16-byte aligned, element accesses (Dn <= 512,
 * Dr <= 64); otherwise CAMP_ERR_NOT_SUPPORTED. The caches must be disjoint from every
 * input and from each other. Errors as for camp_rmsnorm.
 */
CAMP_API camp_status_t camp_kv_rmsnorm_rope_cache(const void* kv, const void* gamma,
                                                  const float* sin, const float* cos,
                                                  const int64_t* slots, void* cache_n,
                                                  void* cache_r, int64_t B, int64_t S,
                                                  int64_t Dn, int64_t Dr, int64_t num_slots,
                                                  float eps, camp_dtype_t dtype, void* stream);

/*
 * Interleaved RoPE with per-token position ids, as in the xserv "phase 4" kernel
 * (csrc/embedding/rope.cu): for each pair (x[2i], x[2i+1]) of every head of token t,
 * at position p = positions[t], with c = cos[p, i] and sn = sin[p, i]:
 *   y[2i]   = round(x[2i] * c - x[2i+1] * sn)
 *   y[2i+1] = round(x[2i] * sn + x[2i+1] * c)
 * (the same compensated fp32 products as camp_rope, one rounding).
 *
 *   x, y       [tokens, H, D]  storage type `dtype`; y == x (in place) is allowed.
 *   sin, cos   [max_pos, D/2]  fp32 tables (camp_rope_tables makes them).
 *   positions  [tokens] int32  device array; a position outside [0, max_pos) leaves the
 *                              token's rows of y unwritten (nothing is read out of bounds).
 *   D even, >= 2; tokens, H >= 0 (0 is a no-op).
 *
 * Pointers must be aligned to one pair (2 elements); CAMP_ERR_NOT_SUPPORTED if a token's
 * heads need more than one CTA even at 8 heads per thread (H * D too large).
 */
CAMP_API camp_status_t camp_rope_interleaved(const void* x, const float* sin, const float* cos,
                                             const int32_t* positions, void* y, int64_t tokens,
                                             int64_t H, int64_t D, int64_t max_pos,
                                             camp_dtype_t dtype, void* stream);

/*
 * Concatenation of cached and new keys (or values) along the sequence, with the head repeat
 * of grouped-query attention, in one pass. The gollamago README (RoPE and RMSNorm notes, the
 * list of what is not handled) leaves attention's repeat_interleave on the PyTorch path:
 * there the cached keys and the new ones are joined with torch.cat and each of the Hk key
 * heads is then repeated n_rep = Hq / Hk times for the Hq query heads, two passes that read
 * and write the whole cache. Here each source element is read once and its n_rep copies are
 * written once, and the new rows can be rotated (rotate-half RoPE) on the way:
 *
 *   out[b, t,     h*n_rep + r, :] = past[b, t, h, :]                           t < P
 *   out[b, P + s, h*n_rep + r, :] = rope(fresh[b, s, h, :], table row P + s)     s < S
 *
 * for every r < n_rep (torch.repeat_interleave order: copies of one head are adjacent).
 *
 *   past     [B, P, Hk, D]   cached rows, storage type `dtype`; may be NULL when P == 0.
 *   fresh    [B, S, Hk, D]   new rows, storage type `dtype`; may be NULL when S == 0.
 *   sin, cos [P + S, D/2]    fp32 tables indexed by absolute position (only rows P .. P+S-1
 *                            are read), or both NULL: the new rows are copied unrotated.
 *                            A longer table (say [max_pos, D/2]) may be passed.
 *   out      [B, P + S, Hk * n_rep, D]  output, disjoint from every input.
 *   B, P, S, Hk >= 0 (B*(P+S)*Hk == 0 is a no-op); D even, >= 2; n_rep >= 1.
 *
 * Copied values are bit-exact; rotated values are camp_rope's arithmetic (compensated fp32
 * products, one rounding). CAMP_ERR_NOT_SUPPORTED when B*(P+S) >= 2^32 or a row's heads need
 * more than one CTA even at 8 heads per thread (Hk * D too large). Errors otherwise as for
 * camp_rope, plus CAMP_ERR_INVALID_ARG when only one of sin and cos is NULL.
 */
CAMP_API camp_status_t camp_kv_cat_repeat(const void* past, const void* fresh, const float* sin,
                                          const float* cos, void* out, int64_t B, int64_t P,
                                          int64_t S, int64_t Hk, int64_t D, int64_t n_rep,
                                          camp_dtype_t dtype, void* stream);

/*
 * RoPE tables on the device: sin[p, i] and cos[p, i] for p < max_pos, i < D/2, with
 * angle = p * theta^(-2i/D) (the table of the xserv compute_rope_cache kernel; theta is
 * 10000 in the original Llama and 500000 in Llama 3). Computed in fp64 with CUDA's
 * double-precision pow and sincos, each value rounded once to fp32 (an fp32 angle is off
 * by about 4e-3 rad at position 65536). The tables serve camp_rope, camp_rope_qk,
 * camp_rope_interleaved and camp_kv_rmsnorm_rope_cache alike.
 *
 *   sin, cos  [max_pos, D/2] fp32 outputs (disjoint). max_pos >= 0 (0 is a no-op);
 *   D even, >= 2; theta finite and > 0. Errors: CAMP_ERR_INVALID_ARG, CAMP_ERR_RUNTIME.
 */
CAMP_API camp_status_t camp_rope_tables(float* sin, float* cos, int64_t max_pos, int64_t D,
                                        double theta, void* stream);

/*
 * LayerNorm forward: y = gamma * (x - mean) / sqrt(var + eps) + beta per row, with the
 * population variance (xserv "phase 4", csrc/normalization/layernorm.cu).
 *
 *   x, y   [rows, cols]  storage type `dtype`; y == x (in place) is allowed.
 *   gamma, beta [cols]   storage type `dtype`; y must not overlap them.
 *
 * The row is held in registers (camp_rmsnorm's rows kernel layout: x read once, y written
 * once) and the statistics are taken in two passes over the registers, in fp32: with
 * K = x[row, 0], mu = sum(x - K) / n and d = (x - K) - mu, var = sum(d^2) / n and
 * y = fma(d * rsqrt(var + eps), gamma, beta), rounded once to the storage type. Rows of
 * more than 4096 16-byte vectors (32768 bf16/f16 / 16384 fp32 columns), or of more than
 * 2048 when there are at most 1024 rows (all pointers and the row pitch 16-byte aligned),
 * leave the registers: in 16-bit storage they are spread over a cluster of up to 16 CTAs,
 * each holding its whole chunk of the row in shared memory (up to about 1.7 M columns); in
 * fp32 they are staged in shared memory by persistent clusters of CTAs (up to 16 x 2048
 * vectors: 131072 columns), and spread like 16-bit rows where the staged chunks would
 * leave a fifth or more of the threads' vector slots empty, or past the staged kernel.
 * Rows wider still, and rows past 16384 columns on the element path, take one CTA per row
 * (any width). In 16-bit storage any of these kernels may take the
 * variance as sum((x - K)^2) / n - mu^2 (one pass) for a row where mu^2 <= 4 times that
 * value. Errors as for camp_rmsnorm.
 */
CAMP_API camp_status_t camp_layernorm(const void* x, const void* gamma, const void* beta,
                                      void* y, int64_t rows, int64_t cols, float eps,
                                      camp_dtype_t dtype, void* stream);

/*
 * The library's device error word: bit CAMP_DEVICE_ERROR_WAIT_TIMEOUT is set by a kernel
 * whose bounded wait (on an asynchronous copy; one second at most) ran out, in which case
 * that kernel's output is incomplete. Correct operation never sets it. *flags receives the
 * word; clear != 0 resets it to 0. Synchronizes the device (it reads device memory).
 * Errors: CAMP_ERR_INVALID_ARG for a NULL flags; CAMP_ERR_RUNTIME if the read fails.
 */
#define CAMP_DEVICE_ERROR_WAIT_TIMEOUT 1u
CAMP_API camp_status_t camp_device_errors(uint32_t* flags, int clear);

/* A static, human-readable name for a status code (never NULL). */
CAMP_API const char* camp_status_string(camp_status_t status);

/*
 * The cudaError_t value behind the most recent CAMP_ERR_RUNTIME returned on the calling
 * thread (0 if none). Reading it does not clear it.
 */
CAMP_API int camp_last_cuda_error(void);

/* ------------------------------------------------------------------ kernel plans
 * A plan names the kernel variant that a call with the given shapes and pointers runs.
 * Planning is host-only arithmetic (no CUDA call), so it works without a GPU; the
 * benchmark and the tests use it to label and to enumerate kernel variants. A *_with_plan
 * call given a plan whose kernel the operation does not have, or a variant that is not
 * built or does not cover the row, returns CAMP_ERR_NOT_SUPPORTED without launching.
 */
typedef enum {
    CAMP_KERNEL_RMSNORM_ROWS = 1,   /* a group of threads per row, row held in registers */
    CAMP_KERNEL_RMSNORM_WIDE = 2,   /* one CTA per row, two sweeps over x (very wide rows) */
    CAMP_KERNEL_ROPE = 3,           /* tiled: a CTA covers whole positions, all their heads */
    CAMP_KERNEL_ROPE_FLAT = 4,      /* any shape: one work item per (position, heads, vector) */
    CAMP_KERNEL_ROPE_SPLIT = 5,     /* camp_rope_qk only: Q and K as two separate launches */
    CAMP_KERNEL_RMSNORM_CLUSTER = 6, /* a cluster of CTAs per row, sums combined over DSMEM */
    CAMP_KERNEL_KV_CACHE = 7,       /* camp_kv_rmsnorm_rope_cache: one warp per token */
    CAMP_KERNEL_ROPE_INTERLEAVED = 8, /* camp_rope_interleaved: tiled like CAMP_KERNEL_ROPE */
    CAMP_KERNEL_LAYERNORM_ROWS = 9, /* camp_layernorm: a group of threads per row, registers */
    CAMP_KERNEL_KV_CAT = 10,        /* camp_kv_cat_repeat: tiled like CAMP_KERNEL_ROPE */
    CAMP_KERNEL_RMSNORM_STAGED = 11, /* persistent clusters, rows staged in shared memory by
                                        bulk asynchronous copies, `per_thread` buffers deep */
    CAMP_KERNEL_LAYERNORM_STAGED = 12, /* camp_layernorm: the same, for the widest rows */
    CAMP_KERNEL_LAYERNORM_WIDE = 13, /* camp_layernorm: one CTA per row, block-stride sweeps
                                        over x, for rows no other kernel holds (any width) */
    CAMP_KERNEL_RMSNORM_SPREAD = 14, /* camp_rmsnorm and camp_add_rmsnorm: a cluster of CTAs
                                        per row, each holding its whole chunk (of x, and of
                                        r) in shared memory (rows past the staged kernel) */
    CAMP_KERNEL_LAYERNORM_SPREAD = 15 /* camp_layernorm: the same */
} camp_kernel_t;

typedef struct {
    int32_t kernel;        /* camp_kernel_t */
    int32_t vec_bytes;     /* bytes per vector access of x and y: 16, 8, 4 or 2 */
    int32_t group;         /* RMSNorm: threads per row (staged kernel: 16-byte vectors of a
                              row per CTA). RoPE, KV concat: heads per thread.
                              KV cache: rope access bytes per half and lane */
    int32_t per_thread;    /* RMSNorm: vector accesses per thread per row (staged kernel:
                              shared-memory buffers per CTA). RoPE: unused (0) */
    int32_t block;         /* threads per CTA */
    int32_t cluster;       /* CTAs per cluster (RMSNorm cluster kernel: 2..16), else 1 */
    int64_t grid;          /* CTAs launched. Staged and spread kernels (persistent
                              clusters): the planner's estimate from shared memory and
                              registers per SM; the launch takes the clusters the device
                              holds at once (cudaOccupancyMaxActiveClusters), at most one a
                              row */
    int32_t rows_per_step; /* staged LayerNorm: rows one step takes (1 or 2; 0 on input means
                              1); other kernels: 0 */
} camp_plan_t;

/*
 * Fill *plan with the variant camp_rmsnorm would launch for these arguments. Validation
 * is the same as camp_rmsnorm's (pointers are only inspected, never dereferenced).
 */
CAMP_API camp_status_t camp_rmsnorm_plan(const void* x, const void* w, const void* y,
                                         int64_t rows, int64_t cols, camp_dtype_t dtype,
                                         camp_plan_t* plan);

/* Like camp_rmsnorm_plan, for camp_rope. */
CAMP_API camp_status_t camp_rope_plan(const void* x, const float* sin, const float* cos,
                                      const void* y, int64_t B, int64_t S, int64_t H,
                                      int64_t D, camp_dtype_t dtype, camp_plan_t* plan);

/*
 * camp_rmsnorm with an explicit plan (kernel, vec_bytes, group, per_thread, and cluster for
 * the cluster kernel; block and grid are derived), for tuning sweeps and for tests that
 * cover every compiled variant.
 * Returns CAMP_ERR_NOT_SUPPORTED if no compiled variant matches or if the plan cannot
 * hold the row (vec_bytes must divide the row pitch and every pointer's alignment).
 */
CAMP_API camp_status_t camp_rmsnorm_with_plan(const void* x, const void* w, void* y,
                                              int64_t rows, int64_t cols, float eps,
                                              camp_dtype_t dtype, const camp_plan_t* plan,
                                              void* stream);

/* camp_rope with an explicit plan (kernel, vec_bytes and group = heads per thread). */
CAMP_API camp_status_t camp_rope_with_plan(const void* x, const float* sin, const float* cos,
                                           void* y, int64_t B, int64_t S, int64_t H, int64_t D,
                                           camp_dtype_t dtype, const camp_plan_t* plan,
                                           void* stream);

/* Like camp_rope_plan, for camp_rope_qk. */
CAMP_API camp_status_t camp_rope_qk_plan(const void* q, const void* k, const float* sin,
                                         const float* cos, const void* yq, const void* yk,
                                         int64_t B, int64_t S, int64_t Hq, int64_t Hk,
                                         int64_t D, camp_dtype_t dtype, camp_plan_t* plan);

/* camp_rope_qk with an explicit plan: only the single fused launch (CAMP_KERNEL_ROPE). */
CAMP_API camp_status_t camp_rope_qk_with_plan(const void* q, const void* k, const float* sin,
                                              const float* cos, void* yq, void* yk, int64_t B,
                                              int64_t S, int64_t Hq, int64_t Hk, int64_t D,
                                              camp_dtype_t dtype, const camp_plan_t* plan,
                                              void* stream);

/* Like camp_rmsnorm_plan, for camp_add_rmsnorm (same kernels, add variants). */
CAMP_API camp_status_t camp_add_rmsnorm_plan(const void* x, const void* r, const void* w,
                                             const void* h, const void* y, int64_t rows,
                                             int64_t cols, camp_dtype_t dtype,
                                             camp_plan_t* plan);

/* camp_add_rmsnorm with an explicit plan, as camp_rmsnorm_with_plan. */
CAMP_API camp_status_t camp_add_rmsnorm_with_plan(const void* x, const void* r, const void* w,
                                                  void* h, void* y, int64_t rows, int64_t cols,
                                                  float eps, camp_dtype_t dtype,
                                                  const camp_plan_t* plan, void* stream);

/* Like camp_rmsnorm_plan, for camp_kv_rmsnorm_rope_cache: one warp per token; vec_bytes =
 * norm access width (16 or the element size), per_thread = norm accesses per lane, group =
 * rope access width per half and lane (4, 8 or 16 bytes with 16-byte norm accesses, the
 * element size otherwise). */
CAMP_API camp_status_t camp_kv_rmsnorm_rope_cache_plan(
    const void* kv, const void* gamma, const float* sin, const float* cos, const int64_t* slots,
    const void* cache_n, const void* cache_r, int64_t B, int64_t S, int64_t Dn, int64_t Dr,
    int64_t num_slots, camp_dtype_t dtype, camp_plan_t* plan);

/* camp_kv_rmsnorm_rope_cache with an explicit plan (vec_bytes, per_thread, group; group 0
 * takes the default rope width for vec_bytes); NULL plan = the default one. */
CAMP_API camp_status_t camp_kv_rmsnorm_rope_cache_with_plan(
    const void* kv, const void* gamma, const float* sin, const float* cos, const int64_t* slots,
    void* cache_n, void* cache_r, int64_t B, int64_t S, int64_t Dn, int64_t Dr,
    int64_t num_slots, float eps, camp_dtype_t dtype, const camp_plan_t* plan, void* stream);

/* Like camp_rope_plan, for camp_rope_interleaved (vec_bytes; group = heads per thread). */
CAMP_API camp_status_t camp_rope_interleaved_plan(const void* x, const float* sin,
                                                  const float* cos, const int32_t* positions,
                                                  const void* y, int64_t tokens, int64_t H,
                                                  int64_t D, int64_t max_pos, camp_dtype_t dtype,
                                                  camp_plan_t* plan);

/* camp_rope_interleaved with an explicit plan (vec_bytes, group); NULL plan = the default. */
CAMP_API camp_status_t camp_rope_interleaved_with_plan(const void* x, const float* sin,
                                                       const float* cos,
                                                       const int32_t* positions, void* y,
                                                       int64_t tokens, int64_t H, int64_t D,
                                                       int64_t max_pos, camp_dtype_t dtype,
                                                       const camp_plan_t* plan, void* stream);

/* Like camp_rope_plan, for camp_kv_cat_repeat (vec_bytes = access bytes per half;
 * group = heads per thread). */
CAMP_API camp_status_t camp_kv_cat_repeat_plan(const void* past, const void* fresh,
                                               const float* sin, const float* cos,
                                               const void* out, int64_t B, int64_t P, int64_t S,
                                               int64_t Hk, int64_t D, int64_t n_rep,
                                               camp_dtype_t dtype, camp_plan_t* plan);

/* camp_kv_cat_repeat with an explicit plan (vec_bytes, group); NULL plan = the default. */
CAMP_API camp_status_t camp_kv_cat_repeat_with_plan(const void* past, const void* fresh,
                                                    const float* sin, const float* cos,
                                                    void* out, int64_t B, int64_t P, int64_t S,
                                                    int64_t Hk, int64_t D, int64_t n_rep,
                                                    camp_dtype_t dtype, const camp_plan_t* plan,
                                                    void* stream);

/* Like camp_rmsnorm_plan, for camp_layernorm (kernel CAMP_KERNEL_LAYERNORM_ROWS). */
CAMP_API camp_status_t camp_layernorm_plan(const void* x, const void* gamma, const void* beta,
                                           const void* y, int64_t rows, int64_t cols,
                                           camp_dtype_t dtype, camp_plan_t* plan);

/* camp_layernorm with an explicit plan (vec_bytes, group, per_thread); NULL = default. */
CAMP_API camp_status_t camp_layernorm_with_plan(const void* x, const void* gamma,
                                                const void* beta, void* y, int64_t rows,
                                                int64_t cols, float eps, camp_dtype_t dtype,
                                                const camp_plan_t* plan, void* stream);

/*
 * The same diagnostic for RMSNorm without the residual add (the pages have no counterpart):
 * the staged RMSNorm kernel (plan == NULL: the staged plan for these arguments, whichever
 * kernel camp_rmsnorm would take) or the kernel of `plan` (staged or spread, checked as
 * camp_rmsnorm_with_plan checks it), with every mbarrier wait bounded by `wait_ns` and each
 * CTA's first row copy left unissued; the outcome is as for camp_layernorm_wait_probe below
 * (the timeout bit set, y untouched, the next call normal). Arguments, validation and errors
 * as camp_rmsnorm; in addition CAMP_ERR_INVALID_ARG if wait_ns is outside
 * [1000, 1000000000], and CAMP_ERR_NOT_SUPPORTED for a plan of another kernel or one that
 * does not hold the row, or, with plan == NULL, unless the staged kernel holds the row
 * (16-byte-aligned pointers and rows of more than 4096 16-byte vectors, up to 16 x 2048).
 */
CAMP_API camp_status_t camp_rmsnorm_wait_probe(const void* x, const void* w, void* y,
                                               int64_t rows, int64_t cols, float eps,
                                               camp_dtype_t dtype, const camp_plan_t* plan,
                                               uint64_t wait_ns, void* stream);

/*
 * Diagnostic of the bounded waits (the pages have no counterpart; it exists so that the
 * failure path of the staged and spread kernels can be exercised without faulting
 * anything). Runs the staged LayerNorm kernel (plan == NULL: the staged plan for these
 * arguments, whichever kernel camp_layernorm would take) or the kernel of `plan` (staged
 * or spread, checked as camp_layernorm_with_plan checks it) on these arguments, with every
 * mbarrier wait bounded by `wait_ns` nanoseconds instead of one second and with the bulk
 * copy of each CTA's first row left unissued (its barrier still expects the bytes), so
 * every CTA's first wait runs out. Each CTA then sets CAMP_DEVICE_ERROR_WAIT_TIMEOUT in the
 * device error word, stores nothing into y, keeps exchanging its (zero) partials so that
 * no peer waits for it, waits (bounded again) for the copies it did issue, and returns: y
 * is left untouched and the next call runs normally. Arguments, validation and errors as
 * camp_layernorm; in addition CAMP_ERR_INVALID_ARG if wait_ns is outside
 * [1000, 1000000000], and CAMP_ERR_NOT_SUPPORTED for a plan of another kernel or one that
 * does not hold the row, or, with plan == NULL, unless the staged kernel holds the row
 * (16-byte-aligned pointers and rows of more than 4096 16-byte vectors, or 2048 with at
 * most 1024 rows, up to 16 x 2048). Each CTA spends about two times wait_ns.
 */
CAMP_API camp_status_t camp_layernorm_wait_probe(const void* x, const void* gamma,
                                                 const void* beta, void* y, int64_t rows,
                                                 int64_t cols, float eps, camp_dtype_t dtype,
                                                 const camp_plan_t* plan, uint64_t wait_ns,
                                                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CAMP_H_ */
