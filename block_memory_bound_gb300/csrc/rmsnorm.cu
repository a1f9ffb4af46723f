// RMSNorm forward (no residual add): the plain instantiations of rmsnorm_kernels.cuh, the
// table of compiled variants, and the dispatch entry points both paths share.
#include "rmsnorm_kernels.cuh"

namespace camp {

bool rmsnorm_rows_compiled(bool add, DType t, int vec_bytes, int group, int per_thread) {
    if (!rows_variant_compiled(add, vec_bytes, group, per_thread)) return false;
    const bool groups = group == 32 || group == 64 || group == 128 || group == 256 ||
                        group == 512 || group == 1024;
    if (vec_bytes == 16)
        return groups && (per_thread == 1 || per_thread == 2 || per_thread == 3 ||
                          per_thread == 4 || per_thread == 6 || per_thread == 8);
    if (vec_bytes == elem_bytes(t))
        return (group == 32 || group == 256 || group == 1024) &&
               (per_thread == 1 || per_thread == 2 || per_thread == 4 || per_thread == 8 ||
                per_thread == 16);
    return false;
}

cudaError_t rmsnorm_rows_launch(bool add, DType t, int vec_bytes, int group, int per_thread,
                                const RmsnormArgs& a, int64_t grid, cudaStream_t s) {
    if (add) return add_path::rows_launch(t, vec_bytes, group, per_thread, a, grid, s);
    return rms::Tables<false>::rows(t, vec_bytes, group, per_thread, a, grid, s);
}

bool rmsnorm_cluster_compiled(DType, int per_thread) {
    return per_thread == 1 || per_thread == 2 || per_thread == 3 || per_thread == 4 ||
           per_thread == 6 || per_thread == 8;
}

cudaError_t rmsnorm_cluster_launch(bool add, DType t, int per_thread, int cluster,
                                   const RmsnormArgs& a, cudaStream_t s) {
    if (add) return add_path::cluster_launch(t, per_thread, cluster, a, s);
    return rms::Tables<false>::cluster(t, per_thread, cluster, a, s);
}

bool rmsnorm_wide_compiled(DType t, int vec_bytes) {
    return vec_bytes == 16 || vec_bytes == elem_bytes(t);
}

cudaError_t rmsnorm_wide_launch(bool add, DType t, int vec_bytes, const RmsnormArgs& a,
                                int64_t grid, cudaStream_t s) {
    if (add) return add_path::wide_launch(t, vec_bytes, a, grid, s);
    return rms::Tables<false>::wide(t, vec_bytes, a, grid, s);
}

}  // namespace camp
