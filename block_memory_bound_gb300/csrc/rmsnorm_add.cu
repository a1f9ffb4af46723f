// RMSNorm with a fused residual add: the add-path instantiations of rmsnorm_kernels.cuh
// (own translation unit, so that both halves compile in parallel).
#include "rmsnorm_kernels.cuh"

namespace camp {
namespace add_path {

cudaError_t rows_launch(DType t, int vec_bytes, int group, int per_thread, const RmsnormArgs& a,
                        int64_t grid, cudaStream_t s) {
    return rms::Tables<true>::rows(t, vec_bytes, group, per_thread, a, grid, s);
}

cudaError_t cluster_launch(DType t, int per_thread, int cluster, const RmsnormArgs& a,
                           cudaStream_t s) {
    return rms::Tables<true>::cluster(t, per_thread, cluster, a, s);
}

cudaError_t wide_launch(DType t, int vec_bytes, const RmsnormArgs& a, int64_t grid,
                        cudaStream_t s) {
    return rms::Tables<true>::wide(t, vec_bytes, a, grid, s);
}

}  // namespace add_path
}  // namespace camp
