// Instantiations of the db-product (db = (dy.h) S_U) with dy staged inside
// the kernel by its stager warps, with the per-token scales and the dh sums
// (blr_stager.cuh).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_stg_bwd(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    return launch_gemm_stg<kEpiBwd1, 2>(plan, maps, args, s);
}

}  // namespace blr
