// Instantiations of the a-product (a = (x.g) S_V) with x staged inside the
// kernel by its stager warps (blr_stager.cuh).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_stg_fwd(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    return launch_gemm_stg<kEpiFwd1, 1>(plan, maps, args, s);
}

}  // namespace blr
