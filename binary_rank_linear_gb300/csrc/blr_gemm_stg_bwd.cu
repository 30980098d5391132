// Instantiations of the db-product (db = dy16 S_U / s_t) with dy16 =
// f16(dy.h.s_t) staged inside the kernel by its stager warps, which also add
// the dh partial sums (blr_stager.cuh).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_stg_bwd(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    if (!plan.pair) return cudaErrorInvalidValue;  // CTA-pair tiles only
    return launch_gemm_stg<kEpiBwd1, 2>(plan, maps, args, s);
}

}  // namespace blr
