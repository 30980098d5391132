// Instantiations of the blr GEMM for the two backward products
// (db = (dy.h) S_U and dx' = (db.l) S_V^T).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_bwd(int epi, const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    if (epi == kEpiBwd1) return launch_gemm_epi<kEpiBwd1>(plan, maps, args, s);
    if (epi == kEpiBwd2) return launch_gemm_epi<kEpiBwd2>(plan, maps, args, s);
    return cudaErrorInvalidValue;
}

}  // namespace blr
