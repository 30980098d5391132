// Instantiations of the blr GEMM for the two forward products
// (a = (x.g) S_V and c = (a.l) S_U^T).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_fwd(int epi, const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    if (epi == kEpiFwd1) return launch_gemm_epi<kEpiFwd1>(plan, maps, args, s);
    if (epi == kEpiFwd2) return launch_gemm_epi<kEpiFwd2>(plan, maps, args, s);
    return cudaErrorInvalidValue;
}

}  // namespace blr
