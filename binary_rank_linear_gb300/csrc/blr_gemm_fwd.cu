// Instantiations of the blr GEMM for the two forward products
// (a = (x.g) S_V and c = (a.l) S_U^T).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_fwd(int epi, int bn, const CUtensorMap &tmap_a, const EpiMaps &emaps, const GemmArgs &args,
                            int grid, cudaStream_t s) {
    if (epi == kEpiFwd1) return launch_gemm_epi<kEpiFwd1>(bn, tmap_a, emaps, args, grid, s);
    if (epi == kEpiFwd2) return launch_gemm_epi<kEpiFwd2>(bn, tmap_a, emaps, args, grid, s);
    return cudaErrorInvalidValue;
}

}  // namespace blr
