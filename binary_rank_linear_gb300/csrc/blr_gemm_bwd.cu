// Instantiations of the blr GEMM for the two backward products
// (db = (dy.h) S_U and dx' = (db.l) S_V^T).
#include "blr_gemm.cuh"

namespace blr {

cudaError_t launch_gemm_bwd(int epi, int bn, const CUtensorMap &tmap_a, const EpiMaps &emaps, const GemmArgs &args,
                            int grid, cudaStream_t s) {
    if (epi == kEpiBwd1) return launch_gemm_epi<kEpiBwd1>(bn, tmap_a, emaps, args, grid, s);
    if (epi == kEpiBwd2) return launch_gemm_epi<kEpiBwd2>(bn, tmap_a, emaps, args, grid, s);
    return cudaErrorInvalidValue;
}

}  // namespace blr
