// Launchers shared between the translation units of the blr library.
// Host-side declarations only; every launcher queues work on `stream` and
// returns the cudaError_t of the launch.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace blr {

// Launch with programmatic stream serialization (see pdl_wait in
// blr_device.cuh) and the maximum shared-memory carveout, so that consecutive
// kernels of a pass overlap their setup and never reconfigure L1/shared
// memory between each other.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Sets the maximum dynamic shared memory and the carveout of `kernel` once.
template <typename... KArgs>
cudaError_t prepare_kernel(void (*kernel)(KArgs...), int max_dyn_smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

// Optional per-kernel event tracing (see blr_trace_begin in blr.h).
void trace_before(const char *name, cudaStream_t stream);
void trace_after(cudaStream_t stream);

// ---- sign bitmaps -------------------------------------------------------
cudaError_t launch_pack_signs(const float *src, uint32_t *bits, int rows, int r, cudaStream_t s);
cudaError_t launch_unpack_signs(const uint32_t *bits, uint16_t *dst, int rows, int r, cudaStream_t s);

// Re-layout of one bitmap into the GEMM's "pair-ready" operand order
// [ceil(K/64)][N][2] u32 (see sign_word_pair_ready):
//  - kind 0 ("direct"): src is [N][K/32], bits already run along K;
//  - kind 1 ("transpose"): src is [K][N/32], bits run along N.
struct SignPrep {
    const uint32_t *src;
    uint32_t *dst;
    int N;     // operand rows (output features)
    int K;     // reduction length
    int kind;  // 0 direct, 1 transpose
};

// Forward prologue, one launch: clear the device status word, re-lay two
// bitmaps and stage x16 = f16(x.g).
cudaError_t launch_fwd_prologue(SignPrep p0, SignPrep p1, const float *x, const float *g, uint16_t *x16, int M,
                                int d_in, uint32_t *status, cudaStream_t s);

// Backward prologue, two parts in one launch: re-lay two bitmaps, and stage
// dy16 = f16(dy.h.s_t) with per-token scales, dh partials and sigma_t.
struct StageDyArgs {
    const float *dy;       // [M][d_out]
    const float *h;        // [d_out]
    const uint16_t *c16;   // [M][d_out] forward tape (f16 bits)
    const float *l;        // [r]
    uint16_t *dy16;        // [M][d_out] out
    float *s_inv;          // [M] out: 1/s_t
    float *sig;            // [M] out: sigma_t (scale of db.l)
    float *sig_inv;        // [M] out: 1/sigma_t
    float *part_dh;        // [stage_dy_blocks(M, d_out)][d_out] out
    float gscale;          // > 0 fixed, <= 0 dynamic
    int M, d_out, r;
    int *rows_used;        // host out: dh partial rows the launch wrote
};
int stage_dy_blocks(int M, int d_out);  // dh partial rows reserved in the workspace
cudaError_t launch_bwd_prologue(SignPrep p0, SignPrep p1, const StageDyArgs &a, cudaStream_t s);

// out[f] += sum_p part[p][f] over three independent segments, fixed order.
struct ReduceSeg {
    const float *part;
    float *out;
    int rows;
    int n;
};
cudaError_t launch_reduce_partials(ReduceSeg a, ReduceSeg b, ReduceSeg c, cudaStream_t s);

// ---- tcgen05 GEMMs --------------------------------------------------------
enum GemmEpi : int { kEpiFwd1 = 0, kEpiFwd2 = 1, kEpiBwd1 = 2, kEpiBwd2 = 3 };

struct GemmArgs {
    int M;                   // tokens
    int N;                   // features = operand rows of the sign matrix
    int K;                   // reduction length
    const uint32_t *bsign;   // pair-ready bitmap [ceil(K/64)][N][2]
    float *out32;            // FWD1 a-tape, FWD2 y, BWD2 dx   [M][N]
    uint16_t *out16;         // FWD1 a.l, FWD2 c, BWD1 db.l.sigma (f16 bits) [M][N]
    const float *colv;       // per-feature factor: FWD1 l, FWD2 h, BWD1 l, BWD2 g
    const float *aux;        // BWD1 a-tape, BWD2 x   [M][N]
    const float *row_inv;    // BWD1 1/s_t, BWD2 1/sigma_t  [M]
    const float *row_scale;  // BWD1 sigma_t  [M]
    float *part;             // BWD1 dl partials, BWD2 dg partials  [ceil(M/128)][N]
    int accumulate;          // FWD2 y +=, BWD2 dx +=
    uint32_t *status;        // device status word
};

// Extra TMA descriptors of the wide-output products (c and dx'); unused by
// the other two.
struct EpiMaps {
    CUtensorMap out32;  // f32 [M][N], box 32 x 32, 128-byte swizzle (y or dx)
    CUtensorMap out16;  // f16 [M][N], box 32 x 32, 64-byte swizzle (c)
    CUtensorMap in32;   // f32 [M][N], box 32 x 32, 128-byte swizzle (x, or y to accumulate)
};

// `tmap_a`: the f16 activation operand [M][K], box 64 x 128, 128-B swizzle.
// bn: 32, 64, 128 or 256 (must divide N). grid: number of persistent CTAs.
cudaError_t launch_gemm(int epi, int bn, const CUtensorMap &tmap_a, const EpiMaps &emaps, const GemmArgs &args,
                        int grid, cudaStream_t s);

}  // namespace blr
