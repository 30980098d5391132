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

// Per-device launch facts, thread-safe (a process may drive several GPUs from
// several threads): the current device's SM count; a kernel's resident blocks
// per SM at a block size and shared-memory size (queried once per device and
// configuration); and, once per (device, kernel), the kernel's maximum
// dynamic shared memory and the maximum shared-memory carveout.
int current_device_sms();
int occupancy_blocks(const void *kernel, int threads, size_t smem);
cudaError_t prepare_once(const void *kernel, int max_dyn_smem);
template <typename... KArgs>
cudaError_t prepare_kernel_once(void (*kernel)(KArgs...), int max_dyn_smem) {
    return prepare_once(reinterpret_cast<const void *>(kernel), max_dyn_smem);
}

// Optional per-kernel event tracing (see blr_trace_begin in blr.h).
void trace_before(const char *name, cudaStream_t stream);
void trace_after(cudaStream_t stream);

// ---- sign bitmaps -------------------------------------------------------
cudaError_t launch_pack_signs(const float *src, uint32_t *bits, int rows, int r, cudaStream_t s);
cudaError_t launch_unpack_signs(const uint32_t *bits, uint16_t *dst, int rows, int r, cudaStream_t s);

// Re-layout of one bitmap into the GEMM's "pair-ready" operand order
// [2 ceil(K/128)][Ns][2] u32 (see sign_word_pair_ready); rows N .. Ns-1 and
// words past K are written as all -1 signs (they only ever meet zero
// activations or are never stored):
//  - kind 0 ("direct"): src is [N][K/32], bits already run along K;
//  - kind 1 ("transpose"): src is [K][N/32], bits run along N.
//  - kind 2 ("plane"): src is [N][K/32] with K = r, dst the +-1 f16 plane
//    [N][K] (as u32 pairs) that plane-mode GEMMs read by TMA; Ns unused.
struct SignPrep {
    const uint32_t *src;
    uint32_t *dst;
    int N;     // operand rows (output features; plane: bitmap rows)
    int K;     // reduction length (plane: r)
    int kind;  // 0 direct, 1 transpose, 2 plane
    int Ns;    // destination row stride, sign_rows(N)
};

// Grouped launches of a multi-path layer run one stage of the pass for up to
// kMaxGroupPaths paths of the same shape: the prologues and the reduction
// with gridDim.y = paths (block row p takes entry p of its group), the GEMMs
// with the path in their tile sequence (GemmArgs.paths).
constexpr int kMaxGroupPaths = 8;

// Forward prologue, one launch: clear the device status word, re-lay two
// bitmaps and stage x16 = f16(x.g), for each path of the group.
struct FwdPathArgs {
    SignPrep p0, p1;
    const float *g;
    uint16_t *x16;
    uint32_t *status;
};
struct FwdGroup {
    FwdPathArgs e[kMaxGroupPaths];
    int n;
};
cudaError_t launch_fwd_prologue(const FwdGroup &grp, const float *x, int M, int d_in, cudaStream_t s);
inline cudaError_t launch_fwd_prologue(SignPrep p0, SignPrep p1, const float *x, const float *g, uint16_t *x16,
                                       int M, int d_in, uint32_t *status, cudaStream_t s) {
    FwdGroup grp{};
    grp.e[0] = FwdPathArgs{p0, p1, g, x16, status};
    grp.n = 1;
    return launch_fwd_prologue(grp, x, M, d_in, s);
}

// Prologue of a pass whose first product stages its own operand (GemmPlan
// stg): re-lay two bitmaps, clear the device status word (when `status` is
// not null: the forward) and zero the stagers' ncnt row counters.
cudaError_t launch_prep(SignPrep p0, SignPrep p1, uint32_t *status, unsigned int *cnt, int ncnt, const char *name,
                        cudaStream_t s);
// The same for each path of a group (block row p: entry p's re-layouts and
// status word, and the ncnt counters at cnt0 + p * pstride bytes).
cudaError_t launch_prep_group(const FwdGroup &grp, unsigned int *cnt0, long long pstride, int ncnt, const char *name,
                              cudaStream_t s);

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
    float2 *blkmax;        // [stage blocks] out: per block (max 1/s_t, max 1/sigma_t) over its rows with
                           // nonzero finite dy.h (0 if none); the sign-gradient products rescale by them
    float gscale;          // > 0 fixed, <= 0 dynamic
    int M, d_out, r;
    int *rows_used;        // host out: dh partial rows the launch wrote
    uint32_t *status;      // device status word (bounded waits of the streaming staging)
    unsigned int *red_cnt; // zeroed by the launch (the dx'-product's reduction counter), or null
    // scale pass (dy staged inside the db-product, STG = 2): the launch writes
    // only s_inv, sig, sig_inv and blkmax (no dy16, no dh sums; c16 unread),
    // and zeroes n_cnt stager counters at zero_cnt and n_part floats of dh
    // partial rows at zero_part
    unsigned int *zero_cnt;
    int n_cnt;
    float *zero_part;
    long long n_part;
};
int stage_dy_blocks(int M, int d_out);  // dh partial rows reserved in the workspace
// per path of a group; M, d_out, r, gscale, dy and rows_used are taken from
// entry 0 (the paths share them)
struct BwdPathArgs {
    SignPrep p0, p1;
    StageDyArgs sd;
};
struct BwdGroup {
    BwdPathArgs e[kMaxGroupPaths];
    int n;
};
cudaError_t launch_bwd_prologue(const BwdGroup &grp, cudaStream_t s);
inline cudaError_t launch_bwd_prologue(SignPrep p0, SignPrep p1, const StageDyArgs &a, cudaStream_t s) {
    BwdGroup grp{};
    grp.e[0] = BwdPathArgs{p0, p1, a};
    grp.n = 1;
    return launch_bwd_prologue(grp, s);
}
// The scale pass only (a.zero_cnt / a.zero_part set): per-row scales, block
// maxima, the bitmap re-layouts; the db-product then stages dy itself.
cudaError_t launch_bwd_scales(const BwdGroup &grp, cudaStream_t s);
inline cudaError_t launch_bwd_scales(SignPrep p0, SignPrep p1, const StageDyArgs &a, cudaStream_t s) {
    BwdGroup grp{};
    grp.e[0] = BwdPathArgs{p0, p1, a};
    grp.n = 1;
    return launch_bwd_scales(grp, s);
}

// out[f] += sum_p part[p][f] over three independent segments, fixed order.
struct ReduceSeg {
    const float *part;
    float *out;
    int rows;
    int n;
};
// per path of a group: its dh, dl and dg segments (same widths for every path)
struct ReduceGroup {
    ReduceSeg a[kMaxGroupPaths], b[kMaxGroupPaths], c[kMaxGroupPaths];
    int n;
};
cudaError_t launch_reduce_partials(const ReduceGroup &grp, cudaStream_t s);
inline cudaError_t launch_reduce_partials(ReduceSeg a, ReduceSeg b, ReduceSeg c, cudaStream_t s) {
    ReduceGroup grp{};
    grp.a[0] = a;
    grp.b[0] = b;
    grp.c[0] = c;
    grp.n = 1;
    return launch_reduce_partials(grp, s);
}

// ---- tcgen05 GEMMs --------------------------------------------------------
enum GemmEpi : int { kEpiFwd1 = 0, kEpiFwd2 = 1, kEpiBwd1 = 2, kEpiBwd2 = 3 };

// Epilogue warps of a product's GEMM: one per TMEM lane quarter, or two
// (taking alternate chunks) for dx', whose epilogue (x in, dx out) outlasts its
// short main loop. Measured on GB300, two warps per quarter did not shorten
// the c-product (with eight expander warps, 18 warps at 96 registers, it
// lengthened it for K > 512; with four, 14 warps at 128 registers, the
// 12288-wide c-product took 316 against 308 us). Each epilogue warp writes its
// own row of token partial sums, so dx' has two partial rows per token tile.
__host__ __device__ constexpr int epi_warps(int epi) { return epi == kEpiBwd2 ? 8 : 4; }
__host__ __device__ constexpr int epi_part_rows_per_tile(int epi) { return epi_warps(epi) / 4; }

// In-kernel staging of the a-product's activation operand (GEMM template
// STG = 1: x16 = f16(x.g)): stager warps of every CTA write the f16 operand
// ahead of the MMA pipeline, in the order the persistent grid consumes token
// tiles, and count the rows they finish per (token tile, column chunk) in
// `cnt`; a tile's loads wait for its counts (blr_stager.cuh).
// Columns per readiness chunk (two 128-deep k-steps); the host sizes and
// zeroes the counters with it.
constexpr int kStageChunkCols = 256;
// dh partial rows per CTA of a db-product that stages dy (one per converter warp)
constexpr int kDyPartRowsPerCta = 4;
// CTAs such a launch may have: the workspace reserves dh partial rows for them
constexpr int kDyStageMaxCtas = 160;
inline int stage_counters(int M, int bt, int K) {
    return (M + bt - 1) / bt * ((K + kStageChunkCols - 1) / kStageChunkCols);
}
// The stagers index items and rounds in 32-bit arithmetic: stage in the
// kernel only while token tiles x (feature tiles + column chunks x 3 row
// groups) stays below 2^31 (beyond any x that fits on the device).
inline bool stage_fits(int M, int bt, int K, int f_tiles, int paths = 1) {
    const long long t = (long long)paths * ((M + bt - 1) / bt);
    return t * ((long long)f_tiles + 3ll * ((K + kStageChunkCols - 1) / kStageChunkCols)) < (1ll << 31);
}

// A grid barrier on a counter in global memory: barrier k waits for
// k * grid + extra arrivals, for at most wait_ns of wall time (extra is 0
// except in the test that makes the waits run out; see blr_api.cu). Used by
// the fused small-M kernels and by the dx'-product's folded reduction.
struct GridBarrier {
    unsigned int *gbar;
    unsigned int extra;
    unsigned long long wait_ns;
};

struct StageArgs {
    const float *src;      // x [M][K] f32 (STG = 2: dy [M][d_out])
    const float *col;      // g [K] (STG = 2: h [d_out])
    uint16_t *dst;         // x16 [M][K] (STG = 2: dy16)
    unsigned int *cnt;     // [token tiles][column chunks] rows staged (zeroed before the launch)
    // dy staged inside the db-product (STG = 2): each row's 1/s_t (written by
    // the scale pass before the launch), and the dh partial rows,
    // kDyPartRowsPerCta per CTA (part + (blockIdx.x * kDyPartRowsPerCta + w) * K
    // floats for converter warp w, zeroed before the launch; each warp adds its
    // items' column sums of dy.c into its own row)
    const float *row_sinv;
    float *part;
    // multi-path launches (paths > 1): path p's g at col_p[p], its x16 and
    // counters at p * pstride bytes after path 0's; the stagers take the
    // paths' token tiles in the product's path-major order
    int paths;
    long long pstride;
    const float *col_p[kMaxGroupPaths];
};

struct GemmArgs {
    int M;                   // tokens
    int N;                   // features = rows of the sign operand
    int K;                   // reduction length
    int Ns;                  // row stride of the re-laid bitmap (N rounded up to 256)
    const uint32_t *bsign;   // pair-ready bitmap [2 ceil(K/128)][Ns][2]
    float *out32;            // FWD1 a-tape, FWD2 y, BWD2 dx   [M][N]
    uint16_t *out16;         // FWD1 a.l, FWD2 c, BWD1 db.l.sigma (f16 bits) [M][N]
    const float *colv;       // per-feature factor: FWD1 l, FWD2 h, BWD1 l, BWD2 g
    const float *row_inv;    // BWD1 1/s_t, BWD2 1/sigma_t  [M]
    const float *row_scale;  // BWD1 sigma_t  [M]
    float *part;             // BWD1 dl partials, BWD2 dg partials  [token tiles][N]
    int accumulate;          // FWD2 y +=, BWD2 dx +=
    uint32_t *status;        // device status word
    StageArgs stg;           // in-kernel staging (STG kernels only)
    // multi-path launches: `paths` paths (0 or 1: one); path p's bsign,
    // row_inv, row_scale and part at p * pstride bytes after path 0's (its
    // workspace slice), its colv at colv_p[p]; the activation, out16 and
    // per-path f32 maps take the path as third coordinate
    int paths;
    long long pstride;
    const float *colv_p[kMaxGroupPaths];
    // dx'-product only (fold = 1): the pass's partial-sum reduction runs in
    // the kernel's tail. Every CTA adds its arrival to red.gbar (zeroed by the
    // backward prologue) once its dg partial rows are written; when the whole
    // grid has arrived (grid + red.extra arrivals, waited for at most
    // red.wait_ns: the persistent grid is resident together), the CTAs share
    // out the columns of every path's dh, dl and dg: out += the fixed-order
    // sum of the partial rows, red_part_h / red_part_l / part (path p at
    // p * pstride) with red_rows_h / red_rows_l / red_rows_g rows of d_out /
    // r / N columns.
    int fold;
    GridBarrier red;
    const float *red_part_h, *red_part_l;
    int red_rows_h, red_rows_l, red_rows_g, red_n_h, red_n_l;
    float *red_out_h[kMaxGroupPaths], *red_out_l[kMaxGroupPaths], *red_out_g[kMaxGroupPaths];
};

// Rows of the re-laid bitmap of a product with N features (a multiple of the
// widest feature tile, so that tile loads stay inside the buffer).
inline int sign_rows(int N) { return (N + 255) / 256 * 256; }

// TMA descriptors of one GEMM launch. act: the f16 activation operand [M][K],
// box 64 x (BT/2 for CTA pairs, BT otherwise), 128-byte swizzle. The
// epilogue's chunk maps are [M][N] with a 32 x 32 box and no swizzle: in32
// the f32 input (a-tape for db, x for dx', y when c accumulates into it),
// out32 / out16 the f32 and f16 outputs (a and a.l, y and c, -, dx and -).
// Maps a product does not use are left zero.
// sgn: the sign plane of a plane-mode GEMM, f16 with 128-byte swizzle: for
// the a- and db-products [K][N] read MN-major (box 64 features x 64 K), for
// the c- and dx'-products [N][K] read K-major (box 64 K x 128 features).
struct GemmMaps {
    CUtensorMap act, in32, out32, out16, sgn;
    CUtensorMap aux;  // STG = 2: the c tape in 256 x 16 boxes (unused otherwise)
};

// Tile plan of one GEMM launch: CTA pairs (tcgen05 cta_group::2) with 160 or
// 192 tokens per tile, or single CTAs with 128; grid = persistent CTAs (even
// for pairs); part_rows = token tiles (the epilogue writes
// epi_part_rows_per_tile rows of partial sums per token tile).
// plane = true: the sign operand is a +-1 f16 plane read by TMA (single CTAs,
// bt = 128, 192 or 256); false: bitmap words expanded into TMEM.
// split = 4: split-K over clusters of four single CTAs (one tile each; the
// a- and db-products of problems with few tiles), grid = tiles * 4.
// stg = 1 (a-product only): the activation operand is staged inside the
// kernel (args.stg), not by a pass before it.
struct GemmPlan {
    bool pair;
    int bt;
    int grid;
    int part_rows;
    bool plane;
    int split;
    int stg;
};

// TMEM-expansion tiles. Single-CTA token tiles are halved from 128 down to
// min_bt (64 or 32; the fused small-M kernels take 128) while the tiles would
// fill at most half the SMs. tile_cost: a tile's fixed cost in token units
// (CTA-pair tile choice).
GemmPlan plan_gemm(int M, int N, int sms, int min_bt = 64, int tile_cost = 0, int paths = 1);
// The c-product (K = r, output d_out wide) has a large fixed cost per tile:
// fitted on GB300 to the attention-sized layer at 160- and 192-token pair
// tiles, a round takes about 4.1 us + 0.0125 us per token of the tile, i.e.
// a fixed cost worth about 330 tokens. Counting it picks 192-token tiles there
// (67.5 -> 65.4 us; 16384 tokens, 12288 -> 4096: 124.9 -> 116.6 us). The
// dx'-product, same shape but a heavier epilogue, measured faster at 160.
constexpr int kWideTileCost = 330;
GemmPlan plan_gemm_plane(int M, int N, int sms);  // plane tiles

cudaError_t launch_gemm(int epi, const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s);

// ---- fused small-M path (blr_small.cu) ---------------------------------------
// One cooperative launch (grid = one CTA per SM) per pass; the GEMM phases use
// single-CTA 128-token tiles (plans with pair = false, bt = 128). `gb.gbar`
// is a grid-barrier counter in the workspace header, zeroed by the launcher.

struct SmallFwdArgs {
    SignPrep pv, pu;    // re-layouts of S_V (a-product) and S_U (c-product)
    const float *x, *g;
    uint16_t *x16;
    int M, d_in;
    uint32_t *status;
    GridBarrier gb;
    GemmArgs f1, f2;    // the a- and c-products
};

struct SmallBwdArgs {
    SignPrep pu, pv;    // re-layouts of S_U (db-product) and S_V (dx'-product)
    StageDyArgs sd;     // dy staging (its part_dh has stage_blocks rows)
    int stage_tpr;      // threads per token row in the staging (power of two <= 256); set by the launcher
    int stage_nthr;     // staging threads per CTA (a multiple of stage_tpr); set by the launcher
    int stage_blocks;   // CTAs that stage (dh partial rows written); set by the launcher
    GridBarrier gb;
    GemmArgs b1, b2;    // the db- and dx'-products
    ReduceSeg rh, rl, rg;
};

cudaError_t launch_small_fwd(const GemmMaps &m1, const GemmMaps &m2, const SmallFwdArgs &a, int grid,
                             cudaStream_t s);
// The launcher fills in the staging geometry and rh.rows (dh partial rows:
// at most rows_dh_reserved, the rows the workspace holds).
cudaError_t launch_small_bwd(const GemmMaps &m1, const GemmMaps &m2, SmallBwdArgs a, int grid, int rows_dh_reserved,
                             cudaStream_t s);
bool small_bwd_fits(int d_out);  // the fused backward stages rows of d_out floats

// ---- sign gradients (blr_sign.cu) -------------------------------------------
// ---- dense tensor-core products (blr_dense.cu) --------------------------------
// TMA descriptors of up to two products, [0] and [1]:
// a = the M-side operand: MN-major [K][F] (box 64 rows x 64 K) or K-major
//     [F][K] (box 64 K x 128 rows), f16, 128-byte swizzle;
// b = the N-side operand: MN-major [K][R] (box 64 x 64) or K-major [R][K]
//     (box 64 K x BN rows), f16, 128-byte swizzle;
// o = the f32 output [F][R] (box 32 x 32, 128-byte swizzle).
// o16: mode 1's f16 output c [F][R] (box 32 x 32, 64-byte swizzle).
struct DenseGemmMaps {
    CUtensorMap a[2], b[2], o[2], o16;
};

// Column tile of the dense products: 256 when R >= 256, else 128.
inline int dense_bn(int R) { return R >= 256 ? 256 : 128; }

// out_j = scale_j * dscale_j (if given) * sum_k A_j B_j, stored or (accumulate)
// added by TMA reduce-add into the outputs the maps o describe.
struct DenseGemmLaunch {
    DenseGemmMaps maps;
    int F[2];                      // rows of each product (F[1] = 0: one product)
    float scale[2];
    const float *dscale[2];        // device scalars or null
    int R, K, accumulate;
    bool a_mn, b_mn;               // operand majorness (A MN-major needs B MN-major)
    uint32_t *status;
    int sms;
    int epm;                       // epilogue mode (blr_dense.cu): 0 plain, 1 the c-product, 2 the dx'-product
    const float *colv, *row_inv, *xin;  // modes 1, 2: h or g; 1/sigma_t; x
    float *part;                   // mode 2: dg partial rows [ceil(F0/128) * 4][R]
};
cudaError_t launch_dense_gemm(const DenseGemmLaunch &L, const char *name, cudaStream_t s);

// ---- sign gradients (blr_sign.cu) -------------------------------------------
// G_U = dense product of dy16 [M][d_out] and the rank-side operand [M][r], G_V
// of x16 [M][d_in] and [M][r]: K = tokens, both operands MN-major.

// Dynamic gradient scale: rescale the rank-side operands to one scale each,
//   bu[t][k] = al16[t][k] * (1/s_t) / max_t (1/s_t)
//   bv[t][k] = db16[t][k] * (1/sigma_t) / max_t (1/sigma_t)
// (powers of two <= 1), maxima from the staging's per-block maxima; gmax[0..1]
// receives the two maxima (a zero maximum, all dy zero, counts as 1).
struct SignRescaleArgs {
    const uint16_t *al16, *db16;   // [M][r]
    const float *s_inv, *sig_inv;  // [M]
    const float2 *blkmax;          // [nblk]
    int nblk, M, r;
    uint16_t *bu, *bv;             // [M][r] out
    float *gmax;                   // [2] out
};
cudaError_t launch_sign_rescale(const SignRescaleArgs &a, int sms, cudaStream_t s);


// ---- plane_linear (blr_plane.cu) ----------------------------------------------
// act16 = f16(x * scale) over n values (n a multiple of 8); clears *status.
cudaError_t launch_plane_stage(const float *x, uint16_t *act16, long long n, float scale, uint32_t *status, int sms,
                               cudaStream_t s);

// ---- Adam (blr_adam.cu) -------------------------------------------------------
struct AdamArgs {
    float *w;             // [n] parameters, updated
    const float *grad;    // [n]
    float *m1, *m2;       // [n] first and second moments, updated
    const float *mask;    // [n] or null; 0 = frozen entry
    long long n;
    float lr, b1, b2, eps, gmul, rel;
    float bc1, bc2;       // 1 - b1^t, 1 - b2^t
};
cudaError_t launch_adam(const AdamArgs &a, int sms, cudaStream_t s);

}  // namespace blr
