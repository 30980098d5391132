// Bandwidth kernels of the blr layer on sm_103a: sign packing/expansion, the
// one-per-call re-layout of the bitmaps into the GEMMs' operand order, the
// f32 -> f16 staging of x and dy (with the dh token sums fused into the dy
// staging), and the fixed-order reduction of per-tile partial sums.
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "blr_device.cuh"
#include "blr_kernels.h"
#include "blr_stage.cuh"

namespace blr {

// ====================================================== pack / unpack ======
// train_mm.rs (cortiq-engine 0.8.21), test helper `pack_bits`: bit (row, k)
// is 1 iff src[row][k] > 0. One warp per output word; lane j votes for rank
// 32w+j of the row.
__global__ void pack_signs_kernel(const float *__restrict__ src, uint32_t *__restrict__ bits, int rows, int r) {
    pdl_wait();
    const int words = (r + 31) / 32;
    const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    for (long long wi = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; wi < (long long)rows * words;
         wi += nwarps) {
        const long long row = wi / words;
        const int w = (int)(wi % words);
        const int k = 32 * w + lane;
        bool pos = false;
        if (k < r) pos = src[row * r + k] > 0.0f;  // NaN compares false
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, pos);
        if (lane == 0) bits[wi] = word;
    }
}

// train_mm.rs, `expand` kernel: bitmap -> +-1 f16, through the same
// pair-ready transform and pair expansion the GEMM expanders use.
__global__ void unpack_signs_kernel(const uint32_t *__restrict__ bits, uint16_t *__restrict__ dst, int rows,
                                    int r) {
    pdl_wait();
    const int words = (r + 31) / 32;
    const long long total = (long long)rows * words;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / words;
        const int w = (int)(i % words);
        const uint32_t p = sign_word_pair_ready(bits[i]);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const uint32_t pair = sign_pair(p, q);
            const int k = 32 * w + 2 * q;
            if (k < r) dst[row * r + k] = (uint16_t)(pair & 0xFFFFu);
            if (k + 1 < r) dst[row * r + k + 1] = (uint16_t)(pair >> 16);
        }
    }
}

// Blocks [0, stage_blocks) stage; when the grid has more, the extra blocks do
// the bitmap re-layouts alone (off the staging's critical path), otherwise
// every block does its share of them first.
__device__ __forceinline__ bool prologue_prep(const SignPrep &p0, const SignPrep &p1, int stage_blocks) {
    const int extra = (int)gridDim.x - stage_blocks;
    if (extra > 0) {
        if ((int)blockIdx.x < stage_blocks) return false;
        prep_share(p0, p1, (int)blockIdx.x - stage_blocks, extra);
        return true;  // a re-layout-only block
    }
    prep_share(p0, p1, blockIdx.x, stage_blocks);
    return false;
}

// (Forward and backward prologues: block row blockIdx.y works for path
// blockIdx.y of the group.)
__global__ void __launch_bounds__(256) fwd_prologue_kernel(const FwdGroup grp, const float *x, int M, int d_in,
                                                           int stage_blocks) {
    const FwdPathArgs &a = grp.e[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    if (prologue_prep(a.p0, a.p1, stage_blocks)) return;
    stage_x_run(x, a.g, a.x16, M, d_in, blockIdx.x, stage_blocks);
}

// The same prologue with x staged by rows (d_in up to kSxMaxCols).
template <int KQ>
__global__ void __launch_bounds__(512) fwd_prologue_rows_kernel(const FwdGroup grp, const float *x, int M,
                                                                int d_in, int stage_blocks) {
    const FwdPathArgs &a = grp.e[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    if (prologue_prep(a.p0, a.p1, stage_blocks)) return;
    stage_x_rows<KQ>(x, a.g, a.x16, M, d_in, blockIdx.x, stage_blocks);
}

// The same prologue with x streamed through a shared-memory ring (one block
// per SM; blocks past stage_blocks only do bitmap re-layouts).
template <int KQ>
__global__ void __launch_bounds__(kSxsThreads, 1)
    fwd_prologue_stream_kernel(const FwdGroup grp, const float *x, int M, int d_in, int stage_blocks) {
    extern __shared__ __align__(128) unsigned char smem_b[];
    const FwdPathArgs &a = grp.e[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    const int extra = (int)gridDim.x - stage_blocks;
    if (extra > 0 && (int)blockIdx.x >= stage_blocks) {
        prep_share(a.p0, a.p1, (int)blockIdx.x - stage_blocks, extra);
        return;
    }
    stage_x_stream<KQ>(x, a.g, a.x16, M, d_in, blockIdx.x, stage_blocks, smem_b, a.status, a.p0, a.p1,
                       extra > 0 ? 0 : stage_blocks);
}

// Prologue of a pass whose staging runs in its first product: the status
// word, the stagers' row counters and the two bitmap re-layouts.
__global__ void __launch_bounds__(256) prep_kernel(SignPrep p0, SignPrep p1, uint32_t *status, unsigned int *cnt,
                                                   int ncnt) {
    pdl_wait();
    pdl_launch_dependents();
    if (status && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ncnt; i += gridDim.x * blockDim.x) cnt[i] = 0u;
    prep_share(p0, p1, blockIdx.x, gridDim.x);
}

// The same for each path of a group (block row blockIdx.y).
__global__ void __launch_bounds__(256) prep_group_kernel(const FwdGroup grp, unsigned int *cnt0, long long pstride,
                                                         int ncnt) {
    const FwdPathArgs &a = grp.e[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    unsigned int *cnt = reinterpret_cast<unsigned int *>(reinterpret_cast<char *>(cnt0) + blockIdx.y * pstride);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ncnt; i += gridDim.x * blockDim.x) cnt[i] = 0u;
    prep_share(a.p0, a.p1, blockIdx.x, gridDim.x);
}

// The scale pass zeroes the db-product's stager counters and dh partial rows
// before any of its other work.
__device__ __forceinline__ void scale_pass_zero(const StageDyArgs &a) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    for (long long i = tid; i < a.n_cnt; i += nth) a.zero_cnt[i] = 0u;
    float4 *p = reinterpret_cast<float4 *>(a.zero_part);
    for (long long i = tid; i < a.n_part / 4; i += nth) p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int GPT, int THREADS>
__global__ void __launch_bounds__(THREADS, (THREADS <= 512 && GPT <= 8 ? 2 : 1))
    bwd_prologue_kernel(const BwdGroup grp, int stage_blocks) {
    extern __shared__ __align__(16) float smem_f[];
    const BwdPathArgs &e = grp.e[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0 && e.sd.red_cnt) *e.sd.red_cnt = 0u;
    if (prologue_prep(e.p0, e.p1, stage_blocks)) return;
    stage_dy_run<GPT>(e.sd, blockIdx.x, stage_blocks, smem_f, stage_tpr(e.sd.d_out, THREADS), THREADS);
}

// ============================================== scale pass (STG = 2) =======
// Ahead of a db-product that stages dy itself: per row the scales of the
// dy staging (s_t from max |dy.h|, sigma_t from sum |dy.h| max |l|, the same
// rules and arithmetic per element as stage_dy_run), written as s_inv, sig,
// sig_inv, and per block the maxima blkmax. One warp per row, 128-bit
// streaming loads straight from global memory (four in flight per lane), no
// shared-memory ring: nothing of the row is kept. Blocks past stage_blocks
// do the bitmap re-layouts; every thread first zeroes its share of the
// db-product's stager counters and dh partial rows.
constexpr int kScaleThreads = 1024;
__global__ void __launch_bounds__(kScaleThreads, 1) bwd_scale_kernel(const BwdGroup grp, int stage_blocks) {
    const BwdPathArgs &e = grp.e[0];
    const StageDyArgs &a = e.sd;
    __shared__ float2 red[kScaleThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.red_cnt) *a.red_cnt = 0u;
    scale_pass_zero(a);
    if (prologue_prep(e.p0, e.p1, stage_blocks)) return;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, nw = kScaleThreads / 32;
    const bool dynamic = !(a.gscale > 0.0f);
    const float ginv = dynamic ? 1.0f : 1.0f / a.gscale;
    float lmax = 0.0f;
    if (dynamic) {
        for (int k = lane; k < a.r; k += 32) lmax = fmaxf(lmax, fabsf(__ldg(a.l + k)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    }
    const int G = a.d_out / 4;
    const float4 *dy4 = reinterpret_cast<const float4 *>(a.dy);
    const float4 *h4 = reinterpret_cast<const float4 *>(a.h);
    const int row0 = (int)((long long)blockIdx.x * a.M / stage_blocks);
    const int row1 = (int)((long long)(blockIdx.x + 1) * a.M / stage_blocks);
    float2 mx = make_float2(0.0f, 0.0f);
    for (int t = row0 + warp; t < row1; t += nw) {
        const float4 *src = dy4 + (size_t)t * G;
        float amax = 0.0f, l1 = 0.0f;
        int c = lane;
        for (; c + 96 < G; c += 128) {
            float4 d[4], f[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                d[i] = __ldcs(src + c + 32 * i);
                f[i] = __ldg(h4 + c + 32 * i);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float vx = fabsf(d[i].x * f[i].x), vy = fabsf(d[i].y * f[i].y);
                const float vz = fabsf(d[i].z * f[i].z), vw = fabsf(d[i].w * f[i].w);
                amax = fmaxf(amax, fmaxf(fmaxf(vx, vy), fmaxf(vz, vw)));
                l1 += (vx + vy) + (vz + vw);
            }
        }
        for (; c < G; c += 32) {
            const float4 d = __ldcs(src + c), f = __ldg(h4 + c);
            const float vx = fabsf(d.x * f.x), vy = fabsf(d.y * f.y), vz = fabsf(d.z * f.z), vw = fabsf(d.w * f.w);
            amax = fmaxf(amax, fmaxf(fmaxf(vx, vy), fmaxf(vz, vw)));
            l1 += (vx + vy) + (vz + vw);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
        }
        if (lane == 0) {
            float s = a.gscale, sig = a.gscale;
            bool counts = true;
            if (dynamic) {
                const bool fin = amax > 0.0f && amax <= 3.402823466e38f;
                counts = fin;
                s = fin ? pow2i(14 - ceil_log2_pos(amax)) : 1.0f;
                sig = s;
                const float bound = l1 * lmax;  // bound on |db_t . l|, unscaled
                if (fin && bound > 0.0f && bound <= 3.402823466e38f) sig = pow2i(15 - ceil_log2_pos(bound));
            }
            const float si = dynamic ? pow2_recip(s) : ginv, gi = dynamic ? pow2_recip(sig) : ginv;
            a.s_inv[t] = si;
            a.sig[t] = sig;
            a.sig_inv[t] = gi;
            if (counts) mx = make_float2(fmaxf(mx.x, si), fmaxf(mx.y, gi));
        }
    }
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < nw; ++i) {
            mx.x = fmaxf(mx.x, red[i].x);
            mx.y = fmaxf(mx.y, red[i].y);
        }
        a.blkmax[blockIdx.x] = mx;
    }
}

// Streaming form of the same prologue (rows up to kSdMaxCols wide): one block
// per SM, a producer warp feeding row batches through a shared-memory ring.
// Blocks past stage_blocks only do bitmap re-layouts.
template <int Q>
__global__ void __launch_bounds__(kSdThreads, 1)
    bwd_stream_kernel(const BwdGroup grp, int stage_blocks) {
    extern __shared__ __align__(128) unsigned char smem_b[];
    const BwdPathArgs &e = grp.e[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0 && e.sd.red_cnt) *e.sd.red_cnt = 0u;
    const int extra = (int)gridDim.x - stage_blocks;
    if (extra > 0 && (int)blockIdx.x >= stage_blocks) {
        prep_share(e.p0, e.p1, (int)blockIdx.x - stage_blocks, extra);
        return;
    }
    stage_dy_stream<Q>(e.sd, blockIdx.x, stage_blocks, smem_b, e.p0, e.p1, extra > 0 ? 0 : stage_blocks);
}

int stage_dy_blocks(int M, int d_out) {
    const int rb = kStageThreads / stage_tpr(d_out);
    const int batches = (M + rb - 1) / rb;
    return batches < kStageMaxBlocks ? batches : kStageMaxBlocks;
}

// ============================================================== reduce =====
// out[f] += sum_p part[p][f]. A block of 32 warps owns 128 consecutive columns
// of one segment (a float4 per lane); warp w sums rows w, w+32, ... (their
// loads issued together: about one memory round trip for the row counts of
// the layer's partials) and the 32 warp sums are added in warp order, so the
// result does not depend on scheduling. Segment widths are multiples of 32.
constexpr int kReduceWarps = 32;
constexpr int kReduceCols = 128;

__global__ void __launch_bounds__(kReduceWarps * 32) reduce_partials_kernel(const ReduceGroup grp) {
    __shared__ float4 red[kReduceWarps][32];
    // block row blockIdx.y: the segments of path blockIdx.y of the group
    const ReduceSeg &a = grp.a[blockIdx.y], &b = grp.b[blockIdx.y], &c = grp.c[blockIdx.y];
    pdl_wait();
    pdl_launch_dependents();
    const int nba = (a.n + kReduceCols - 1) / kReduceCols, nbb = (b.n + kReduceCols - 1) / kReduceCols;
    const float *part;
    float *out;
    int rows, n, col0;
    if ((int)blockIdx.x < nba) {
        part = a.part, out = a.out, rows = a.rows, n = a.n, col0 = blockIdx.x * kReduceCols;
    } else if ((int)blockIdx.x < nba + nbb) {
        part = b.part, out = b.out, rows = b.rows, n = b.n, col0 = (blockIdx.x - nba) * kReduceCols;
    } else {
        part = c.part, out = c.out, rows = c.rows, n = c.n, col0 = (blockIdx.x - nba - nbb) * kReduceCols;
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int col = col0 + 4 * lane;  // n is a multiple of 32: a lane's float4 is wholly in or out
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < n) {
#pragma unroll 8
        for (int p = w; p < rows; p += kReduceWarps) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(part + (long long)p * n + col));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    red[w][lane] = acc;
    __syncthreads();
    if (w == 0 && col < n) {
        float4 t = red[0][lane];
#pragma unroll
        for (int i = 1; i < kReduceWarps; ++i) {
            const float4 o = red[i][lane];
            t.x += o.x;
            t.y += o.y;
            t.z += o.z;
            t.w += o.w;
        }
        float4 *dst = reinterpret_cast<float4 *>(out + col);
        float4 d = *dst;
        d.x += t.x;
        d.y += t.y;
        d.z += t.z;
        d.w += t.w;
        *dst = d;
    }
}

// ============================================================ launchers ====
namespace {
std::mutex g_launch_mu;
std::map<std::tuple<int, const void *, int, size_t>, int> g_occupancy;
std::map<std::pair<int, const void *>, int> g_prepared;
}  // namespace

int current_device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

int occupancy_blocks(const void *kernel, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const auto key = std::make_tuple(dev, kernel, threads, smem);
    std::lock_guard<std::mutex> lk(g_launch_mu);
    auto it = g_occupancy.find(key);
    if (it != g_occupancy.end()) return it->second;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess) per_sm = 1;
    if (per_sm < 1) per_sm = 1;
    g_occupancy[key] = per_sm;
    return per_sm;
}

cudaError_t prepare_once(const void *kernel, int max_dyn_smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_launch_mu);
    auto key = std::make_pair(dev, kernel);
    auto it = g_prepared.find(key);
    if (it != g_prepared.end() && it->second >= max_dyn_smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    g_prepared[key] = max_dyn_smem;
    return cudaSuccess;
}

static int grid_for(long long items, int per_block, int cap = 1 << 20) {
    long long g = (items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

cudaError_t launch_pack_signs(const float *src, uint32_t *bits, int rows, int r, cudaStream_t s) {
    const long long words = (long long)rows * ((r + 31) / 32);
    trace_before("pack_signs", s);
    cudaError_t e = launch_k(pack_signs_kernel, dim3(grid_for(words, 8, 65535)), dim3(256), 0, s, src, bits, rows, r);
    trace_after(s);
    return e;
}

cudaError_t launch_unpack_signs(const uint32_t *bits, uint16_t *dst, int rows, int r, cudaStream_t s) {
    const long long words = (long long)rows * ((r + 31) / 32);
    trace_before("unpack_signs", s);
    cudaError_t e = launch_k(unpack_signs_kernel, dim3(grid_for(words, 256, 65535)), dim3(256), 0, s, bits, dst, rows, r);
    trace_after(s);
    return e;
}

template <int KQ>
static cudaError_t launch_fwd_prologue_rows(const FwdGroup &grp, const float *x, int M, int d_in, cudaStream_t s) {
    cudaError_t pe = prepare_kernel_once(fwd_prologue_rows_kernel<KQ>, 0);
    if (pe != cudaSuccess) return pe;
    const int T = sx_threads(d_in);
    const int wave = occupancy_blocks(reinterpret_cast<const void *>(fwd_prologue_rows_kernel<KQ>), T, 0) *
                     current_device_sms();
    const int nchunks = (M + sx_rows(KQ) - 1) / sx_rows(KQ);
    const int bs = nchunks < wave ? nchunks : wave;
    const int pb = prep_blocks(grp.e[0].p0, T) + prep_blocks(grp.e[0].p1, T);
    const int grid = bs + pb <= wave ? bs + pb : bs;
    trace_before("fwd_prologue", s);
    cudaError_t e = launch_k(fwd_prologue_rows_kernel<KQ>, dim3(grid, grp.n), dim3(T), 0, s, grp, x, M, d_in, bs);
    trace_after(s);
    return e;
}

template <int KQ>
static cudaError_t launch_fwd_prologue_stream(const FwdGroup &grp, const float *x, int M, int d_in, cudaStream_t s) {
    cudaError_t pe = prepare_kernel_once(fwd_prologue_stream_kernel<KQ>, kSxsHeadBytes + kSxsRingBytes);
    if (pe != cudaSuccess) return pe;
    const int sms = current_device_sms();
    const SxPlan pl = sxs_plan(d_in);
    int sb = (M + pl.rs - 1) / pl.rs;
    if (sb > sms) sb = sms;
    const int pb = prep_blocks(grp.e[0].p0, kSxsThreads) + prep_blocks(grp.e[0].p1, kSxsThreads);
    const int grid = sb + pb <= sms ? sb + pb : sb;
    trace_before("fwd_prologue", s);
    cudaError_t e = launch_k(fwd_prologue_stream_kernel<KQ>, dim3(grid, grp.n), dim3(kSxsThreads),
                             sxs_smem_bytes(d_in), s, grp, x, M, d_in, sb);
    trace_after(s);
    return e;
}

cudaError_t launch_fwd_prologue(const FwdGroup &grp, const float *x, int M, int d_in, cudaStream_t s) {
    if (grp.n < 1 || grp.n > kMaxGroupPaths) return cudaErrorInvalidValue;
    // Streaming for large x (measured on GB300: 134 MB of x 43 -> 39 us, 805 MB
    // 233 -> 190 us), rows for small ones (8 MB: 8.2 us rows, 10.4 streamed).
    // BLR_X_STAGE=stream|rows|flat forces a form.
    const char *form = std::getenv("BLR_X_STAGE");
    const bool want_stream = form ? std::strcmp(form, "stream") == 0 : (long long)M * d_in * 4 >= (64ll << 20);
    if (d_in <= kSxMaxCols && want_stream && sxs_plan(d_in).nst >= 2) {
        switch (sx_kq(d_in)) {
            case 1: return launch_fwd_prologue_stream<1>(grp, x, M, d_in, s);
            case 2: return launch_fwd_prologue_stream<2>(grp, x, M, d_in, s);
            case 4: return launch_fwd_prologue_stream<4>(grp, x, M, d_in, s);
            case 6: return launch_fwd_prologue_stream<6>(grp, x, M, d_in, s);
            default: return launch_fwd_prologue_stream<8>(grp, x, M, d_in, s);
        }
    }
    if (d_in <= kSxMaxCols && !(form && std::strcmp(form, "flat") == 0)) {
        switch (sx_kq(d_in)) {
            case 1: return launch_fwd_prologue_rows<1>(grp, x, M, d_in, s);
            case 2: return launch_fwd_prologue_rows<2>(grp, x, M, d_in, s);
            case 4: return launch_fwd_prologue_rows<4>(grp, x, M, d_in, s);
            case 6: return launch_fwd_prologue_rows<6>(grp, x, M, d_in, s);
            default: return launch_fwd_prologue_rows<8>(grp, x, M, d_in, s);
        }
    }
    cudaError_t pe = prepare_kernel_once(fwd_prologue_kernel, 0);
    if (pe != cudaSuccess) return pe;
    // one wave of persistent blocks (each does its share of the re-layouts, then
    // grid-strides over x), but no more blocks than 8-group shares of x
    const int wave = occupancy_blocks(reinterpret_cast<const void *>(fwd_prologue_kernel), 256, 0) *
                     current_device_sms();
    const long long groups = (long long)M * (d_in / 4);
    const int bs = grid_for(groups, 256 * 8, wave);
    // re-layout-only blocks where the wave has room for them
    const int pb = prep_blocks(grp.e[0].p0, 256) + prep_blocks(grp.e[0].p1, 256);
    const int grid = bs + pb <= wave ? bs + pb : bs;
    trace_before("fwd_prologue", s);
    cudaError_t e = launch_k(fwd_prologue_kernel, dim3(grid, grp.n), dim3(256), 0, s, grp, x, M, d_in, bs);
    trace_after(s);
    return e;
}

template <int GPT, int THREADS = kStageThreads>
static cudaError_t launch_bwd_prologue_t(const BwdGroup &grp, cudaStream_t s) {
    const StageDyArgs &a = grp.e[0].sd;
    const SignPrep &p0 = grp.e[0].p0, &p1 = grp.e[0].p1;
    const int tpr = stage_tpr(a.d_out, THREADS);
    const int rb_n = THREADS / tpr;
    const size_t smem = stage_dy_smem_bytes(a.d_out, tpr, rb_n * tpr);
    cudaError_t pe = prepare_kernel_once(bwd_prologue_kernel<GPT, THREADS>, 200 * 1024);
    if (pe != cudaSuccess) return pe;
    const int per_sm = occupancy_blocks(reinterpret_cast<const void *>(bwd_prologue_kernel<GPT, THREADS>), THREADS,
                                        smem);
    const int sms = current_device_sms();
    int sb = stage_dy_blocks(a.M, a.d_out);
    if (sb > per_sm * sms) sb = per_sm * sms;
    // re-layout-only blocks where the wave has room for them
    const int pb = prep_blocks(p0, THREADS) + prep_blocks(p1, THREADS);
    const int grid = sb + pb <= per_sm * sms ? sb + pb : sb;
    trace_before("bwd_prologue", s);
    cudaError_t e = launch_k(bwd_prologue_kernel<GPT, THREADS>, dim3(grid, grp.n), dim3(THREADS), smem, s, grp, sb);
    trace_after(s);
    if (e == cudaSuccess && a.rows_used) *a.rows_used = sb;
    return e;
}

template <int Q>
static cudaError_t launch_bwd_stream_t(const BwdGroup &grp, cudaStream_t s) {
    const StageDyArgs &a = grp.e[0].sd;
    const SignPrep &p0 = grp.e[0].p0, &p1 = grp.e[0].p1;
    cudaError_t pe = prepare_kernel_once(bwd_stream_kernel<Q>, kSdHeadBytes + kSdRingBytes);
    if (pe != cudaSuccess) return pe;
    const int sms = current_device_sms();
    const SdPlan pl = sd_plan(a.d_out);
    int sb = (a.M + pl.ngrp - 1) / pl.ngrp;
    if (sb > sms) sb = sms;
    const int cap = stage_dy_blocks(a.M, a.d_out);
    if (sb > cap) sb = cap;
    // re-layout-only blocks on SMs the staging leaves idle
    const int pb = prep_blocks(p0, kSdThreads) + prep_blocks(p1, kSdThreads);
    const int grid = sb + pb <= sms ? sb + pb : sb;
    trace_before("bwd_prologue", s);
    cudaError_t e = launch_k(bwd_stream_kernel<Q>, dim3(grid, grp.n), dim3(kSdThreads), sd_smem_bytes(a.d_out), s,
                             grp, sb);
    trace_after(s);
    if (e == cudaSuccess && a.rows_used) *a.rows_used = sb;
    return e;
}

// BLR_DY_STAGE=rows selects the register-staged row kernel for every width
// (the streaming kernel is used for rows up to kSdMaxCols otherwise).
static bool dy_stage_rows_forced() {
    const char *e = std::getenv("BLR_DY_STAGE");
    return e && std::strcmp(e, "rows") == 0;
}

cudaError_t launch_bwd_prologue(const BwdGroup &grp, cudaStream_t s) {
    if (grp.n < 1 || grp.n > kMaxGroupPaths) return cudaErrorInvalidValue;
    const StageDyArgs &a = grp.e[0].sd;
    if (sd_supported(a.d_out) && !dy_stage_rows_forced()) {
        switch (sd_plan(a.d_out).Q) {
            case 2: return launch_bwd_stream_t<2>(grp, s);
            case 4: return launch_bwd_stream_t<4>(grp, s);
            case 6: return launch_bwd_stream_t<6>(grp, s);
            default: return launch_bwd_stream_t<8>(grp, s);
        }
    }
    switch (stage_gpt(a.d_out)) {
        case 1: return launch_bwd_prologue_t<1>(grp, s);
        case 2: return launch_bwd_prologue_t<2>(grp, s);
        case 3:
        case 4: return launch_bwd_prologue_t<4>(grp, s);
        case 5:
        case 6:
        case 7:
        case 8: return launch_bwd_prologue_t<8>(grp, s);
        default: break;
    }
    // rows wider than 16384: 1024-thread blocks, 8 groups per thread (measured
    // on GB300, 4000 rows of 32768: 271 -> 228 us against 512 threads with 16;
    // at 12288 the 512-thread blocks stay faster, 293 against 310 us)
    if (stage_gpt(a.d_out, 1024) <= 8) return launch_bwd_prologue_t<8, 1024>(grp, s);
    return cudaErrorInvalidValue;
}

// The scale pass ahead of a db-product that stages dy itself (StageDyArgs
// zero_cnt, zero_part): one block of bwd_scale_kernel per SM, plus blocks
// for the bitmap re-layouts where the wave has room for them.
cudaError_t launch_bwd_scales(const BwdGroup &grp, cudaStream_t s) {
    if (grp.n != 1) return cudaErrorInvalidValue;
    const StageDyArgs &a = grp.e[0].sd;
    const SignPrep &p0 = grp.e[0].p0, &p1 = grp.e[0].p1;
    const int sms = current_device_sms();
    int sb = sms;
    const int cap = stage_dy_blocks(a.M, a.d_out);  // blkmax rows of the workspace
    if (sb > cap) sb = cap;
    if (sb > a.M) sb = a.M;
    const int pb = prep_blocks(p0, kScaleThreads) + prep_blocks(p1, kScaleThreads);
    const int grid = sb + pb <= sms ? sb + pb : sb;
    trace_before("bwd_scales", s);
    cudaError_t e = launch_k(bwd_scale_kernel, dim3(grid), dim3(kScaleThreads), 0, s, grp, sb);
    trace_after(s);
    if (e == cudaSuccess && a.rows_used) *a.rows_used = sb;
    return e;
}

cudaError_t launch_prep(SignPrep p0, SignPrep p1, uint32_t *status, unsigned int *cnt, int ncnt, const char *name,
                        cudaStream_t s) {
    cudaError_t pe = prepare_kernel_once(prep_kernel, 0);
    if (pe != cudaSuccess) return pe;
    const int wave = occupancy_blocks(reinterpret_cast<const void *>(prep_kernel), 256, 0) * current_device_sms();
    int grid = prep_blocks(p0, 256) + prep_blocks(p1, 256);
    if (grid < (ncnt + 255) / 256) grid = (ncnt + 255) / 256;
    if (grid > wave) grid = wave;
    if (grid < 1) grid = 1;
    trace_before(name, s);
    cudaError_t e = launch_k(prep_kernel, dim3(grid), dim3(256), 0, s, p0, p1, status, cnt, ncnt);
    trace_after(s);
    return e;
}

cudaError_t launch_prep_group(const FwdGroup &grp, unsigned int *cnt0, long long pstride, int ncnt, const char *name,
                              cudaStream_t s) {
    if (grp.n < 1 || grp.n > kMaxGroupPaths) return cudaErrorInvalidValue;
    cudaError_t pe = prepare_kernel_once(prep_group_kernel, 0);
    if (pe != cudaSuccess) return pe;
    const int wave = occupancy_blocks(reinterpret_cast<const void *>(prep_group_kernel), 256, 0) *
                     current_device_sms();
    int grid = prep_blocks(grp.e[0].p0, 256) + prep_blocks(grp.e[0].p1, 256);
    if (grid < (ncnt + 255) / 256) grid = (ncnt + 255) / 256;
    if (grid * grp.n > wave) grid = (wave + grp.n - 1) / grp.n;
    if (grid < 1) grid = 1;
    trace_before(name, s);
    cudaError_t e = launch_k(prep_group_kernel, dim3(grid, grp.n), dim3(256), 0, s, grp, cnt0, pstride, ncnt);
    trace_after(s);
    return e;
}

cudaError_t launch_reduce_partials(const ReduceGroup &grp, cudaStream_t s) {
    if (grp.n < 1 || grp.n > kMaxGroupPaths) return cudaErrorInvalidValue;
    const ReduceSeg &a = grp.a[0], &b = grp.b[0], &c = grp.c[0];
    const int blocks = (a.n + kReduceCols - 1) / kReduceCols + (b.n + kReduceCols - 1) / kReduceCols +
                       (c.n + kReduceCols - 1) / kReduceCols;
    cudaError_t pe = prepare_kernel_once(reduce_partials_kernel, 0);
    if (pe != cudaSuccess) return pe;
    trace_before("reduce_partials", s);
    cudaError_t e = launch_k(reduce_partials_kernel, dim3(blocks, grp.n), dim3(kReduceWarps * 32), 0, s, grp);
    trace_after(s);
    return e;
}

}  // namespace blr
