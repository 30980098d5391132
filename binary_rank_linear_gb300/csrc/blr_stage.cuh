// Bandwidth stages of the blr layer as device functions, shared by the
// stand-alone prologue kernels (blr_aux.cu) and the fused small-M kernels
// (blr_small.cu): bitmap re-layout, x staging, dy staging with the dh sums,
// and the fixed-order reduction of per-tile partial sums.
#pragma once

#include <cuda_fp16.h>

#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

// ============================================ bitmap re-layout (prep) ======
// Destination order [kb][n][2] u32 (kb < 2 ceil(K/128), n < Ns): word
// (n, 2kb + w) covers reduction indices 64kb + 32w .. +31 of operand row n,
// pair-ready. Rows past N and words past K are written from an all-zero word.
__host__ __device__ __forceinline__ int prep_kwords(int K) { return 4 * ((K + 127) / 128); }

__host__ __device__ __forceinline__ int prep_blocks(const SignPrep &p, int threads) {
    if (p.kind == 2) {
        const long long words = (long long)p.N * (p.K / 32);
        return (int)((words + threads - 1) / threads);
    }
    if (p.kind == 0) {
        const long long units = (long long)p.Ns * prep_kwords(p.K);
        return (int)((units + threads - 1) / threads);
    }
    const long long warps = (long long)prep_kwords(p.K) * (p.Ns / 32);
    return (int)((warps + threads / 32 - 1) / (threads / 32));
}

__device__ inline void prep_run(const SignPrep &p, int block, int threads);

// This block's share of the two re-layouts: virtual prep blocks block,
// block + nblocks, ... (done first by every block of a prologue, so that the
// re-layout never runs as a tail after the staging).
__device__ inline void prep_share(const SignPrep &p0, const SignPrep &p1, int block, int nblocks) {
    const int b0 = prep_blocks(p0, blockDim.x), b1 = prep_blocks(p1, blockDim.x);
    for (int v = block; v < b0 + b1; v += nblocks) {
        if (v < b0)
            prep_run(p0, v, blockDim.x);
        else
            prep_run(p1, v - b0, blockDim.x);
    }
}

__device__ inline void prep_run(const SignPrep &p, int block, int threads) {
    if (p.kind == 2) {
        // plane: one bitmap word -> 32 f16 signs (64 bytes) of its row, through
        // the pair-ready transform and pair expansion of the TMEM expanders
        const int words = p.K / 32;
        const long long u = (long long)block * threads + threadIdx.x;
        if (u >= (long long)p.N * words) return;
        const uint32_t w = sign_word_pair_ready(p.src[u]);
        uint4 *dst = reinterpret_cast<uint4 *>(p.dst + u * 16);  // row n, ranks 32(u % words) ..
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(sign_pair(w, 4 * i), sign_pair(w, 4 * i + 1), sign_pair(w, 4 * i + 2),
                                sign_pair(w, 4 * i + 3));
        return;
    }
    const int kw_total = prep_kwords(p.K);
    if (p.kind == 0) {
        // direct: src [N][K/32]
        const int words = p.K / 32;
        const long long u = (long long)block * threads + threadIdx.x;
        if (u >= (long long)p.Ns * kw_total) return;
        const int n = (int)(u % p.Ns);
        const int kw = (int)(u / p.Ns);
        const uint32_t w = (kw < words && n < p.N) ? p.src[(long long)n * words + kw] : 0u;
        p.dst[((long long)(kw >> 1) * p.Ns + n) * 2 + (kw & 1)] = sign_word_pair_ready(w);
    } else {
        // transpose: src [K][N/32]; one warp per 32 x 32 bit block.
        const int nwords = p.N / 32;
        const int nwords_s = p.Ns / 32;
        const long long wi = (long long)block * (threads / 32) + threadIdx.x / 32;
        if (wi >= (long long)kw_total * nwords_s) return;
        const int kw = (int)(wi / nwords_s);
        const int nw = (int)(wi % nwords_s);
        const int lane = threadIdx.x & 31;
        const bool in = kw < p.K / 32 && nw < nwords;
        const uint32_t mine = in ? p.src[(long long)(32 * kw + lane) * nwords + nw] : 0u;
        uint32_t keep = 0;
#pragma unroll
        for (int b = 0; b < 32; ++b) {
            const uint32_t col = __ballot_sync(0xFFFFFFFFu, (mine >> b) & 1u);
            if (lane == b) keep = col;
        }
        const int n = 32 * nw + lane;
        p.dst[((long long)(kw >> 1) * p.Ns + n) * 2 + (kw & 1)] = sign_word_pair_ready(keep);
    }
}

// Re-layout work interleaved with a streaming kernel's consumers: a cursor
// over this block's share of the virtual prep blocks (each `threads` wide,
// threads = the consumer count), which a consumer warp advances by doing its
// own part of one virtual block (its 32 threads; kind 1 is a warp-wide
// transpose). Warps advance independently; every part is done once.
struct PrepCursor {
    int v, b0, b1, nblocks, threads;
    __device__ PrepCursor(const SignPrep &p0, const SignPrep &p1, int block, int nblocks_, int threads_, bool on)
        : v(block), b0(on ? prep_blocks(p0, threads_) : 0), b1(on ? prep_blocks(p1, threads_) : 0),
          nblocks(nblocks_), threads(threads_) {}
    __device__ bool done() const { return v >= b0 + b1; }
    __device__ void step(const SignPrep &p0, const SignPrep &p1) {
        if (v < b0)
            prep_run(p0, v, threads);
        else
            prep_run(p1, v - b0, threads);
        v += nblocks;
    }
};

// ============================================================ stage x ======
// train_mm.rs, `cvt_col` staging: x16 = f16(x . g), forward unscaled.
// A thread walks float4 groups (row-major [M][d_in/4]) with a grid stride,
// four groups per round (four loads in flight); row and column advance by
// precomputed steps, so the loop does no division.
__device__ inline void stage_x_run(const float *__restrict__ x, const float *__restrict__ g, uint16_t *__restrict__ x16,
                            int M, int d_in, int block, int nblocks) {
    const int g4n = d_in / 4;
    const long long groups = (long long)M * g4n;
    const long long stride = (long long)nblocks * blockDim.x;  // groups between a thread's consecutive visits
    const int step_col = (int)(stride % g4n);
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const float4 *gg = reinterpret_cast<const float4 *>(g);
    uint2 *o = reinterpret_cast<uint2 *>(x16);
    long long i = (long long)block * blockDim.x + threadIdx.x;
    int col = (int)(i % g4n);
    constexpr int kU = 8;
    for (; i < groups; i += kU * stride) {
        float4 v[kU], f[kU];
        long long idx[kU];
        long long ii = i;
        int cc = col;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            idx[u] = ii;
            if (ii < groups) {
                v[u] = __ldcs(x4 + ii);
                f[u] = __ldg(gg + cc);
            }
            ii += stride;
            cc += step_col;
            if (cc >= g4n) cc -= g4n;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (idx[u] < groups) {
                uint2 out;
                out.x = pack_half2(v[u].x * f[u].x, v[u].y * f[u].y);
                out.y = pack_half2(v[u].z * f[u].z, v[u].w * f[u].w);
                o[idx[u]] = out;
            }
        }
        col = cc;
    }
}

// x staging by rows (d_in up to kSxMaxCols): a block of T threads walks
// chunks of R consecutive rows; thread t owns the float4 columns t, t + T, ..
// (KQ of them) and keeps their g factors in registers, so the loop is R * KQ
// streaming loads in flight, the products and 8-byte stores.
constexpr int kSxMaxCols = 16384;

__host__ __device__ inline int sx_kq(int d_in) {
    const int q = (d_in / 4 + 511) / 512;  // blocks of at most 512 threads
    return q <= 2 ? q : (q <= 4 ? 4 : (q <= 6 ? 6 : 8));
}

__host__ __device__ inline int sx_threads(int d_in) {
    const int kq = sx_kq(d_in);
    const int t = (d_in / 4 + kq - 1) / kq;
    return (t + 31) / 32 * 32;
}

__host__ __device__ constexpr int sx_rows(int kq) { return (8 + kq - 1) / kq; }

template <int KQ>
__device__ void stage_x_rows(const float *__restrict__ x, const float *__restrict__ g, uint16_t *__restrict__ x16,
                             int M, int d_in, int block, int nblocks) {
    constexpr int R = sx_rows(KQ);
    const int G = d_in / 4;
    const int T = blockDim.x;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    uint2 *o = reinterpret_cast<uint2 *>(x16);
    float4 gv[KQ];
#pragma unroll
    for (int k = 0; k < KQ; ++k) {
        const int col = threadIdx.x + k * T;
        gv[k] = col < G ? __ldg(reinterpret_cast<const float4 *>(g) + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int nchunks = (M + R - 1) / R;
    for (int c = block; c < nchunks; c += nblocks) {
        float4 v[R][KQ];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int row = c * R + j;
#pragma unroll
            for (int k = 0; k < KQ; ++k) {
                const int col = threadIdx.x + k * T;
                if (row < M && col < G) v[j][k] = __ldcs(x4 + (size_t)row * G + col);
            }
        }
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int row = c * R + j;
#pragma unroll
            for (int k = 0; k < KQ; ++k) {
                const int col = threadIdx.x + k * T;
                if (row < M && col < G) {
                    uint2 out;
                    out.x = pack_half2(v[j][k].x * gv[k].x, v[j][k].y * gv[k].y);
                    out.y = pack_half2(v[j][k].z * gv[k].z, v[j][k].w * gv[k].w);
                    o[(size_t)row * G + col] = out;
                }
            }
        }
    }
}

// x staging as a stream of row batches (d_in up to kSxMaxCols), the ring and
// producer of the streaming dy staging below without its row reductions: a
// producer warp bulk-copies batches of consecutive rows of x into a
// shared-memory ring; the consumer threads form row groups of T threads (T as
// in stage_x_rows) that own fixed float4 columns, keep their g factors in
// registers, and write f16(x.g) with 8-byte stores.
constexpr int kSxsWarps = 16;
constexpr int kSxsThreads = (kSxsWarps + 1) * 32;
constexpr int kSxsRingBytes = 200 * 1024;
constexpr int kSxsHeadBytes = 256;

struct SxPlan {
    int T;      // threads per row group
    int ngr;    // row groups
    int rs;     // rows per batch (a multiple of ngr)
    int nst;    // ring stages
};

__host__ __device__ inline SxPlan sxs_plan(int d_in) {
    SxPlan p;
    p.T = sx_threads(d_in);
    p.ngr = (kSxsWarps * 32) / p.T;
    int m = 32768 / (p.ngr * d_in * 4);
    if (m < 1) m = 1;
    p.rs = p.ngr * m;
    p.nst = kSxsRingBytes / (p.rs * d_in * 4);
    if (p.nst > 8) p.nst = 8;
    return p;
}

__host__ __device__ inline size_t sxs_smem_bytes(int d_in) {
    const SxPlan p = sxs_plan(d_in);
    return (size_t)kSxsHeadBytes + (size_t)p.nst * p.rs * d_in * 4;
}

// The block does its share (1 of prep_nblocks) of the two bitmap re-layouts
// while its consumers wait for data.
template <int KQ>
__device__ void stage_x_stream(const float *__restrict__ x, const float *__restrict__ g, uint16_t *__restrict__ x16,
                               int M, int d_in, int block, int nblocks, unsigned char *smem, uint32_t *status,
                               const SignPrep &p0, const SignPrep &p1, int prep_nblocks) {
    const SxPlan pl = sxs_plan(d_in);
    const int G = d_in / 4;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [8]
    uint64_t *empty = full + 8;                            // [8]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 128);
    unsigned char *ring = smem + kSxsHeadBytes;
    const uint32_t stage_bytes = (uint32_t)pl.rs * d_in * 4;
    const int row0 = (int)((long long)block * M / nblocks);
    const int row1 = (int)((long long)(block + 1) * M / nblocks);
    const int nbatch = (row1 - row0 + pl.rs - 1) / pl.rs;

    if (threadIdx.x == 0) {
        for (int i = 0; i < pl.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kSxsWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool producer = warp == kSxsWarps && lane == 0;
    uint64_t pol = 0;
    int issued = 0;
    auto issue = [&](int i) {
        const int st = i % pl.nst;
        const int r = row0 + i * pl.rs;
        const int nr = row1 - r < pl.rs ? row1 - r : pl.rs;
        mbar_arrive_expect_tx(&full[st], (uint32_t)nr * d_in * 4);
        bulk_load_hint(ring + (size_t)st * stage_bytes, x + (size_t)r * d_in, (uint32_t)nr * d_in * 4, &full[st], pol);
        issued = i + 1;
    };
    if (producer) {
        pol = l2_policy_evict_first();
        for (int i = 0; i < nbatch && i < pl.nst; ++i) issue(i);
    }
    __syncwarp();
    if (warp == kSxsWarps) {
        if (lane != 0) return;
        for (int i = issued; i < nbatch; ++i) {
            const int st = i % pl.nst;
            if (!mbar_wait(&empty[st], (uint32_t)((i / pl.nst - 1) & 1), abort_flag)) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(status, kStTimeoutStage);
                }
                break;
            }
            issue(i);
        }
        // every issued copy lands before the block may exit
        for (int j = issued - pl.nst < 0 ? 0 : issued - pl.nst; j < issued; ++j)
            if (!mbar_wait(&full[j % pl.nst], (uint32_t)((j / pl.nst) & 1), abort_flag, false))
                atomicOr(status, kStTimeoutDrain);
        return;
    }
    // ---- consumers ----
    const int grp = threadIdx.x / pl.T;
    const int ti = threadIdx.x % pl.T;
    const bool active = grp < pl.ngr;
    float4 gv[KQ];
#pragma unroll
    for (int k = 0; k < KQ; ++k) {
        const int col = ti + k * pl.T;
        gv[k] = active && col < G ? __ldg(reinterpret_cast<const float4 *>(g) + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint2 *o = reinterpret_cast<uint2 *>(x16);
    // the block's share of the re-layouts fills the consumers' waits for data
    PrepCursor prep(p0, p1, block, prep_nblocks, kSxsWarps * 32, prep_nblocks > 0);
    for (int i = 0; i < nbatch; ++i) {
        const int st = i % pl.nst;
        const uint32_t par = (uint32_t)((i / pl.nst) & 1);
        while (!prep.done() && !__shfl_sync(0xFFFFFFFFu, (int)mbar_test_wait(&full[st], par), 0)) prep.step(p0, p1);
        if (!mbar_wait(&full[st], par, abort_flag)) {
            if (!*abort_flag) {
                *abort_flag = 1;
                atomicOr(status, kStTimeoutStage);
            }
            break;
        }
        const int r = row0 + i * pl.rs;
        const int nr = row1 - r < pl.rs ? row1 - r : pl.rs;
        const float4 *sx = reinterpret_cast<const float4 *>(ring + (size_t)st * stage_bytes);
        if (active) {
            for (int j = grp; j < nr; j += pl.ngr) {
#pragma unroll
                for (int k = 0; k < KQ; ++k) {
                    const int col = ti + k * pl.T;
                    if (col < G) {
                        const float4 v = sx[(size_t)j * G + col];
                        uint2 out;
                        out.x = pack_half2(v.x * gv[k].x, v.y * gv[k].y);
                        out.y = pack_half2(v.z * gv[k].z, v.w * gv[k].w);
                        o[(size_t)(r + j) * G + col] = out;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    while (!prep.done()) prep.step(p0, p1);
}

// =========================================================== stage dy ======
// Backward staging (train_mm.rs, `blr_backward`: cvt of dy with the column
// factor h under the gradient scale, and `colsum_prod` of dy and c for dh).
// The first `nthr` threads of a block own whole token rows: `tpr` threads
// share a row and the block works on nthr/tpr rows at a time, visiting rows
// in a grid-stride loop (the other threads of the block only keep step with
// its barriers). Per row t (one joint block reduction of the pair (max, sum)):
//   A_t     = max_i |dy_ti h_i|,  L_t = sum_i |dy_ti h_i|
//   s_t     = gscale, or 2^(14 - ceil(log2 A_t))   (1 if A_t is 0 or not finite)
//   dy16_t  = f16(dy_t . h . s_t)
//   sigma_t = gscale, or 2^(15 - ceil(log2(L_t max_k |l_k|)))
// sigma_t scales the staged db.l in the next product. Since
// |db_tk| = |sum_i dy16_ti S_ik| / s_t <= L_t (1 + 2^-11), every staged value
// |db_tk l_k sigma_t| stays below 2^15 (1 + 2^-11), under the f16 maximum
// 65504 whatever the data, while sigma_t is as large as that bound allows.
// The block accumulates sum_t dy_ti c_ti for its rows in shared memory and
// writes one partial row of dh, and the largest 1/s_t and 1/sigma_t of its
// rows with nonzero finite A_t (rows of zeros carry no gradient, and their
// scale 1 must not set the common scale of the sign-gradient products).
constexpr int kStageThreads = 512;
// floats of the staging's shared reduction buffer: float2 [2][32 warps], for
// blocks of up to 1024 threads (the dh row sums follow it)
constexpr int kStageRedFloats = 2 * 32 * 2;
constexpr int kStageMaxBlocks = 2 * 160;  // partial rows reserved per call

__host__ __device__ inline int stage_tpr(int d_out, int cap = kStageThreads) {
    const int G = d_out / 4;  // float4 groups per row
    int t = 32;
    while (t * 8 < G && t < cap) t *= 2;  // at most 8 groups per thread when possible
    return t;
}

__host__ __device__ inline int stage_gpt(int d_out, int cap = kStageThreads) {
    const int tpr = stage_tpr(d_out, cap);
    return (d_out / 4 + tpr - 1) / tpr;
}

// ceil(log2(v)) for finite v > 0.
__device__ __forceinline__ int ceil_log2_pos(float v) {
    int e;
    const float m = frexpf(v, &e);  // v = m * 2^e, m in [0.5, 1)
    return (m == 0.5f) ? e - 1 : e;
}

__device__ __forceinline__ float pow2i(int e) {
    e = e < -126 ? -126 : (e > 127 ? 127 : e);
    return __int_as_float((e + 127) << 23);
}

// Shared memory stage_dy_run needs (floats) for `tpr` threads per row.
__host__ __device__ inline size_t stage_dy_smem_bytes(int d_out, int tpr, int nthr) {
    return (kStageRedFloats + (size_t)(nthr / tpr) * d_out) * sizeof(float);
}

template <int GPT>
__device__ void stage_dy_run(const StageDyArgs &a, int block, int nblocks, float *smem, int tpr, int nthr) {
    const int rb_n = nthr / tpr;
    const int wpr = tpr / 32;  // warps per row
    const bool active = (int)threadIdx.x < nthr;
    const int rb = active ? (int)threadIdx.x / tpr : 0;
    const int ti = threadIdx.x % tpr;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int G = a.d_out / 4;
    float2 *red = reinterpret_cast<float2 *>(smem);                    // [2][32 warps]
    float4 *dh_s = reinterpret_cast<float4 *>(smem + kStageRedFloats);  // [rb_n][G]
    const bool dynamic = !(a.gscale > 0.0f);

    float lmax = 0.0f;
    if (dynamic) {
        for (int k = lane; k < a.r; k += 32) lmax = fmaxf(lmax, fabsf(__ldg(a.l + k)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    }

    const float4 *dy4 = reinterpret_cast<const float4 *>(a.dy);
    const float4 *h4 = reinterpret_cast<const float4 *>(a.h);
    const uint2 *c4 = reinterpret_cast<const uint2 *>(a.c16);
    uint2 *o4 = reinterpret_cast<uint2 *>(a.dy16);
#pragma unroll
    for (int g = 0; g < GPT; ++g) {
        const int col = g * tpr + ti;
        if (active && col < G) dh_s[rb * G + col] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const int batches = (a.M + rb_n - 1) / rb_n;
    // the block reduces and stores a batch before it loads the next one: the
    // next batch's rows of dy and c are prefetched into L2 meanwhile
    auto prefetch_batch = [&](int bt) {
        if (threadIdx.x != 0 || bt >= batches) return;
        const int r0 = bt * rb_n;
        const int nr = a.M - r0 < rb_n ? a.M - r0 : rb_n;
        bulk_prefetch_l2(a.dy + (size_t)r0 * a.d_out, (uint32_t)((size_t)nr * a.d_out * 4));
        bulk_prefetch_l2(a.c16 + (size_t)r0 * a.d_out, (uint32_t)((size_t)nr * a.d_out * 2));
    };
    prefetch_batch(block);
    int buf = 0;
    float2 mx = make_float2(0.0f, 0.0f);  // this thread's rows: max 1/s_t, max 1/sigma_t
    for (int bt = block; bt < batches; bt += nblocks, buf ^= 1) {
        prefetch_batch(bt + nblocks);
        const int t = bt * rb_n + rb;
        const bool valid = active && t < a.M;
        float4 v[GPT];
        float amax = 0.0f, l1 = 0.0f;
#pragma unroll
        for (int g = 0; g < GPT; ++g) {
            const int col = g * tpr + ti;
            v[g] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid && col < G) {
                const long long idx = (long long)t * G + col;
                const float4 d = __ldcs(dy4 + idx);
                const uint2 cw = __ldcs(c4 + idx);
                const float4 f = __ldg(h4 + col);
                v[g] = make_float4(d.x * f.x, d.y * f.y, d.z * f.z, d.w * f.w);
                const float2 c0 = __half22float2(*reinterpret_cast<const __half2 *>(&cw.x));
                const float2 c1 = __half22float2(*reinterpret_cast<const __half2 *>(&cw.y));
                float4 acc = dh_s[rb * G + col];
                acc.x += d.x * c0.x;
                acc.y += d.y * c0.y;
                acc.z += d.z * c1.x;
                acc.w += d.w * c1.y;
                dh_s[rb * G + col] = acc;
                const float4 q = make_float4(fabsf(v[g].x), fabsf(v[g].y), fabsf(v[g].z), fabsf(v[g].w));
                amax = fmaxf(amax, fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)));
                l1 += (q.x + q.y) + (q.z + q.w);
            }
        }
        float s = a.gscale, sig = a.gscale;
        bool counts = true;  // the row takes part in the block's maxima
        if (dynamic) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
            }
            if (lane == 0 && active) red[buf * 32 + warp] = make_float2(amax, l1);
            __syncthreads();
            float2 r = red[buf * 32 + rb * wpr];
            for (int i = 1; i < wpr; ++i) {
                const float2 o = red[buf * 32 + rb * wpr + i];
                r.x = fmaxf(r.x, o.x);
                r.y += o.y;
            }
            const bool fin = r.x > 0.0f && r.x <= 3.402823466e38f;
            counts = fin;
            s = fin ? pow2i(14 - ceil_log2_pos(r.x)) : 1.0f;
            sig = s;
            const float bound = r.y * lmax;  // bound on |db_t . l|, unscaled
            if (fin && bound > 0.0f && bound <= 3.402823466e38f) sig = pow2i(15 - ceil_log2_pos(bound));
        }
#pragma unroll
        for (int g = 0; g < GPT; ++g) {
            const int col = g * tpr + ti;
            if (valid && col < G) {
                uint2 st;
                st.x = pack_half2(v[g].x * s, v[g].y * s);
                st.y = pack_half2(v[g].z * s, v[g].w * s);
                __stcs(o4 + (long long)t * G + col, st);
            }
        }
        if (valid && ti == 0) {
            a.s_inv[t] = 1.0f / s;
            a.sig[t] = sig;
            a.sig_inv[t] = 1.0f / sig;
            if (counts) mx = make_float2(fmaxf(mx.x, 1.0f / s), fmaxf(mx.y, 1.0f / sig));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx.x = fmaxf(mx.x, __shfl_xor_sync(0xFFFFFFFFu, mx.x, o));
        mx.y = fmaxf(mx.y, __shfl_xor_sync(0xFFFFFFFFu, mx.y, o));
    }
    __syncthreads();  // every read of red in the loop is done
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < (int)(blockDim.x >> 5); ++i) {
            mx.x = fmaxf(mx.x, red[i].x);
            mx.y = fmaxf(mx.y, red[i].y);
        }
        a.blkmax[block] = mx;
    }
    // fixed-order combine of the row groups' dh sums into the block's partial row
    float4 *dst = reinterpret_cast<float4 *>(a.part_dh + (long long)block * a.d_out);
    for (int col = threadIdx.x; col < G; col += blockDim.x) {
        float4 acc = dh_s[col];
        for (int q = 1; q < rb_n; ++q) {
            const float4 o = dh_s[q * G + col];
            acc.x += o.x;
            acc.y += o.y;
            acc.z += o.z;
            acc.w += o.w;
        }
        dst[col] = acc;
    }
}

// ================================================ stage dy (streaming) ======
// The same staging, as a stream of row batches that a producer warp moves
// into a shared-memory ring with 1-D bulk copies (cp.async.bulk), so that
// HBM sees several batches in flight per SM whatever the consumers' register
// budget. Rows up to kSdMaxCols wide. Layout of the work:
//  - a block owns a contiguous range of token rows;
//  - its kSdWarps consumer warps form NGRP row groups of W warps; a group
//    stages one row of a batch (a batch is NGRP consecutive rows, one bulk
//    copy of dy and one of c per batch);
//  - lane i of a group owns the float4 columns i, i + 32W, ... (Q of them)
//    for the whole kernel, so the dh sums of its columns live in registers
//    and are combined over the groups once, at the end, in a fixed order.
// Per row: pass 1 over the row in shared memory gives max |dy.h| and
// sum |dy.h| (shuffles, then a barrier of the group's warps), pass 2 writes
// f16(dy.h.s_t) with direct 8-byte stores.
constexpr int kSdWarps = 16;                     // consumer warps
constexpr int kSdThreads = (kSdWarps + 1) * 32;  // + one producer warp
constexpr int kSdMaxCols = 8191;  // wider rows: the register-staged row kernel (faster there, measured)
constexpr int kSdRingBytes = 200 * 1024;
constexpr int kSdHeadBytes = 1024;  // barriers, flags, reduction buffers

struct SdPlan {
    int W;        // warps per row group
    int ngrp;     // row groups (rows per batch)
    int Q;        // float4 columns per lane, rounded up to the kernel's template value
    int nst;      // ring stages
    int batch_bytes;
};

__host__ __device__ inline SdPlan sd_plan(int d_out) {
    SdPlan p;
    int w = d_out / 512;
    p.W = 1;
    while (p.W * 2 <= w && p.W < kSdWarps) p.W *= 2;
    p.ngrp = kSdWarps / p.W;
    const int q = (d_out / 4 + 32 * p.W - 1) / (32 * p.W);
    p.Q = q <= 2 ? 2 : (q <= 4 ? 4 : (q <= 6 ? 6 : 8));
    p.batch_bytes = p.ngrp * d_out * 6;
    p.nst = kSdRingBytes / p.batch_bytes;
    if (p.nst > 8) p.nst = 8;
    return p;
}

__host__ __device__ inline bool sd_supported(int d_out) {
    return d_out <= kSdMaxCols && sd_plan(d_out).nst >= 2 && (d_out / 4 + 32 * sd_plan(d_out).W - 1) /
                                                                   (32 * sd_plan(d_out).W) <= 8;
}

// 1/2^k for a power-of-two scale 2^k, k in [-126, 127], exactly (2^-127 is subnormal).
__device__ __forceinline__ float pow2_recip(float s) {
    const int k = ((__float_as_int(s) >> 23) & 0xFF) - 127;
    return k <= 126 ? __int_as_float((127 - k) << 23) : __int_as_float(1 << 22);
}

__host__ __device__ inline size_t sd_smem_bytes(int d_out) {
    const SdPlan p = sd_plan(d_out);
    return (size_t)kSdHeadBytes + (size_t)p.nst * p.batch_bytes;
}

// The block first does its share (1 of prep_nblocks) of the two bitmap
// re-layouts, while the producer's first copies are in flight (interleaving
// it with the consumers' waits, as the x staging does, measured slower here:
// the consumers' registers are short).
template <int Q>
__device__ void stage_dy_stream(const StageDyArgs &a, int block, int nblocks, unsigned char *smem,
                                const SignPrep &p0, const SignPrep &p1, int prep_nblocks) {
    const SdPlan pl = sd_plan(a.d_out);
    const int G = a.d_out / 4;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);      // [8]
    uint64_t *empty = full + 8;                                // [8]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 128);
    float2 *red = reinterpret_cast<float2 *>(smem + 256);     // [2][kSdWarps] row sums, then block maxima
    unsigned char *ring = smem + kSdHeadBytes;

    const int row0 = (int)((long long)block * a.M / nblocks);
    const int row1 = (int)((long long)(block + 1) * a.M / nblocks);
    const int nbatch = (row1 - row0 + pl.ngrp - 1) / pl.ngrp;
    const uint32_t dy_bytes = (uint32_t)pl.ngrp * a.d_out * 4;  // offset of the c part in a stage

    if (threadIdx.x == 0) {
        for (int i = 0; i < pl.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kSdWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ---- producer: one lane of the last warp ----
    const bool producer = warp == kSdWarps && lane == 0;
    uint64_t pol = 0;
    int issued = 0;
    auto issue = [&](int i) {
        const int st = i % pl.nst;
        const int r = row0 + i * pl.ngrp;
        const int nr = row1 - r < pl.ngrp ? row1 - r : pl.ngrp;
        unsigned char *dst = ring + (size_t)st * pl.batch_bytes;
        mbar_arrive_expect_tx(&full[st], (uint32_t)nr * a.d_out * 6);
        bulk_load_hint(dst, a.dy + (size_t)r * a.d_out, (uint32_t)nr * a.d_out * 4, &full[st], pol);
        bulk_load_hint(dst + dy_bytes, a.c16 + (size_t)r * a.d_out, (uint32_t)nr * a.d_out * 2, &full[st], pol);
        issued = i + 1;
    };
    if (producer) {
        pol = l2_policy_evict_first();
        for (int i = 0; i < nbatch && i < pl.nst; ++i) issue(i);
    }
    __syncwarp();
    if (prep_nblocks > 0) prep_share(p0, p1, block, prep_nblocks);
    if (warp == kSdWarps) {
        if (lane != 0) return;
        for (int i = issued; i < nbatch; ++i) {
            const int st = i % pl.nst;
            if (!mbar_wait(&empty[st], (uint32_t)((i / pl.nst - 1) & 1), abort_flag)) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(a.status, kStTimeoutStage);
                }
                break;
            }
            issue(i);
        }
        // every issued copy lands before the block may exit
        for (int j = issued - pl.nst < 0 ? 0 : issued - pl.nst; j < issued; ++j)
            if (!mbar_wait(&full[j % pl.nst], (uint32_t)((j / pl.nst) & 1), abort_flag, false))
                atomicOr(a.status, kStTimeoutDrain);
        return;
    }

    // ---- consumers ----
    const int grp = warp / pl.W;            // row group
    const int ti = threadIdx.x % (32 * pl.W);  // index in the group
    const int wg = warp % pl.W;             // warp in the group
    const int gthreads = 32 * pl.W;
    const bool dynamic = !(a.gscale > 0.0f);
    const float ginv = dynamic ? 1.0f : 1.0f / a.gscale;
    float lmax = 0.0f;
    if (dynamic) {
        for (int k = lane; k < a.r; k += 32) lmax = fmaxf(lmax, fabsf(__ldg(a.l + k)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    }
    const float4 *h4 = reinterpret_cast<const float4 *>(a.h);
    float4 hv[Q], dh[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        const int col = ti + k * gthreads;
        hv[k] = col < G ? __ldg(h4 + col) : make_float4(0.f, 0.f, 0.f, 0.f);
        dh[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint2 *o4 = reinterpret_cast<uint2 *>(a.dy16);
    float2 mx = make_float2(0.0f, 0.0f);  // this thread's rows: max 1/s_t, max 1/sigma_t
    bool failed = false;
    for (int i = 0; i < nbatch; ++i) {
        const int st = i % pl.nst;
        bool ok = mbar_wait(&full[st], (uint32_t)((i / pl.nst) & 1), abort_flag);
        if (!ok && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(a.status, kStTimeoutStage);
        }
        const int t = row0 + i * pl.ngrp + grp;
        const bool valid = ok && t < row1;
        const float4 *sdy = reinterpret_cast<const float4 *>(ring + (size_t)st * pl.batch_bytes) + (size_t)grp * G;
        const uint2 *sc = reinterpret_cast<const uint2 *>(ring + (size_t)st * pl.batch_bytes + dy_bytes) +
                          (size_t)grp * G;
        float amax = 0.0f, l1 = 0.0f;
        if (valid) {
#pragma unroll
            for (int k = 0; k < Q; ++k) {
                const int col = ti + k * gthreads;
                if (col < G) {
                    const float4 d = sdy[col];
                    const uint2 cw = sc[col];
                    const float2 c0 = __half22float2(*reinterpret_cast<const __half2 *>(&cw.x));
                    const float2 c1 = __half22float2(*reinterpret_cast<const __half2 *>(&cw.y));
                    dh[k].x += d.x * c0.x;
                    dh[k].y += d.y * c0.y;
                    dh[k].z += d.z * c1.x;
                    dh[k].w += d.w * c1.y;
                    const float vx = fabsf(d.x * hv[k].x), vy = fabsf(d.y * hv[k].y);
                    const float vz = fabsf(d.z * hv[k].z), vw = fabsf(d.w * hv[k].w);
                    amax = fmaxf(amax, fmaxf(fmaxf(vx, vy), fmaxf(vz, vw)));
                    l1 += (vx + vy) + (vz + vw);
                }
            }
        }
        float s = a.gscale, sig = a.gscale;
        bool counts = true;
        if (dynamic) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
            }
        }
        if (pl.W > 1) {
            // the group's warps exchange their sums and agree on whether to go on
            if (dynamic && lane == 0) red[(i & 1) * kSdWarps + warp] = make_float2(amax, l1);
            failed = named_bar_or(1 + grp, gthreads, !ok || *abort_flag);
            if (dynamic) {
                float2 r = red[(i & 1) * kSdWarps + grp * pl.W];
                for (int q = 1; q < pl.W; ++q) {
                    const float2 o = red[(i & 1) * kSdWarps + grp * pl.W + q];
                    r.x = fmaxf(r.x, o.x);
                    r.y += o.y;
                }
                amax = r.x;
                l1 = r.y;
            }
        } else {
            failed = !ok || *abort_flag;
        }
        (void)wg;
        if (dynamic) {
            const bool fin = amax > 0.0f && amax <= 3.402823466e38f;
            counts = fin;
            s = fin ? pow2i(14 - ceil_log2_pos(amax)) : 1.0f;
            sig = s;
            const float bound = l1 * lmax;  // bound on |db_t . l|, unscaled
            if (fin && bound > 0.0f && bound <= 3.402823466e38f) sig = pow2i(15 - ceil_log2_pos(bound));
        }
        if (valid) {
#pragma unroll
            for (int k = 0; k < Q; ++k) {
                const int col = ti + k * gthreads;
                if (col < G) {
                    const float4 d = sdy[col];  // re-read: fewer live registers than keeping dy.h
                    const float4 v = make_float4(d.x * hv[k].x, d.y * hv[k].y, d.z * hv[k].z, d.w * hv[k].w);
                    uint2 o;
                    o.x = pack_half2(v.x * s, v.y * s);
                    o.y = pack_half2(v.z * s, v.w * s);
                    o4[(size_t)t * G + col] = o;
                }
            }
            if (ti == 0) {
                const float si = dynamic ? pow2_recip(s) : ginv, gi = dynamic ? pow2_recip(sig) : ginv;
                a.s_inv[t] = si;
                a.sig[t] = sig;
                a.sig_inv[t] = gi;
                if (counts) mx = make_float2(fmaxf(mx.x, si), fmaxf(mx.y, gi));
            }
        }
        // the stage's shared memory is read: hand it back to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (failed) break;
    }
    // ---- block end: maxima and the dh partial row, fixed order ----
    const int cthreads = kSdWarps * 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx.x = fmaxf(mx.x, __shfl_xor_sync(0xFFFFFFFFu, mx.x, o));
        mx.y = fmaxf(mx.y, __shfl_xor_sync(0xFFFFFFFFu, mx.y, o));
    }
    if (named_bar_or(9, cthreads, *abort_flag != 0)) return;  // every consumer is done with the ring
    if (lane == 0) red[2 * kSdWarps + warp] = mx;
    float4 *dst = reinterpret_cast<float4 *>(a.part_dh + (size_t)block * a.d_out);
    if (pl.ngrp == 1) {
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const int col = ti + k * gthreads;
            if (col < G) dst[col] = dh[k];
        }
    } else {
        float4 *acc = reinterpret_cast<float4 *>(ring);  // [ngrp][G]
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const int col = ti + k * gthreads;
            if (col < G) acc[(size_t)grp * G + col] = dh[k];
        }
    }
    named_bar_sync(9, cthreads);
    if (threadIdx.x == 0) {
        float2 m = red[2 * kSdWarps];
        for (int q = 1; q < kSdWarps; ++q) {
            m.x = fmaxf(m.x, red[2 * kSdWarps + q].x);
            m.y = fmaxf(m.y, red[2 * kSdWarps + q].y);
        }
        a.blkmax[block] = m;
    }
    if (pl.ngrp > 1) {
        const float4 *acc = reinterpret_cast<const float4 *>(ring);
        for (int col = threadIdx.x; col < G; col += cthreads) {
            float4 v = acc[col];
            for (int q = 1; q < pl.ngrp; ++q) {
                const float4 o = acc[(size_t)q * G + col];
                v.x += o.x;
                v.y += o.y;
                v.z += o.z;
                v.w += o.w;
            }
            dst[col] = v;
        }
    }
}

// ============================================================== reduce =====
// out[f] += sum_p part[p][f] over three segments, 32 columns per work item:
// warp w of the block sums rows w, w + nwarps, ... and the warp sums are
// added in warp order, so the result depends only on the block size. `red`
// is nwarps x 32 floats of shared memory.
__device__ __forceinline__ void reduce_partials_run(const ReduceSeg &a, const ReduceSeg &b, const ReduceSeg &c,
                                                    int block, int nblocks, float *red) {
    const int nba = (a.n + 31) / 32, nbb = (b.n + 31) / 32, nbc = (c.n + 31) / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int item = block; item < nba + nbb + nbc; item += nblocks) {
        // the segment's fields by value (selecting a parameter by reference
        // would copy the parameters to local memory)
        const float *part;
        float *out;
        int rows, n, col0;
        if (item < nba) {
            part = a.part, out = a.out, rows = a.rows, n = a.n, col0 = 32 * item;
        } else if (item < nba + nbb) {
            part = b.part, out = b.out, rows = b.rows, n = b.n, col0 = 32 * (item - nba);
        } else {
            part = c.part, out = c.out, rows = c.rows, n = c.n, col0 = 32 * (item - nba - nbb);
        }
        const int col = col0 + lane;
        float acc = 0.0f;
        if (col < n) {
#pragma unroll 4
            for (int p = w; p < rows; p += nwarps) acc += __ldcs(part + (long long)p * n + col);
        }
        red[w * 32 + lane] = acc;
        __syncthreads();
        if (w == 0 && col < n) {
            float t = red[lane];
            for (int i = 1; i < nwarps; ++i) t += red[i * 32 + lane];
            out[col] += t;
        }
        __syncthreads();
    }
}

}  // namespace blr
