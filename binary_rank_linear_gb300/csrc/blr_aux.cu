// Bandwidth kernels of the blr layer on sm_103a: sign packing/expansion, the
// one-per-call re-layout of the bitmaps into the GEMMs' operand order, the
// f32 -> f16 staging of x and dy (with the dh token sums fused into the dy
// staging), and the fixed-order reduction of per-tile partial sums.
#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

// ====================================================== pack / unpack ======
// train_mm.rs (cortiq-engine 0.8.21), test helper `pack_bits`: bit (row, k)
// is 1 iff src[row][k] > 0. One warp per output word; lane j votes for rank
// 32w+j of the row.
__global__ void pack_signs_kernel(const float *__restrict__ src, uint32_t *__restrict__ bits, int rows, int r) {
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

// ============================================ bitmap re-layout (prep) ======
// Destination order [ks][n][2] u32: word (n, 2ks + w) covers reduction
// indices 64ks + 32w .. +31 of operand row n, pair-ready.
__device__ __forceinline__ int prep_blocks(const SignPrep &p, int threads) {
    if (p.kind == 0) {
        const long long units = (long long)p.N * 2 * ((p.K + 63) / 64);
        return (int)((units + threads - 1) / threads);
    }
    const long long warps = (long long)(p.K / 32) * (p.N / 32);
    return (int)((warps + threads / 32 - 1) / (threads / 32));
}

__device__ void prep_run(const SignPrep &p, int block, int threads) {
    if (p.kind == 0) {
        // direct: src [N][K/32]
        const int words = p.K / 32;
        const int kw_total = 2 * ((p.K + 63) / 64);
        const long long u = (long long)block * threads + threadIdx.x;
        if (u >= (long long)p.N * kw_total) return;
        const int n = (int)(u % p.N);
        const int kw = (int)(u / p.N);
        const uint32_t w = kw < words ? p.src[(long long)n * words + kw] : 0u;
        p.dst[((long long)(kw >> 1) * p.N + n) * 2 + (kw & 1)] = sign_word_pair_ready(w);
    } else {
        // transpose: src [K][N/32]; one warp per 32 x 32 bit block.
        const int nwords = p.N / 32;
        const long long wi = (long long)block * (threads / 32) + threadIdx.x / 32;
        if (wi >= (long long)(p.K / 32) * nwords) return;
        const int kw = (int)(wi / nwords);
        const int nw = (int)(wi % nwords);
        const int lane = threadIdx.x & 31;
        const uint32_t mine = p.src[(long long)(32 * kw + lane) * nwords + nw];
        uint32_t keep = 0;
#pragma unroll
        for (int b = 0; b < 32; ++b) {
            const uint32_t col = __ballot_sync(0xFFFFFFFFu, (mine >> b) & 1u);
            if (lane == b) keep = col;
        }
        const int n = 32 * nw + lane;
        p.dst[((long long)(kw >> 1) * p.N + n) * 2 + (kw & 1)] = sign_word_pair_ready(keep);
    }
}

// ============================================================ stage x ======
// train_mm.rs, `cvt_col` staging: x16 = f16(x . g), forward unscaled.
__device__ void stage_x_run(const float *__restrict__ x, const float *__restrict__ g, uint16_t *__restrict__ x16,
                            int M, int d_in, int block, int nblocks) {
    const long long groups = (long long)M * (d_in / 4);
    const int g4n = d_in / 4;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const float4 *gg = reinterpret_cast<const float4 *>(g);
    uint2 *o = reinterpret_cast<uint2 *>(x16);
    for (long long i = (long long)block * blockDim.x + threadIdx.x; i < groups; i += (long long)nblocks * blockDim.x) {
        const float4 v = __ldcs(x4 + i);
        const float4 f = __ldg(gg + (int)(i % g4n));
        uint2 out;
        out.x = pack_half2(v.x * f.x, v.y * f.y);
        out.y = pack_half2(v.z * f.z, v.w * f.w);
        o[i] = out;
    }
}

__global__ void __launch_bounds__(256) fwd_prologue_kernel(SignPrep p0, SignPrep p1, const float *x, const float *g,
                                                           uint16_t *x16, int M, int d_in) {
    const int b0 = prep_blocks(p0, blockDim.x);
    const int b1 = prep_blocks(p1, blockDim.x);
    const int b = blockIdx.x;
    if (b < b0) {
        prep_run(p0, b, blockDim.x);
    } else if (b < b0 + b1) {
        prep_run(p1, b - b0, blockDim.x);
    } else {
        stage_x_run(x, g, x16, M, d_in, b - b0 - b1, gridDim.x - b0 - b1);
    }
}

// =========================================================== stage dy ======
// Backward staging (train_mm.rs, `blr_backward`: cvt of dy with the column
// factor h under the gradient scale, and `colsum_prod` of dy and c for dh).
// A block of 1024 threads owns whole token rows; `tpr` threads share a row
// and a block works on 1024/tpr rows at a time. Per row t:
//   s_t     = gscale, or 2^(14 - ceil(log2 max_i |dy_ti h_i|))  (1 if the max is 0)
//   dy16_t  = f16(dy_t . h . s_t)
//   sigma_t = gscale, or s_t * 2^(15 - ceil(log2(L1_t * max|l|))) with
//             L1_t = sum_i |dy16_ti|, which bounds |db_t . l . sigma_t| by 2^15
// and the block accumulates sum_t dy_ti c_ti into one partial row of dh.
constexpr int kStageThreads = 1024;
constexpr int kStageRowsPerBlock = 32;

__host__ __device__ inline int stage_tpr(int d_out) {
    const int G = d_out / 4;
    int t = 32;
    while (t * 2 <= G / 4 && t < kStageThreads) t *= 2;
    return t;
}

int stage_dy_blocks(int M, int d_out) {
    const int rb = kStageThreads / stage_tpr(d_out);
    const int rows = rb > kStageRowsPerBlock ? rb : kStageRowsPerBlock;
    return (M + rows - 1) / rows;
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

// Reduce `v` over the `tpr` consecutive threads sharing a row (tpr >= 32, a
// power of two). Every thread of the block must call it.
template <bool kMax>
__device__ __forceinline__ float row_reduce(float v, float *red, int tpr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = kMax ? fmaxf(v, u) : v + u;
    }
    const int warp = threadIdx.x / 32;
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    const int wpr = tpr / 32;
    const int first = (threadIdx.x / tpr) * wpr;
    float r = red[first];
    for (int i = 1; i < wpr; ++i) r = kMax ? fmaxf(r, red[first + i]) : r + red[first + i];
    __syncthreads();
    return r;
}

template <int GPT>
__device__ void stage_dy_run(const StageDyArgs &a, int block, float *smem) {
    float *red = smem;             // [32]
    float *dh_red = smem + 32;     // [d_out]
    const int tpr = stage_tpr(a.d_out);
    const int rb_n = kStageThreads / tpr;
    const int rows_per_block = rb_n > kStageRowsPerBlock ? rb_n : kStageRowsPerBlock;
    const int rb = threadIdx.x / tpr;
    const int ti = threadIdx.x % tpr;
    const int G = a.d_out / 4;
    const int row0 = block * rows_per_block;
    const int row_end = min(row0 + rows_per_block, a.M);
    const bool dynamic = !(a.gscale > 0.0f);

    float lmax = 0.0f;
    if (dynamic) {
        for (int k = threadIdx.x; k < a.r; k += blockDim.x) lmax = fmaxf(lmax, fabsf(__ldg(a.l + k)));
        lmax = row_reduce<true>(lmax, red, kStageThreads < 1024 ? kStageThreads : 1024);
    }

    const float4 *dy4 = reinterpret_cast<const float4 *>(a.dy);
    const float4 *h4 = reinterpret_cast<const float4 *>(a.h);
    const uint2 *c4 = reinterpret_cast<const uint2 *>(a.c16);
    uint2 *o4 = reinterpret_cast<uint2 *>(a.dy16);

    float4 acc[GPT];
#pragma unroll
    for (int g = 0; g < GPT; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int base = row0; base < row_end; base += rb_n) {
        const int t = base + rb;
        const bool valid = t < row_end;
        float s = a.gscale;
        if (dynamic) {
            float amax = 0.0f;
#pragma unroll
            for (int g = 0; g < GPT; ++g) {
                const int col = g * tpr + ti;
                if (valid && col < G) {
                    const float4 v = __ldg(dy4 + (long long)t * G + col);
                    const float4 f = __ldg(h4 + col);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x * f.x), fabsf(v.y * f.y)),
                                             fmaxf(fabsf(v.z * f.z), fabsf(v.w * f.w))));
                }
            }
            amax = row_reduce<true>(amax, red, tpr);
            s = (amax > 0.0f && amax <= 3.402823466e38f) ? pow2i(14 - ceil_log2_pos(amax)) : 1.0f;
        }
        float l1 = 0.0f;
#pragma unroll
        for (int g = 0; g < GPT; ++g) {
            const int col = g * tpr + ti;
            if (valid && col < G) {
                const long long idx = (long long)t * G + col;
                const float4 v = __ldg(dy4 + idx);
                const float4 f = __ldg(h4 + col);
                uint2 st;
                st.x = pack_half2(v.x * f.x * s, v.y * f.y * s);
                st.y = pack_half2(v.z * f.z * s, v.w * f.w * s);
                o4[idx] = st;
                const __half2 s0 = *reinterpret_cast<const __half2 *>(&st.x);
                const __half2 s1 = *reinterpret_cast<const __half2 *>(&st.y);
                const float2 q0 = __half22float2(s0), q1 = __half22float2(s1);
                l1 += fabsf(q0.x) + fabsf(q0.y) + fabsf(q1.x) + fabsf(q1.y);
                const uint2 cw = __ldg(c4 + idx);
                const float2 c0 = __half22float2(*reinterpret_cast<const __half2 *>(&cw.x));
                const float2 c1 = __half22float2(*reinterpret_cast<const __half2 *>(&cw.y));
                acc[g].x += v.x * c0.x;
                acc[g].y += v.y * c0.y;
                acc[g].z += v.z * c1.x;
                acc[g].w += v.w * c1.y;
            }
        }
        float sig = a.gscale;
        if (dynamic) {
            l1 = row_reduce<false>(l1, red, tpr);
            const float bound = l1 * lmax;
            sig = s;
            if (bound > 0.0f && bound <= 3.402823466e38f) {
                int e_s;
                frexpf(s, &e_s);  // s = 0.5 * 2^e_s
                sig = pow2i((e_s - 1) + 15 - ceil_log2_pos(bound));
            }
        }
        if (valid && ti == 0) {
            a.s_inv[t] = 1.0f / s;
            a.sig[t] = sig;
            a.sig_inv[t] = 1.0f / sig;
        }
    }

    // combine the row groups' dh sums in a fixed order, then store the block's partial row
    for (int q = 0; q < rb_n; ++q) {
        if (rb == q) {
#pragma unroll
            for (int g = 0; g < GPT; ++g) {
                const int col = g * tpr + ti;
                if (col < G) {
                    float4 *d = reinterpret_cast<float4 *>(dh_red) + col;
                    if (q == 0) {
                        *d = acc[g];
                    } else {
                        float4 o = *d;
                        o.x += acc[g].x;
                        o.y += acc[g].y;
                        o.z += acc[g].z;
                        o.w += acc[g].w;
                        *d = o;
                    }
                }
            }
        }
        __syncthreads();
    }
    float4 *dst = reinterpret_cast<float4 *>(a.part_dh + (long long)block * a.d_out);
    for (int col = threadIdx.x; col < G; col += blockDim.x) dst[col] = reinterpret_cast<float4 *>(dh_red)[col];
}

template <int GPT>
__global__ void __launch_bounds__(kStageThreads, 1)
    bwd_prologue_kernel(SignPrep p0, SignPrep p1, StageDyArgs a, int stage_blocks) {
    extern __shared__ __align__(16) float smem_f[];
    const int b = blockIdx.x;
    if (b < stage_blocks) {
        stage_dy_run<GPT>(a, b, smem_f);
        return;
    }
    const int b0 = prep_blocks(p0, blockDim.x);
    const int rest = b - stage_blocks;
    if (rest < b0) {
        prep_run(p0, rest, blockDim.x);
    } else {
        prep_run(p1, rest - b0, blockDim.x);
    }
}

// ============================================================== reduce =====
__global__ void reduce_partials_kernel(ReduceSeg a, ReduceSeg b, ReduceSeg c) {
    const long long total = (long long)a.n + b.n + c.n;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const float *part;
        float *out;
        int rows, n, f;
        if (i < a.n) {
            part = a.part, out = a.out, rows = a.rows, n = a.n, f = (int)i;
        } else if (i < (long long)a.n + b.n) {
            part = b.part, out = b.out, rows = b.rows, n = b.n, f = (int)(i - a.n);
        } else {
            part = c.part, out = c.out, rows = c.rows, n = c.n, f = (int)(i - a.n - b.n);
        }
        float acc = 0.0f;
        for (int p = 0; p < rows; ++p) acc += part[(long long)p * n + f];
        out[f] += acc;
    }
}

// ============================================================ launchers ====
static int grid_for(long long items, int per_block, int cap = 1 << 20) {
    long long g = (items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

cudaError_t launch_pack_signs(const float *src, uint32_t *bits, int rows, int r, cudaStream_t s) {
    const long long words = (long long)rows * ((r + 31) / 32);
    trace_before("pack_signs", s);
    pack_signs_kernel<<<grid_for(words, 8, 65535), 256, 0, s>>>(src, bits, rows, r);
    trace_after(s);
    return cudaGetLastError();
}

cudaError_t launch_unpack_signs(const uint32_t *bits, uint16_t *dst, int rows, int r, cudaStream_t s) {
    const long long words = (long long)rows * ((r + 31) / 32);
    trace_before("unpack_signs", s);
    unpack_signs_kernel<<<grid_for(words, 256, 65535), 256, 0, s>>>(bits, dst, rows, r);
    trace_after(s);
    return cudaGetLastError();
}

static int host_prep_blocks(const SignPrep &p, int threads) {
    if (p.kind == 0) {
        const long long units = (long long)p.N * 2 * ((p.K + 63) / 64);
        return (int)((units + threads - 1) / threads);
    }
    const long long warps = (long long)(p.K / 32) * (p.N / 32);
    return (int)((warps + threads / 32 - 1) / (threads / 32));
}

cudaError_t launch_fwd_prologue(SignPrep p0, SignPrep p1, const float *x, const float *g, uint16_t *x16, int M,
                                int d_in, cudaStream_t s) {
    const int b0 = host_prep_blocks(p0, 256), b1 = host_prep_blocks(p1, 256);
    const long long groups = (long long)M * (d_in / 4);
    int bs = grid_for(groups, 256 * 4, 152 * 16);
    trace_before("fwd_prologue", s);
    fwd_prologue_kernel<<<b0 + b1 + bs, 256, 0, s>>>(p0, p1, x, g, x16, M, d_in);
    trace_after(s);
    return cudaGetLastError();
}

template <int GPT>
static cudaError_t launch_bwd_prologue_t(SignPrep p0, SignPrep p1, const StageDyArgs &a, cudaStream_t s) {
    const int sb = stage_dy_blocks(a.M, a.d_out);
    const int b0 = host_prep_blocks(p0, kStageThreads), b1 = host_prep_blocks(p1, kStageThreads);
    const size_t smem = (32 + (size_t)a.d_out) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(bwd_prologue_kernel<GPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    trace_before("bwd_prologue", s);
    bwd_prologue_kernel<GPT><<<sb + b0 + b1, kStageThreads, smem, s>>>(p0, p1, a, sb);
    trace_after(s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_prologue(SignPrep p0, SignPrep p1, const StageDyArgs &a, cudaStream_t s) {
    const int tpr = stage_tpr(a.d_out);
    const int gpt = (a.d_out / 4 + tpr - 1) / tpr;
    if (gpt <= 1) return launch_bwd_prologue_t<1>(p0, p1, a, s);
    if (gpt <= 2) return launch_bwd_prologue_t<2>(p0, p1, a, s);
    if (gpt <= 4) return launch_bwd_prologue_t<4>(p0, p1, a, s);
    if (gpt <= 8) return launch_bwd_prologue_t<8>(p0, p1, a, s);
    if (gpt <= 16) return launch_bwd_prologue_t<16>(p0, p1, a, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_partials(ReduceSeg a, ReduceSeg b, ReduceSeg c, cudaStream_t s) {
    const long long total = (long long)a.n + b.n + c.n;
    trace_before("reduce_partials", s);
    reduce_partials_kernel<<<grid_for(total, 256, 4096), 256, 0, s>>>(a, b, c);
    trace_after(s);
    return cudaGetLastError();
}

}  // namespace blr
