// Dense f16 tensor-core products (see the comment below): the kernel behind
// the sign gradients and plane_linear.
#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

// Dense f16 products on the tensor cores, f32 out:
//     out[f][c] (+)= scale * dscale * sum_k A(f, k) B(c, k)
// for up to two independent products ("jobs") in one persistent launch over
// the tiles of both. A tile is 128 rows f (the MMA's M side) x BN columns c
// (its N side), K in 64-deep k-steps. Each operand is read by TMA either
// K-major (the reduction index contiguous: rows of A or B are K-vectors) or
// MN-major (f or c contiguous, K strided), as it lies in memory, so no
// operand is ever transposed. Users: the sign gradients (K = tokens; both
// operands MN-major, the pass's token-major staging) and the dense frozen
// linear plane_linear (K = the input width; A K-major, B K-major for y =
// x plane^T or MN-major for the transpose y = x plane).
//
// Warp 0 TMA producer, warp 1 MMA issuer (tcgen05 kind::f16), warps 2-5
// epilogue (thread = one row f): each 32 x 32 chunk is staged in shared
// memory (128-byte swizzle) and written by a TMA store, or by a TMA reduce-add
// store in accumulate mode. Epilogue modes (EPM):
//  0: out = acc * scale;
//  1: the layer's c-product read token-major (rows = tokens, columns =
//     output features, B = the S_U plane): y = h[c] * acc and c16 = f16(acc)
//     (train_mm.rs, blr_forward: mm into cbuf, scale_acc with h);
//  2: its dx'-product read token-major (B = the S_V plane): dx' = acc /
//     sigma_t, dx = g[c] * dx', and the token sums of x * dx' for dg, one
//     partial row per warp (32 tokens) of the tile (blr_backward: mm into t1,
//     colsum_prod for dg, scale_acc with g).
// Per-column factors are the same for every row: each thread reads the
// chunk's 32 with eight broadcast 16-byte loads.
//
// Shared-memory operand tiles, as TMA writes them with the 128-byte swizzle:
//  - K-major: rows of 64 K values (128 bytes), 8-row groups 1024 bytes apart
//    (stride byte offset); the k-th MMA (K = 16) of a k-step starts 32 k
//    bytes in;
//  - MN-major: blocks of [64 K][64 M or N] (8 KB; row = K index, 128 bytes);
//    8-row groups along K 1024 bytes apart (stride byte offset), 64-element
//    blocks along M or N 8 KB apart (leading byte offset); the k-th MMA
//    starts 2048 k bytes in.
struct DenseGemmArgs {
    int F0, F1;                  // rows (M side) of the two products; F1 = 0: one product
    float scale0, scale1;
    const float *dscale0, *dscale1;
    int R;                       // columns (N side), both products
    int K;                       // reduction length
    int accumulate;              // reduce-add into the output instead of storing
    uint32_t *status;
    const float *colv;           // EPM 1, 2: per-column factor (h or g) [R]
    const float *row_inv;        // EPM 2: per-row 1/sigma_t [F0]
    const float *xin;            // EPM 2: x [F0][R] f32
    float *part;                 // EPM 2: dg partial rows [row tiles * 4][R]
};

constexpr int kSgThreads = 192;
constexpr int kSgEpi0 = 2;

template <int BN, int EPM = 0>
struct DenseGemmShape {
    static constexpr int kABytes = 2 * kMnBlockBytes;
    static constexpr int kBBytes = (BN / 64) * kMnBlockBytes;
    static constexpr int kStage = kABytes + kBBytes;
    // epilogue chunk slots per warp: two 4 KB f32 slots (modes 0 and 2), or
    // one 6 KB slot of f32 y and f16 c (mode 1), which keeps four operand stages
    static constexpr int kSlotBytes = EPM == 1 ? 6144 : 4096;
    static constexpr int kSlots = EPM == 1 ? 1 : 2;
    static constexpr int kEpiBytes = 4 * kSlots * kSlotBytes;
    static constexpr int kNBRaw = (227 * 1024 - 1024 - 256 - kEpiBytes) / kStage;
    static constexpr int kNB = kNBRaw > 8 ? 8 : kNBRaw;
    static constexpr int kNumBars = 2 * kNB + 4 + 1;
    static constexpr int kSmemBytes = 1024 + kNB * kStage + kEpiBytes + kNumBars * 8 + 16;
    static_assert(kNB >= 2, "pipeline depth");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Descriptor of an operand tile and its per-MMA advance (16 K values).
template <bool MN>
__device__ __forceinline__ uint64_t dense_sdesc(uint32_t saddr) {
    if constexpr (MN)
        return umma_sdesc_sw128_mn(saddr);
    else
        return umma_sdesc_sw128(saddr);
}
template <bool MN>
constexpr uint64_t kDenseDescK = MN ? (2048u >> 4) : (32u >> 4);

__device__ __forceinline__ int sw128_chunk_off(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }
// 64-byte rows (32 f16) in the 64-byte swizzle: 16-byte chunk c of row r
__device__ __forceinline__ int sw64_chunk_off(int row, int c) { return row * 64 + ((c ^ ((row >> 1) & 3)) << 4); }

// Lane l of the warp returns sum over the 32 lanes of v[l] (a transposing
// butterfly: 31 shuffles, each step halving the values a lane carries).
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, s);
        }
    }
    return v[0];
}

template <int BN, bool A_MN, bool B_MN, int EPM>
__global__ void __launch_bounds__(kSgThreads, 1)
    dense_gemm_kernel(const __grid_constant__ DenseGemmMaps maps, const DenseGemmArgs args) {
    using S = DenseGemmShape<BN, EPM>;
    constexpr int NB = S::kNB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sS = smem;                          // [NB][A | B]
    uint8_t *sE = sS + NB * S::kStage;           // [4 warps][kSlots][slot]
    uint64_t *full = reinterpret_cast<uint64_t *>(sE + S::kEpiBytes);
    uint64_t *empty = full + NB;
    uint64_t *tmem_full = empty + NB;
    uint64_t *tmem_empty = tmem_full + 2;
    uint64_t *drain_bar = tmem_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int r_tiles = (args.R + BN - 1) / BN;
    const int tiles0 = ((args.F0 + 127) / 128) * r_tiles;
    const int num_tiles = tiles0 + ((args.F1 + 127) / 128) * r_tiles;
    const int num_ks = (args.K + 63) / 64;
    // tile -> (product, row tile, column tile); column tile varies fastest
    auto decode = [&](int tile, int &jb, int &f0, int &k0) {
        jb = tile >= tiles0 ? 1 : 0;
        const int tl = tile - (jb ? tiles0 : 0);
        f0 = (tl / r_tiles) * 128;
        k0 = (tl % r_tiles) * BN;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NB; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tmem_full[i], 1);
            mbar_init(&tmem_empty[i], 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < 2; ++i) {
            tma_prefetch_desc(&maps.a[i]);
            tma_prefetch_desc(&maps.b[i]);
            tma_prefetch_desc(&maps.o[i]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();
    auto fail = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(args.status, code);
    };

    if (warp == 0) {
        if (lane == 0) {
            int sb = 0;
            uint32_t pb = 0, issued = 0, parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int jb, f0, k0;
                decode(tile, jb, f0, k0);
                const CUtensorMap *ma = jb ? &maps.a[1] : &maps.a[0];
                const CUtensorMap *mb = jb ? &maps.b[1] : &maps.b[0];
                for (int ks = 0; ks < num_ks; ++ks) {
                    if (!mbar_wait(&empty[sb], pb ^ 1u, abort_flag)) {
                        fail(kStTimeoutTma);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[sb], S::kStage);
                    uint8_t *st = sS + sb * S::kStage;
                    const int t0 = ks * 64;  // first K index of the k-step
                    if constexpr (A_MN) {
                        tma_load_2d(st, ma, &full[sb], f0, t0);
                        tma_load_2d(st + kMnBlockBytes, ma, &full[sb], f0 + 64, t0);
                    } else {
                        tma_load_2d(st, ma, &full[sb], t0, f0);  // box 64 K x 128 rows
                    }
                    if constexpr (B_MN) {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(st + S::kABytes + j * kMnBlockBytes, mb, &full[sb], k0 + 64 * j, t0);
                    } else {
                        tma_load_2d(st + S::kABytes, mb, &full[sb], t0, k0);  // box 64 K x BN rows
                    }
                    issued |= 1u << sb;
                    parity = (parity & ~(1u << sb)) | (pb << sb);
                    if (++sb == NB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
            }
            for (int s = 0; s < NB; ++s)
                if (((issued >> s) & 1u) && !mbar_wait(&full[s], (parity >> s) & 1u, abort_flag, false))
                    atomicOr(args.status, kStTimeoutDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32_major(128, BN, A_MN, B_MN);
            int sb = 0;
            uint32_t pb = 0;
            bool ok = true;
            int local = 0;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
                if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)) {
                    fail(kStTimeoutMma);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int ks = 0; ks < num_ks; ++ks) {
                    if (!mbar_wait(&full[sb], pb, abort_flag)) {
                        fail(kStTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = dense_sdesc<A_MN>(smem_u32(sS + sb * S::kStage));
                    const uint64_t bdesc = dense_sdesc<B_MN>(smem_u32(sS + sb * S::kStage + S::kABytes));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16(d_tmem, adesc + kDenseDescK<A_MN> * k, bdesc + kDenseDescK<B_MN> * k, idesc,
                                 (ks > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[sb]);
                    if (++sb == NB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tmem_full[acc]);
            }
            umma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, abort_flag, false)) atomicOr(args.status, kStTimeoutDrain);
        }
        __syncwarp();
    } else {
        // ---- epilogue: thread = one row f of the tile ------------------------
        const int q = warp & 3;
        uint8_t *ebuf = sE + (warp - kSgEpi0) * S::kSlots * S::kSlotBytes;
        int gch = 0, local = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
            int jb, f0, k0;
            decode(tile, jb, f0, k0);
            const int jF = jb ? args.F1 : args.F0;
            const float *jds = jb ? args.dscale1 : args.dscale0;
            const CUtensorMap *mo = jb ? &maps.o[1] : &maps.o[0];
            const float scale = (jb ? args.scale1 : args.scale0) * (jds ? *jds : 1.0f);
            const int acc = local & 1;
            const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
            const int fr = f0 + q * 32;  // this warp's 32 rows
            const int f = fr + lane;
            const bool fvalid = f < jF;
            // mode 2: this row's 1/sigma_t, and x of the tile's first chunk
            const float ri = (EPM == 2 && fvalid) ? __ldg(args.row_inv + f) : 0.0f;
            float4 xa[8];
            auto load_x = [&](int kc, float4 (&xr)[8]) {
                const bool in = fvalid && kc < args.R;
                const float4 *src = reinterpret_cast<const float4 *>(args.xin + (size_t)f * args.R + kc);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) xr[j4] = in ? __ldcs(src + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
            };
            if constexpr (EPM == 2) load_x(k0, xa);
            const bool got = mbar_wait(&tmem_full[acc], acc_phase, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) fail(kStTimeoutEpi);
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c, ++gch) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + 32 * c), v);
                const int kc = k0 + 32 * c;  // first column of the chunk
                float4 xn[8];
                if constexpr (EPM == 2) {
                    if (c + 1 < BN / 32) load_x(kc + 32, xn);  // next chunk's x, in flight meanwhile
                }
                tmem_wait_ld_regs(v);
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tmem_empty[acc]);
                }
                uint8_t *buf = ebuf + (gch % S::kSlots) * S::kSlotBytes;
                // the store that last used buf has read it
                if (lane == 0) {
                    if constexpr (S::kSlots == 1)
                        bulk_wait_group_read<0>();
                    else
                        bulk_wait_group_read<1>();
                }
                __syncwarp();
                const bool cvalid = kc < args.R;
                if constexpr (EPM == 0) {
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 o = make_float4(
                            __uint_as_float(v[4 * j4]) * scale, __uint_as_float(v[4 * j4 + 1]) * scale,
                            __uint_as_float(v[4 * j4 + 2]) * scale, __uint_as_float(v[4 * j4 + 3]) * scale);
                        *reinterpret_cast<float4 *>(buf + sw128_chunk_off(lane, j4)) = o;
                    }
                } else if constexpr (EPM == 1) {
                    // y = h * acc (f32, 128-byte swizzle), c = f16(acc) (64-byte swizzle)
                    const float4 *h4 = reinterpret_cast<const float4 *>(args.colv + kc);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 hv = cvalid ? __ldg(h4 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
                        const float4 o = make_float4(__uint_as_float(v[4 * j4]) * hv.x, __uint_as_float(v[4 * j4 + 1]) * hv.y,
                                                     __uint_as_float(v[4 * j4 + 2]) * hv.z,
                                                     __uint_as_float(v[4 * j4 + 3]) * hv.w);
                        *reinterpret_cast<float4 *>(buf + sw128_chunk_off(lane, j4)) = o;
                    }
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) {
                        uint4 w;
                        w.x = pack_half2(__uint_as_float(v[8 * c16]), __uint_as_float(v[8 * c16 + 1]));
                        w.y = pack_half2(__uint_as_float(v[8 * c16 + 2]), __uint_as_float(v[8 * c16 + 3]));
                        w.z = pack_half2(__uint_as_float(v[8 * c16 + 4]), __uint_as_float(v[8 * c16 + 5]));
                        w.w = pack_half2(__uint_as_float(v[8 * c16 + 6]), __uint_as_float(v[8 * c16 + 7]));
                        *reinterpret_cast<uint4 *>(buf + 4096 + sw64_chunk_off(lane, c16)) = w;
                    }
                } else {
                    // dx' = acc / sigma_t; dx = g * dx'; dg partial = sum over the warp's rows of x * dx'
                    const float4 *g4 = reinterpret_cast<const float4 *>(args.colv + kc);
                    float prod[32];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 gv = cvalid ? __ldg(g4 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
                        const float d0 = __uint_as_float(v[4 * j4]) * ri, d1 = __uint_as_float(v[4 * j4 + 1]) * ri;
                        const float d2 = __uint_as_float(v[4 * j4 + 2]) * ri, d3 = __uint_as_float(v[4 * j4 + 3]) * ri;
                        prod[4 * j4] = xa[j4].x * d0;
                        prod[4 * j4 + 1] = xa[j4].y * d1;
                        prod[4 * j4 + 2] = xa[j4].z * d2;
                        prod[4 * j4 + 3] = xa[j4].w * d3;
                        *reinterpret_cast<float4 *>(buf + sw128_chunk_off(lane, j4)) =
                            make_float4(gv.x * d0, gv.y * d1, gv.z * d2, gv.w * d3);
                    }
                    const float colsum = warp_transpose_sum(prod);  // lane l: column kc + l
                    if (cvalid) args.part[((size_t)(f0 / 128) * 4 + q) * args.R + kc + lane] = colsum;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) xa[j4] = xn[j4];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (fr < jF && cvalid) {
                        if (args.accumulate)
                            tma_reduce_add_2d(mo, buf, kc, fr);
                        else
                            tma_store_2d(mo, buf, kc, fr);
                        if constexpr (EPM == 1) tma_store_2d(&maps.o16, buf + 4096, kc, fr);
                    }
                    bulk_commit_group();
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 2 * BN);
}

// ------------------------------------------------------------ launcher ---
template <int BN, bool A_MN, bool B_MN, int EPM>
static cudaError_t launch_dense_t(const DenseGemmLaunch &L, const DenseGemmArgs &ga, int grid, cudaStream_t s) {
    using S = DenseGemmShape<BN, EPM>;
    const cudaError_t e = prepare_kernel_once(dense_gemm_kernel<BN, A_MN, B_MN, EPM>, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_k(dense_gemm_kernel<BN, A_MN, B_MN, EPM>, dim3(grid), dim3(kSgThreads), S::kSmemBytes, s, L.maps,
                    ga);
}

cudaError_t launch_dense_gemm(const DenseGemmLaunch &L, const char *name, cudaStream_t s) {
    DenseGemmArgs ga{};
    ga.F0 = L.F[0];
    ga.F1 = L.F[1];
    ga.scale0 = L.scale[0];
    ga.scale1 = L.scale[1];
    ga.dscale0 = L.dscale[0];
    ga.dscale1 = L.dscale[1];
    ga.R = L.R;
    ga.K = L.K;
    ga.accumulate = L.accumulate;
    ga.status = L.status;
    ga.colv = L.colv;
    ga.row_inv = L.row_inv;
    ga.xin = L.xin;
    ga.part = L.part;
    const int bn = L.epm ? 256 : dense_bn(L.R);
    const long long tiles = (long long)(((L.F[0] + 127) / 128) + ((L.F[1] + 127) / 128)) * ((L.R + bn - 1) / bn);
    const int grid = (int)(tiles < L.sms ? tiles : L.sms);
    if (grid < 1) return cudaSuccess;
    cudaError_t e = cudaErrorInvalidValue;
    trace_before(name, s);
    if (L.epm == 1 && !L.a_mn && !L.b_mn)
        e = launch_dense_t<256, false, false, 1>(L, ga, grid, s);
    else if (L.epm == 2 && !L.a_mn && !L.b_mn)
        e = launch_dense_t<256, false, false, 2>(L, ga, grid, s);
    else if (L.epm != 0)
        e = cudaErrorInvalidValue;
    else if (L.a_mn && L.b_mn)
        e = bn == 256 ? launch_dense_t<256, true, true, 0>(L, ga, grid, s)
                      : launch_dense_t<128, true, true, 0>(L, ga, grid, s);
    else if (!L.a_mn && !L.b_mn)
        e = bn == 256 ? launch_dense_t<256, false, false, 0>(L, ga, grid, s)
                      : launch_dense_t<128, false, false, 0>(L, ga, grid, s);
    else if (!L.a_mn && L.b_mn)
        e = bn == 256 ? launch_dense_t<256, false, true, 0>(L, ga, grid, s)
                      : launch_dense_t<128, false, true, 0>(L, ga, grid, s);
    trace_after(s);
    return e;
}

}  // namespace blr
