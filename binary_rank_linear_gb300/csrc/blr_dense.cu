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
// epilogue: out = acc * scale (+ out), each 32 x 32 chunk staged in shared
// memory (128-byte swizzle) and written by a TMA store.
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
    float *out0, *out1;          // [F][R] (read when accumulating)
    int R;                       // columns (N side), both products
    int K;                       // reduction length
    int accumulate;
    uint32_t *status;
};

constexpr int kSgThreads = 192;
constexpr int kSgEpi0 = 2;

template <int BN>
struct DenseGemmShape {
    static constexpr int kABytes = 2 * kMnBlockBytes;
    static constexpr int kBBytes = (BN / 64) * kMnBlockBytes;
    static constexpr int kStage = kABytes + kBBytes;
    static constexpr int kEpiBytes = 4 * 2 * 4096;
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

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kSgThreads, 1)
    dense_gemm_kernel(const __grid_constant__ DenseGemmMaps maps, const DenseGemmArgs args) {
    using S = DenseGemmShape<BN>;
    constexpr int NB = S::kNB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sS = smem;                          // [NB][A | B]
    uint8_t *sE = sS + NB * S::kStage;           // [4 warps][2][32 x 32 f32]
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
        uint8_t *ebuf = sE + (warp - kSgEpi0) * 2 * 4096;
        int gch = 0, local = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
            int jb, f0, k0;
            decode(tile, jb, f0, k0);
            const int jF = jb ? args.F1 : args.F0;
            const float *jds = jb ? args.dscale1 : args.dscale0;
            float *jout = jb ? args.out1 : args.out0;
            const CUtensorMap *mo = jb ? &maps.o[1] : &maps.o[0];
            const float scale = (jb ? args.scale1 : args.scale0) * (jds ? *jds : 1.0f);
            const int acc = local & 1;
            const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
            const int fr = f0 + q * 32;  // this warp's 32 rows
            const int f = fr + lane;
            const bool fvalid = f < jF;
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
                tmem_wait_ld_regs(v);
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tmem_empty[acc]);
                }
                const int kc = k0 + 32 * c;  // first column of the chunk
                uint8_t *buf = ebuf + (gch & 1) * 4096;
                if (lane == 0) bulk_wait_group_read<1>();  // the store that last used buf has read it
                __syncwarp();
                const bool accum = args.accumulate && fvalid && kc < args.R;
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float4 o = make_float4(__uint_as_float(v[4 * j4]) * scale, __uint_as_float(v[4 * j4 + 1]) * scale,
                                           __uint_as_float(v[4 * j4 + 2]) * scale,
                                           __uint_as_float(v[4 * j4 + 3]) * scale);
                    if (accum) {
                        const float4 old =
                            *reinterpret_cast<const float4 *>(jout + (size_t)f * args.R + kc + 4 * j4);
                        o.x += old.x;
                        o.y += old.y;
                        o.z += old.z;
                        o.w += old.w;
                    }
                    *reinterpret_cast<float4 *>(buf + sw128_chunk_off(lane, j4)) = o;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (fr < jF && kc < args.R) tma_store_2d(mo, buf, kc, fr);
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
template <int BN, bool A_MN, bool B_MN>
static cudaError_t launch_dense_t(const DenseGemmLaunch &L, const DenseGemmArgs &ga, int grid, cudaStream_t s) {
    static bool prepared = false;
    if (!prepared) {
        const cudaError_t e = prepare_kernel(dense_gemm_kernel<BN, A_MN, B_MN>, DenseGemmShape<BN>::kSmemBytes);
        if (e != cudaSuccess) return e;
        prepared = true;
    }
    return launch_k(dense_gemm_kernel<BN, A_MN, B_MN>, dim3(grid), dim3(kSgThreads), DenseGemmShape<BN>::kSmemBytes,
                    s, L.maps, ga);
}

cudaError_t launch_dense_gemm(const DenseGemmLaunch &L, const char *name, cudaStream_t s) {
    DenseGemmArgs ga{};
    ga.F0 = L.F[0];
    ga.F1 = L.F[1];
    ga.scale0 = L.scale[0];
    ga.scale1 = L.scale[1];
    ga.dscale0 = L.dscale[0];
    ga.dscale1 = L.dscale[1];
    ga.out0 = L.out[0];
    ga.out1 = L.out[1];
    ga.R = L.R;
    ga.K = L.K;
    ga.accumulate = L.accumulate;
    ga.status = L.status;
    const int bn = dense_bn(L.R);
    const long long tiles = (long long)(((L.F[0] + 127) / 128) + ((L.F[1] + 127) / 128)) * ((L.R + bn - 1) / bn);
    const int grid = (int)(tiles < L.sms ? tiles : L.sms);
    if (grid < 1) return cudaSuccess;
    cudaError_t e = cudaErrorInvalidValue;
    trace_before(name, s);
    if (L.a_mn && L.b_mn)
        e = bn == 256 ? launch_dense_t<256, true, true>(L, ga, grid, s) : launch_dense_t<128, true, true>(L, ga, grid, s);
    else if (!L.a_mn && !L.b_mn)
        e = bn == 256 ? launch_dense_t<256, false, false>(L, ga, grid, s)
                      : launch_dense_t<128, false, false>(L, ga, grid, s);
    else if (!L.a_mn && L.b_mn)
        e = bn == 256 ? launch_dense_t<256, false, true>(L, ga, grid, s)
                      : launch_dense_t<128, false, true>(L, ga, grid, s);
    trace_after(s);
    return e;
}

}  // namespace blr
