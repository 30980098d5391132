// Persistent tcgen05 GEMM of the blr layer on sm_103a:
//
//     acc[t][n] = sum_k act16[t][k] * S[n][k]        (S = +-1, exact in f16)
//
// for one 128-token x BN-feature tile at a time, with a fused epilogue per
// pass. The activation operand is an f16 matrix [M][K] brought in by TMA
// (128-byte swizzle, box 64 x 128). The sign operand is never stored as a
// dense matrix anywhere: expander warps read the pair-ready bitmap words and
// write +-1 f16 straight into the shared-memory operand tile, in the same
// 128-byte-swizzled K-major layout TMA produces. One thread issues the MMAs;
// the accumulators live in TMEM, double-buffered so that the epilogue of one
// tile overlaps the main loop of the next.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 sign expanders, warps 6-9 epilogue (warp w reads TMEM
// lanes 32*(w%4) .. +31, i.e. tokens 32*(w%4) .. +31 of the tile).
//
// Every wait is bounded (blr_device.cuh): a wait that runs out sets the
// shared abort flag and a status bit, the other roles leave their loops, the
// TMA producer drains its in-flight loads, the MMA issuer drains its MMAs, and
// the CTA frees its TMEM and returns.
#pragma once

#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kGemmThreads = 320;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpExp0 = 2;
constexpr int kNumExpWarps = 4;
constexpr int kWarpEpi0 = 6;
constexpr int kNumEpiWarps = 4;

template <int BN>
struct GemmShape {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStagesRaw = (192 * 1024) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : (kStagesRaw < 2 ? 2 : kStagesRaw);
    static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr int kBarBytes = (3 * kStages + 5) * 8;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + 16;
};

// Sum of p[j] over the 32 lanes of the warp, returned in lane j (a
// transpose-reduce: 31 shuffles, fixed order, so deterministic).
__device__ __forceinline__ float warp_column_sums(float (&p)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? p[i] : p[i + o];
            const float keep = upper ? p[i + o] : p[i];
            p[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
    }
    return p[0];
}

__device__ __forceinline__ void fail_status(const GemmArgs &a, volatile int *abort_flag, uint32_t code) {
    *abort_flag = 1;
    atomicOr(a.status, code);
}

// Epilogue of one 32-column chunk. f[] = accumulator of token t (this
// thread's TMEM lane), columns col0 .. col0+31.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs &a, float (&f)[32], long long t, bool valid, int col0,
                                               int part_row, float row_inv, float row_scale) {
    const long long rowoff = t * (long long)a.N + col0;
    const float4 *cv = reinterpret_cast<const float4 *>(a.colv + col0);
    if constexpr (EPI == kEpiFwd1) {
        // a (f32 tape) and a.l staged to f16 for the second forward product
        uint32_t hp[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 lv = __ldg(cv + j);
            hp[2 * j] = pack_half2(f[4 * j] * lv.x, f[4 * j + 1] * lv.y);
            hp[2 * j + 1] = pack_half2(f[4 * j + 2] * lv.z, f[4 * j + 3] * lv.w);
        }
        if (valid) {
            float4 *d = reinterpret_cast<float4 *>(a.out32 + rowoff);
#pragma unroll
            for (int j = 0; j < 8; ++j) d[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
            uint4 *d16 = reinterpret_cast<uint4 *>(a.out16 + rowoff);
#pragma unroll
            for (int j = 0; j < 4; ++j) d16[j] = make_uint4(hp[4 * j], hp[4 * j + 1], hp[4 * j + 2], hp[4 * j + 3]);
        }
    } else if constexpr (EPI == kEpiFwd2) {
        // y (+)= h.c, and c saved in f16 for dh
        if (valid) {
            float4 *d = reinterpret_cast<float4 *>(a.out32 + rowoff);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 hv = __ldg(cv + j);
                float4 y = make_float4(hv.x * f[4 * j], hv.y * f[4 * j + 1], hv.z * f[4 * j + 2], hv.w * f[4 * j + 3]);
                if (a.accumulate) {
                    const float4 o = d[j];
                    y.x += o.x;
                    y.y += o.y;
                    y.z += o.z;
                    y.w += o.w;
                }
                d[j] = y;
            }
            uint4 *d16 = reinterpret_cast<uint4 *>(a.out16 + rowoff);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                d16[j] = make_uint4(pack_half2(f[8 * j], f[8 * j + 1]), pack_half2(f[8 * j + 2], f[8 * j + 3]),
                                    pack_half2(f[8 * j + 4], f[8 * j + 5]), pack_half2(f[8 * j + 6], f[8 * j + 7]));
            }
        }
    } else if constexpr (EPI == kEpiBwd1) {
        // db = acc / s_t; dl partial sum_t a.db; db.l staged under sigma_t
        float p[32];
        uint32_t hp[16];
        const float4 *ap = reinterpret_cast<const float4 *>(a.aux + rowoff);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 av = valid ? __ldg(ap + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 lv = __ldg(cv + j);
            const float d0 = f[4 * j] * row_inv, d1 = f[4 * j + 1] * row_inv;
            const float d2 = f[4 * j + 2] * row_inv, d3 = f[4 * j + 3] * row_inv;
            p[4 * j] = av.x * d0;
            p[4 * j + 1] = av.y * d1;
            p[4 * j + 2] = av.z * d2;
            p[4 * j + 3] = av.w * d3;
            hp[2 * j] = pack_half2(d0 * lv.x * row_scale, d1 * lv.y * row_scale);
            hp[2 * j + 1] = pack_half2(d2 * lv.z * row_scale, d3 * lv.w * row_scale);
        }
        if (valid) {
            uint4 *d16 = reinterpret_cast<uint4 *>(a.out16 + rowoff);
#pragma unroll
            for (int j = 0; j < 4; ++j) d16[j] = make_uint4(hp[4 * j], hp[4 * j + 1], hp[4 * j + 2], hp[4 * j + 3]);
        }
        const float s = warp_column_sums(p);
        a.part[(long long)part_row * a.N + col0 + (threadIdx.x & 31)] = s;
    } else {
        // dx' = acc / sigma_t; dg partial sum_t x.dx'; dx (+)= g.dx'
        float p[32];
        const float4 *xp = reinterpret_cast<const float4 *>(a.aux + rowoff);
        float4 *d = reinterpret_cast<float4 *>(a.out32 + rowoff);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 xv = valid ? __ldg(xp + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 gv = __ldg(cv + j);
            const float d0 = f[4 * j] * row_inv, d1 = f[4 * j + 1] * row_inv;
            const float d2 = f[4 * j + 2] * row_inv, d3 = f[4 * j + 3] * row_inv;
            p[4 * j] = xv.x * d0;
            p[4 * j + 1] = xv.y * d1;
            p[4 * j + 2] = xv.z * d2;
            p[4 * j + 3] = xv.w * d3;
            if (valid) {
                float4 o = make_float4(gv.x * d0, gv.y * d1, gv.z * d2, gv.w * d3);
                if (a.accumulate) {
                    const float4 old = d[j];
                    o.x += old.x;
                    o.y += old.y;
                    o.z += old.z;
                    o.w += old.w;
                }
                d[j] = o;
            }
        }
        const float s = warp_column_sums(p);
        a.part[(long long)part_row * a.N + col0 + (threadIdx.x & 31)] = s;
    }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    blr_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs args) {
    using S = GemmShape<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + S::kStages * S::kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + S::kStages * S::kBBytes);
    uint64_t *full_a = bars;
    uint64_t *full_b = bars + S::kStages;
    uint64_t *empty = bars + 2 * S::kStages;
    uint64_t *tmem_full = bars + 3 * S::kStages;
    uint64_t *tmem_empty = tmem_full + 2;
    uint64_t *drain_bar = tmem_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int M = args.M, N = args.N;
    const int m_tiles = (M + kBM - 1) / kBM;
    const int n_tiles = N / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int num_kb = (args.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(&full_a[s], 1);
            mbar_init(&full_b[s], kNumExpWarps);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tmem_full[i], 1);
            mbar_init(&tmem_empty[i], kNumEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpTma && lane == 0) tma_prefetch_desc(&tmap_a);
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, S::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kWarpTma) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const int m0 = (tile / n_tiles) * kBM;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutTma);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_a[stage], S::kABytes);
                    tma_load_2d(sA + stage * S::kABytes, &tmap_a, &full_a[stage], kb * kBK, m0);
                    issued |= 1u << stage;
                    parity = (parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == S::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // drain: every load issued must have landed before the CTA exits
            for (int s = 0; s < S::kStages; ++s) {
                if (((issued >> s) & 1u) && !mbar_wait(&full_a[s], (parity >> s) & 1u, abort_flag, false))
                    atomicOr(args.status, kStTimeoutDrain);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
                if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)) {
                    fail_status(args, abort_flag, kStTimeoutMma);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full_a[stage], phase, abort_flag) || !mbar_wait(&full_b[stage], phase, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = umma_sdesc_sw128(smem_u32(sA + stage * S::kABytes));
                    const uint64_t bdesc = umma_sdesc_sw128(smem_u32(sB + stage * S::kBBytes));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // advance 16 f16 (32 bytes) along K inside the swizzled rows
                        umma_f16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == S::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tmem_full[acc]);
            }
            // drain: no MMA may still be running when TMEM is freed
            umma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, abort_flag, false)) atomicOr(args.status, kStTimeoutDrain);
        }
        __syncwarp();
    } else if (warp < kWarpEpi0) {
        // ---- sign expanders: bitmap words -> +-1 f16 operand tile --------
        constexpr int kUnits = BN * 2;  // (operand row, word) pairs per k-step
        constexpr int kUpt = (kUnits + 127) / 128;
        const int e = threadIdx.x - kWarpExp0 * 32;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const int n0 = (tile % n_tiles) * BN;
            for (int kb = 0; kb < num_kb; ++kb) {
                const uint32_t *src = args.bsign + ((size_t)kb * N + n0) * 2;
                uint32_t wv[kUpt];
#pragma unroll
                for (int i = 0; i < kUpt; ++i) {
                    const int u = e + 128 * i;
                    wv[i] = (u < kUnits) ? __ldg(src + u) : 0u;
                }
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    if (lane == 0) fail_status(args, abort_flag, kStTimeoutExpand);
                    ok = false;
                    break;
                }
                uint8_t *tile_b = sB + stage * S::kBBytes;
#pragma unroll
                for (int i = 0; i < kUpt; ++i) {
                    const int u = e + 128 * i;
                    if (u < kUnits) {
                        const int row = u >> 1;
                        const int w = u & 1;
                        const uint32_t p = wv[i];
                        uint8_t *rowp = tile_b + row * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 v = make_uint4(sign_pair(p, 4 * j), sign_pair(p, 4 * j + 1),
                                                       sign_pair(p, 4 * j + 2), sign_pair(p, 4 * j + 3));
                            const int chunk = (4 * w + j) ^ (row & 7);
                            *reinterpret_cast<uint4 *>(rowp + chunk * 16) = v;
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_b[stage]);
                if (++stage == S::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ---- epilogue ------------------------------------------------------
        const int q = warp & 3;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
            const int mt = tile / n_tiles;
            const int n0 = (tile % n_tiles) * BN;
            const bool got = mbar_wait(&tmem_full[acc], acc_phase, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) fail_status(args, abort_flag, kStTimeoutEpi);
                break;
            }
            tc_fence_after();
            const long long t = (long long)mt * kBM + q * 32 + lane;
            const bool valid = t < M;
            float row_inv = 1.0f, row_scale = 1.0f;
            if constexpr (EPI == kEpiBwd1 || EPI == kEpiBwd2) {
                if (valid) row_inv = __ldg(args.row_inv + t);
            }
            if constexpr (EPI == kEpiBwd1) {
                if (valid) row_scale = __ldg(args.row_scale + t);
            }
            const int part_row = mt * 4 + q;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + ch * 32), v);
                tmem_wait_ld();
                if (ch == BN / 32 - 1) {
                    // accumulator fully read: hand it back to the MMA issuer
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tmem_empty[acc]);
                }
                float f[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
                epilogue_chunk<EPI>(args, f, t, valid, n0 + ch * 32, part_row, row_inv, row_scale);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem_base, S::kTmemCols);
}

template <int BN, int EPI>
cudaError_t launch_gemm_t(const CUtensorMap &tmap_a, const GemmArgs &args, int grid, cudaStream_t s) {
    using S = GemmShape<BN>;
    static_assert(S::kSmemBytes <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(blr_gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         S::kSmemBytes);
    if (e != cudaSuccess) return e;
    blr_gemm_kernel<BN, EPI><<<grid, kGemmThreads, S::kSmemBytes, s>>>(tmap_a, args);
    return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_gemm_epi(int bn, const CUtensorMap &tmap_a, const GemmArgs &args, int grid, cudaStream_t s) {
    switch (bn) {
        case 32: return launch_gemm_t<32, EPI>(tmap_a, args, grid, s);
        case 64: return launch_gemm_t<64, EPI>(tmap_a, args, grid, s);
        case 128: return launch_gemm_t<128, EPI>(tmap_a, args, grid, s);
        case 256: return launch_gemm_t<256, EPI>(tmap_a, args, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace blr
