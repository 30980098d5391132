// Sign gradients of the blr layer (train_mm.rs, blr_backward documentation
// and its test helper host_sign_grads):
//
//     G_U[i][k] = h_i l_k sum_t dy[t][i] a[t][k]        [d_out][r]
//     G_V[j][k] = g_j l_k sum_t x[t][j]  b[t][k]        [d_in][r],  b = db
//
// Two dense products with the tokens as the reduction dimension. The pass
// already holds every factor in f16, token-major: dy16 = dy.h.s_t,
// x16 = x.g, al16 = a.l, db16 = db.l.sigma_t. The pages transpose their
// operands into token-contiguous copies first (`cvt_t`); here the MMAs read
// the token-major arrays as they are, as MN-major operands (the feature or
// rank index contiguous, K = tokens strided), so no transposed copy exists.
//
// A product over tokens needs one gradient scale. With a fixed scale the
// staged arrays serve directly. With per-token powers of two, the rank-side
// operands are rescaled first: bu = al16 (1/s_t)/max(1/s_t) and
// bv = db16 (1/sigma_t)/max(1/sigma_t), powers of two <= 1 (exact unless a
// value falls into the f16 subnormals); the maxima multiply the products back.
#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

// ------------------------------------------------------------ rescale -----
// 8 f16 per thread step (16-byte accesses); every block first reduces the
// staging's per-block maxima (a few hundred pairs, from L2).
__global__ void __launch_bounds__(256) sign_rescale_kernel(const SignRescaleArgs a) {
    __shared__ float2 mx_s;
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x < 32) {
        float2 m = make_float2(0.0f, 0.0f);
        for (int i = threadIdx.x; i < a.nblk; i += 32) {
            const float2 v = a.blkmax[i];
            m.x = fmaxf(m.x, v.x);
            m.y = fmaxf(m.y, v.y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m.x = fmaxf(m.x, __shfl_xor_sync(0xFFFFFFFFu, m.x, o));
            m.y = fmaxf(m.y, __shfl_xor_sync(0xFFFFFFFFu, m.y, o));
        }
        if (threadIdx.x == 0) {
            // no row with a nonzero gradient: every operand row is zero, any scale will do
            if (!(m.x > 0.0f)) m.x = 1.0f;
            if (!(m.y > 0.0f)) m.y = 1.0f;
            mx_s = m;
            if (blockIdx.x == 0) {
                a.gmax[0] = m.x;
                a.gmax[1] = m.y;
            }
        }
    }
    __syncthreads();
    const float inv_u = 1.0f / mx_s.x, inv_v = 1.0f / mx_s.y;  // powers of two
    const int vpr = a.r / 8;                                      // 16-byte groups per row
    const long long n = (long long)a.M * vpr;
    const uint4 *al = reinterpret_cast<const uint4 *>(a.al16);
    const uint4 *db = reinterpret_cast<const uint4 *>(a.db16);
    uint4 *bu = reinterpret_cast<uint4 *>(a.bu);
    uint4 *bv = reinterpret_cast<uint4 *>(a.bv);
    auto scale8 = [](uint4 w, float f) {
        uint32_t *p = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&p[i]));
            p[i] = pack_half2(v.x * f, v.y * f);
        }
        return w;
    };
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / vpr);
        const float fu = __ldg(a.s_inv + t) * inv_u;
        const float fv = __ldg(a.sig_inv + t) * inv_v;
        bu[i] = scale8(al[i], fu);
        bv[i] = scale8(db[i], fv);
    }
}

// ------------------------------------------------------ the products ------
// One persistent launch over the tiles of both products: tile = 128 features
// x BN ranks, K = tokens in 64-token k-steps. Warp 0 TMA producer, warp 1
// MMA issuer (tcgen05 kind::f16, both operands MN-major in shared memory),
// warps 2-5 epilogue: G = acc * scale, each 32 x 32 chunk staged in shared
// memory (128-byte swizzle) and written by a TMA store.
//
// Shared-memory operand tiles, as TMA writes them with the 128-byte swizzle:
// blocks of [64 tokens][64 features] f16 (8 KB; row = token, 128 bytes),
// two blocks for the 128 features of A, BN/64 blocks for the ranks of B. In
// the MN-major canonical layout the 8-token row groups are 1024 bytes apart
// (stride byte offset) and the 64-element blocks 8 KB apart (leading byte
// offset); one MMA (K = 16) takes two row groups, so the k-th MMA of a
// k-step starts 2048 k bytes into the tiles.
struct SignGemmArgs {
    int F0, F1;                  // features of the two products
    float scale0, scale1;
    const float *dscale0, *dscale1;
    float *out0, *out1;          // [F][R] (read when accumulating)
    int R;                       // ranks
    int M;                       // tokens
    int accumulate;
    uint32_t *status;
};

constexpr int kSgThreads = 192;
constexpr int kSgEpi0 = 2;
constexpr uint32_t kMnBlockBytes = 64 * 64 * 2;

template <int BN>
struct SignGemmShape {
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

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle
// layout (fields as in umma_sdesc_sw128): leading byte offset = stride of the
// 64-element blocks along M or N, stride byte offset = stride of the 8-row
// groups along K.
__device__ __forceinline__ uint64_t umma_sdesc_sw128_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(kMnBlockBytes >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor with both operands MN-major (transpose bits 15, 16).
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32_mn(int m, int n) {
    return umma_idesc_f16_f32(m, n) | (1u << 15) | (1u << 16);
}

__device__ __forceinline__ int sw128_chunk_off(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }

template <int BN>
__global__ void __launch_bounds__(kSgThreads, 1)
    sign_gemm_kernel(const __grid_constant__ SignGemmMaps maps, const SignGemmArgs args) {
    using S = SignGemmShape<BN>;
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
    const int num_ks = (args.M + 63) / 64;
    // tile -> (product, feature tile, rank tile); rank tile varies fastest
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
                    const int t0 = ks * 64;
                    tma_load_2d(st, ma, &full[sb], f0, t0);
                    tma_load_2d(st + kMnBlockBytes, ma, &full[sb], f0 + 64, t0);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(st + S::kABytes + j * kMnBlockBytes, mb, &full[sb], k0 + 64 * j, t0);
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
            constexpr uint32_t idesc = umma_idesc_f16_f32_mn(128, BN);
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
                    const uint64_t adesc = umma_sdesc_sw128_mn(smem_u32(sS + sb * S::kStage));
                    const uint64_t bdesc = umma_sdesc_sw128_mn(smem_u32(sS + sb * S::kStage + S::kABytes));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16(d_tmem, adesc + (uint64_t)(128 * k), bdesc + (uint64_t)(128 * k), idesc,
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
        // ---- epilogue: thread = one feature row of the tile ----------------
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
            const int fr = f0 + q * 32;  // this warp's 32 feature rows
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
                const int kc = k0 + 32 * c;  // first rank of the chunk
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

// ------------------------------------------------------------ launchers ---
cudaError_t launch_sign_rescale(const SignRescaleArgs &a, int sms, cudaStream_t s) {
    const long long n = (long long)a.M * (a.r / 8);
    long long blocks = (n + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    trace_before("sign_rescale", s);
    const cudaError_t e = launch_k(sign_rescale_kernel, dim3((unsigned)blocks), dim3(256), 0, s, a);
    trace_after(s);
    return e;
}

cudaError_t launch_sign_gemm(const SignGemmLaunch &L, cudaStream_t s) {
    static bool prepared = false;
    if (!prepared) {
        cudaError_t e = prepare_kernel(sign_gemm_kernel<128>, SignGemmShape<128>::kSmemBytes);
        if (e == cudaSuccess) e = prepare_kernel(sign_gemm_kernel<256>, SignGemmShape<256>::kSmemBytes);
        if (e != cudaSuccess) return e;
        prepared = true;
    }
    SignGemmArgs ga{};
    ga.F0 = L.F[0];
    ga.F1 = L.F[1];
    ga.scale0 = L.scale[0];
    ga.scale1 = L.scale[1];
    ga.dscale0 = L.dscale[0];
    ga.dscale1 = L.dscale[1];
    ga.out0 = L.out[0];
    ga.out1 = L.out[1];
    ga.R = L.r;
    ga.M = L.M;
    ga.accumulate = L.accumulate;
    ga.status = L.status;
    const int bn = sign_bn(L.r);
    const long long tiles = (long long)(((L.F[0] + 127) / 128) + ((L.F[1] + 127) / 128)) * ((L.r + bn - 1) / bn);
    const int grid = (int)(tiles < L.sms ? tiles : L.sms);
    cudaError_t e;
    trace_before("sign_gemm", s);
    if (bn == 256)
        e = launch_k(sign_gemm_kernel<256>, dim3(grid), dim3(kSgThreads), SignGemmShape<256>::kSmemBytes, s, L.maps,
                     ga);
    else
        e = launch_k(sign_gemm_kernel<128>, dim3(grid), dim3(kSgThreads), SignGemmShape<128>::kSmemBytes, s, L.maps,
                     ga);
    trace_after(s);
    return e;
}

}  // namespace blr
