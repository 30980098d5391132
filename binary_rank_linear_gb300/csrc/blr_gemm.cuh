// Persistent tcgen05 GEMM of the blr layer on sm_103a:
//
//     acc[t][n] = sum_k act16[t][k] * S[n][k]        (S = +-1, exact in f16)
//
// for one 128-token x BN-feature tile at a time, with a fused epilogue per
// pass. The activation operand is an f16 matrix [M][K] brought in by TMA
// (128-byte swizzle, box 64 x 128). The sign operand is never stored as a
// dense matrix anywhere: the TMA producer bulk-copies each k-step's
// pair-ready bitmap words (BN x 8 bytes) next to the activation tile, and
// expander warps turn them into +-1 f16 straight in a shared-memory operand
// tile, in the same 128-byte-swizzled K-major layout TMA produces. One thread
// issues the MMAs; the accumulators live in TMEM, double-buffered so that the
// epilogue of one tile overlaps the main loop of the next.
//
// Two rings feed the MMAs: a deep "A ring" (activation tile + bitmap words,
// filled by TMA, so that load latency is hidden) and a shallow "B ring" of
// expanded sign tiles (filled by the expanders from the A ring's words).
//
// Warp roles (448 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-9 sign expanders, warps 10-13 epilogue (warp w reads TMEM
// lanes 32*(w%4) .. +31, i.e. tokens 32*(w%4) .. +31 of the tile).
//
// Per k-step the MMA issuer waits on one barrier (full_b: the expanders
// finished the sign tile; they had waited for the stage's activation tile
// and bitmap words on full_a, so full_b implies full_a) and commits once
// (empty_a). An expander reuses sign slot i % NB once the MMAs of k-step
// i - NB completed, which is the completion of empty_a for that k-step.
//
// Epilogues: the two products with a wide output (c and dx', N = d_out or
// d_in, K = r) stage each 32 x 32 output chunk in per-warp shared memory and
// write it with TMA stores; their input chunks (x for dg, y for accumulation)
// arrive by TMA into the same buffers, double-buffered. The two products with
// a narrow output (a and db, N = r) write straight from registers.
//
// Every wait is bounded (blr_device.cuh): a wait that runs out sets the
// shared abort flag and a status bit, the other roles leave their loops, the
// TMA producer drains its in-flight loads, the epilogue drains its copies,
// the MMA issuer drains its MMAs, and the CTA frees its TMEM and returns.
#pragma once

#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kGemmThreads = 448;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpExp0 = 2;
constexpr int kNumExpWarps = 8;
constexpr int kWarpEpi0 = 10;
constexpr int kNumEpiWarps = 4;

template <int BN, int EPI, bool PAIR>
struct GemmShape {
    static constexpr bool kTmaEpi = (EPI == kEpiFwd2 || EPI == kEpiBwd2);
    static constexpr int kKB = PAIR ? 2 : 1;            // 64-wide K blocks per k-step
    static constexpr int kStepK = kKB * kBK;            // K per k-step
    static constexpr int kBRows = PAIR ? BN / 2 : BN;   // sign-tile rows this CTA expands
    static constexpr int kABlock = kBM * kBK * 2;       // one 128 x 64 activation box
    static constexpr int kABytes = kKB * kABlock;       // activation tile of a k-step
    static constexpr int kBitsBlock = kBRows * 8;       // bitmap words of one 64-wide block
    static constexpr int kBitsBytes = kKB * kBitsBlock;
    static constexpr int kBBlock = kBRows * kBK * 2;    // one 64-wide block of the sign tile
    static constexpr int kBBytes = kKB * kBBlock;       // expanded sign tile (this CTA's rows)
    static constexpr int kEpiF32 = 32 * 32 * 4;
    static constexpr int kEpiF16 = (EPI == kEpiFwd2) ? 32 * 32 * 2 : 0;
    static constexpr int kEpiBuf = kEpiF32 + kEpiF16;
    static constexpr int kEpiBytes = kTmaEpi ? kNumEpiWarps * 2 * kEpiBuf : 0;
    static constexpr int kBudget = (PAIR ? 220 : 205) * 1024 - kEpiBytes;
    static constexpr int kNB = kTmaEpi ? 2 : (PAIR ? 3 : (kBRows >= 128 ? 3 : 4));
    static constexpr int kNARaw = (kBudget - kNB * kBBytes) / (kABytes + kBitsBytes);
    static constexpr int kNA = kNARaw > 8 ? 8 : kNARaw;
    static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr int kBitsRegion = ((kNA * kBitsBytes + 1023) / 1024) * 1024;
    static constexpr int kNumBars = 2 * kNA + kNB + 4 + 1 + kNumEpiWarps * 2;
    static constexpr int kSmemBytes =
        1024 + kNA * kABytes + kNB * kBBytes + kEpiBytes + kBitsRegion + kNumBars * 8 + 16;
    static_assert(kNA >= 2, "activation ring too shallow");
    // an expander frees sign slot i % NB by waiting on the activation slot of
    // k-step i - NB; that wait is unambiguous only if the activation ring is at
    // least as deep as the sign ring
    static_assert(kNA >= kNB, "activation ring must be at least as deep as the sign ring");
    static_assert(kBitsBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(!PAIR || BN >= 64, "a pair splits the sign tile in two halves of >= 32 rows");
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

// Byte offset of 16-byte chunk c of row `row` in a box with 128-byte rows in
// the 128-byte swizzle (the layout TMA reads and writes).
__device__ __forceinline__ int sw128_off(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }
// Same for 64-byte rows and the 64-byte swizzle.
__device__ __forceinline__ int sw64_off(int row, int c) { return row * 64 + ((c ^ ((row >> 1) & 3)) << 4); }

// Epilogue of one 32-column chunk of a narrow-output product (N = r), written
// straight from registers. f[] = accumulator of token t (this thread's TMEM
// lane), columns col0 .. col0+31.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk_direct(const GemmArgs &a, float (&f)[32], long long t, bool valid,
                                                      int col0, int part_row, float row_inv, float row_scale) {
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
    } else {
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
    }
}

// Epilogue of one 32-column chunk of a wide-output product, through the
// warp's shared-memory chunk buffer `buf` (f32 part in the 128-byte swizzle;
// for the forward an f16 part at +4096 in the 64-byte swizzle). When `has_in`
// the f32 part already holds the chunk's input (x for the backward, y for an
// accumulating forward); outputs overwrite the buffer in place.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk_smem(const GemmArgs &a, float (&f)[32], uint8_t *buf, long long t,
                                                    bool valid, int col0, int part_row, float row_inv,
                                                    bool has_in) {
    const int row = threadIdx.x & 31;
    const float4 *cv = reinterpret_cast<const float4 *>(a.colv + col0);
    if constexpr (EPI == kEpiFwd2) {
        // y (+)= h.c, c saved in f16
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 hv = __ldg(cv + j);
            float4 y = make_float4(hv.x * f[4 * j], hv.y * f[4 * j + 1], hv.z * f[4 * j + 2], hv.w * f[4 * j + 3]);
            float4 *slot = reinterpret_cast<float4 *>(buf + sw128_off(row, j));
            if (has_in) {
                const float4 o = *slot;
                y.x += o.x;
                y.y += o.y;
                y.z += o.z;
                y.w += o.w;
            }
            *slot = y;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint4 *>(buf + 4096 + sw64_off(row, j)) =
                make_uint4(pack_half2(f[8 * j], f[8 * j + 1]), pack_half2(f[8 * j + 2], f[8 * j + 3]),
                           pack_half2(f[8 * j + 4], f[8 * j + 5]), pack_half2(f[8 * j + 6], f[8 * j + 7]));
        }
    } else {
        // dx' = acc / sigma_t; dg partial sum_t x.dx'; dx (+)= g.dx'
        float p[32];
        const long long rowoff = t * (long long)a.N + col0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 *slot = reinterpret_cast<float4 *>(buf + sw128_off(row, j));
            const float4 xv = *slot;  // rows past M arrive as zeros
            const float4 gv = __ldg(cv + j);
            const float d0 = f[4 * j] * row_inv, d1 = f[4 * j + 1] * row_inv;
            const float d2 = f[4 * j + 2] * row_inv, d3 = f[4 * j + 3] * row_inv;
            p[4 * j] = xv.x * d0;
            p[4 * j + 1] = xv.y * d1;
            p[4 * j + 2] = xv.z * d2;
            p[4 * j + 3] = xv.w * d3;
            float4 o = make_float4(gv.x * d0, gv.y * d1, gv.z * d2, gv.w * d3);
            if (a.accumulate && valid) {
                const float4 old = *reinterpret_cast<const float4 *>(a.out32 + rowoff + 4 * j);
                o.x += old.x;
                o.y += old.y;
                o.z += old.z;
                o.w += old.w;
            }
            *slot = o;
        }
        const float s = warp_column_sums(p);
        a.part[(long long)part_row * a.N + col0 + (threadIdx.x & 31)] = s;
    }
}

// PAIR = false: one CTA per 128-token tile (tcgen05 cta_group::1).
// PAIR = true: a cluster of two CTAs per 256-token tile (cta_group::2). Each
// CTA loads its own 128 activation rows and expands half of the sign tile;
// the leader (rank 0) issues the M=256 MMAs, which read both CTAs' shared
// memory and write each CTA's TMEM. Within each CTA the producer, expanders
// and epilogue signal local barriers only; the peer's MMA warp waits until a
// k-step's sign half is in place (which follows its activation tile) and then
// makes the one cluster-scope arrival on the leader's full_b (a cluster-scope
// release costs a memory barrier, so it is paid once per k-step, not per
// warp). The peer's epilogue warps release their TMEM half to the leader
// remotely, once per tile. The leader's commits are multicast to both CTAs'
// barriers.
template <int BN, int EPI, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    blr_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ EpiMaps emaps,
                    const GemmArgs args) {
    using S = GemmShape<BN, EPI, PAIR>;
    constexpr int NA = S::kNA, NB = S::kNB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                                                 // [NA][kABytes]
    uint8_t *sB = sA + NA * S::kABytes;                                 // [NB][kBBytes]
    uint8_t *sE = sB + NB * S::kBBytes;                                 // [4 warps][2][kEpiBuf]
    uint32_t *sBits = reinterpret_cast<uint32_t *>(sE + S::kEpiBytes);  // [NA][BN*2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sBits) + S::kBitsRegion);
    uint64_t *full_a = bars;
    uint64_t *empty_a = full_a + NA;
    uint64_t *full_b = empty_a + NA;
    uint64_t *tmem_full = full_b + NB;
    uint64_t *tmem_empty = tmem_full + 2;
    uint64_t *drain_bar = tmem_full + 4;
    uint64_t *eload = drain_bar + 1;  // [4 warps][2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(eload + kNumEpiWarps * 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int M = args.M, N = args.N;
    constexpr int kUnitRows = PAIR ? 2 * kBM : kBM;  // token rows per tile
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // tile worker (CTA or pair)
    const int num_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int m_tiles = (M + kUnitRows - 1) / kUnitRows;
    const int n_tiles = N / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int num_kb = (args.K + S::kStepK - 1) / S::kStepK;  // k-steps per tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < NA; ++s) {
            mbar_init(&full_a[s], 1);
            mbar_init(&empty_a[s], 1);
        }
        for (int s = 0; s < NB; ++s) mbar_init(&full_b[s], (PAIR && leader) ? kNumExpWarps + 1 : kNumExpWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tmem_full[i], 1);
            mbar_init(&tmem_empty[i], PAIR ? 2 * kNumEpiWarps : kNumEpiWarps);
        }
        mbar_init(drain_bar, 1);
        for (int i = 0; i < kNumEpiWarps * 2; ++i) mbar_init(&eload[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpTma && lane == 0) tma_prefetch_desc(&tmap_a);
    if constexpr (S::kTmaEpi) {
        if (warp == kWarpEpi0 && lane == 0) {
            tma_prefetch_desc(&emaps.out32);
            tma_prefetch_desc(&emaps.in32);
            if constexpr (EPI == kEpiFwd2) tma_prefetch_desc(&emaps.out16);
        }
    }
    if constexpr (PAIR) {
        cluster_sync();  // both CTAs' barriers exist before any remote arrival
        if (warp == kWarpMma) {
            tmem_alloc_pair(tmem_slot, S::kTmemCols);
            tmem_relinquish_pair();
        }
    } else {
        if (warp == kWarpMma) {
            tmem_alloc(tmem_slot, S::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the leader's copy of a barrier, as a cluster address (PAIR only)
    auto leader_bar = [&](uint64_t *bar) -> uint32_t { return mapa_shared(smem_u32(bar), 0); };
    // setup above overlaps the previous kernel; global memory only after this
    pdl_wait();
    pdl_launch_dependents();

    if (warp == kWarpTma) {
        if (lane == 0) {
            int sa = 0;
            uint32_t pa = 0, issued = 0, parity = 0;
            bool ok = true;
            for (int tile = unit; tile < num_tiles && ok; tile += num_units) {
                const int m0 = (tile / n_tiles) * kUnitRows + (int)rank * kBM;
                const int nb0 = (tile % n_tiles) * BN + (int)rank * S::kBRows;  // this CTA's sign rows
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty_a[sa], pa ^ 1u, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutTma);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_a[sa], S::kABytes + S::kBitsBytes);
#pragma unroll
                    for (int kk = 0; kk < S::kKB; ++kk) {
                        const int blk = kb * S::kKB + kk;  // 64-wide K block (the bitmap layout pads to kKB)
                        tma_load_2d(sA + sa * S::kABytes + kk * S::kABlock, &tmap_a, &full_a[sa], blk * kBK, m0);
                        bulk_load(sBits + sa * (S::kBitsBytes / 4) + kk * (S::kBitsBlock / 4),
                                  args.bsign + ((size_t)blk * N + nb0) * 2, S::kBitsBlock, &full_a[sa]);
                    }
                    issued |= 1u << sa;
                    parity = (parity & ~(1u << sa)) | (pa << sa);
                    if (++sa == NA) {
                        sa = 0;
                        pa ^= 1u;
                    }
                }
            }
            // drain: every load issued must have landed before the CTA exits
            for (int s = 0; s < NA; ++s) {
                if (((issued >> s) & 1u) && !mbar_wait(&full_a[s], (parity >> s) & 1u, abort_flag, false))
                    atomicOr(args.status, kStTimeoutDrain);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(PAIR ? 2 * kBM : kBM, BN);
            int sa = 0, sb = 0;
            uint32_t pa = 0, pb = 0;
            bool ok = true;
            int local = 0;
            for (int tile = unit; tile < num_tiles && ok; tile += num_units, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
                const bool got = PAIR ? mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)
                                      : mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag);
                if (!got) {
                    fail_status(args, abort_flag, kStTimeoutMma);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    const bool ready = PAIR ? mbar_wait_cluster(&full_b[sb], pb, abort_flag)
                                            : mbar_wait(&full_b[sb], pb, abort_flag);
                    if (!ready) {
                        fail_status(args, abort_flag, kStTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < S::kKB; ++kk) {
                        const uint64_t adesc = umma_sdesc_sw128(smem_u32(sA + sa * S::kABytes + kk * S::kABlock));
                        const uint64_t bdesc = umma_sdesc_sw128(smem_u32(sB + sb * S::kBBytes + kk * S::kBBlock));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // advance 16 f16 (32 bytes) along K inside the swizzled rows
                            const uint32_t acc_in = (kb > 0 || kk > 0 || k > 0) ? 1u : 0u;
                            if constexpr (PAIR)
                                umma_f16_pair(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                                              acc_in);
                            else
                                umma_f16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc, acc_in);
                        }
                    }
                    if constexpr (PAIR)
                        umma_commit_pair_multicast(&empty_a[sa], 3);
                    else
                        umma_commit(&empty_a[sa]);
                    if (++sa == NA) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sb == NB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    umma_commit_pair_multicast(&tmem_full[acc], 3);
                else
                    umma_commit(&tmem_full[acc]);
            }
            // drain: no MMA may still be running when TMEM is freed
            if constexpr (PAIR)
                umma_commit_pair_multicast(drain_bar, 1);
            else
                umma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, abort_flag, false)) atomicOr(args.status, kStTimeoutDrain);
        } else if (PAIR && lane == 0) {
            // the peer's MMA warp: once a k-step's sign half is in this CTA's
            // shared memory (after its activation tile), one arrival on the leader
            int sb = 0;
            uint32_t pb = 0;
            bool ok = true;
            for (int tile = unit; tile < num_tiles && ok; tile += num_units) {
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full_b[sb], pb, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutMma);
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(leader_bar(&full_b[sb]));
                    if (++sb == NB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < kWarpEpi0) {
        // ---- sign expanders: bitmap words -> +-1 f16 operand tile --------
        constexpr int kUnits = S::kBRows * 2 * S::kKB;  // (operand row, word) pairs per k-step
        constexpr int kExpThreads = kNumExpWarps * 32;
        constexpr int kUpt = (kUnits + kExpThreads - 1) / kExpThreads;
        const int e = threadIdx.x - kWarpExp0 * 32;
        int sa = 0, sb = 0;
        uint32_t pa = 0;
        int lag = -NB;              // k-step whose MMAs must have freed this sign slot
        int ls = 0;                 // its activation slot
        uint32_t lp = 0;            // and that slot's phase parity
        bool ok = true;
        for (int tile = unit; tile < num_tiles && ok; tile += num_units) {
            for (int kb = 0; kb < num_kb; ++kb) {
                bool got = mbar_wait(&full_a[sa], pa, abort_flag);
                if (got && lag >= 0) got = mbar_wait(&empty_a[ls], lp, abort_flag);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    if (lane == 0) fail_status(args, abort_flag, kStTimeoutExpand);
                    ok = false;
                    break;
                }
                const uint32_t *bits = sBits + sa * (S::kBitsBytes / 4);
                uint8_t *tile_b = sB + sb * S::kBBytes;
#pragma unroll
                for (int i = 0; i < kUpt; ++i) {
                    const int u = e + kExpThreads * i;
                    if (u < kUnits) {
                        const int kk = u / (S::kBRows * 2);  // 64-wide block
                        const int v = u - kk * (S::kBRows * 2);
                        const int row = v >> 1;
                        const int w = v & 1;
                        const uint32_t p = bits[u];
                        uint8_t *rowp = tile_b + kk * S::kBBlock + row * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 q4 = make_uint4(sign_pair(p, 4 * j), sign_pair(p, 4 * j + 1),
                                                        sign_pair(p, 4 * j + 2), sign_pair(p, 4 * j + 3));
                            const int chunk = (4 * w + j) ^ (row & 7);
                            *reinterpret_cast<uint4 *>(rowp + chunk * 16) = q4;
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_b[sb]);
                if (++sa == NA) {
                    sa = 0;
                    pa ^= 1u;
                }
                if (++sb == NB) sb = 0;
                if (++lag > 0) {
                    if (++ls == NA) {
                        ls = 0;
                        lp ^= 1u;
                    }
                }
            }
        }
    } else {
        // ---- epilogue ------------------------------------------------------
        const int q = warp & 3;
        constexpr int kChunks = BN / 32;
        uint8_t *ebuf = sE + (warp - kWarpEpi0) * 2 * S::kEpiBuf;
        uint64_t *ebar = eload + (warp - kWarpEpi0) * 2;
        const bool has_in = (EPI == kEpiBwd2) || (EPI == kEpiFwd2 && args.accumulate);
        uint32_t ephase = 0u;   // bit b: phase of buffer b's next input load
        uint32_t pending = 0u;  // bit b: an input load in flight into buffer b (lane 0's view)
        int gch = 0;                       // running chunk count: buffer = gch & 1
        int local = 0;
        bool ok = true;
        for (int tile = unit; tile < num_tiles && ok; tile += num_units, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
            const int mt = (tile / n_tiles) * (PAIR ? 2 : 1) + (int)rank;  // 128-row tile index
            const int n0 = (tile % n_tiles) * BN;
            const int row0 = mt * kBM + q * 32;
            if constexpr (S::kTmaEpi) {
                // this tile's first two input chunks, once the buffers' last stores have read them
                if (has_in && lane == 0) {
                    bulk_wait_group_read<0>();
                    for (int c = 0; c < 2 && c < kChunks; ++c) {
                        const int b = (gch + c) & 1;
                        mbar_arrive_expect_tx(&ebar[b], S::kEpiF32);
                        tma_load_2d(ebuf + b * S::kEpiBuf, &emaps.in32, &ebar[b], n0 + 32 * c, row0);
                        pending |= 1u << b;
                    }
                }
            }
            const bool got = mbar_wait(&tmem_full[acc], acc_phase, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) fail_status(args, abort_flag, kStTimeoutEpi);
                ok = false;
                break;
            }
            tc_fence_after();
            const long long t = (long long)row0 + lane;
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
            for (int ch = 0; ch < kChunks; ++ch, ++gch) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + ch * 32), v);
                tmem_wait_ld();
                if (ch == kChunks - 1) {
                    // accumulator fully read: hand it back to the MMA issuer
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_remote(leader_bar(&tmem_empty[acc]));
                        else
                            mbar_arrive(&tmem_empty[acc]);
                    }
                }
                float f[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
                if constexpr (S::kTmaEpi) {
                    const int b = gch & 1;
                    uint8_t *buf = ebuf + b * S::kEpiBuf;
                    if (has_in) {
                        const bool in_ok = mbar_wait(&ebar[b], (ephase >> b) & 1u, abort_flag);
                        ephase ^= 1u << b;
                        pending &= ~(1u << b);
                        if (!__all_sync(0xFFFFFFFFu, in_ok)) {
                            if (lane == 0) fail_status(args, abort_flag, kStTimeoutEpi);
                            ok = false;
                            break;
                        }
                    } else {
                        // the store that last used this buffer must have read it
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                    }
                    epilogue_chunk_smem<EPI>(args, f, buf, t, valid, n0 + ch * 32, part_row, row_inv, has_in);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&emaps.out32, buf, n0 + ch * 32, row0);
                        if constexpr (EPI == kEpiFwd2) tma_store_2d(&emaps.out16, buf + 4096, n0 + ch * 32, row0);
                        bulk_commit_group();
                        if (has_in && ch + 2 < kChunks) {
                            // chunk ch+2 uses this buffer again: load it once the store has read it
                            bulk_wait_group_read<0>();
                            mbar_arrive_expect_tx(&ebar[b], S::kEpiF32);
                            tma_load_2d(buf, &emaps.in32, &ebar[b], n0 + 32 * (ch + 2), row0);
                            pending |= 1u << b;
                        }
                    }
                    __syncwarp();
                } else {
                    epilogue_chunk_direct<EPI>(args, f, t, valid, n0 + ch * 32, part_row, row_inv, row_scale);
                }
            }
        }
        if constexpr (S::kTmaEpi) {
            // drain: stores complete, and input loads issued but not consumed have landed
            if (lane == 0) {
                bulk_wait_group_all();
                for (int b = 0; b < 2; ++b)
                    if (((pending >> b) & 1u) && !mbar_wait(&ebar[b], (ephase >> b) & 1u, abort_flag, false))
                        atomicOr(args.status, kStTimeoutDrain);
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    if constexpr (PAIR) {
        // neither CTA leaves while the pair's MMAs or remote arrivals may still touch it
        cluster_sync();
        tc_fence_after();
        if (warp == kWarpMma) tmem_dealloc_pair(tmem_base, S::kTmemCols);
    } else {
        __syncthreads();
        tc_fence_after();
        if (warp == kWarpMma) tmem_dealloc(tmem_base, S::kTmemCols);
    }
}

template <int BN, int EPI, bool PAIR>
cudaError_t launch_gemm_t(const CUtensorMap &tmap_a, const EpiMaps &emaps, const GemmArgs &args, int grid,
                          cudaStream_t s) {
    using S = GemmShape<BN, EPI, PAIR>;
    static bool attr_set = false;  // set once, outside any later stream capture
    if (!attr_set) {
        cudaError_t e = prepare_kernel(blr_gemm_kernel<BN, EPI, PAIR>, S::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if constexpr (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kGemmThreads);
        cfg.dynamicSmemBytes = S::kSmemBytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, blr_gemm_kernel<BN, EPI, PAIR>, tmap_a, emaps, args);
    } else {
        return launch_k(blr_gemm_kernel<BN, EPI, PAIR>, dim3(grid), dim3(kGemmThreads), S::kSmemBytes, s, tmap_a,
                        emaps, args);
    }
}

// bn > 0: one CTA per 128-token tile of width bn; bn < 0: CTA pairs, tiles of
// 256 tokens x |bn| features (|bn| = 128 or 256). `grid` counts CTAs (even for
// pairs).
template <int EPI>
cudaError_t launch_gemm_epi(int bn, const CUtensorMap &tmap_a, const EpiMaps &emaps, const GemmArgs &args,
                            int grid, cudaStream_t s) {
    switch (bn) {
        case 32: return launch_gemm_t<32, EPI, false>(tmap_a, emaps, args, grid, s);
        case 64: return launch_gemm_t<64, EPI, false>(tmap_a, emaps, args, grid, s);
        case 128: return launch_gemm_t<128, EPI, false>(tmap_a, emaps, args, grid, s);
        case 256: return launch_gemm_t<256, EPI, false>(tmap_a, emaps, args, grid, s);
        case -128: return launch_gemm_t<128, EPI, true>(tmap_a, emaps, args, grid, s);
        case -256: return launch_gemm_t<256, EPI, true>(tmap_a, emaps, args, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace blr
