// In-kernel staging of the a- and db-products' activation operand.
//
// The separate staging passes of the layer (x16 = f16(x.g) before the
// a-product; dy16 = f16(dy.h.s_t) with the dh sums before the db-product) are
// HBM streams that leave the tensor cores idle, while the r-wide products
// they feed leave most of the HBM bandwidth idle. Here the staging runs inside
// those products' persistent kernels, on two stager warps of every CTA, ahead
// of the MMA pipeline:
//
//  - Work items are blocks of token rows and columns, taken in the order the
//    persistent grid consumes token tiles: round by round (a round is the
//    token tiles whose feature tiles the units start together), then column
//    chunk by column chunk (x only), then token tile and row group. CTA c
//    stages items c, c + grid, c + 2 grid, ...
//  - Stager thread 0 bulk-copies the items' f32 row segments into a 48 KB
//    shared-memory ring (cp.async.bulk, full/empty mbarriers) several units
//    ahead, and asks L2 to prefetch the units after those; the 64 stager
//    threads convert from shared memory and write f16 with plain 8-byte
//    stores, so the staged tiles sit in L2 when the products' TMA loads come.
//  - After an item, the stagers publish the rows they finished on a counter
//    of its (token tile, column chunk): stores, a proxy fence (the consumer
//    reads by TMA), a barrier of the stager warps, then one release add. The
//    TMA producer acquires the counter of each chunk of a tile before its
//    loads (bounded wait), then fences the async proxy.
//  - x needs no row-wide quantity, so its counters are per 256-column chunk
//    and a product starts as soon as the first chunk of its first round is
//    staged. dy's per-token scale needs the whole row first, so a dy item is 4
//    whole rows in two passes (statistics and dh sums, then the f16 rows, dy
//    read again from L2), and its counters are per token tile.
//
// Stagers never wait for another CTA: every counter completes once the
// stagers of the grid have run (the CTAs of the persistent grid are resident
// together). A bounded wait that runs out, or the CTA's abort flag, stops
// them between items; thread 0 then waits for the copies it issued.
#pragma once

#include <cuda_fp16.h>

#include "blr_device.cuh"
#include "blr_kernels.h"
#include "blr_stage.cuh"

namespace blr {

constexpr int kStgWarps = 2;
constexpr int kStgThreads = kStgWarps * 32;
constexpr int kStgBar = 8;          // named barrier of the stager warps (0 is __syncthreads)
constexpr int kStgKC = kStageChunkCols;  // columns per chunk: one float4 per stager thread
constexpr int kStgRingBytes = 48 * 1024;
constexpr int kStgSlotsMax = 8;
// x: items of 8 rows x 256 columns (8 KB f32), one ring slot each
constexpr int kStgRowsX = 8;
constexpr int kStgSlotX = kStgRowsX * kStgKC * 4;
constexpr int kStgSlotsX = kStgRingBytes / kStgSlotX;
// dy: items of 4 whole rows; a ring unit is one 256-column chunk of them, dy
// (4 KB) and c (2 KB) in the first pass, dy alone in the second
constexpr int kStgRowsDy = 4;
constexpr int kStgSlotDy = kStgRowsDy * kStgKC * 6;
constexpr int kStgSlotsDy = kStgRingBytes / kStgSlotDy;
constexpr int kStgPrefetchUnits = 6;  // units prefetched into L2 beyond those in the ring
static_assert(kStgSlotsX >= 2 && kStgSlotsX <= kStgSlotsMax && kStgSlotsDy >= 2 && kStgSlotsDy <= kStgSlotsMax,
              "stager ring");

__host__ __device__ constexpr int stg_chunks(int K, int mode) { return mode == 1 ? (K + kStgKC - 1) / kStgKC : 1; }
static_assert(kStgKC == 4 * kStgThreads, "a chunk is one float4 per stager thread");

// Shared-memory scratch of the stager warps, inside the GEMM control block.
struct StgScratch {
    float2 red[kStgWarps][kStgRowsDy];  // per-warp (max |dy.h|, sum |dy.h|) of the item's rows
    float lmax[kStgWarps];
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned int *p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *cnt >= target (acquire). False when the wait ran out or
// the CTA's abort flag was raised.
__device__ __forceinline__ bool wait_count(const unsigned int *cnt, unsigned int target,
                                           const volatile int *abort_flag) {
    if (ld_acquire_u32(cnt) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(100);
        if (ld_acquire_u32(cnt) >= target) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// Consumption order of the persistent GEMM grid and the stager items.
struct StgGeom {
    int M, K, BT, t_tiles, f_tiles, units, n_kc, R, n_rg;

    __device__ StgGeom(int M_, int K_, int BT_, int f_tiles_, int units_, int mode)
        : M(M_), K(K_), BT(BT_), t_tiles((M_ + BT_ - 1) / BT_), f_tiles(f_tiles_), units(units_),
          n_kc(stg_chunks(K_, mode)), R(mode == 1 ? kStgRowsX : kStgRowsDy), n_rg((BT_ + R - 1) / R) {}
    // round of a token tile: the units start tiles u, u + units, ... with the
    // feature tile varying fastest, so token tile tt first appears in round
    // floor(tt * f_tiles / units)
    __device__ int round_of(int tt) const { return (int)(((long long)tt * f_tiles) / units); }
    // first token tile of round r: ceil(r * units / f_tiles)
    __device__ int tt_begin(int r) const {
        const long long v = ((long long)r * units + f_tiles - 1) / f_tiles;
        return v < t_tiles ? (int)v : t_tiles;
    }
    __device__ long long items() const { return (long long)t_tiles * n_kc * n_rg; }
    // item i -> (token tile, column chunk, row group); rounds partition the
    // token tiles in order, so the items before round r are tt_begin(r) * n_kc * n_rg
    __device__ void item(long long i, int &tt, int &kc, int &rg) const {
        const long long P = (long long)n_kc * n_rg;
        const int r = round_of((int)(i / P));
        const int lo = tt_begin(r), hi = tt_begin(r + 1);
        const long long ii = i - (long long)lo * P;
        const long long per_kc = (long long)(hi - lo) * n_rg;
        kc = (int)(ii / per_kc);
        const long long rem = ii - (long long)kc * per_kc;
        tt = lo + (int)(rem / n_rg);
        rg = (int)(rem % n_rg);
    }
    // first row and row count of an item
    __device__ void rows(int tt, int rg, int &r0, int &nr) const {
        r0 = tt * BT + rg * R;
        int r1 = r0 + R;
        if (r1 > tt * BT + BT) r1 = tt * BT + BT;
        if (r1 > M) r1 = M;
        nr = r1 > r0 ? r1 - r0 : 0;
    }
};

__device__ __forceinline__ uint2 pack4_f16(float4 v, float4 f, float s) {
    uint2 o;
    o.x = pack_half2(v.x * f.x * s, v.y * f.y * s);
    o.y = pack_half2(v.z * f.z * s, v.w * f.w * s);
    return o;
}

// Thread 0: wait for the copies it issued into the ring (units issued, of
// which the first `done` were consumed) before the CTA may exit.
__device__ __forceinline__ void stager_drain(uint64_t *full, long long done, long long issued, int slots,
                                             const volatile int *abort_flag, uint32_t *status) {
    for (long long u = done; u < issued; ++u)
        if (!mbar_wait(&full[u % slots], (uint32_t)((u / slots) & 1), abort_flag, false))
            atomicOr(status, kStTimeoutDrain);
}

// ---- x: x16 = f16(x.g), items of 8 rows x 256 columns ----------------------
__device__ inline void stager_x(const StageArgs &a, const StgGeom &G, int t, volatile int *abort_flag,
                                uint8_t *ring, uint64_t *full, uint64_t *empty, uint32_t *status) {
    const int cta = blockIdx.x, nctas = gridDim.x;
    const long long n = G.items();
    const long long mine = cta < n ? (n - cta + nctas - 1) / nctas : 0;  // this CTA's items: cta + j grid
    constexpr int S = kStgSlotsX;
    const uint64_t once = l2_policy_evict_first();
    auto segs = [&](long long j, int &r0, int &nr, int &c0, int &w, int &tt, int &kc) {
        int rg;
        G.item(cta + j * nctas, tt, kc, rg);
        G.rows(tt, rg, r0, nr);
        c0 = kc * kStgKC;
        w = G.K - c0 < kStgKC ? G.K - c0 : kStgKC;
    };
    long long issued = 0;
    auto issue = [&](long long j) {  // thread 0: item j into slot j % S
        int r0, nr, c0, w, tt, kc;
        segs(j, r0, nr, c0, w, tt, kc);
        const int sl = (int)(j % S);
        if (j >= S && !mbar_wait(&empty[sl], (uint32_t)(((j / S) - 1) & 1), abort_flag)) return false;
        mbar_arrive_expect_tx(&full[sl], (uint32_t)(nr * w * 4));
        for (int q = 0; q < nr; ++q)
            bulk_load_hint(ring + sl * kStgSlotX + q * kStgKC * 4, a.src + (size_t)(r0 + q) * G.K + c0,
                           (uint32_t)w * 4, &full[sl], once);
        issued = j + 1;
        return true;
    };
    auto prefetch = [&](long long j) {
        if (j >= mine) return;
        int r0, nr, c0, w, tt, kc;
        segs(j, r0, nr, c0, w, tt, kc);
        for (int q = 0; q < nr; ++q) bulk_prefetch_l2(a.src + (size_t)(r0 + q) * G.K + c0, (uint32_t)w * 4);
    };
    bool ok = true;
    if (t == 0) {
        for (long long j = 0; j < mine && j < S && ok; ++j) ok = issue(j);
        for (long long j = S; j < S + kStgPrefetchUnits; ++j) prefetch(j);
    }
    long long j = 0, first_bad = -1;  // first item whose copy this thread did not see land
    for (; j < mine; ++j) {
        int r0, nr, c0, w, tt, kc;
        segs(j, r0, nr, c0, w, tt, kc);
        const int sl = (int)(j % S);
        const bool got = mbar_wait(&full[sl], (uint32_t)((j / S) & 1), abort_flag);
        if (!got && first_bad < 0) first_bad = j;
        if (!got && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(status, kStTimeoutStage);
        }
        const int col = c0 + 4 * t;
        if (got && col < G.K) {
            const float4 gv = __ldg(reinterpret_cast<const float4 *>(a.col + col));
            const float4 *src = reinterpret_cast<const float4 *>(ring + sl * kStgSlotX) + t;
#pragma unroll
            for (int q = 0; q < kStgRowsX; ++q)
                if (q < nr)
                    *reinterpret_cast<uint2 *>(a.dst + (size_t)(r0 + q) * G.K + col) =
                        pack4_f16(src[q * (kStgKC / 4)], gv, 1.0f);
        }
        // the slot is read: hand it back (only if the whole warp has read it: a
        // slot whose copy may still be landing is never handed back); the rows
        // are written: publish them
        const bool warp_got = __all_sync(0xFFFFFFFFu, got);
        if (warp_got && (t & 31) == 0) mbar_arrive(&empty[sl]);
        fence_proxy_async_global();
        const bool stop = named_bar_or(kStgBar, kStgThreads, !ok || *abort_flag != 0);
        if (stop) {
            ++j;
            break;
        }
        if (t == 0) {
            if (nr > 0) red_release_add_u32(a.cnt + (size_t)tt * G.n_kc + kc, (unsigned int)nr);
            if (ok && j + S < mine) ok = issue(j + S);
            prefetch(j + S + kStgPrefetchUnits);
        }
    }
    if (t == 0) stager_drain(full, first_bad >= 0 ? first_bad : j, issued, S, abort_flag, status);
}

// ---- dy: dy16 = f16(dy.h.s_t), s_t, sigma_t, dh sums; items of 4 whole rows --
// Per row t (the formulas of the stand-alone staging, blr_stage.cuh):
//   A_t = max_i |dy_ti h_i|, L_t = sum_i |dy_ti h_i|
//   s_t = gscale, or 2^(14 - ceil(log2 A_t))   (1 if A_t is 0 or not finite)
//   sigma_t = gscale, or 2^(15 - ceil(log2(L_t max_k |l_k|)))
// dh partial sums: each CTA adds the sums over its rows of dy.c into its own
// row part_dh[cta] (thread t owns the columns 256 c + 4 t of every chunk c, so
// a column is only ever updated by one thread: fixed order, deterministic).
// Ring units of item j: 2C of them (C = chunks of 256 columns), the first C
// bring dy and c (statistics and dh), the last C dy again (the f16 rows).
__device__ inline void stager_dy(const StageArgs &a, const StgGeom &G, int t, volatile int *abort_flag,
                                 StgScratch *sc, uint8_t *ring, uint64_t *full, uint64_t *empty, uint32_t *status) {
    const int cta = blockIdx.x, nctas = gridDim.x;
    const int warp = t / 32, lane = t & 31;
    const long long n = G.items();
    const long long mine = cta < n ? (n - cta + nctas - 1) / nctas : 0;
    const bool dynamic = !(a.gscale > 0.0f);
    const int K = G.K;
    const int C = (K + kStgKC - 1) / kStgKC;
    constexpr int S = kStgSlotsDy;
    const long long units = mine * 2 * C;
    float *pdh = a.part_dh + (size_t)cta * K;
    for (int c0 = 0; c0 < K; c0 += kStgKC)
        if (c0 + 4 * t < K) *reinterpret_cast<float4 *>(pdh + c0 + 4 * t) = make_float4(0.f, 0.f, 0.f, 0.f);
    float lmax = 0.0f;
    if (dynamic) {
        for (int k = t; k < a.r; k += kStgThreads) lmax = fmaxf(lmax, fabsf(__ldg(a.l + k)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
        if (lane == 0) sc->lmax[warp] = lmax;
        named_bar_sync(kStgBar, kStgThreads);
        lmax = fmaxf(sc->lmax[0], sc->lmax[1]);
    }
    const uint64_t once = l2_policy_evict_first();
    // unit u -> item j, pass p (0: statistics, 1: f16 rows), chunk c
    auto unit = [&](long long u, int &r0, int &nr, int &tt, int &p, int &c0, int &w) {
        const long long j = u / (2 * C);
        const int rem = (int)(u - j * 2 * C);
        p = rem / C;
        c0 = (rem % C) * kStgKC;
        w = K - c0 < kStgKC ? K - c0 : kStgKC;
        int kc, rg;
        G.item(cta + j * nctas, tt, kc, rg);
        G.rows(tt, rg, r0, nr);
    };
    long long issued = 0;
    auto issue = [&](long long u) {  // thread 0: unit u into slot u % S
        int r0, nr, tt, p, c0, w;
        unit(u, r0, nr, tt, p, c0, w);
        const int sl = (int)(u % S);
        if (u >= S && !mbar_wait(&empty[sl], (uint32_t)(((u / S) - 1) & 1), abort_flag)) return false;
        uint8_t *dst = ring + sl * kStgSlotDy;
        mbar_arrive_expect_tx(&full[sl], (uint32_t)(nr * w * (p == 0 ? 6 : 4)));
        for (int q = 0; q < nr; ++q) {
            // the first pass keeps dy in L2 for the second; c is read once
            if (p == 0)
                bulk_load(dst + q * kStgKC * 4, a.src + (size_t)(r0 + q) * K + c0, (uint32_t)w * 4, &full[sl]);
            else
                bulk_load_hint(dst + q * kStgKC * 4, a.src + (size_t)(r0 + q) * K + c0, (uint32_t)w * 4, &full[sl],
                               once);
            if (p == 0)
                bulk_load_hint(dst + kStgRowsDy * kStgKC * 4 + q * kStgKC * 2, a.c16 + (size_t)(r0 + q) * K + c0,
                               (uint32_t)w * 2, &full[sl], once);
        }
        issued = u + 1;
        return true;
    };
    auto prefetch = [&](long long u) {
        if (u >= units) return;
        int r0, nr, tt, p, c0, w;
        unit(u, r0, nr, tt, p, c0, w);
        if (p != 0) return;  // the second pass finds dy in L2
        for (int q = 0; q < nr; ++q) {
            bulk_prefetch_l2(a.src + (size_t)(r0 + q) * K + c0, (uint32_t)w * 4);
            bulk_prefetch_l2(a.c16 + (size_t)(r0 + q) * K + c0, (uint32_t)w * 2);
        }
    };
    bool ok = true;
    if (t == 0) {
        for (long long u = 0; u < units && u < S && ok; ++u) ok = issue(u);
        for (long long u = S; u < S + kStgPrefetchUnits; ++u) prefetch(u);
    }
    float2 mx = make_float2(0.0f, 0.0f);  // thread 0: this CTA's max 1/s_t, max 1/sigma_t (rows that count)
    float amax[kStgRowsDy], l1[kStgRowsDy], s[kStgRowsDy];
#pragma unroll
    for (int q = 0; q < kStgRowsDy; ++q) amax[q] = l1[q] = s[q] = 0.0f;
    long long u = 0, first_bad = -1;  // first unit whose copy this thread did not see land
    for (; u < units; ++u) {
        int r0, nr, tt, p, c0, w;
        unit(u, r0, nr, tt, p, c0, w);
        const int sl = (int)(u % S);
        const int c = c0 / kStgKC;
        if (p == 0 && c == 0) {
#pragma unroll
            for (int q = 0; q < kStgRowsDy; ++q) amax[q] = l1[q] = 0.0f;
        }
        // a wait that runs out raises the CTA's abort flag, so that the waits
        // of the item's remaining units end at once; the item then stops at
        // its next uniform decision below
        const bool got = mbar_wait(&full[sl], (uint32_t)((u / S) & 1), abort_flag);
        if (!got && first_bad < 0) first_bad = u;
        if (!got && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(status, kStTimeoutStage);
        }
        const int col = c0 + 4 * t;
        if (got && col < K) {
            const float4 hv = __ldg(reinterpret_cast<const float4 *>(a.col + col));
            const float4 *sd = reinterpret_cast<const float4 *>(ring + sl * kStgSlotDy) + t;
            if (p == 0) {
                const uint2 *scw = reinterpret_cast<const uint2 *>(ring + sl * kStgSlotDy + kStgRowsDy * kStgKC * 4) + t;
                float4 acc = *reinterpret_cast<float4 *>(pdh + col);
#pragma unroll
                for (int q = 0; q < kStgRowsDy; ++q)
                    if (q < nr) {
                        const float4 d = sd[q * (kStgKC / 4)];
                        const uint2 cw = scw[q * (kStgKC / 4)];
                        const float2 c0f = __half22float2(*reinterpret_cast<const __half2 *>(&cw.x));
                        const float2 c1f = __half22float2(*reinterpret_cast<const __half2 *>(&cw.y));
                        acc.x += d.x * c0f.x;
                        acc.y += d.y * c0f.y;
                        acc.z += d.z * c1f.x;
                        acc.w += d.w * c1f.y;
                        const float vx = fabsf(d.x * hv.x), vy = fabsf(d.y * hv.y);
                        const float vz = fabsf(d.z * hv.z), vw = fabsf(d.w * hv.w);
                        amax[q] = fmaxf(amax[q], fmaxf(fmaxf(vx, vy), fmaxf(vz, vw)));
                        l1[q] += (vx + vy) + (vz + vw);
                    }
                *reinterpret_cast<float4 *>(pdh + col) = acc;
            } else {
#pragma unroll
                for (int q = 0; q < kStgRowsDy; ++q)
                    if (q < nr)
                        *reinterpret_cast<uint2 *>(a.dst + (size_t)(r0 + q) * K + col) =
                            pack4_f16(sd[q * (kStgKC / 4)], hv, s[q]);
            }
        }
        // the slot goes back to the producer only if the whole warp has read
        // it (a slot whose copy may still be landing is never handed back)
        const bool warp_got = __all_sync(0xFFFFFFFFu, got);
        if (warp_got && lane == 0) mbar_arrive(&empty[sl]);
        bool stop = false;
        if (p == 0 && c == C - 1) {
            // end of the first pass: the rows' scales, reduced over the stager threads
            if (dynamic) {
#pragma unroll
                for (int q = 0; q < kStgRowsDy; ++q) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        amax[q] = fmaxf(amax[q], __shfl_xor_sync(0xFFFFFFFFu, amax[q], o));
                        l1[q] += __shfl_xor_sync(0xFFFFFFFFu, l1[q], o);
                    }
                    if (lane == 0) sc->red[warp][q] = make_float2(amax[q], l1[q]);
                }
            }
            stop = named_bar_or(kStgBar, kStgThreads, !ok || *abort_flag != 0);
            const float ginv = dynamic ? 1.0f : 1.0f / a.gscale;
#pragma unroll
            for (int q = 0; q < kStgRowsDy; ++q) {
                float sg = a.gscale;
                bool counts = true;
                s[q] = a.gscale;
                if (dynamic) {
                    const float2 ra = sc->red[0][q], rb = sc->red[1][q];
                    const float am = fmaxf(ra.x, rb.x), l1s = ra.y + rb.y;
                    const bool fin = am > 0.0f && am <= 3.402823466e38f;
                    counts = fin;
                    s[q] = fin ? pow2i(14 - ceil_log2_pos(am)) : 1.0f;
                    sg = s[q];
                    const float bound = l1s * lmax;  // bound on |db_t . l|, unscaled
                    if (fin && bound > 0.0f && bound <= 3.402823466e38f) sg = pow2i(15 - ceil_log2_pos(bound));
                }
                if (t == 0 && q < nr) {
                    const float si = dynamic ? pow2_recip(s[q]) : ginv, gi = dynamic ? pow2_recip(sg) : ginv;
                    a.s_inv[r0 + q] = si;
                    a.sig[r0 + q] = sg;
                    a.sig_inv[r0 + q] = gi;
                    if (counts) mx = make_float2(fmaxf(mx.x, si), fmaxf(mx.y, gi));
                }
            }
            // every thread has read the reduction buffer before the next item writes it
            named_bar_sync(kStgBar, kStgThreads);
        } else if (p == 1 && c == C - 1) {
            // end of the item: publish its rows (and their scales)
            fence_proxy_async_global();
            stop = named_bar_or(kStgBar, kStgThreads, !ok || *abort_flag != 0);
            if (!stop && t == 0 && nr > 0) red_release_add_u32(a.cnt + tt, (unsigned int)nr);
        }
        if (stop) {
            ++u;
            break;
        }
        if (t == 0) {
            if (ok && u + S < units) ok = issue(u + S);
            prefetch(u + S + kStgPrefetchUnits);
        }
    }
    if (t == 0) {
        stager_drain(full, first_bad >= 0 ? first_bad : u, issued, S, abort_flag, status);
        a.blkmax[cta] = mx;
    }
}

}  // namespace blr
