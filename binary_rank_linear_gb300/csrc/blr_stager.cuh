// In-kernel staging of the a-product's activation operand.
//
// The separate x staging pass of the layer (x16 = f16(x.g) before the
// a-product) is an HBM stream that leaves the tensor cores idle, while the
// a-product it feeds (K = d_in, r outputs) leaves most of the HBM bandwidth
// idle. Here the staging runs inside the a-product's persistent kernel, on
// six stager warps of every CTA, ahead of the MMA pipeline:
//
//  - Work items are blocks of 64 token rows x 256 columns of x, taken in the
//    order the persistent grid consumes them: round by round (a round is the
//    token tiles whose feature tiles the units start together), then column
//    chunk by column chunk, then token tile and row group. CTA c stages
//    items c, c + grid, c + 2 grid, ...
//  - One stager lane (the copy producer) loads the items' f32 tiles into a
//    51 KB shared-memory ring by TMA (three slots of one 256 x 16 box, a
//    16-row unit, plus the item's 256 g factors and the unit's geometry;
//    full/empty mbarriers); another (the publisher) asks L2 to prefetch whole
//    items (one 256 x 64 box) two items ahead and publishes finished items;
//    four converter warps convert from shared memory and write f16 with
//    16-byte stores, so the staged tiles sit in L2 when the product's TMA
//    loads come. (Measured on
//    GB300 with in-kernel clock counters: converters that also issued the
//    TMA copies and the releases spent most of their time there; each TMA
//    instruction costs its thread several hundred cycles in this kernel.)
//  - After an item, the stagers publish its rows on the counter of its
//    (token tile, column chunk): stores, a proxy fence (the consumer reads by
//    TMA), the converter warps' arrivals on a shared-memory counter, then
//    one release add by the publisher. The TMA
//    producer acquires the counter of each chunk of a tile before its loads
//    (bounded wait), then fences the async proxy. A product starts as soon as
//    the first chunk of its first round is staged.
//
// Stagers never wait for another CTA: every counter completes once the
// stagers of the grid have run (the CTAs of the persistent grid are resident
// together). A bounded wait that runs out, or the CTA's abort flag, stops
// them; the copy producer then waits for the copies it issued.
//
// The db-product's operand dy16 = f16(dy.h.s_t) is staged the same way
// (GEMM template STG = 2) once a scale pass has written each row's 1/s_t:
// a ring unit then also carries the c tape's 16 x 256 tile and the rows'
// scales, and the converters add each item's column sums of dy.c (the dh
// partial sums) into partial rows of their own (one per converter warp and
// CTA), so that no two warps ever add into the same row.
#pragma once

#include <cuda_fp16.h>

#include "blr_device.cuh"
#include "blr_kernels.h"
#include "blr_stage.cuh"

namespace blr {

constexpr int kStgConvWarps = 4;                 // converter warps
constexpr int kStgConvThreads = kStgConvWarps * 32;
constexpr int kStgWarps = kStgConvWarps + 2;     // + the copy producer and the publisher
constexpr int kStgThreads = kStgWarps * 32;
constexpr int kStgKC = kStageChunkCols;  // columns per chunk: one float4 per stager thread
constexpr int kStgSlotsMax = 8;
// items of 64 rows x 256 columns, ring units of 16 rows: a slot holds the
// unit's f32 tile (16 KB, one TMA box: x is read through a tensor map with a
// 256 x 16 box) and the item's 256 g factors (1 KB)
constexpr int kStgRowsX = 64;
constexpr int kStgUnitRows = 16;
constexpr int kStgUnitsX = kStgRowsX / kStgUnitRows;
constexpr int kStgTileBytes = kStgUnitRows * kStgKC * 4;
constexpr int kStgSlotX = kStgTileBytes + kStgKC * 4;
constexpr int kStgSlotsX = 3;
constexpr int kStgRingBytes = kStgSlotsX * kStgSlotX;
constexpr int kStgPrefetchItems = 2;  // items prefetched into L2 ahead of the one being converted
static_assert(kStgSlotsX >= 2 && kStgSlotsX <= kStgSlotsMax, "stager ring");
// dy items (STG = 2): a slot holds the unit's dy tile (256 x 16 f32), its c
// tile (256 x 16 f16), the chunk's 256 h factors and the unit's 16 row scales
// 1/s_t; slots stay 128-byte aligned for the TMA boxes
constexpr int kStgCOff = kStgTileBytes;
constexpr int kStgHOff = kStgCOff + kStgUnitRows * kStgKC * 2;
constexpr int kStgSOff = kStgHOff + kStgKC * 4;
constexpr int kStgSlotDy = kStgSOff + 128;
constexpr int kStgSlotsDy = 3;
constexpr int kStgRingBytesDy = kStgSlotsDy * kStgSlotDy;
static_assert(kStgSlotDy % 128 == 0 && kStgCOff % 128 == 0, "stager slots hold TMA boxes");
static_assert(kStgSlotsDy >= 2 && kStgSlotsDy <= kStgSlotsMax, "stager ring");
static_assert(kStgConvWarps == kDyPartRowsPerCta, "one dh partial row per converter warp");

__host__ __device__ constexpr int stg_chunks(int K) { return (K + kStgKC - 1) / kStgKC; }
static_assert(kStgKC == 8 * 32, "a chunk row is eight columns per lane of a converter warp");
static_assert(kStgUnitRows % kStgConvWarps == 0, "the converter warps share a unit's rows evenly");

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

// Consumption order of the persistent GEMM grid and the stager items (32-bit
// arithmetic: the host stages in the kernel only while the item count and
// token tiles x feature tiles stay below 2^31, see stage_fits). With several
// paths the grid takes the paths' tiles path-major, so the token tiles are
// virtual: tile vt is token tile vt % t_path of path vt / t_path.
struct StgGeom {
    unsigned M, K, BT, t_path, t_tiles, f_tiles, units, n_kc, R, n_rg;

    __device__ StgGeom(int M_, int K_, int BT_, int f_tiles_, int units_, int paths)
        : M(M_), K(K_), BT(BT_), t_path((M_ + BT_ - 1) / BT_), t_tiles(t_path * (unsigned)(paths > 1 ? paths : 1)),
          f_tiles(f_tiles_), units(units_), n_kc(stg_chunks(K_)), R(kStgRowsX),
          n_rg((BT_ + kStgRowsX - 1) / kStgRowsX) {}
    // round of a token tile: the units start tiles u, u + units, ... with the
    // feature tile varying fastest, so token tile tt first appears in round
    // floor(tt * f_tiles / units)
    __device__ unsigned round_of(unsigned tt) const { return tt * f_tiles / units; }
    // first token tile of round r: ceil(r * units / f_tiles)
    __device__ unsigned tt_begin(unsigned r) const {
        const unsigned v = (r * units + f_tiles - 1) / f_tiles;
        return v < t_tiles ? v : t_tiles;
    }
    __device__ unsigned items() const { return t_tiles * n_kc * n_rg; }
    // item i -> (token tile, column chunk, row group); rounds partition the
    // token tiles in order, so the items before round r are tt_begin(r) * n_kc * n_rg
    __device__ void item(unsigned i, int &tt, int &kc, int &rg) const {
        const unsigned P = n_kc * n_rg;
        const unsigned r = round_of(i / P);
        const unsigned lo = tt_begin(r), hi = tt_begin(r + 1);
        const unsigned ii = i - lo * P;
        const unsigned per_kc = (hi - lo) * n_rg;
        kc = (int)(ii / per_kc);
        const unsigned rem = ii - (unsigned)kc * per_kc;
        tt = (int)(lo + rem / n_rg);
        rg = (int)(rem % n_rg);
    }
    // the path and first row of x of an item, and its row count (virtual
    // token tile vt, row group rg)
    __device__ void rows(int vt, int rg, int &p, int &r0, int &nr) const {
        p = vt / (int)t_path;
        const int tt = vt - p * (int)t_path;
        r0 = tt * (int)BT + rg * (int)R;
        int r1 = r0 + (int)R;
        if (r1 > tt * (int)BT + (int)BT) r1 = tt * (int)BT + (int)BT;
        if (r1 > (int)M) r1 = (int)M;
        nr = r1 > r0 ? r1 - r0 : 0;
    }
};

// f16 bits of (a * b) for two f32 pairs: one paired multiply (mul.rn.f32x2,
// each product rounded as by a plain f32 multiply) and one packed conversion
// (round to nearest even).
__device__ __forceinline__ uint32_t mul_pack_half2(float a0, float a1, float b0, float b1) {
    unsigned long long a = ((unsigned long long)__float_as_uint(a1) << 32) | __float_as_uint(a0);
    unsigned long long b = ((unsigned long long)__float_as_uint(b1) << 32) | __float_as_uint(b0);
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return pack_half2(__uint_as_float((uint32_t)d), __uint_as_float((uint32_t)(d >> 32)));
}

// ---- x: x16 = f16(x.g), items of 64 rows x 256 columns ---------------------
// An item is kStgUnitsX ring units of 8 rows (8 KB f32 each). The consumer
// side decodes an item once, loads its 256 g factors (one float4 per
// thread) once, converts unit by unit, and publishes the item with one
// fence, one barrier and one release. Thread 0 also runs two cursors ahead of
// the consumers over the same unit sequence: the bulk copies into the ring
// (S units ahead) and the L2 prefetches (S + kStgPrefetchUnits ahead).
struct XCursor {
    unsigned j;   // this CTA's item index (CTA item cta + j * grid)
    int s;        // unit of the item
    int r0, nr, c0, w, tt, kc, p;  // (tt: the virtual token tile; p: the path)
};

__device__ __forceinline__ void x_cursor_load(XCursor &c, const StgGeom &G, unsigned mine, int cta, int nctas) {
    if (c.j >= mine) return;
    int rg;
    G.item((unsigned)cta + c.j * (unsigned)nctas, c.tt, c.kc, rg);
    G.rows(c.tt, rg, c.p, c.r0, c.nr);
    c.c0 = c.kc * kStgKC;
    c.w = G.K - c.c0 < kStgKC ? G.K - c.c0 : kStgKC;
}

__device__ __forceinline__ void x_cursor_next(XCursor &c, const StgGeom &G, unsigned mine, int cta, int nctas) {
    if (++c.s == kStgUnitsX) {
        c.s = 0;
        ++c.j;
        x_cursor_load(c, G, mine, cta, nctas);
    }
}

// Roles of the stager warps (kStgThreads threads, t = 0 ..): warps 0 ..
// kStgConvWarps - 1 convert; the next warp's lane 0 copies ring units by TMA
// (stager_x_producer); the last warp's lane 0 prefetches items into L2 and
// publishes finished items (stager_x_publisher). The converters count the
// items they finish on a shared-memory counter (one arrival per converter
// warp and item, release at CTA scope), which the publisher acquires before
// its release add at GPU scope; nothing in the stagers waits on a named
// barrier, so a converter that stops early (an abort) cannot hang another.
__device__ __forceinline__ unsigned int ld_acquire_shared_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_shared_add_u32(unsigned int *p, unsigned int v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

struct StgX {
    const StageArgs &a;
    const StgGeom &G;
    unsigned mine;  // this CTA's items: cta + j * grid, j < mine
    long long units;
    int cta, nctas;
    __device__ StgX(const StageArgs &a_, const StgGeom &G_) : a(a_), G(G_) {
        cta = blockIdx.x;
        nctas = gridDim.x;
        const unsigned n = G.items();
        mine = (unsigned)cta < n ? (n - cta + nctas - 1) / nctas : 0;
        units = (long long)mine * kStgUnitsX;
    }
};

// Where a ring unit's rows go (written by the copy producer with the unit's
// copies, read by the converters after the slot's full barrier).
struct StgGeo {
    int q0;  // first row
    int nq;  // rows of x in the unit (0 .. 16)
    int c0;  // first column
    int p;   // path
};

// lane 0 of the producer warp: ring units by TMA, S ahead of the converters,
// each with its geometry and the item's g factors
__device__ inline void stager_x_producer(const StgX &X, const CUtensorMap *tmap_x, volatile int *abort_flag,
                                         uint8_t *ring, uint64_t *full, uint64_t *empty, StgGeo *geo,
                                         uint32_t *status) {
    constexpr int S = kStgSlotsX;
    const uint64_t once = l2_policy_evict_first();
    XCursor ci{0, 0, 0, 0, 0, 0, 0, 0, 0};
    x_cursor_load(ci, X.G, X.mine, X.cta, X.nctas);
    long long u = 0;
    for (; u < X.units; ++u) {
        const int sl = (int)(u % S);
        if (u >= S && !mbar_wait(&empty[sl], (uint32_t)(((u / S) - 1) & 1), abort_flag)) break;
        const int q0 = ci.r0 + kStgUnitRows * ci.s;
        int nq = ci.r0 + ci.nr - q0;
        nq = nq < 0 ? 0 : (nq > kStgUnitRows ? kStgUnitRows : nq);
        geo[sl] = StgGeo{q0, nq, ci.c0, ci.p};
        // one box of 256 columns x 16 rows (rows and columns past x read
        // zero), and the chunk's g factors (the unit's path's)
        const float *g = X.a.paths > 1 ? X.a.col_p[ci.p] : X.a.col;
        mbar_arrive_expect_tx(&full[sl], (uint32_t)(kStgTileBytes + ci.w * 4));
        tma_load_2d_hint(ring + sl * kStgSlotX, tmap_x, &full[sl], ci.c0, q0, once);
        bulk_load(ring + sl * kStgSlotX + kStgTileBytes, g + ci.c0, (uint32_t)ci.w * 4, &full[sl]);
        x_cursor_next(ci, X.G, X.mine, X.cta, X.nctas);
    }
    // every copy issued lands before the CTA may exit: for each slot, the
    // phase of the last unit copied into it
    for (long long v = (u > S ? u - S : 0); v < u; ++v)
        if (!mbar_wait(&full[v % S], (uint32_t)((v / S) & 1), abort_flag, false)) atomicOr(status, kStTimeoutDrain);
}

// lane 0 of the publisher warp: L2 prefetches two items ahead, and the
// release add of each item once every converter warp has finished it
__device__ inline void stager_x_publisher(const StgX &X, const CUtensorMap *tmap_pf, volatile int *abort_flag,
                                          const unsigned int *done, uint32_t *status) {
    auto prefetch_item = [&](unsigned j) {
        if (j >= X.mine) return;
        XCursor c{j, 0, 0, 0, 0, 0, 0, 0, 0};
        x_cursor_load(c, X.G, X.mine, X.cta, X.nctas);
        if (c.nr > 0) tma_prefetch_l2_2d(tmap_pf, c.c0, c.r0);  // one 256 x 64 box
    };
    for (unsigned j = 0; j < kStgPrefetchItems; ++j) prefetch_item(j);
    for (unsigned j = 0; j < X.mine; ++j) {
        prefetch_item(j + kStgPrefetchItems);
        XCursor c{j, 0, 0, 0, 0, 0, 0, 0, 0};
        x_cursor_load(c, X.G, X.mine, X.cta, X.nctas);
        const unsigned target = (j + 1) * kStgConvWarps;
        if (ld_acquire_shared_u32(done) < target) {
            const uint64_t t0 = globaltimer_ns();
            bool ok = true;
            for (uint32_t i = 1; ld_acquire_shared_u32(done) < target; ++i) {
                __nanosleep(64);
                if ((i & 15u) == 0 && (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(status, kStTimeoutStage);
                }
                return;
            }
        }
        if (c.nr > 0) {
            // the counter of (token tile, chunk) in the item's path's slice
            unsigned int *cnt = reinterpret_cast<unsigned int *>(reinterpret_cast<char *>(X.a.cnt) +
                                                                 (size_t)c.p * (size_t)X.a.pstride);
            const int tt = c.tt - c.p * (int)X.G.t_path;
            red_release_add_u32(cnt + (size_t)tt * X.G.n_kc + c.kc, (unsigned int)c.nr);
        }
    }
}

// converter warps: thread t < kStgConvThreads converts columns 8 (t % 32) ..
// + 7 of the chunk in the rows t / 32, t / 32 + kStgConvWarps, ... of each
// unit (one 16-byte store each); a unit's geometry and g factors come with
// its slot. Software-pipelined over the units: the next unit's shared-memory
// loads are in flight while the current unit converts.
__device__ inline void stager_x_convert(const StgX &X, int t, volatile int *abort_flag, uint8_t *ring,
                                        uint64_t *full, uint64_t *empty, const StgGeo *geo, unsigned int *done,
                                        uint32_t *status) {
    constexpr int S = kStgSlotsX;
    constexpr int kRows = kStgUnitRows / kStgConvWarps;
    const int cg = t & 31, rp = t >> 5, lane = t & 31;
    const int K = (int)X.G.K;
    // wait for unit u's copy and load this thread's rows of it
    auto fetch = [&](long long u, float4 (&v)[kRows][2]) -> bool {
        const int sl = (int)(u % S);
        const bool got = mbar_wait(&full[sl], (uint32_t)((u / S) & 1), abort_flag);
        if (!got && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(status, kStTimeoutStage);
        }
        if (got) {
            const float4 *src = reinterpret_cast<const float4 *>(ring + sl * kStgSlotX) + 2 * cg + rp * (kStgKC / 4);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                v[i][0] = src[i * kStgConvWarps * (kStgKC / 4)];
                v[i][1] = src[i * kStgConvWarps * (kStgKC / 4) + 1];
            }
        }
        return got;
    };
    float4 va[kRows][2], vb[kRows][2];
    bool got_a = X.units > 0 && fetch(0, va);
    bool ok = true;
    for (long long u = 0; u < X.units; ++u) {
        const int sl = (int)(u % S);
        // the next unit's loads go out first
        const bool got_b = u + 1 < X.units && fetch(u + 1, vb);
        if (got_a) {
            const StgGeo gq = geo[sl];
            const int col = gq.c0 + 8 * cg;
            if (col < K) {
                const float4 *gs = reinterpret_cast<const float4 *>(ring + sl * kStgSlotX + kStgTileBytes) + 2 * cg;
                const float4 g0 = gs[0], g1 = gs[1];
                uint16_t *dst = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(X.a.dst) +
                                                             (size_t)gq.p * (size_t)X.a.pstride) +
                                (size_t)(gq.q0 + rp) * K + col;
#pragma unroll
                for (int i = 0; i < kRows; ++i)
                    if (rp + kStgConvWarps * i < gq.nq) {
                        uint4 o;
                        o.x = mul_pack_half2(va[i][0].x, va[i][0].y, g0.x, g0.y);
                        o.y = mul_pack_half2(va[i][0].z, va[i][0].w, g0.z, g0.w);
                        o.z = mul_pack_half2(va[i][1].x, va[i][1].y, g1.x, g1.y);
                        o.w = mul_pack_half2(va[i][1].z, va[i][1].w, g1.z, g1.w);
                        *reinterpret_cast<uint4 *>(dst + (size_t)i * kStgConvWarps * K) = o;
                    }
            }
        }
        // unit u's slot goes back to the producer once the whole warp has
        // converted it (a slot whose copy may still be landing is never handed back)
        const bool warp_got = __all_sync(0xFFFFFFFFu, got_a);
        if (warp_got && lane == 0) mbar_arrive(&empty[sl]);
        ok = ok && warp_got;
        if (u % kStgUnitsX == kStgUnitsX - 1) {
            if (!ok || *abort_flag) break;
            // the item's rows are written: proxy fence (the TMA loads of other
            // CTAs read them), then one arrival of this warp on the item counter
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) red_release_shared_add_u32(done, 1u);
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            va[i][0] = vb[i][0];
            va[i][1] = vb[i][1];
        }
        got_a = got_b;
    }
}


// ---- dy: dy16 = f16(dy.h.s_t) and the dh partial sums (STG = 2) -----------
// lane 0 of the producer warp: ring units by TMA (the dy tile and the c tile),
// S ahead of the converters, with the chunk's h factors and the unit's row
// scales. Single-path launches only.
__device__ inline void stager_dy_producer(const StgX &X, const CUtensorMap *tmap_dy, const CUtensorMap *tmap_c,
                                          volatile int *abort_flag, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                          StgGeo *geo, uint32_t *status) {
    constexpr int S = kStgSlotsDy;
    const uint64_t once = l2_policy_evict_first();
    XCursor ci{0, 0, 0, 0, 0, 0, 0, 0, 0};
    x_cursor_load(ci, X.G, X.mine, X.cta, X.nctas);
    long long u = 0;
    for (; u < X.units; ++u) {
        const int sl = (int)(u % S);
        if (u >= S && !mbar_wait(&empty[sl], (uint32_t)(((u / S) - 1) & 1), abort_flag)) break;
        const int q0 = ci.r0 + kStgUnitRows * ci.s;
        int nq = ci.r0 + ci.nr - q0;
        nq = nq < 0 ? 0 : (nq > kStgUnitRows ? kStgUnitRows : nq);
        geo[sl] = StgGeo{q0, nq, ci.c0, 0};
        uint8_t *slot = ring + sl * kStgSlotDy;
        // boxes past dy's rows read zero; a unit with no rows takes row 0's
        // scales (never used), so that the copy stays inside the scale array
        mbar_arrive_expect_tx(&full[sl], (uint32_t)(kStgTileBytes + kStgUnitRows * kStgKC * 2 + ci.w * 4 +
                                                    kStgUnitRows * 4));
        tma_load_2d_hint(slot, tmap_dy, &full[sl], ci.c0, q0, once);
        tma_load_2d_hint(slot + kStgCOff, tmap_c, &full[sl], ci.c0, q0, once);
        bulk_load(slot + kStgHOff, X.a.col + ci.c0, (uint32_t)ci.w * 4, &full[sl]);
        bulk_load(slot + kStgSOff, X.a.row_sinv + (nq > 0 ? q0 : 0), kStgUnitRows * 4, &full[sl]);
        x_cursor_next(ci, X.G, X.mine, X.cta, X.nctas);
    }
    // every copy issued lands before the CTA may exit
    for (long long v = (u > S ? u - S : 0); v < u; ++v)
        if (!mbar_wait(&full[v % S], (uint32_t)((v / S) & 1), abort_flag, false)) atomicOr(status, kStTimeoutDrain);
}

// converter warps: as for x, thread t converts columns 8 (t % 32) .. + 7 of
// the chunk in rows t / 32, t / 32 + kStgConvWarps, ... of each unit (16-byte
// stores), and sums dy.c of those columns over the item's rows; each warp
// adds its sums into a partial row of its own (kStgConvWarps rows per CTA),
// so the warp's item order fixes every column's summation order.
__device__ inline void stager_dy_convert(const StgX &X, int t, volatile int *abort_flag, uint8_t *ring,
                                         uint64_t *full, uint64_t *empty, const StgGeo *geo, unsigned int *done,
                                         uint32_t *status) {
    constexpr int S = kStgSlotsDy;
    constexpr int kRows = kStgUnitRows / kStgConvWarps;
    const int cg = t & 31, rp = t >> 5, lane = t & 31;
    const int K = (int)X.G.K;
    float *prow = X.a.part + ((size_t)blockIdx.x * kStgConvWarps + rp) * K;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    int col = 0;
    bool ok = true;
    for (long long u = 0; u < X.units; ++u) {
        const int sl = (int)(u % S);
        const bool got = mbar_wait(&full[sl], (uint32_t)((u / S) & 1), abort_flag);
        if (!got && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(status, kStTimeoutStage);
        }
        if (got) {
            const StgGeo gq = geo[sl];
            const uint8_t *slot = ring + sl * kStgSlotDy;
            col = gq.c0 + 8 * cg;
            if (col < K) {
                const float4 *sd = reinterpret_cast<const float4 *>(slot) + 2 * cg;
                const uint4 *sc = reinterpret_cast<const uint4 *>(slot + kStgCOff) + cg;
                const float4 h0 = reinterpret_cast<const float4 *>(slot + kStgHOff)[2 * cg];
                const float4 h1 = reinterpret_cast<const float4 *>(slot + kStgHOff)[2 * cg + 1];
                const float *sv = reinterpret_cast<const float *>(slot + kStgSOff);
                float4 d0[kRows], d1[kRows];
                uint4 cw[kRows];
                float sr[kRows];
#pragma unroll
                for (int i = 0; i < kRows; ++i) {
                    const int row = rp + kStgConvWarps * i;
                    if (row < gq.nq) {
                        d0[i] = sd[row * (kStgKC / 4)];
                        d1[i] = sd[row * (kStgKC / 4) + 1];
                        cw[i] = sc[row * (kStgKC / 8)];
                        sr[i] = sv[row];
                    }
                }
                uint16_t *dst = X.a.dst + (size_t)(gq.q0 + rp) * K + col;
#pragma unroll
                for (int i = 0; i < kRows; ++i) {
                    if (rp + kStgConvWarps * i < gq.nq) {
                        // f16(round(dy.h) s_t): s_t is a power of two, so the
                        // scaling is exact and the bits match the prologue's
                        const float s = pow2_recip(sr[i]);
                        const float v[8] = {d0[i].x * h0.x, d0[i].y * h0.y, d0[i].z * h0.z, d0[i].w * h0.w,
                                            d1[i].x * h1.x, d1[i].y * h1.y, d1[i].z * h1.z, d1[i].w * h1.w};
                        uint4 o;
                        o.x = pack_half2(v[0] * s, v[1] * s);
                        o.y = pack_half2(v[2] * s, v[3] * s);
                        o.z = pack_half2(v[4] * s, v[5] * s);
                        o.w = pack_half2(v[6] * s, v[7] * s);
                        *reinterpret_cast<uint4 *>(dst + (size_t)i * kStgConvWarps * K) = o;
                        const uint32_t cws[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
                        const float dv[8] = {d0[i].x, d0[i].y, d0[i].z, d0[i].w, d1[i].x, d1[i].y, d1[i].z, d1[i].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 c2 = __half22float2(*reinterpret_cast<const __half2 *>(&cws[j]));
                            acc[2 * j] += dv[2 * j] * c2.x;
                            acc[2 * j + 1] += dv[2 * j + 1] * c2.y;
                        }
                    }
                }
            }
        }
        // unit u's slot goes back to the producer once the whole warp has read it
        const bool warp_got = __all_sync(0xFFFFFFFFu, got);
        if (warp_got && lane == 0) mbar_arrive(&empty[sl]);
        ok = ok && warp_got;
        if (u % kStgUnitsX == kStgUnitsX - 1) {
            if (!ok || *abort_flag) break;
            // the item's column sums into this warp's partial row
            if (col < K) {
                float4 *pr = reinterpret_cast<float4 *>(prow + col);
                float4 a0 = pr[0], a1 = pr[1];
                a0.x += acc[0];
                a0.y += acc[1];
                a0.z += acc[2];
                a0.w += acc[3];
                a1.x += acc[4];
                a1.y += acc[5];
                a1.z += acc[6];
                a1.w += acc[7];
                pr[0] = a0;
                pr[1] = a1;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
            // the item's rows are written: proxy fence (other CTAs' TMA loads
            // read them), then this warp's arrival on the item counter
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) red_release_shared_add_u32(done, 1u);
        }
    }
}

}  // namespace blr
