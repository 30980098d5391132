// Persistent tcgen05 GEMM of the blr layer on sm_103a, in feature-major form:
//
//     acc[n][t] = sum_k S[n][k] * act16[t][k]        (S = +-1, exact in f16)
//
// n runs over the product's output features (rows of the sign matrix), t over
// tokens. One tile is 128 features (256 for a CTA pair) x BT tokens; the MMA's
// M side is the sign matrix and its N side the tokens.
//
// The sign operand never exists as a dense matrix anywhere but in tensor
// memory: the TMA producer bulk-copies each k-step's pair-ready bitmap words
// (128 rows x 16 bytes) next to the activation tile, and expander warps turn
// them into +-1 f16 in registers and write them with tcgen05.st straight into
// a TMEM stage, which the MMA reads as its A operand. Shared memory carries
// only the activation tiles (TMA in, MMA out); with CTA pairs each SM holds
// and reads half of them.
//
// Tile shape, measured on GB300: an MMA whose operands change from one
// instruction to the next takes max(N/2, ~77) cycles, so N = 128 runs at 83%
// of the tensor rate (and lower still while expanders store to TMEM) while
// N >= 160 runs at full rate. BT is 160 or 192 tokens for CTA pairs and 128
// for single CTAs (small problems).
//
// TMEM (512 columns): two f32 accumulators of BT columns (the epilogue of one
// tile overlaps the main loop of the next) and the remaining columns as sign
// stages of 64 columns (one 128-deep k-step each, two f16 per column).
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 sign expanders (warp w writes TMEM lanes 32*(w%4) .. +31
// of both of the k-step's 64-wide blocks), warps 6-9 epilogue (warp w reads
// lanes 32*(w%4) .. +31: each thread owns one feature of the tile and walks
// its tokens, so the token sums dl and dg are per-thread running sums). The
// dx'-product runs eight epilogue warps (two per quarter, alternate chunks);
// the kernels that stage x add six stager warps. (Measured on GB300, four
// expander warps of two blocks each against eight of one: db-product of the
// 4096 -> 12288 MLP layer 262 against 278 us, c-product 303 against 309, the
// attention-sized db-product 63.4 against 67.5; half as many arrivals on each
// sign stage's barrier.)
// The epilogue stages each 32-token x 32-feature chunk in shared memory
// ([token][feature], the layout of the row-major outputs) and writes it with
// a TMA store; inputs (the a-tape, x, or y to accumulate) arrive by TMA into
// the same chunk slots, prefetched two chunks ahead.
//
// Rings: the activation ring (TMA; NB stages, full_b / empty_b) is at least
// as deep as the sign ring (TMEM; NS stages, full_s). An expander computes a
// stage's signs as soon as its words land (full_b), then waits for the MMAs
// that last read its sign stage, which committed to the activation slot of
// k-step i - NS (empty_b); the MMA issuer waits on full_s only (it implies
// full_b) and commits once per k-step to empty_b.
//
// CTA pairs (tcgen05 cta_group::2): the leader issues M=256 MMAs reading A
// from both CTAs' TMEM (rows 0-127 leader, 128-255 peer) and B from both
// CTAs' shared memory (tokens 0 .. BT/2-1 leader, the rest peer); each CTA's
// TMEM receives its 128 feature rows of the accumulator. The peer's expander
// warps arrive on the leader's full_s directly (remote arrivals); the leader's
// commits are multicast to both CTAs.
//
// Every wait is bounded (blr_device.cuh): a wait that runs out sets the
// shared abort flag and a status bit, the other roles leave their loops, the
// TMA producer drains its in-flight loads, the epilogue drains its copies,
// the MMA issuer drains its MMAs, and the CTA frees its TMEM and returns.
#pragma once

#include <cuda_fp16.h>

#include "blr_device.cuh"
#include "blr_kernels.h"
#include "blr_stage.cuh"
#include "blr_stager.cuh"

namespace blr {

constexpr int kFM = 128;          // feature rows per CTA (TMEM lanes)
constexpr int kBK = 64;           // K of one TMA box / bitmap block
constexpr int kKB = 2;            // 64-wide blocks per k-step
constexpr int kStepK = kKB * kBK;  // K per k-step (one MMA-issuer wait and one commit)
constexpr int kSignCols = kStepK / 2;  // TMEM columns of one sign stage
constexpr int kTmemCols = 512;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpExp0 = 2;
constexpr int kNumExpWarps = 4;  // one per TMEM lane quarter, both 64-wide blocks of a k-step
constexpr int kWarpEpi0 = 6;
constexpr int kGemmThreads = (kWarpEpi0 + 8) * 32;  // the fused small-M kernels' block (every phase fits)
constexpr int kCtlBytes = 1024;   // shared-memory control block ahead of a phase's layout
static_assert(kNumExpWarps == 4, "one expander warp per TMEM lane quarter");
static_assert(kWarpExp0 % 4 == 2, "expander and epilogue warps cover the four TMEM lane quarters in turn");

// PLANE selects where the sign operand comes from: false, bitmap words
// expanded into TMEM by expander warps (above); true, a +-1 f16 sign plane
// in global memory (written once per pass by the prologue, L2-resident) read
// by TMA like the activations, so both MMA operands come from shared memory
// and no expander warps exist. Plane mode takes one 64-deep block per k-step,
// and the plane tile is K-major (the c- and dx'-products: plane rows are the
// features) or MN-major (the a- and db-products: plane rows run along K). In
// a CTA pair each CTA loads its own 128 plane rows and half the tokens, and
// the peer's MMA warp, idle otherwise, forwards each stage's arrival to the
// leader (full_p) once the peer's loads have landed.
// STG: 0, the activation operand is staged before the launch; 1, stager
// warps after the epilogue warps stage x inside the a-product's kernel
// (blr_stager.cuh), with a 51 KB ring of their own; 2, the same for the
// db-product's dy (75 KB ring: each unit also brings its c tile and scales).
template <int EPI, bool PAIR, int BT, bool PLANE = false, int STG = 0>
struct GemmShape {
    static constexpr int kKBm = PLANE ? 1 : kKB;           // 64-wide blocks per k-step
    static constexpr int kStepKm = kKBm * kBK;             // K per k-step
    // expander warps: one per TMEM lane quarter, covering both 64-wide blocks
    // of a k-step (with the stager warps or the dx'-product's second epilogue
    // warp per quarter a CTA stays at 16 warps or fewer, which keeps every
    // role at 128 registers; more would cap them at 96)
    static constexpr int kNExp = PLANE ? 0 : kNumExpWarps;
    static constexpr int kEpi0 = PLANE ? 2 : kWarpExp0 + kNExp;  // first epilogue warp
    static constexpr bool kPlaneMN = EPI == kEpiFwd1 || EPI == kEpiBwd1;  // plane rows run along K
    static constexpr int kAccCols = BT;                    // TMEM columns of one accumulator
    static constexpr int kSignCol0 = 2 * BT;               // first sign-stage column
    static constexpr int kChunks = BT / 32;                // epilogue chunks per tile
    static constexpr int kTokRows = PAIR ? BT / 2 : BT;    // activation rows this CTA loads per tile
    static constexpr int kBBlock = kTokRows * kBK * 2;     // one 64-wide activation box
    static constexpr int kBBytes = kKBm * kBBlock;         // activation tile of a k-step
    static constexpr int kBitsBlock = kFM * 8;             // bitmap words of 128 rows, one block
    static constexpr int kABlock = kFM * kBK * 2;          // plane tile of 128 rows x 64 K (PLANE)
    static constexpr int kBitsBytes = PLANE ? kABlock : kKB * kBitsBlock;  // per stage: words or plane tile
    static constexpr int kEW = epi_warps(EPI);             // epilogue warps
    static constexpr int kSplit = kEW / 4;                 // epilogue warps per TMEM lane quarter
    static constexpr int kStg0 = kEpi0 + kEW;              // first stager warp
    static constexpr int kThreads = (kEpi0 + kEW + (STG ? kStgWarps : 0)) * 32;
    static constexpr bool kHas16 = EPI != kEpiBwd2;        // f16 output: a.l, c, db.l
    static constexpr bool kHas32 = EPI != kEpiBwd1;        // f32 output: a, y, dx
    static constexpr int kSlot32 = 32 * 32 * 4;            // f32 chunk: input, then output in place
    static constexpr int kSlotBytes = kSlot32 + (kHas16 ? 32 * 32 * 2 : 0);
    // chunk slots per epilogue warp; inputs are prefetched kNE - 2 of the
    // warp's chunks ahead (a slot is free once the store of the warp's chunk two
    // before has read it). dx' streams x in and dx out at HBM rate
    // (plane mode leaves more room to the operand ring, which measured faster
    // than deeper chunk buffering: no input prefetch but for dx')
    // (with in-kernel staging the stager ring takes 51 KB: the a-product keeps
    // two chunk slots, measured as fast as four for the forward products)
    static constexpr int kNE = STG ? 2
                             : PLANE ? (EPI == kEpiBwd2 ? 3 : 2)
                                     : (EPI == kEpiBwd2 ? 4 : (kSplit == 2 ? 2 : 4));
    static constexpr int kEpiBytes = kEW * kNE * kSlotBytes;
    static constexpr int kStgBytes = STG == 1 ? kStgRingBytes : (STG == 2 ? kStgRingBytesDy : 0);
    static constexpr int kStgSlots = STG == 1 ? kStgSlotsX : (STG == 2 ? kStgSlotsDy : 0);
    static constexpr int kBudget = (PLANE ? 224 : 221) * 1024 - kEpiBytes - kStgBytes;
    static constexpr int kNBRaw = kBudget / (kBBytes + kBitsBytes);
    static constexpr int kNB = kNBRaw > 10 ? 10 : kNBRaw;
    static constexpr int kNSMax = (kTmemCols - 2 * BT) / kSignCols;
    static constexpr int kNS = PLANE ? 0 : (kNSMax < kNB ? kNSMax : kNB);  // sign stages in TMEM
    static constexpr int kNumBars = 2 * kNB + kNS + 2 + 2 + 1 + kEW * kNE + (PLANE && PAIR ? kNB : 0) + 2 * kStgSlots;
    static_assert(kNE >= 2, "double-buffered chunk staging");
    static constexpr int kPhaseBytes = kNB * kBBytes + kEpiBytes + kNB * kBitsBytes + kStgBytes + kNumBars * 8;
    static constexpr int kSmemBytes = 1024 + kCtlBytes + kPhaseBytes;  // alignment slack, control block, phase
    static_assert(BT % 32 == 0 && BT >= 32 && BT <= 256 && (!PAIR || BT % 16 == 0), "token tile");
    static_assert(kTokRows % 8 == 0, "activation boxes hold whole 8-row swizzle groups");
    static_assert(PLANE || kNS >= 2, "at least two sign stages");
    static_assert(kNB >= 2, "at least two operand stages");
    // an expander frees sign stage i % NS by waiting on the activation slot of
    // k-step i - NS; that wait is unambiguous only if the activation ring is at
    // least as deep as the sign ring
    static_assert(kNB >= kNS, "activation ring must be at least as deep as the sign ring");
    static_assert(kBBlock % 1024 == 0, "swizzled boxes stay 1024-byte aligned");
    static_assert(kSlotBytes % 1024 == 0, "chunk slots stay 1024-byte aligned");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Path p's copy of a workspace array of a multi-path launch: `stride` bytes
// per path after path 0's.
template <typename T>
__device__ __forceinline__ T *path_at(T *base, int p, long long stride) {
    return reinterpret_cast<T *>(reinterpret_cast<uintptr_t>(base) + (uintptr_t)((long long)p * stride));
}

// Shared-memory control block at the (1024-aligned) start of dynamic shared
// memory; a GEMM phase's own layout starts kCtlBytes after it.
struct GemmCtl {
    uint32_t tmem_slot;  // TMEM base address written by tcgen05.alloc
    int abort_flag;      // set by any role whose bounded wait ran out
    unsigned int stg_done;  // items finished by the converter warps, one count per warp (STG kernels)
    StgGeo stg_geo[kStgSlotsMax];  // geometry of the units in the stager ring (STG kernels)
    int red_go;          // the folded reduction's grid barrier completed (dx'-product)
};
static_assert(sizeof(GemmCtl) <= kCtlBytes, "control block");

// Shared-memory layout of one GEMM phase (from a 1024-aligned base).
template <int EPI, bool PAIR, int BT, bool PLANE = false, int STG = 0>
struct GemmLayout {
    using S = GemmShape<EPI, PAIR, BT, PLANE, STG>;
    uint8_t *sB;       // [NB][kBBytes] activation tiles
    uint8_t *sE;       // [4 warps][kNE][slot] epilogue chunks
    uint32_t *sBits;   // [NB][2][128][2] bitmap words, or [NB][plane tile] (PLANE)
    uint8_t *sStg;     // stager ring (STG)
    uint64_t *full_b, *empty_b, *full_s, *tmem_full, *tmem_empty, *drain_bar, *eload, *full_p, *stg_full, *stg_empty;
    __device__ explicit GemmLayout(uint8_t *base) {
        sB = base;
        sE = sB + S::kNB * S::kBBytes;
        sBits = reinterpret_cast<uint32_t *>(sE + S::kEpiBytes);
        sStg = reinterpret_cast<uint8_t *>(sBits) + S::kNB * S::kBitsBytes;
        full_b = reinterpret_cast<uint64_t *>(sStg + S::kStgBytes);
        empty_b = full_b + S::kNB;
        full_s = empty_b + S::kNB;
        tmem_full = full_s + S::kNS;
        tmem_empty = tmem_full + 2;
        drain_bar = tmem_empty + 2;
        eload = drain_bar + 1;  // [epilogue warps][kNE]
        full_p = eload + S::kEW * S::kNE;  // [NB] (plane pairs: the peer's stage has landed)
        stg_full = full_p + (PLANE && PAIR ? S::kNB : 0);  // [stager slots]
        stg_empty = stg_full + S::kStgSlots;
    }
    // one thread: initialise every barrier of the phase
    __device__ void init_barriers() const {
        for (int s = 0; s < S::kNB; ++s) {
            mbar_init(&full_b[s], 1);
            mbar_init(&empty_b[s], 1);
        }
        for (int s = 0; s < S::kNS; ++s) mbar_init(&full_s[s], PAIR ? 2 * S::kNExp : S::kNExp);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tmem_full[i], 1);
            mbar_init(&tmem_empty[i], PAIR ? 2 * S::kEW : S::kEW);
        }
        mbar_init(drain_bar, 1);
        for (int i = 0; i < S::kEW * S::kNE; ++i) mbar_init(&eload[i], 1);
        if (PLANE && PAIR)
            for (int s = 0; s < S::kNB; ++s) mbar_init(&full_p[s], 1);
        for (int s = 0; s < S::kStgSlots; ++s) {
            mbar_init(&stg_full[s], 1);
            mbar_init(&stg_empty[s], kStgConvWarps);
        }
    }
    // one thread, once every role of the phase has finished with the barriers
    __device__ void inval_barriers() const {
        for (uint64_t *b = full_b; b < stg_empty + S::kStgSlots; ++b) mbar_inval(b);
    }
};

__device__ __forceinline__ void fail_status(const GemmArgs &a, volatile int *abort_flag, uint32_t code) {
    *abort_flag = 1;
    atomicOr(a.status, code);
}

__device__ __forceinline__ uint16_t f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }

// The four roles of one GEMM phase over the tiles unit, unit + num_units, ...
// (a CTA, or a CTA pair, per unit). Barriers must be initialised (and, for a
// pair, both CTAs' barriers visible) and TMEM allocated before the call; on
// return every load, MMA and store the phase issued has completed.
// SPLIT > 1 (single CTAs, one tile per CTA, clusters of SPLIT along K): CTA
// kj of the cluster reduces k-steps [kj n / SPLIT, (kj + 1) n / SPLIT) of the
// tile into its TMEM, stages the chunks it does not own in shared memory, and
// after a cluster barrier adds the peers' copies of chunk kj (read over DSMEM)
// into its TMEM; its epilogue then runs the tile's chunk kj only. For
// problems with few tiles and long K this cuts both the k-loop and the
// epilogue a CTA runs by SPLIT.
template <int EPI, bool PAIR, int BT, bool PLANE = false, int SPLIT = 1, int STG = 0>
__device__ __forceinline__ void gemm_roles(const GemmLayout<EPI, PAIR, BT, PLANE, STG> &L, const CUtensorMap &tmap_act,
                                           const CUtensorMap &tmap_in, const CUtensorMap &tmap_out32,
                                           const CUtensorMap &tmap_out16, const GemmArgs &args,
                                           uint32_t tmem_base, volatile int *abort_flag, int unit, int num_units,
                                           const CUtensorMap *tmap_sgn = nullptr, GemmCtl *ctl = nullptr,
                                           const CUtensorMap *tmap_aux = nullptr) {
    using S = GemmShape<EPI, PAIR, BT, PLANE, STG>;
    static_assert(STG == 0 || (STG == 1 && SPLIT == 1 && !PLANE && EPI == kEpiFwd1) ||
                      (STG == 2 && SPLIT == 1 && !PLANE && EPI == kEpiBwd1),
                  "in-kernel staging: the a-product stages x, the db-product dy");
    constexpr int kKB = S::kKBm, kStepK = S::kStepKm, kWarpEpi0 = S::kEpi0;
    constexpr int NB = S::kNB, NS = S::kNS, kChunks = S::kChunks, kNE = S::kNE;
    uint8_t *sB = L.sB;
    uint8_t *sE = L.sE;
    uint32_t *sBits = L.sBits;
    uint64_t *full_b = L.full_b, *empty_b = L.empty_b, *full_s = L.full_s, *tmem_full = L.tmem_full,
             *tmem_empty = L.tmem_empty, *drain_bar = L.drain_bar, *eload = L.eload;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int M = args.M, N = args.N;
    constexpr int kUnitF = PAIR ? 2 * kFM : kFM;  // features per tile
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int f_tiles = (N + kUnitF - 1) / kUnitF;
    const int t_tiles = (M + BT - 1) / BT;
    const int num_tiles = f_tiles * t_tiles;  // feature tile varies fastest: neighbours share activations
    // Multi-path launches. The products that add into y or dx compute each
    // tile for every path in turn on the same unit (local tile lt: tile
    // unit + (lt / P) * num_units, path lt % P), so that the paths' chunks of
    // an output tile are added in path order; the others spread the P x
    // num_tiles (path, tile) pairs over the units, path-major. Path p's
    // workspace arrays lie p * pstride bytes after path 0's, its TMA boxes at
    // third coordinate p, its column factors at args.colv_p[p].
    constexpr bool kPathMinor = EPI == kEpiFwd2 || EPI == kEpiBwd2;
    const int P = args.paths > 1 ? args.paths : 1;
    const int n_virt = num_tiles * P;
    const int n_local = kPathMinor ? (unit < num_tiles ? (num_tiles - unit + num_units - 1) / num_units : 0) * P
                                   : (unit < n_virt ? (n_virt - unit + num_units - 1) / num_units : 0);
    auto tile_of = [&](int lt) {
        return kPathMinor ? unit + (lt / P) * num_units : (unit + lt * num_units) % num_tiles;
    };
    auto path_of = [&](int lt) { return kPathMinor ? lt % P : (unit + lt * num_units) / num_tiles; };
    const int num_ks = (args.K + kStepK - 1) / kStepK;
    static_assert(SPLIT == 1 || (!PAIR && !PLANE), "split-K runs single TMEM-expansion CTAs");
    const int kj = SPLIT > 1 ? (int)cluster_ctarank() : 0;  // this CTA's share of K
    const int ks0 = kj * num_ks / SPLIT, ks1 = (kj + 1) * num_ks / SPLIT;
    // the leader's copy of a barrier, as a cluster address (PAIR only)
    auto leader_bar = [&](uint64_t *bar) -> uint32_t { return mapa_shared(smem_u32(bar), 0); };

    if (warp == kWarpTma) {
        if (lane == 0) {
            int sb = 0;
            uint32_t pb = 0, issued = 0, parity = 0;
            bool ok = true;
            for (int lt = 0; lt < n_local && ok; ++lt) {
                const int tile = tile_of(lt), pz = path_of(lt);
                const int t0 = (tile / f_tiles) * BT + (int)rank * S::kTokRows;  // this CTA's token rows
                const int f0 = (tile % f_tiles) * kUnitF + (int)rank * kFM;      // this CTA's sign rows
                const uint32_t *bsign = path_at(args.bsign, pz, args.pstride);
                for (int ks = ks0; ks < ks1; ++ks) {
                    if constexpr (STG != 0) {
                        // the stagers publish a tile's rows per column chunk:
                        // acquire the count before the chunk's loads
                        constexpr int kChunkSteps = kStgKC / kStepK;
                        if (ks % kChunkSteps == 0) {
                            const int tt = tile / f_tiles;
                            const int kc = ks / kChunkSteps;
                            const unsigned int need = (unsigned int)(M - tt * BT < BT ? M - tt * BT : BT);
                            if (!wait_count(path_at(args.stg.cnt, pz, args.pstride) + (size_t)tt * stg_chunks(args.K) + kc,
                                            need, abort_flag)) {
                                fail_status(args, abort_flag, kStTimeoutStage);
                                ok = false;
                                break;
                            }
                            fence_proxy_async_global();
                        }
                    }
                    if (!mbar_wait(&empty_b[sb], pb ^ 1u, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutTma);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_b[sb], S::kBBytes + S::kBitsBytes);
                    if constexpr (PLANE) {
                        // one 64-deep block: the activation box and the plane tile
                        // (rows and K past the plane's extent read zero)
                        const int k0 = ks * kBK;
                        uint8_t *sa = reinterpret_cast<uint8_t *>(sBits) + sb * S::kBitsBytes;
                        tma_load_3d(sB + sb * S::kBBytes, &tmap_act, &full_b[sb], k0, t0, pz);
                        if constexpr (S::kPlaneMN) {
                            // plane [K][N]: two 64-feature blocks of 64 K rows
                            tma_load_2d(sa, tmap_sgn, &full_b[sb], f0, k0);
                            tma_load_2d(sa + S::kABlock / 2, tmap_sgn, &full_b[sb], f0 + 64, k0);
                        } else {
                            // plane [N][K]: 128 feature rows of 64 K
                            tma_load_2d(sa, tmap_sgn, &full_b[sb], k0, f0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kKB; ++kk) {
                            // 64-wide K block; blocks past K read zero activations (and padded words)
                            const int blk = ks * kKB + kk;
                            tma_load_3d(sB + sb * S::kBBytes + kk * S::kBBlock, &tmap_act, &full_b[sb], blk * kBK,
                                        t0, pz);
                            bulk_load(sBits + sb * (S::kBitsBytes / 4) + kk * (S::kBitsBlock / 4),
                                      bsign + ((size_t)blk * args.Ns + f0) * 2, S::kBitsBlock, &full_b[sb]);
                        }
                    }
                    issued |= 1u << sb;
                    parity = (parity & ~(1u << sb)) | (pb << sb);
                    if (++sb == NB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
            }
            // drain: every load issued must have landed before the CTA exits
            for (int s = 0; s < NB; ++s) {
                if (((issued >> s) & 1u) && !mbar_wait(&full_b[s], (parity >> s) & 1u, abort_flag, false))
                    atomicOr(args.status, kStTimeoutDrain);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma && PLANE) {
        if constexpr (PLANE) {
            if (lane == 0 && leader) {
                // both operands in shared memory: 4 MMAs (K = 16 each) per 64-deep block
                constexpr uint32_t idesc = umma_idesc_f16_f32_major(PAIR ? 2 * kFM : kFM, BT, S::kPlaneMN, false);
                constexpr uint64_t kAdvA = S::kPlaneMN ? (2048u >> 4) : (32u >> 4);
                const uint64_t bdesc0 = umma_sdesc_sw128(smem_u32(sB));
                const uint32_t abase = smem_u32(sBits);
                int sb = 0;
                uint32_t pb = 0;
                bool ok = true;
                for (int local = 0; local < n_local && ok; ++local) {
                    const int acc = local & 1;
                    const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
                    if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutMma);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(acc * S::kAccCols);
                    uint32_t acc_in = 0u;
                    for (int ks = ks0; ks < ks1; ++ks) {
                        bool got = mbar_wait(&full_b[sb], pb, abort_flag);
                        if (PAIR && got) got = mbar_wait(&L.full_p[sb], pb, abort_flag);
                        if (!got) {
                            fail_status(args, abort_flag, kStTimeoutMma);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = abase + (uint32_t)(sb * S::kBitsBytes);
                        const uint64_t adesc = S::kPlaneMN ? umma_sdesc_sw128_mn(a_addr) : umma_sdesc_sw128(a_addr);
                        const uint64_t bdesc = bdesc0 + (uint64_t)sb * (S::kBBytes >> 4);
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            if constexpr (PAIR)
                                umma_f16_pair(d_tmem, adesc + kAdvA * k, bdesc + (uint64_t)(2 * k), idesc, acc_in);
                            else
                                umma_f16(d_tmem, adesc + kAdvA * k, bdesc + (uint64_t)(2 * k), idesc, acc_in);
                            acc_in = 1u;
                        }
                        if constexpr (PAIR)
                            umma_commit_pair_multicast(&empty_b[sb], 3);
                        else
                            umma_commit(&empty_b[sb]);
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
                if constexpr (PAIR)
                    umma_commit_pair_multicast(drain_bar, 1);
                else
                    umma_commit(drain_bar);
                if (!mbar_wait(drain_bar, 0, abort_flag, false)) atomicOr(args.status, kStTimeoutDrain);
            } else if (PAIR && lane == 0) {
                // peer: forward each stage's landing (its own full_b) to the leader's full_p
                int sb = 0;
                uint32_t pb = 0;
                bool ok = true;
                for (int lt = 0; lt < n_local && ok; ++lt) {
                    for (int ks = ks0; ks < ks1; ++ks) {
                        if (!mbar_wait(&full_b[sb], pb, abort_flag)) {
                            fail_status(args, abort_flag, kStTimeoutMma);
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote(leader_bar(&L.full_p[sb]));
                        if (++sb == NB) {
                            sb = 0;
                            pb ^= 1u;
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(PAIR ? 2 * kFM : kFM, BT);
            // descriptors and TMEM addresses advance by constants per k-step, so
            // the issuer's path between two k-steps stays a handful of instructions
            const uint64_t bdesc0 = umma_sdesc_sw128(smem_u32(sB));
            constexpr uint64_t kDescStage = S::kBBytes >> 4, kDescBlock = S::kBBlock >> 4;
            const uint32_t sign0 = tmem_base + (uint32_t)S::kSignCol0;
            int sa = 0, sb = 0;
            uint32_t pa = 0;
            bool ok = true;
            for (int local = 0; local < n_local && ok; ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
                // (the peer's arrivals on tmem_empty and full_s are released at CTA
                // scope, see mbar_arrive_remote; they are awaited at CTA scope too)
                if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)) {
                    fail_status(args, abort_flag, kStTimeoutMma);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * S::kAccCols);
                uint32_t acc_in = 0u;  // the tile's first MMA overwrites the accumulator
                for (int ks = ks0; ks < ks1; ++ks) {
                    if (!mbar_wait(&full_s[sa], pa, abort_flag)) {
                        fail_status(args, abort_flag, kStTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = sign0 + (uint32_t)(sa * kSignCols);
                    const uint64_t bdesc = bdesc0 + (uint64_t)sb * kDescStage;
#pragma unroll
                    for (int kk = 0; kk < kKB; ++kk) {
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // 16 K values per MMA: 8 TMEM columns of A, 32 bytes along B's swizzled rows
                            const uint32_t a_k = a_tmem + (uint32_t)(kk * (kBK / 2) + k * 8);
                            const uint64_t b_k = bdesc + (uint64_t)kk * kDescBlock + (uint64_t)(2 * k);
                            if constexpr (PAIR)
                                umma_f16_ts_pair(d_tmem, a_k, b_k, idesc, acc_in);
                            else
                                umma_f16_ts(d_tmem, a_k, b_k, idesc, acc_in);
                            acc_in = 1u;
                        }
                    }
                    if constexpr (PAIR)
                        umma_commit_pair_multicast(&empty_b[sb], 3);
                    else
                        umma_commit(&empty_b[sb]);
                    if (++sa == NS) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sb == NB) sb = 0;
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
        }
        __syncwarp();
    } else if (warp < kWarpEpi0) {
      if constexpr (!PLANE) {
        // ---- sign expanders: bitmap words -> +-1 f16 A operand in TMEM -----
        constexpr int kBlocks = 4 * kKB / S::kNExp;  // 64-wide blocks of a k-step per warp
        const int quarter = warp & 3;
        const int kk0 = (warp - kWarpExp0) / 4 * kBlocks;  // the warp's first 64-wide block of the k-step
        const int row = quarter * 32 + lane;    // sign row within the CTA's 128
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        int sb = 0, sa = 0;
        uint32_t pb = 0;
        int lag = -NS;    // k-step whose MMAs must have finished reading this sign stage
        int ls = 0;       // its activation slot
        uint32_t lp = 0;  // and that slot's phase parity
        bool ok = true;
        for (int lt = 0; lt < n_local && ok; ++lt) {
            for (int ks = ks0; ks < ks1; ++ks) {
                bool got = mbar_wait(&full_b[sb], pb, abort_flag);
                uint32_t v[kBlocks][32];
                if (got) {
                    // signs first: they only need the words, not the free stage
#pragma unroll
                    for (int b = 0; b < kBlocks; ++b) {
                        const uint2 w = reinterpret_cast<const uint2 *>(sBits + sb * (S::kBitsBytes / 4) +
                                                                        (kk0 + b) * (S::kBitsBlock / 4))[row];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            v[b][q] = sign_pair(w.x, q);       // K 2q, 2q+1 of the block
                            v[b][16 + q] = sign_pair(w.y, q);  // K 32+2q, 32+2q+1
                        }
                    }
                }
                if (got && lag >= 0) got = mbar_wait(&empty_b[ls], lp, abort_flag);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    if (lane == 0) fail_status(args, abort_flag, kStTimeoutExpand);
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    // the warp's blocks are adjacent column ranges of the stage
                    const uint32_t col =
                        tmem_base + lane_addr + (uint32_t)(S::kSignCol0 + sa * kSignCols + kk0 * (kBK / 2));
                    if constexpr (kBlocks == 2) {
                        tmem_st_32x32b_x64(col, v);  // one 64-column store (measured 2% faster than two)
                    } else {
#pragma unroll
                        for (int b = 0; b < kBlocks; ++b) tmem_st_32x32b_x32(col + (uint32_t)(b * (kBK / 2)), v[b]);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // the leader's MMAs read both CTAs' stages: the peer's warps
                    // arrive on the leader's barrier directly
                    if (PAIR && !leader)
                        mbar_arrive_remote(leader_bar(&full_s[sa]));
                    else
                        mbar_arrive(&full_s[sa]);
                }
                if (++sb == NB) {
                    sb = 0;
                    pb ^= 1u;
                }
                if (++sa == NS) sa = 0;
                if (++lag > 0) {
                    if (++ls == NB) {
                        ls = 0;
                        lp ^= 1u;
                    }
                }
            }
        }
      }
    } else if (warp < kWarpEpi0 + S::kEW) {
        // ---- epilogue: thread = one feature of the tile, BT tokens ----------
        // With two warps per lane quarter (kSplit = 2), the warp `half` takes
        // the tile's chunks half, half + 2, ...; g counts the warp's own chunks.
        constexpr int kSplit = S::kSplit;
        constexpr int kMaxNc = (kChunks + kSplit - 1) / kSplit;  // chunks per tile of the busier warp
        const int q = warp & 3;
        const int ew = warp - kWarpEpi0;
        const int half = ew / 4;
        // this warp's first chunk of a tile and its chunks per tile (split-K: chunk kj only)
        const int cb = SPLIT > 1 ? kj : half;
        const int nc = SPLIT > 1 ? 1 : (kChunks - half + kSplit - 1) / kSplit;
        uint8_t *slots = sE + ew * kNE * S::kSlotBytes;
        uint64_t *ebar = eload + ew * kNE;
        // inputs: the a-tape (db) or x (dx'); y and dx accumulate by reduce-add stores
        const bool has_in = (EPI == kEpiBwd1) || (EPI == kEpiBwd2);
        // which chunk maps hold one plane per path: the a-tape in and out, and
        // every f16 output; y, dx and x are the paths' common tensors
        constexpr bool kIn32PerPath = EPI == kEpiBwd1, kOut32PerPath = EPI == kEpiFwd1;
        // chunks per tile of the less busy warp of a lane quarter
        constexpr int kMinNc = kChunks / kSplit;
        static_assert(kMinNc >= 1, "every epilogue warp has a chunk per tile");
        uint32_t pending = 0u;  // lane 0: slots with an input load not yet waited on
        uint32_t ppar = 0u;     // and that load's phase parity
        // the warp's chunk g: local tile g / nc, chunk half + kSplit * (g % nc)
        auto chunk_at = [&](int g, int &fq, int &tok, int &pz) -> bool {
            const int lt = g / nc;
            if (lt >= n_local) return false;
            const int tile = tile_of(lt);
            pz = path_of(lt);
            fq = (tile % f_tiles) * kUnitF + (int)rank * kFM + q * 32;
            tok = (tile / f_tiles) * BT + 32 * (cb + kSplit * (g - lt * nc));
            return true;
        };
        // L2 policy of the streams this epilogue reads or writes once (the
        // a-tape, x, y, dx, c); the f16 operands of the next product (a.l,
        // db.l) keep the default so that its CTAs find them in L2
        const uint64_t once = l2_policy_evict_first();
        auto load_chunk = [&](int g) {  // lane 0
            int fq, tok, pz;
            if (!chunk_at(g, fq, tok, pz)) return;
            const int sl = g % kNE;
            const uint32_t par = (uint32_t)(g / kNE) & 1u;
            mbar_arrive_expect_tx(&ebar[sl], S::kSlot32);
            tma_load_3d_hint(slots + sl * S::kSlotBytes, &tmap_in, &ebar[sl], fq, tok, kIn32PerPath ? pz : 0, once);
            pending |= 1u << sl;
            ppar = (ppar & ~(1u << sl)) | (par << sl);
        };
        if (has_in && lane == 0)
            for (int i = 0; i < kNE - 2; ++i) load_chunk(i);
        int g = 0;
        int local = 0;
        bool ok = true;
        if constexpr (SPLIT > 1) {
            // split-K: one tile per CTA. Stage the chunks other CTAs own, then sum
            // this CTA's chunk over the cluster back into TMEM (accumulator 0).
            // Every thread of every role passes the two cluster barriers.
            bool got = unit < num_tiles && mbar_wait(&tmem_full[0], 0, abort_flag);
            got = __all_sync(0xFFFFFFFFu, got);
            if (!got && lane == 0 && unit < num_tiles) fail_status(args, abort_flag, kStTimeoutEpi);
            tc_fence_after();
            const uint32_t acc_addr = tmem_base + ((uint32_t)(q * 32) << 16);
            const int row = q * 32 + lane;  // feature row of the tile
            float *stg = reinterpret_cast<float *>(sB);  // [kChunks][128 rows][32] f32, 16-byte groups swizzled
            uint32_t v[32];
            if (got) {
                for (int c = 0; c < kChunks; ++c) {
                    if (c == kj) continue;
                    tmem_ld_32x32b_x32(acc_addr + (uint32_t)(32 * c), v);
                    tmem_wait_ld_regs(v);
                    float *dst = stg + ((size_t)c * kFM + row) * 32;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4)
                        reinterpret_cast<float4 *>(dst)[j4 ^ (row & 7)] =
                            make_float4(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]),
                                        __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]));
                }
            }
            cluster_sync();  // every CTA's chunks are staged
            if (got) {
                tmem_ld_32x32b_x32(acc_addr + (uint32_t)(32 * kj), v);
                tmem_wait_ld_regs(v);
                const uint32_t mine = smem_u32(stg + ((size_t)kj * kFM + row) * 32);
                for (int p = 0; p < SPLIT; ++p) {
                    if (p == kj) continue;
                    const uint32_t peer = mapa_shared(mine, (uint32_t)p);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 o = ld_shared_cluster_v4(peer + (uint32_t)((j4 ^ (row & 7)) * 16));
                        v[4 * j4] = __float_as_uint(__uint_as_float(v[4 * j4]) + o.x);
                        v[4 * j4 + 1] = __float_as_uint(__uint_as_float(v[4 * j4 + 1]) + o.y);
                        v[4 * j4 + 2] = __float_as_uint(__uint_as_float(v[4 * j4 + 2]) + o.z);
                        v[4 * j4 + 3] = __float_as_uint(__uint_as_float(v[4 * j4 + 3]) + o.w);
                    }
                }
                tmem_st_32x32b_x32(acc_addr + (uint32_t)(32 * kj), v);
                tmem_wait_st();
            }
            cluster_sync();  // no CTA reads a peer's staging any more
            if (!got) ok = false;
        }
        for (; local < n_local && ok; ++local) {
            const int tile = tile_of(local), pz = path_of(local);
            const int acc = local & 1;
            const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
            const int tt = tile / f_tiles;
            // y and dx: path 0 stores (or adds, in accumulate mode), later paths add
            const bool add_out = (EPI == kEpiFwd2 || EPI == kEpiBwd2) && (args.accumulate || pz > 0);
            const int fq = (tile % f_tiles) * kUnitF + (int)rank * kFM + q * 32;  // this warp's 32 features
            const int f = fq + lane;
            const int t0 = tt * BT;
            // per-token scales of this warp's chunks (lane l: token 32c + l of
            // the tile), fetched before the accumulator is ready
            float ri_t[kMaxNc], rs_t[kMaxNc];
#pragma unroll
            for (int i = 0; i < kMaxNc; ++i) {
                const int tl = t0 + 32 * (cb + kSplit * i) + lane;
                const bool use = i < nc && tl < M;
                ri_t[i] = (EPI == kEpiBwd1 || EPI == kEpiBwd2) && use ? __ldg(path_at(args.row_inv, pz, args.pstride) + tl) : 0.0f;
                rs_t[i] = (EPI == kEpiBwd1) && use ? __ldg(path_at(args.row_scale, pz, args.pstride) + tl) : 0.0f;
            }
            const bool fvalid = f < N;
            const float cf = fvalid ? __ldg((P > 1 ? args.colv_p[pz] : args.colv) + f) : 0.0f;
            const bool got = mbar_wait(&tmem_full[acc], acc_phase, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) fail_status(args, abort_flag, kStTimeoutEpi);
                ok = false;
                break;
            }
            tc_fence_after();
            float psum = 0.0f;
            const uint32_t acc_addr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * S::kAccCols);
            // Accumulator columns come in two register sets: the warp's next
            // chunk is loaded from TMEM while the current one is processed.
            uint32_t va[32], vb[32];
            tmem_ld_32x32b_x32(acc_addr + (uint32_t)(32 * cb), va);
#pragma unroll
            for (int i = 0; i < kMaxNc; ++i) {
                if (i >= nc) break;
                const int c = cb + kSplit * i;  // chunk of the tile
                uint32_t(&v)[32] = (i & 1) ? vb : va;
                uint32_t(&vn)[32] = (i & 1) ? va : vb;
                tmem_wait_ld_regs(v);
                if (i + 1 < nc) tmem_ld_32x32b_x32(acc_addr + (uint32_t)(32 * (c + kSplit)), vn);
                if (i + 1 == nc) {
                    // this warp's part of the accumulator is read: one arrival
                    // of the kEW (per CTA) that hand it back to the MMA issuer
                    tmem_wait_ld_regs(vn);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_remote(leader_bar(&tmem_empty[acc]));
                        else
                            mbar_arrive(&tmem_empty[acc]);
                    }
                }
                if (lane == 0) {
                    // the slot of the warp's chunk g + kNE - 2 was last stored from by
                    // its chunk g-2: all stores but the newest (g-1) have read theirs
                    bulk_wait_group_read<1>();
                    if (has_in) load_chunk(g + kNE - 2);
                }
                __syncwarp();
                const int sl = g % kNE;
                float *s32 = reinterpret_cast<float *>(slots + sl * S::kSlotBytes);       // [32 tokens][32 features]
                uint16_t *s16 = reinterpret_cast<uint16_t *>(slots + sl * S::kSlotBytes + S::kSlot32);
                if (has_in) {
                    const bool in_ok = mbar_wait(&ebar[sl], (uint32_t)(g / kNE) & 1u, abort_flag);
                    if (lane == 0) pending &= ~(1u << sl);
                    if (!__all_sync(0xFFFFFFFFu, in_ok)) {
                        if (lane == 0) fail_status(args, abort_flag, kStTimeoutEpi);
                        tmem_wait_ld();  // no TMEM load may be in flight at teardown
                        ok = false;
                        break;
                    }
                }
                const int tc = t0 + 32 * c;
                if constexpr (EPI == kEpiFwd1) {
                    // a (f32 tape) and a.l staged to f16 for the second forward product
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float x = __uint_as_float(v[j]);
                        s32[j * 32 + lane] = x;
                        s16[j * 32 + lane] = f16_bits(x * cf);
                    }
                } else if constexpr (EPI == kEpiFwd2) {
                    // y (+)= h.c (accumulate: the store adds), c saved in f16
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float x = __uint_as_float(v[j]);
                        s32[j * 32 + lane] = cf * x;
                        s16[j * 32 + lane] = f16_bits(x);
                    }
                } else if constexpr (EPI == kEpiBwd1) {
                    // db = acc / s_t; dl partial sum_t a.db; db.l staged under sigma_t
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float ri = __shfl_sync(0xFFFFFFFFu, ri_t[i], j);
                        const float rs = __shfl_sync(0xFFFFFFFFu, rs_t[i], j);
                        const float db = __uint_as_float(v[j]) * ri;
                        psum += s32[j * 32 + lane] * db;
                        s16[j * 32 + lane] = f16_bits(db * cf * rs);
                    }
                } else {
                    // dx' = acc / sigma_t; dg partial sum_t x.dx'; dx (+)= g.dx'
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float ri = __shfl_sync(0xFFFFFFFFu, ri_t[i], j);
                        const float dxp = __uint_as_float(v[j]) * ri;
                        psum += s32[j * 32 + lane] * dxp;
                        s32[j * 32 + lane] = cf * dxp;
                    }
                }
                // chunk staged: one TMA store per output (rows past M and
                // features past N are clipped; wholly outside boxes are skipped)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && tc < M && fq < N) {
                    if constexpr (S::kHas32) {
                        const int z32 = kOut32PerPath ? pz : 0;
                        if ((EPI == kEpiFwd2 || EPI == kEpiBwd2) && pz > 0) {
                            // the previous path's store of this chunk was this warp's
                            // (nc - 1)-th bulk group before this one: it must have
                            // written y or dx before this path's add reads them
                            bulk_wait_group<kMinNc - 1>();
                        }
                        if (add_out)
                            tma_reduce_add_3d_hint(&tmap_out32, s32, fq, tc, z32, once);  // y or dx += the chunk
                        else
                            tma_store_3d_hint(&tmap_out32, s32, fq, tc, z32, once);
                    }
                    if constexpr (S::kHas16) {
                        if (EPI == kEpiFwd2)
                            tma_store_3d_hint(&tmap_out16, s16, fq, tc, pz, once);  // c, read again by the backward only
                        else
                            tma_store_3d(&tmap_out16, s16, fq, tc, pz);  // a.l or db.l: the next product's operand
                    }
                }
                if (lane == 0) bulk_commit_group();
                ++g;
            }
            if (!ok) break;
            if constexpr (EPI == kEpiBwd1 || EPI == kEpiBwd2) {
                // one partial row per (token tile, warp of the quarter)
                if (fvalid)
                    path_at(args.part, pz, args.pstride)[((size_t)tt * (SPLIT > 1 ? SPLIT : kSplit) + (SPLIT > 1 ? kj : half)) * N + f] =
                        psum;
            }
        }
        // drain: stores complete, and input loads issued but not consumed have landed
        if (lane == 0) {
            bulk_wait_group_all();
            for (int sl = 0; sl < kNE; ++sl)
                if (((pending >> sl) & 1u) && !mbar_wait(&ebar[sl], (ppar >> sl) & 1u, abort_flag, false))
                    atomicOr(args.status, kStTimeoutDrain);
        }
        __syncwarp();
    } else {
        if constexpr (STG != 0) {
            // ---- stagers: x16 of later tiles -----------------------------------
            const StgGeom G(M, args.K, BT, f_tiles, num_units, P);
            const StgX X(args.stg, G);
            const int t = (int)threadIdx.x - S::kStg0 * 32;
            // (the a-product has no epilogue input and no sign plane: those two
            // maps are x, f32, in 256 x 16 boxes for the ring and 256 x 64 for
            // the L2 prefetches)
            // (the db-product has no f32 output and no sign plane: those two
            // maps are dy, f32, in 256 x 16 and 256 x 64 boxes; tmap_aux is c)
            if constexpr (STG == 1) {
                if (t < kStgConvThreads)
                    stager_x_convert(X, t, abort_flag, L.sStg, L.stg_full, L.stg_empty, ctl->stg_geo,
                                     &ctl->stg_done, args.status);
                else if (t == kStgConvThreads)
                    stager_x_producer(X, &tmap_in, abort_flag, L.sStg, L.stg_full, L.stg_empty, ctl->stg_geo,
                                      args.status);
            } else {
                if (t < kStgConvThreads)
                    stager_dy_convert(X, t, abort_flag, L.sStg, L.stg_full, L.stg_empty, ctl->stg_geo,
                                      &ctl->stg_done, args.status);
                else if (t == kStgConvThreads)
                    stager_dy_producer(X, &tmap_out32, tmap_aux, abort_flag, L.sStg, L.stg_full, L.stg_empty,
                                       ctl->stg_geo, args.status);
            }
            if (t == kStgConvThreads + 32) stager_x_publisher(X, tmap_sgn, abort_flag, &ctl->stg_done, args.status);
            __syncwarp();
        }
    }
    if constexpr (SPLIT > 1) {
        // the other roles, done with the tile, pass the epilogue's two cluster barriers
        if (warp < kWarpEpi0) {
            cluster_sync();
            cluster_sync();
        }
    }

}

// Prefetch of a phase's tensor-map descriptors (TMA and epilogue lanes).
template <int EPI, bool PAIR, int BT, bool PLANE = false, int STG = 0>
__device__ __forceinline__ void gemm_prefetch_maps(const CUtensorMap &tmap_act, const CUtensorMap &tmap_in,
                                                   const CUtensorMap &tmap_out32, const CUtensorMap &tmap_out16,
                                                   const CUtensorMap *tmap_sgn = nullptr,
                                                   const CUtensorMap *tmap_aux = nullptr) {
    using S = GemmShape<EPI, PAIR, BT, PLANE, STG>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tmap_act);
        if (PLANE || S::kStgSlots) tma_prefetch_desc(tmap_sgn);
        if (STG == 2) {
            tma_prefetch_desc(&tmap_out32);
            tma_prefetch_desc(tmap_aux);
        }
    }
    if (warp == S::kEpi0 && lane == 0) {
        if (EPI != kEpiFwd1 || S::kStgSlots) tma_prefetch_desc(&tmap_in);
        if (S::kHas32) tma_prefetch_desc(&tmap_out32);
        if (S::kHas16) tma_prefetch_desc(&tmap_out16);
    }
}

// Tail of a dx'-product launch with the pass's partial-sum reduction folded
// in (GemmArgs.fold): a grid barrier on args.red.gbar (bounded: the persistent
// grid, at most one CTA per SM, is resident together), then each CTA adds a
// share of the columns of every path's dh, dl and dg, each column's rows in
// a fixed order. Called by every thread after the roles and the TMEM release;
// the phase's shared memory is free again by then.
__device__ __forceinline__ void gemm_fold_reduce(const GemmArgs &args, uint8_t *smem) {
    // (the decision goes through the control block: static shared memory
    // would push the largest phases past the per-CTA limit)
    volatile int *go = &reinterpret_cast<GemmCtl *>(smem)->red_go;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's dg partial rows (written by its epilogue warps) before the arrival
        atomicAdd(args.red.gbar, 1u);
        const uint64_t t0 = globaltimer_ns();
        const unsigned int target = gridDim.x + args.red.extra;
        bool ok = true;
        while (ld_acquire_u32(args.red.gbar) < target) {
            if (globaltimer_ns() - t0 > args.red.wait_ns) {
                ok = false;
                break;
            }
            __nanosleep(128);
        }
        if (!ok) atomicOr(args.status, kStTimeoutGrid);
        __threadfence();
        *go = ok ? 1 : 0;
    }
    __syncthreads();
    if (!*go) return;
    float *red = reinterpret_cast<float *>(smem + kCtlBytes);
    const int P = args.paths > 1 ? args.paths : 1;
    for (int p = 0; p < P; ++p) {
        const ReduceSeg h{path_at(args.red_part_h, p, args.pstride), args.red_out_h[p], args.red_rows_h, args.red_n_h};
        const ReduceSeg l{path_at(args.red_part_l, p, args.pstride), args.red_out_l[p], args.red_rows_l, args.red_n_l};
        const ReduceSeg g{path_at(const_cast<const float *>(args.part), p, args.pstride), args.red_out_g[p],
                          args.red_rows_g, args.N};
        reduce_partials_run(h, l, g, (int)blockIdx.x, (int)gridDim.x, red);
    }
}

__device__ __forceinline__ uint8_t *smem_base_1024() {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
}

template <int EPI, bool PAIR, int BT, bool PLANE, int SPLIT, int STG>
__global__ void __launch_bounds__(GemmShape<EPI, PAIR, BT, PLANE, STG>::kThreads, 1)
    blr_gemm_kernel(const __grid_constant__ CUtensorMap tmap_act, const __grid_constant__ CUtensorMap tmap_in,
                    const __grid_constant__ CUtensorMap tmap_out32, const __grid_constant__ CUtensorMap tmap_out16,
                    const __grid_constant__ CUtensorMap tmap_sgn, const __grid_constant__ CUtensorMap tmap_aux,
                    const GemmArgs args) {
    uint8_t *smem = smem_base_1024();
    GemmCtl *ctl = reinterpret_cast<GemmCtl *>(smem);
    const GemmLayout<EPI, PAIR, BT, PLANE, STG> L(smem + kCtlBytes);
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        L.init_barriers();
        ctl->abort_flag = 0;
        ctl->stg_done = 0;
        fence_mbar_init();
    }
    gemm_prefetch_maps<EPI, PAIR, BT, PLANE, STG>(tmap_act, tmap_in, tmap_out32, tmap_out16, &tmap_sgn, &tmap_aux);
    if constexpr (PAIR) {
        cluster_sync();  // both CTAs' barriers exist before any remote arrival
        if (warp == kWarpMma) {
            tmem_alloc_pair(&ctl->tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        }
    } else {
        if (warp == kWarpMma) {
            tmem_alloc(&ctl->tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_slot;
    // setup above overlaps the previous kernel; global memory only after this
    pdl_wait();
    pdl_launch_dependents();
    // tile worker: a CTA, a CTA pair, or a split-K cluster
    const int per_unit = PAIR ? 2 : SPLIT;
    const int unit = (int)blockIdx.x / per_unit;
    const int num_units = (int)gridDim.x / per_unit;
    gemm_roles<EPI, PAIR, BT, PLANE, SPLIT, STG>(L, tmap_act, tmap_in, tmap_out32, tmap_out16, args, tmem_base,
                                                 reinterpret_cast<volatile int *>(&ctl->abort_flag), unit, num_units,
                                                 &tmap_sgn, ctl, &tmap_aux);
    tc_fence_before();
    if constexpr (PAIR) {
        // neither CTA leaves while the pair's MMAs or remote arrivals may still touch it
        cluster_sync();
        tc_fence_after();
        if (warp == kWarpMma) tmem_dealloc_pair(tmem_base, kTmemCols);
    } else {
        __syncthreads();
        tc_fence_after();
        if (warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
    }
    if constexpr (EPI == kEpiBwd2 && SPLIT == 1) {
        if (args.fold) gemm_fold_reduce(args, smem);
    }
}

template <int EPI, bool PAIR, int BT, bool PLANE = false, int SPLIT = 1, int STG = 0>
cudaError_t launch_gemm_t(const GemmMaps &maps, const GemmArgs &args, int grid, cudaStream_t s) {
    using S = GemmShape<EPI, PAIR, BT, PLANE, STG>;
    cudaError_t pe = prepare_kernel_once(blr_gemm_kernel<EPI, PAIR, BT, PLANE, SPLIT, STG>, S::kSmemBytes);
    if (pe != cudaSuccess) return pe;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(S::kThreads);
    cfg.dynamicSmemBytes = S::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = PAIR ? 2 : SPLIT;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (PAIR || SPLIT > 1) ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, blr_gemm_kernel<EPI, PAIR, BT, PLANE, SPLIT, STG>, maps.act, maps.in32,
                              maps.out32, maps.out16, maps.sgn, maps.aux, args);
}

// Tile configurations: CTA pairs with 160 or 192 tokens per tile, single CTAs
// with 128.
// The same tiles with the activation operand staged inside the kernel.
template <int EPI, int STG>
cudaError_t launch_gemm_stg(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    if (plan.pair && plan.bt == 192) return launch_gemm_t<EPI, true, 192, false, 1, STG>(maps, args, plan.grid, s);
    if (plan.pair && plan.bt == 160) return launch_gemm_t<EPI, true, 160, false, 1, STG>(maps, args, plan.grid, s);
    if (!plan.pair && plan.bt == 128) return launch_gemm_t<EPI, false, 128, false, 1, STG>(maps, args, plan.grid, s);
    if (!plan.pair && plan.bt == 64) return launch_gemm_t<EPI, false, 64, false, 1, STG>(maps, args, plan.grid, s);
    if (!plan.pair && plan.bt == 32) return launch_gemm_t<EPI, false, 32, false, 1, STG>(maps, args, plan.grid, s);
    return cudaErrorInvalidValue;
}

template <int EPI>
cudaError_t launch_gemm_epi(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    if (plan.plane) {
        if (plan.pair && plan.bt == 256) return launch_gemm_t<EPI, true, 256, true>(maps, args, plan.grid, s);
        if (!plan.pair && plan.bt == 128) return launch_gemm_t<EPI, false, 128, true>(maps, args, plan.grid, s);
        return cudaErrorInvalidValue;
    }
    if constexpr (EPI == kEpiFwd1 || EPI == kEpiBwd1) {
        if (plan.split == 4) return launch_gemm_t<EPI, false, 128, false, 4>(maps, args, plan.grid, s);
    }
    if (plan.pair && plan.bt == 192) return launch_gemm_t<EPI, true, 192>(maps, args, plan.grid, s);
    if (plan.pair && plan.bt == 160) return launch_gemm_t<EPI, true, 160>(maps, args, plan.grid, s);
    if (!plan.pair && plan.bt == 128) return launch_gemm_t<EPI, false, 128>(maps, args, plan.grid, s);
    if (!plan.pair && plan.bt == 64) return launch_gemm_t<EPI, false, 64>(maps, args, plan.grid, s);
    if constexpr (EPI == kEpiFwd1 || EPI == kEpiBwd1) {
        if (!plan.pair && plan.bt == 32) return launch_gemm_t<EPI, false, 32>(maps, args, plan.grid, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace blr
