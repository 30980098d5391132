// Host-side shape rule and workspace layout of the blr layer, shared by every
// entry point that carves buffers out of one block of device memory (the
// caller's workspace in blr_api.cu, the library's fixed scratch array in
// blr_noalloc.cu), so that both always agree on sizes and offsets.
#pragma once

#include <cstddef>

#include "blr_kernels.h"

namespace blr {

// Shape rule: M >= 1; d_in, d_out, r multiples of 32 and >= 64; d_out <=
// 32768 (one block stages a dy row); d_in, r <= 65536; M <= 2^28.
inline bool shape_ok(int M, int d_in, int d_out, int r) {
    auto dim_ok = [](int d, int hi) { return d >= 64 && d <= hi && d % 32 == 0; };
    return M >= 1 && M <= (1 << 28) && dim_ok(d_in, 65536) && dim_ok(d_out, 32768) && dim_ok(r, 65536);
}

inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Bytes of a bitmap re-laid for a product with N features and reduction
// length K: [2 ceil(K/128)][sign_rows(N)][2] u32 (pad blocks and rows are only
// ever multiplied by zero activations, or never stored).
inline size_t relaid_bytes(int N, int K) { return (size_t)((K + 127) / 128) * 2 * sign_rows(N) * 8; }

// Byte offsets of the workspace regions (256-byte aligned). The regions a
// forward pass uses come first (header .. c16, ending at fwd_total), then the
// backward's and the optional sign planes.
struct Layout {
    size_t header, bp_f1, bp_f2, x16, a32, al16, c16, stg_cnt, fwd_total;
    size_t bp_b1, bp_b2, dy16, db16, s_inv, sig, sig_inv, blkmax, part_dh, part_dl, part_dg, plane_u, plane_v, total;
    int rows_dh, rows_dl, rows_dg;
};

// Header words (u32 index): 0 the device status word; 16 the grid-barrier
// counter of the fused small-M kernels; 32 the arrival counter of the
// dx'-product's folded reduction (byte offsets below).
constexpr size_t kGridBarOffset = 64;
constexpr size_t kRedCntOffset = 128;


inline Layout make_layout(int M, int d_in, int d_out, int r) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align256(bytes);
        return o;
    };
    const size_t m = (size_t)M;
    L.header = take(256);
    // forward: re-laid S_V (N = r, K = d_in) and S_U (N = d_out, K = r), the
    // staged x, the a tape (f32), a.l (f16) and the c tape (f16)
    L.bp_f1 = take(relaid_bytes(r, d_in));
    L.bp_f2 = take(relaid_bytes(d_out, r));
    L.x16 = take(m * d_in * 2);
    L.a32 = take(m * r * 4);
    L.al16 = take(m * r * 2);
    L.c16 = take(m * d_out * 2);
    // row counters of the in-kernel x and dy staging: one per (token tile of
    // at least 32 tokens, column chunk of d_in or d_out)
    L.stg_cnt = take((size_t)stage_counters(M, 32, d_in > d_out ? d_in : d_out) * 4);
    L.fwd_total = off;
    // backward: re-laid S_U (N = r, K = d_out) and S_V (N = d_in, K = r); the
    // f16 staging of all four products stays in place after the pass (the
    // sign-gradient products read x16, dy16, al16 and db16 again)
    L.bp_b1 = take(relaid_bytes(r, d_out));
    L.bp_b2 = take(relaid_bytes(d_in, r));
    L.dy16 = take(m * d_out * 2);
    L.db16 = take(m * r * 2);
    L.s_inv = take(m * 4);
    L.sig = take(m * 4);
    L.sig_inv = take(m * 4);
    // dh partial rows: the prologue's blocks, or the converter warps of a
    // db-product that stages dy (kDyPartRowsPerCta per CTA)
    L.rows_dh = stage_dy_blocks(M, d_out);
    if (L.rows_dh < kDyPartRowsPerCta * kDyStageMaxCtas) L.rows_dh = kDyPartRowsPerCta * kDyStageMaxCtas;
    L.blkmax = take((size_t)L.rows_dh * 8);
    // partial rows per token tile (tiles of at least 128 tokens; split-K
    // db-products write one per quarter of K, the token-major dx'-product four
    // per 128-token tile)
    L.rows_dl = (int)((m + 127) / 128) * 4;
    L.rows_dg = (int)((m + 127) / 128) * 4;
    L.part_dh = take((size_t)L.rows_dh * d_out * 4);
    L.part_dl = take((size_t)L.rows_dl * r * 4);
    L.part_dg = take((size_t)L.rows_dg * d_in * 4);
    // +-1 f16 sign planes in the bitmaps' own [rows][r] order (plane-mode GEMMs)
    L.plane_u = take((size_t)d_out * r * 2);
    L.plane_v = take((size_t)d_in * r * 2);
    L.total = off;
    return L;
}

// Host-side failure injection for tests: true when the environment variable
// BLR_FAULT names `site` (the entry point then fails with BLR_ERR_CUDA without
// touching the GPU). Defined in blr_api.cu.
bool fault_injected(const char *site);

}  // namespace blr
