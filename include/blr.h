/*
 * blr.h - C ABI of the GB300 (sm_103a) binary low-rank linear layer.
 *
 * The layer (train_mm.rs, cortiq-engine 0.8.21, module documentation) is
 *
 *     W_hat = diag(h) . S_U . diag(l) . S_V^T . diag(g)
 *
 * with S_U [d_out x r] and S_V [d_in x r] sign matrices held as 1-bit bitmaps,
 * and g [d_in], l [r], h [d_out] f32 vectors. Its forward and backward passes
 * (same page, formula block) are
 *
 *     forward   a = (x.g) S_V         c = (a.l) S_U^T      y (+)= h.c
 *     backward  dh = sum_t dy.c       db = (dy.h) S_U      dl = sum_t a.db
 *               dx' = (db.l) S_V^T    dg = sum_t x.dx'     dx (+)= g.dx'
 *
 * where "." is the elementwise product broadcast along tokens and sum_t sums
 * over tokens.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layouts are row-major and unpadded: x, dx [M][d_in]; y, dy [M][d_out]
 *    f32. Token counts need not be multiples of anything; the library pads
 *    internally (the page pads activation rows to 128).
 *  - Sign bitmaps (train_mm.rs, comment of the `expand` kernel): bits_u is
 *    [d_out][ceil(r/32)] u32 and bits_v is [d_in][ceil(r/32)] u32; bit j of
 *    word w is rank 32w+j; a set bit is +1, a clear bit -1.
 *  - Every data pointer is a DEVICE pointer owned by the caller and must be
 *    16-byte aligned. The library never allocates, frees or synchronises on
 *    the hot path; work is queued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and returns before it runs.
 *  - Shape rule: M >= 1; d_in, d_out, r multiples of 32 and >= 64;
 *    d_out <= 32768 (one token row of dy is staged by one thread block);
 *    d_in, r <= 65536.
 *  - Numerics: operands are staged to f16 (round to nearest even), products
 *    accumulate in f32 on the tensor cores, outputs are f32. The forward
 *    stages x.g and a.l unscaled, so |x.g| and |a.l| must stay below 65504.
 *    The backward stages dy.h and db.l under powers of two (see
 *    blr_backward) that the epilogues divide back out exactly.
 *  - Return value: BLR_OK (0) or a negative BLR_ERR_* code. Argument errors
 *    are reported before anything is queued. Device-side failures (a bounded
 *    wait inside a kernel that ran out) do not fault the GPU: the kernel
 *    records a code in the workspace status word and returns; read it with
 *    blr_check_status().
 *  - Calls are thread-safe as long as concurrent calls use distinct
 *    workspaces.
 *  - The device must be compute capability 10.3 (GB300); there is no other
 *    code path and no CPU fallback.
 */
#ifndef BLR_H_
#define BLR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BLR_API __attribute__((visibility("default")))
#else
#define BLR_API
#endif

/* ABI-identical to cudaStream_t; declared here so that this header needs no
 * CUDA header. */
typedef struct CUstream_st *blr_stream_t;

enum {
    BLR_OK = 0,
    BLR_ERR_ARG = -1,                /* null pointer, bad flag, gscale not a power of two */
    BLR_ERR_SHAPE = -2,              /* shape rule violated */
    BLR_ERR_ALIGN = -3,              /* a pointer is not 16-byte aligned */
    BLR_ERR_WORKSPACE = -4,          /* ws_bytes < blr_workspace_bytes(...) */
    BLR_ERR_STATE = -5,              /* backward without a matching forward on this workspace */
    BLR_ERR_CUDA = -6,               /* a CUDA runtime/driver call or a launch failed */
    BLR_ERR_DEVICE_CHECK = -7,       /* a kernel recorded a failure in the status word */
    BLR_ERR_UNSUPPORTED_DEVICE = -8  /* current device is not compute capability 10.3 */
};

/* Bytes of caller-owned device workspace that one layer instance needs for a
 * forward+backward at this shape. The workspace holds the forward's tape (a in
 * f32 [M][r], c in f16 [M][d_out]) for the backward, the f16 staged operands,
 * the re-laid-out sign bitmaps, the per-tile partial sums of dh/dl/dg and a
 * 256-byte header whose first word is the device status. Returns 0 if the
 * shape breaks the shape rule. Pure host arithmetic; needs no GPU. */
BLR_API size_t blr_workspace_bytes(int M, int d_in, int d_out, int r);

/* The library remembers, per workspace address, what the last blr_forward
 * on it recorded there (its shape and input pointers), so that blr_backward
 * and blr_sign_grads can refuse a workspace that holds no matching tape. This
 * record is host memory only; call blr_workspace_release(ws) before freeing a
 * workspace to drop it (otherwise it is dropped when the library holds more
 * than 65536 records, oldest first). Never touches the GPU.
 * Errors: BLR_ERR_ARG for a null pointer. */
BLR_API int blr_workspace_release(const void *ws);

/* Pack signs into a bitmap (train_mm.rs, test helper `pack_bits`).
 *   src  [rows][r] f32, device.
 *   bits [rows][ceil(r/32)] u32, device, written in full: bit (row, k) is 1
 *        iff src[row][k] > 0 (so 0, -0 and NaN give -1); unused high bits of
 *        the last word are 0.
 * rows >= 1, r >= 1. Bit-exact. */
BLR_API int blr_pack_signs(const float *src, uint32_t *bits, int rows, int r, blr_stream_t stream);

/* Expand a bitmap into +-1 f16 (train_mm.rs, `expand` kernel), through the
 * same device expansion code the GEMMs use for their shared-memory operand
 * tiles. For tests: the GEMMs never write dense planes.
 *   bits [rows][ceil(r/32)] u32, device.
 *   dst  [rows][r] f16 bit patterns (0x3C00 = +1, 0xBC00 = -1), device.
 * rows >= 1, r >= 1. Bit-exact. */
BLR_API int blr_unpack_signs(const uint32_t *bits, uint16_t *dst, int rows, int r, blr_stream_t stream);

/* Forward pass (train_mm.rs, `blr_forward` and the formula block).
 *   x [M][d_in] f32 in; bits_u [d_out][ceil(r/32)], bits_v [d_in][ceil(r/32)];
 *   g [d_in], l [r], h [d_out] f32 in.
 *   y [M][d_out] f32 out: y = h.c when accumulate_y == 0 (the page's first
 *     path), y += h.c when accumulate_y == 1 (its later paths).
 *   ws / ws_bytes: workspace of at least blr_workspace_bytes(M, d_in, d_out, r)
 *     bytes; it receives the tape that blr_backward consumes, so it must not
 *     be shared with another layer between the forward and its backward.
 * Errors: BLR_ERR_ARG (null pointer, accumulate_y not 0/1), BLR_ERR_SHAPE,
 *   BLR_ERR_ALIGN, BLR_ERR_WORKSPACE, BLR_ERR_UNSUPPORTED_DEVICE, BLR_ERR_CUDA. */
BLR_API int blr_forward(const float *x, const uint32_t *bits_u, const uint32_t *bits_v,
                const float *g, const float *l, const float *h,
                float *y, int accumulate_y,
                int M, int d_in, int d_out, int r,
                void *ws, size_t ws_bytes, blr_stream_t stream);

/* Backward pass (train_mm.rs, `blr_backward` and the formula block). Must
 * follow blr_forward on the same workspace, shape, x and parameters.
 *   x [M][d_in], dy [M][d_out] f32 in; bitmaps and g, l, h as in the forward.
 *   dx [M][d_in] f32 out: dx = g.dx' (accumulate_dx == 0) or dx += g.dx' (1).
 *   dg [d_in], dl [r], dh [d_out] f32: ALWAYS accumulated (+=), like the
 *     page's column sums, in a fixed order (deterministic).
 *   gscale > 0: the page's semantics: dy.h and db.l are staged times gscale,
 *     which must be a power of two.
 *   gscale <= 0: dynamic per-token powers of two: token t's dy.h is staged
 *     times s_t = 2^(14 - ceil(log2 max_i |dy_ti h_i|)), and its db.l times
 *     the largest power of two that keeps the L1 bound of db_t.l under 2^15,
 *     which keeps gradients out of the f16 subnormals and never overflows.
 * Errors: as blr_forward, plus BLR_ERR_STATE when the last forward on `ws`
 *   was not of this shape or did not take these same x, bits_u, bits_v, g,
 *   l and h pointers (or there was none, or blr_workspace_release forgot
 *   it), and BLR_ERR_ARG when gscale is positive but not a power of two. */
BLR_API int blr_backward(const float *x, const float *dy,
                 const uint32_t *bits_u, const uint32_t *bits_v,
                 const float *g, const float *l, const float *h,
                 float *dx, int accumulate_dx,
                 float *dg, float *dl, float *dh,
                 float gscale,
                 int M, int d_in, int d_out, int r,
                 void *ws, size_t ws_bytes, blr_stream_t stream);

/* Multi-path layers (train_mm.rs, Blr: y = sum_p W_hat_p x over P paths of
 * the same shape; blr_forward / blr_backward loop over the paths, path 0
 * overwriting y and dx and later paths adding, each path with its own
 * bitmaps, g, l, h and gradients dg, dl, dh).
 *
 * blr_paths_workspace_bytes: P single-path workspaces side by side; path p's
 * slice starts at p * blr_workspace_bytes(M, d_in, d_out, r) (a multiple of
 * 256) and holds that path's tape, so blr_sign_grads(..., ws + offset_p, ...)
 * gives path p's sign gradients after blr_backward_paths.
 *
 * blr_forward_paths / blr_backward_paths take host arrays of P device
 * pointers (bits_u[p], ..., dg[p]) and queue the pass on `stream` with one
 * launch per stage for up to 8 paths at a time: one prologue (each path's
 * bitmap re-layouts and staging), one launch of each product covering every
 * path's tiles, one reduction of every path's partial sums. Path 0 overwrites
 * y and dx and each later path adds its contribution, in path order, tile by
 * tile (accumulate_y/accumulate_dx = 1 makes path 0 add too); the sums are
 * the same as from P single-path calls. More than 8 paths run as groups of 8
 * in turn. With BLR_PATHS=loop in the environment, or an option that has no
 * grouped form (BLR_SMALL_PATH=fused, BLR_SIGN_SRC=plane, BLR_WIDE=token,
 * BLR_SPLITK=1), each path's single-path calls run in turn instead. A
 * grouped launch records device-side failures in path 0's status word (the
 * first slice's header). Every argument is checked before the first launch,
 * so an argument error changes nothing; a launch failure part way leaves
 * the earlier groups' results in place. P in [1, 64]; the rest as
 * blr_forward / blr_backward. */
BLR_API size_t blr_paths_workspace_bytes(int P, int M, int d_in, int d_out, int r);
BLR_API int blr_forward_paths(const float *x, int P,
                              const uint32_t *const *bits_u, const uint32_t *const *bits_v,
                              const float *const *g, const float *const *l, const float *const *h,
                              float *y, int accumulate_y, int M, int d_in, int d_out, int r,
                              void *ws, size_t ws_bytes, blr_stream_t stream);
BLR_API int blr_backward_paths(const float *x, const float *dy, int P,
                               const uint32_t *const *bits_u, const uint32_t *const *bits_v,
                               const float *const *g, const float *const *l, const float *const *h,
                               float *dx, int accumulate_dx,
                               float *const *dg, float *const *dl, float *const *dh,
                               float gscale, int M, int d_in, int d_out, int r,
                               void *ws, size_t ws_bytes, blr_stream_t stream);

/* Bytes of the second workspace blr_sign_grads needs for this shape (0 when
 * the shape violates the shape rule): the rank-side f16 operands rescaled to
 * one gradient scale, 4*M*r bytes plus a 256-byte header. */
BLR_API size_t blr_sign_workspace_bytes(int M, int d_in, int d_out, int r);

/* Sign gradients of the layer (train_mm.rs, blr_backward documentation, and
 * its test helper host_sign_grads):
 *
 *     G_U = diag(h) . dy^T . a . diag(l)      gu [d_out][r] f32
 *     G_V = diag(g) . x^T  . b . diag(l)      gv [d_in][r]  f32
 *
 * with a = (x.g) S_V the forward's product and b = (dy.h) S_U the backward's
 * db. With L = <dy, y> these are dL/dS_U and dL/dS_V. The pages form them
 * inside the backward ("with sign"); here they are a separate call after
 * blr_backward on the same workspace `ws`, whose tape it reads: a (forward),
 * and the backward's staged f16 dy.h and db.l with their per-token powers of
 * two. So dy, h and the bitmaps are not arguments; x, g and l must hold the
 * values of that forward/backward pair (the products read only the staging
 * in `ws`, so other buffers with those values serve as well).
 *  - Operands: the pass's own f16 staging, token-major as it is (the tensor
 *    cores read it as MN-major tiles; nothing is transposed): dy.h with x.g
 *    on the feature side, a.l and db.l on the rank side. With a fixed
 *    gscale every token shares one scale and the products are divided by
 *    it. With dynamic per-token scales, a.l and db.l are first rescaled
 *    into `sws` (caller-owned, blr_sign_workspace_bytes(...) bytes,
 *    16-byte aligned) by 1/s_t / max_t(1/s_t) and 1/sigma_t /
 *    max_t(1/sigma_t), over the tokens with a nonzero gradient: powers of
 *    two <= 1, exact unless a value falls into the f16 subnormals (tokens
 *    whose gradient is far below the largest). The products accumulate in
 *    f32 on the tensor cores and the common scales are divided back out.
 *  - accumulate = 0 overwrites gu and gv, 1 adds to them.
 * Errors: as blr_backward; BLR_ERR_STATE when no blr_backward of this shape
 *   has run on `ws` since its last blr_forward; BLR_ERR_WORKSPACE when
 *   ws_bytes or sws_bytes is short. Kernel-side failures go to the status
 *   word of `ws` (blr_check_status). */
BLR_API int blr_sign_grads(const float *x, const float *g, const float *l,
                           float *gu, float *gv, int accumulate,
                           int M, int d_in, int d_out, int r,
                           const void *ws, size_t ws_bytes, void *sws, size_t sws_bytes,
                           blr_stream_t stream);

/* Bytes of the workspace blr_plane_linear needs (0 when the shape violates
 * its rule): a 256-byte header (word 0: device status) and the f16 staging
 * of x, ntok * max(n, k) * 2 bytes. */
BLR_API size_t blr_plane_workspace_bytes(int ntok, int n, int k);

/* A dense frozen f16 linear (train_mm.rs, plane_linear and mm):
 *
 *   transpose = 0:  y [ntok][n] (+)= (f16(x * scale) . plane^T) / scale,  x [ntok][k]
 *   transpose = 1:  y [ntok][k] (+)= (f16(x * scale) . plane)   / scale,  x [ntok][n]
 *
 * plane [n][k] f16 (IEEE binary16 bits, row-major) is the same array in both
 * directions: the transpose (the input gradient through the plane) reads it
 * as MN-major tiles, nothing is transposed in memory. x is staged once into
 * `ws` as f16(x * scale), round to nearest even; the product accumulates in
 * f32 on the tensor cores and is multiplied by 1/scale.
 *  - scale: a positive power of two (the page's caller-chosen scale, 1 for a
 *    forward, a gradient scale for the input gradient); |x * scale| must stay
 *    below 65504 (f16 range), and values below 2^-14 lose precision.
 *  - accumulate = 0 overwrites y, 1 adds to it.
 *  - Shape rule: ntok >= 1; n and k multiples of 32 in [32, 65536].
 *  - All pointers device, caller-owned, 16-byte aligned.
 * Errors: BLR_ERR_ARG (null pointer, flag not 0/1, scale not a positive power
 *   of two), BLR_ERR_SHAPE, BLR_ERR_ALIGN, BLR_ERR_WORKSPACE,
 *   BLR_ERR_UNSUPPORTED_DEVICE, BLR_ERR_CUDA; kernel-side failures go to the
 *   status word of `ws` (blr_check_status). */
BLR_API int blr_plane_linear(const float *x, const uint16_t *plane, float *y,
                             int transpose, int accumulate, float scale,
                             int ntok, int n, int k,
                             void *ws, size_t ws_bytes, blr_stream_t stream);

/* One Adam step over n parameters (train_mm.rs, WGSL adam kernel and its
 * wrapper adam), meant for the layer's vectors g, l and h (for instance kept
 * as one contiguous [d_in + r + d_out] array with its gradient dg | dl | dh):
 *
 *     gr = grad * gmul
 *     m1 = b1 m1 + (1 - b1) gr,   m2 = b2 m2 + (1 - b2) gr^2
 *     st = lr (m1 / (1 - b1^step)) / (sqrt(m2 / (1 - b2^step)) + eps)
 *     w -= st * max(|w|, rel)   if rel > 0 (steps relative to |w|, floored at rel)
 *     w -= st                   otherwise
 *
 * f32 arithmetic as on the page; the bias corrections are formed on the host.
 *  - w, m1, m2 [n] f32 device, updated in place; grad [n] f32 device;
 *    mask [n] f32 device or NULL: entries with mask exactly 0 are frozen (w,
 *    m1 and m2 unchanged). No weight decay. step >= 1 counts updates from 1.
 *  - Pointers need 4-byte alignment; n = 0 is a no-op.
 * Errors: BLR_ERR_ARG (null pointer, step < 1, b1 or b2 outside [0, 1), eps
 *   negative or not finite, lr or gmul not finite, rel NaN), BLR_ERR_SHAPE
 *   (n < 0), BLR_ERR_ALIGN, BLR_ERR_UNSUPPORTED_DEVICE, BLR_ERR_CUDA. */
BLR_API int blr_adam(float *w, const float *grad, float *m1, float *m2, const float *mask,
                     int n, int step, float lr, float b1, float b2, float eps,
                     float gmul, float rel, blr_stream_t stream);

/* Synchronises `stream` and reads the workspace's device status word.
 * Returns BLR_OK if no kernel recorded a failure since the last blr_forward
 * on this workspace, BLR_ERR_DEVICE_CHECK if one did (the code is written to
 * *device_code when it is not NULL), BLR_ERR_CUDA if the stream reports an
 * error. This call blocks; it is meant for tests and diagnostics.
 * Bits of the device code (each names the wait that ran out):
 *   0x01 a product's operand loader (a ring slot never freed),
 *   0x02 a sign expander, 0x04 an MMA issuer, 0x08 an epilogue,
 *   0x10 the drain of copies or MMAs at a kernel's end,
 *   0x20 a launch geometry the kernel does not accept,
 *   0x40 a grid barrier (of the fused small-problem kernels, or before the
 *        dx'-product's reduction of the partial sums),
 *   0x80 a streaming staging kernel (a row batch never arrived or its ring
 *        slot never freed). */
BLR_API int blr_check_status(const void *ws, size_t ws_bytes, blr_stream_t stream, uint32_t *device_code);

/* Static description of a status code. Never NULL. */
BLR_API const char *blr_status_string(int status);

/* Kernel-level timing for benchmarks. blr_trace_begin(capacity) makes every
 * following blr_forward/blr_backward on this thread bracket each kernel it
 * launches with a pair of CUDA events recorded on the launch stream, up to
 * `capacity` kernels; blr_trace_end() stops recording. blr_trace_count()
 * returns the number of kernels recorded; blr_trace_read(i, &ms) synchronises
 * on kernel i's end event and returns its name, with its duration in
 * milliseconds in *ms (NULL if i is out of range). The events are created
 * once, on the first blr_trace_begin. Calls made while their stream is being
 * captured into a CUDA graph put the events into the graph as event-record
 * nodes: each replay records them again, and blr_trace_read after a replay
 * reads that replay's durations (the kernel before and after such a node run
 * without programmatic overlap). Off by default; no effect on results. */
BLR_API int blr_trace_begin(int capacity);
BLR_API int blr_trace_end(void);
BLR_API int blr_trace_count(void);
BLR_API const char *blr_trace_read(int i, float *ms);

/* Size in bytes of the fixed scratch array behind blr_forward_noalloc. */
#define BLR_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Forward pass for callers that cannot allocate device memory. The pages have
 * no counterpart: this is a library convenience. Some callers cannot call
 * cudaMalloc or any allocator, for instance a plugin inside a host application
 * that owns every device allocation, or a real-time inference loop with a
 * fixed memory budget, so they cannot provide blr_forward's workspace.
 * Arguments, layouts and results are those of blr_forward without `ws`: the
 * scratch is a fixed array of BLR_NOALLOC_SCRATCH_BYTES in the library's own
 * device memory, held by every GPU that loads the library until exit. No
 * allocation happens in this call.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - All calls share the one array, which keeps the last call's contents; the
 *    kernels clear what must start at zero. Calls that overlap on the GPU
 *    (other streams, other threads) race on the array: serialise them.
 *  - The tape it leaves is not usable by blr_backward.
 *  - Device-side failures (a bounded wait inside a kernel that ran out) are
 *    recorded in the array's own status word, which the next call clears:
 *    read it with blr_noalloc_check_status before that call.
 * Errors: as blr_forward (BLR_ERR_SHAPE, BLR_ERR_ARG, BLR_ERR_ALIGN,
 *   BLR_ERR_UNSUPPORTED_DEVICE, BLR_ERR_CUDA); BLR_ERR_WORKSPACE when the
 *   shape needs more scratch than BLR_NOALLOC_SCRATCH_BYTES (roughly
 *   M*(2 d_in + 6 r + 2 d_out) bytes plus the re-laid bitmaps). */
BLR_API int blr_forward_noalloc(const float *x, const uint32_t *bits_u, const uint32_t *bits_v,
                                const float *g, const float *l, const float *h,
                                float *y, int accumulate_y,
                                int M, int d_in, int d_out, int r, blr_stream_t stream);

/* Synchronises `stream` and reads the status word of the current device's
 * blr_forward_noalloc scratch array (the counterpart of blr_check_status for
 * the entry point that has no caller workspace; the pages have none either).
 * Returns BLR_OK when the last blr_forward_noalloc on this device recorded
 * no failure, BLR_ERR_DEVICE_CHECK when it did (code in *device_code when not
 * NULL, bits as for blr_check_status), BLR_ERR_STATE when no
 * blr_forward_noalloc has run on this device yet, BLR_ERR_CUDA on a CUDA
 * error. It copies 4 bytes to the host; it allocates nothing. Blocking; for
 * tests and diagnostics. */
BLR_API int blr_noalloc_check_status(blr_stream_t stream, uint32_t *device_code);

#ifdef __cplusplus
}
#endif

#endif /* BLR_H_ */
