// Host side of the blr C ABI (include/blr.h): argument and shape checks,
// workspace layout, TMA descriptors, GEMM tile choice and the launch sequence
// of the forward and backward passes on the caller's stream.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "../../include/blr.h"
#include "blr_kernels.h"
#include "blr_layout.h"

namespace blr {
cudaError_t launch_gemm_fwd(int epi, const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args,
                            cudaStream_t s);
cudaError_t launch_gemm_bwd(int epi, const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args,
                            cudaStream_t s);

// ------------------------------------------------------------ tracing ------
namespace {
struct TraceState {
    bool on = false;
    int cap = 0;
    int n = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<const char *> names;
};
thread_local TraceState g_trace;
}  // namespace

// A trace event on a stream that is being captured into a CUDA graph becomes
// an event-record node of the graph (recorded at each replay), so that the
// kernels of a replayed step can be timed one by one.
static void trace_record(cudaEvent_t e, cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, stream, cudaEventRecordExternal);
    else
        cudaEventRecord(e, stream);
}

void trace_before(const char *name, cudaStream_t stream) {
    TraceState &t = g_trace;
    if (!t.on || t.n >= t.cap) return;
    t.names[t.n] = name;
    trace_record(t.ev[2 * t.n], stream);
}

void trace_after(cudaStream_t stream) {
    TraceState &t = g_trace;
    if (!t.on || t.n >= t.cap) return;
    trace_record(t.ev[2 * t.n + 1], stream);
    ++t.n;
}

cudaError_t launch_gemm_stg_fwd(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s);
cudaError_t launch_gemm_stg_bwd(const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s);

cudaError_t launch_gemm(int epi, const GemmPlan &plan, const GemmMaps &maps, const GemmArgs &args, cudaStream_t s) {
    static const char *names[4] = {"gemm_fwd1", "gemm_fwd2", "gemm_bwd1", "gemm_bwd2"};
    if (plan.stg) {
        // the a-product with x, or the db-product with dy, staged in the kernel
        const bool fwd = plan.stg == 1 && epi == kEpiFwd1, bwd = plan.stg == 2 && epi == kEpiBwd1;
        if (!fwd && !bwd) return cudaErrorInvalidValue;
        trace_before(fwd ? "gemm_fwd1s" : "gemm_bwd1s", s);
        cudaError_t e = fwd ? launch_gemm_stg_fwd(plan, maps, args, s) : launch_gemm_stg_bwd(plan, maps, args, s);
        trace_after(s);
        return e;
    }
    trace_before(names[epi & 3], s);
    cudaError_t e = (epi == kEpiFwd1 || epi == kEpiFwd2) ? launch_gemm_fwd(epi, plan, maps, args, s)
                                                          : launch_gemm_bwd(epi, plan, maps, args, s);
    trace_after(s);
    return e;
}

// ------------------------------------------------------- device checks ------
namespace {
struct DevInfo {
    bool init = false;
    bool supported = false;
    int sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

int device_info(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BLR_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.init) {
        int maj = 0, min = 0, n = 0;
        if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BLR_ERR_CUDA;
        d.supported = (maj == 10 && min == 3);
        d.sms = n;
        d.init = true;
    }
    if (!d.supported) return BLR_ERR_UNSUPPORTED_DEVICE;
    *sms = d.sms;
    return BLR_OK;
}

// ------------------------------------------------------------- TMA ---------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// f16 activation operand [rows][K], box 64 (K) x box_rows, 128-byte swizzle;
// rows past `rows` and columns past K read as zero.
bool make_tmap_act16(CUtensorMap *m, const void *base, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Maps of the layer GEMMs (blr_gemm.cuh), 3-D: [planes][rows][cols] with
// plane p `pstride` bytes after plane 0, one plane per path of a multi-path
// launch (planes = 1 for a single path and for the tensors the paths share).
// act: f16 activation operand, box 64 x box_rows, 128-byte swizzle, rows and
// columns past the extent read zero. chunk: f32 or f16 epilogue chunks, box
// 32 x 32, no swizzle; loads read zeros out of range, stores are clipped.
bool make_gmap(CUtensorMap *m, const void *base, int rows, int cols, bool f16, int box_cols, int box_rows,
               CUtensorMapSwizzle sw, int planes, long long pstride) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || planes < 1) return false;
    const cuuint64_t esz = f16 ? 2 : 4;
    const cuuint64_t plane_bytes = ((cuuint64_t)rows * cols * esz + 15) / 16 * 16;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)cols * esz, planes > 1 ? (cuuint64_t)pstride : plane_bytes};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_gmap_act(CUtensorMap *m, const void *base, int rows, int K, int box_rows, int planes = 1,
                   long long pstride = 0) {
    return make_gmap(m, base, rows, K, true, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B, planes, pstride);
}
bool make_gmap_chunk(CUtensorMap *m, const void *base, int rows, int cols, bool f16, int planes = 1,
                     long long pstride = 0) {
    return make_gmap(m, base, rows, cols, f16, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE, planes, pstride);
}

// x f32 [rows][cols] with a 256 x box_rows box, no swizzle: the in-kernel x
// staging's ring units (16 rows) and L2 prefetches (64 rows); rows and
// columns past the extent read zero.
bool make_tmap_x_stage(CUtensorMap *m, const void *base, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {(cuuint32_t)kStageChunkCols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The c tape [rows][cols] f16 in 256-column boxes of box_rows rows, no
// swizzle: the db-product's dy stagers read it beside dy for the dh sums.
bool make_tmap_c_stage(CUtensorMap *m, const void *base, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kStageChunkCols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][cols] f32 or f16 with a 32 x 32 box, no swizzle: the epilogue's
// chunks (32 tokens x 32 features); loads read zeros out of range and stores
// are clipped to it.
bool make_tmap_chunk(CUtensorMap *m, const void *base, int rows, int cols, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t esz = f16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][cols] f32 with a 32 x 32 box and 128-byte swizzle (the sign
// gradients' output chunks); stores are clipped to the extent.
bool make_tmap_out_sw128(CUtensorMap *m, void *base, int rows, int cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][cols] f16 with a 32 x 32 box and 64-byte swizzle (c from the
// token-major c-product); stores are clipped to the extent.
bool make_tmap_out16_sw64(CUtensorMap *m, void *base, int rows, int cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ layout --------
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Second workspace of blr_sign_grads: header (the two scale maxima), then the
// rank-side operands rescaled to one gradient scale, bu and bv [M][r] f16.
struct SignLayout {
    size_t header, bu, bv, total;
};

SignLayout make_sign_layout(int M, int r) {
    SignLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align_up(bytes, 256);
        return o;
    };
    L.header = take(256);
    L.bu = take((size_t)M * r * 2);
    L.bv = take((size_t)M * r * 2);
    L.total = off;
    return L;
}

// ------------------------------------------------------------ tape ---------
// What the last forward on a workspace recorded there, keyed by the workspace
// pointer: its shape and the device pointers of its inputs. A backward (and
// the sign gradients) must name the same x and parameters as that forward,
// so that a workspace whose address was freed and handed out again for
// another layer of the same shape cannot pass with a stale tape.
struct Tape {
    int M, d_in, d_out, r;
    const void *x, *bits_u, *bits_v, *g, *l, *h;  // the forward's inputs
    unsigned long long gen;  // forward counter when recorded (oldest first out when the registry is full)
    bool backward_done;  // a blr_backward has run on this tape (its staged dy and db are in the workspace)
    float gscale;        // that backward's gradient scale (<= 0: dynamic per-token scales)
    int stage_blocks;    // its staging blocks (entries of the per-block scale maxima)
};
std::mutex g_tape_mu;
std::unordered_map<const void *, Tape> g_tapes;
unsigned long long g_tape_gen = 0;
// Registry bound: beyond this many live workspaces the oldest record is
// dropped (its backward then fails with BLR_ERR_STATE).
constexpr size_t kMaxTapes = 1u << 16;

void record_tape(const void *ws, Tape t) {
    std::lock_guard<std::mutex> lk(g_tape_mu);
    t.gen = ++g_tape_gen;
    g_tapes[ws] = t;
    if (g_tapes.size() > kMaxTapes) {
        auto oldest = g_tapes.begin();
        for (auto it = g_tapes.begin(); it != g_tapes.end(); ++it)
            if (it->second.gen < oldest->second.gen) oldest = it;
        g_tapes.erase(oldest);
    }
}

// The tape of `ws` if it was recorded by a forward of this shape on these inputs.
bool tape_matches(const void *ws, int M, int d_in, int d_out, int r, const void *x, const void *bits_u,
                  const void *bits_v, const void *g, const void *l, const void *h) {
    std::lock_guard<std::mutex> lk(g_tape_mu);
    auto it = g_tapes.find(ws);
    if (it == g_tapes.end()) return false;
    const Tape &t = it->second;
    if (t.M != M || t.d_in != d_in || t.d_out != d_out || t.r != r) return false;
    if (t.x != x || t.g != g || t.l != l) return false;
    return t.bits_u == bits_u && t.bits_v == bits_v && t.h == h;
}

void mark_backward_done(const void *ws, float gscale, int stage_blocks) {
    std::lock_guard<std::mutex> lk(g_tape_mu);
    auto it = g_tapes.find(ws);
    if (it == g_tapes.end()) return;
    it->second.backward_done = true;
    it->second.gscale = gscale;
    it->second.stage_blocks = stage_blocks;
}

bool plane_shape_ok(int ntok, int n, int k) {
    auto dim_ok = [](int d) { return d >= 32 && d <= 65536 && d % 32 == 0; };
    return ntok >= 1 && ntok <= (1 << 28) && dim_ok(n) && dim_ok(k);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_positive(float v) {
    if (!(v > 0.0f) || !std::isfinite(v)) return false;
    int e;
    return std::frexp(v, &e) == 0.5f;
}
}  // namespace

bool fault_injected(const char *site) {
    const char *f = std::getenv("BLR_FAULT");
    return f && std::strcmp(f, site) == 0;
}
}  // namespace blr

namespace blr {

// Tiles of 128 features (256 for a CTA pair) x BT tokens. CTA pairs whenever
// there are at least as many pair tiles as pairs of SMs, with the token tile
// (160 or 192: MMAs of N >= 160 run at full rate) that needs the fewest
// token-rounds of the persistent grid; otherwise single CTAs with 128-token
// tiles, for more tiles in flight on small problems.
// `paths` > 1 plans a grouped launch whose units share the tiles of that many
// paths (the a- and db-products: tiles x paths in all).
GemmPlan plan_gemm(int M, int N, int sms, int min_bt, int tile_cost, int paths) {
    const int pairs = sms / 2;
    const long long fp = (N + 255) / 256 * paths;
    GemmPlan best{false, 0, 0, 0};
    long long best_cost = 0;
    for (int bt : {192, 160}) {
        const long long t_tiles = (M + bt - 1) / bt;
        const long long tiles = t_tiles * fp;
        if (tiles < pairs) continue;
        // rounds x (a tile's fixed cost + its time per token), in tokens
        const long long cost = ((tiles + pairs - 1) / pairs) * (bt + tile_cost);
        if (best.bt == 0 || cost < best_cost) {
            best = GemmPlan{true, bt, 2 * pairs, (int)t_tiles};
            best_cost = cost;
        }
    }
    if (best.bt != 0) return best;
    // few tiles: halving the token tile (down to min_bt) while the tiles fill
    // at most half the SMs puts more SMs to work (a tile's time is set by its
    // k-loop's latency at these sizes, not by its MMA time); BLR_GEMM_BT=128
    // keeps 128-token tiles
    const char *v = std::getenv("BLR_GEMM_BT");
    if (v && std::strcmp(v, "128") == 0) min_bt = 128;
    const long long fs = (N + 127) / 128 * paths;
    int bt = 128;
    while (bt > min_bt && 2 * ((M + bt - 1) / bt) * fs <= sms && M > bt / 2) bt /= 2;
    const long long t_tiles = (M + bt - 1) / bt;
    const long long tiles = t_tiles * fs;
    return GemmPlan{false, bt, (int)(tiles < sms ? tiles : sms), (int)t_tiles};
}

// Plane-mode tiles: CTA pairs of 256 features x 256 tokens (each CTA loads
// half the tokens, which halves the activation bytes a k-step brings per SM)
// when there are at least as many pair tiles as pairs of SMs, single CTAs of
// 128 x 128 otherwise. Measured on GB300, 256 tokens beat 192 and 160 on every
// workload although they leave more of the last round idle.
GemmPlan plan_gemm_plane(int M, int N, int sms) {
    const int pairs = sms / 2;
    const long long t_tiles = (M + 255) / 256;
    const long long tiles = t_tiles * ((N + 255) / 256);
    if (tiles >= pairs) return GemmPlan{true, 256, 2 * pairs, (int)t_tiles, true};
    const long long s_tiles = (M + 127) / 128;
    const long long stiles = s_tiles * ((N + 127) / 128);
    return GemmPlan{false, 128, (int)(stiles < sms ? stiles : sms), (int)s_tiles, true};
}

// Where the general path's GEMMs take the sign operand from: bitmap words
// expanded into TMEM (default), or +-1 f16 planes read by TMA when
// BLR_SIGN_SRC=plane. Measured on GB300: kernel by kernel (serialised, event
// trace) the planes win every product of the passes whose widths are both at
// most 4096 (attention-sized layer: 12 us of 395) and lose on 12288- and
// 32768-wide ones; but timed as CUDA-graph replays, where consecutive kernels
// overlap their setup and tails, the attention-sized step took 393 us with
// planes against 381 with the TMEM expansion, and the small one 62.4 both ways.
bool plane_mode() {
    const char *v = std::getenv("BLR_SIGN_SRC");
    return v && std::strcmp(v, "plane") == 0;
}

// The wide products (c: d_out outputs, dx': d_in outputs, K = r) run
// feature-major on the sign GEMM (one thread per feature), or, with
// BLR_WIDE=token, token-major on the dense tensor-core kernel (rows = tokens,
// the sign plane as B: a thread owns a token row and writes it in 16-byte
// pieces, h and g are per-column broadcasts, sigma_t a per-thread scalar, dg a
// warp transpose-sum). Measured on GB300 the token-major form is slower on
// every workload (attention-sized dx': 105 against 70 us; its epilogue keeps
// one chunk of x in flight per warp, about 16 KB per SM, where the
// feature-major one prefetches 64 KB), so it is not the default.
bool wide_token_major() {
    const char *v = std::getenv("BLR_WIDE");
    return v && std::strcmp(v, "token") == 0;
}

// Split-K for the r-wide products (a and db, K = d_in or d_out) of problems
// whose single-CTA tiles fill at most a quarter of the SMs: clusters of four
// CTAs share each tile's k-steps (each at least one) and reduce over DSMEM.
// Opt-in (BLR_SPLITK=1): measured on GB300 on the small layer (2048 tokens,
// 1024 -> 1024, r = 256) the a-product took 18.4 us split against 12.2 us
// whole, the db-product 20.4 against 14.2; a 32-CTA tile of 8 k-steps is
// dominated by fixed costs (the first loads' round trip, setup, the epilogue's
// first chunk), which the cluster launch, staging and two cluster barriers add to.
GemmPlan plan_split(GemmPlan p, int M, int N, int K, int sms) {
    const char *v = std::getenv("BLR_SPLITK");
    if (!(v && std::strcmp(v, "1") == 0)) return p;
    if (p.pair || p.plane) return p;
    const long long t_tiles = (M + 127) / 128;
    const long long tiles = t_tiles * ((N + 127) / 128);
    if (tiles * 4 > sms || (K + 127) / 128 < 4) return p;
    return GemmPlan{false, 128, (int)(tiles * 4), (int)t_tiles, false, 4};
}

// Grid of the fused small-M kernels: enough CTAs for the larger GEMM phase's
// tiles (at least 16, for the staging phases), at most one per SM.
int small_grid(const GemmPlan &p1, int N1, const GemmPlan &p2, int N2, int M, int sms) {
    const int t = (M + 127) / 128;
    int tiles = t * ((N1 + 127) / 128);
    const int t2 = t * ((N2 + 127) / 128);
    if (t2 > tiles) tiles = t2;
    if (tiles < 16) tiles = 16;
    (void)p1;
    (void)p2;
    return tiles < sms ? tiles : sms;
}

// The fused small-M kernels (blr_small.cu) are used for small problems only
// when BLR_SMALL_PATH=fused is set: measured on GB300 they match the
// stand-alone kernels on per-kernel time but lose under CUDA-graph replay,
// where the stand-alone kernels overlap each other's setup and tails.
bool fused_small_enabled() {
    const char *v = std::getenv("BLR_SMALL_PATH");
    return v && std::strcmp(v, "fused") == 0;
}

// Where the a-product's activation operand x16 is staged: inside the
// product's kernel by its stager warps for x of 64 MB or more, by a
// stand-alone pass before it otherwise. Measured on GB300 (CUDA-graph steps):
// in the kernel, the 12288 -> 4096 MLP layer's pass and a-product take 357
// against 460 us, the attention-sized layer's 78 against 106; for the small
// layer (8 MB of x) the pass keeps its bitmap re-layouts hidden behind the
// staging and the step is 50.6 against 54.0 us. BLR_STAGE=kernel or
// BLR_STAGE=pass forces a form.
// Where the backward's partial sums of dh, dl and dg are reduced: by a launch
// of its own after the dx'-product (default), or in the dx'-product's tail
// with BLR_REDUCE=fold (its CTAs meet at a grid barrier and share out the
// columns; not for the token-major dx'-product). Measured on GB300 (CUDA-graph
// steps), the folded form is slower everywhere: tiny 33.7 against 30.4 us,
// small 54.8 against 52.6, attention-sized 349.6 against 344.8, the MLP pair
// 2241 against 2197 (the 12288 -> 4096 dx'-product grows from 343 to 371 us
// where the stand-alone reduction takes 11): the reduction starts only when
// the slowest CTA arrives and runs on the product's 14 warps per CTA.
bool reduce_folded() {
    const char *v = std::getenv("BLR_REDUCE");
    return v && std::strcmp(v, "fold") == 0;
}

bool stage_in_kernel(long long x_bytes) {
    const char *v = std::getenv("BLR_STAGE");
    if (v && std::strcmp(v, "pass") == 0) return false;
    if (v && std::strcmp(v, "kernel") == 0) return true;
    return x_bytes >= (64ll << 20);
}

// dy16 staged inside the db-product (after a scale pass) with
// BLR_DY_STAGE=kernel, wherever the db-product runs CTA-pair tiles of one
// path; by the backward prologue otherwise (the default). Measured on GB300:
// the 12288-wide MLP layer's scale pass, staged db-product and reduction take
// 146 + 401 + 16 us against 307 + 264 + 12 for the prologue form, but the
// CUDA-graph step of the MLP pair is no faster (2.207 ms at 1995 MHz against
// 2.189 at 2010); at 4096-wide rows the prologue form is faster outright
// (attention-sized 35 + 96 against 61 + 65 us).
bool dy_stage_in_kernel() {
    const char *v = std::getenv("BLR_DY_STAGE");
    return v && std::strcmp(v, "kernel") == 0;
}

// Grid barriers of the fused small-M kernels and of the dx'-product's folded
// reduction. Their waits give up after 2 s (BLR_WAIT_LIMIT_NS=<ns> sets
// another limit, from 1 us to 10 s). For the test of that path,
// BLR_FAULT=grid_barrier makes every barrier expect one arrival more than the
// grid makes, so each wait runs out: the kernels then record kStTimeoutGrid
// in the status word, leave their remaining work early and return (their
// results are then meaningless).
GridBarrier grid_barrier(unsigned int *gbar) {
    GridBarrier b{gbar, 0u, 2000000000ull};
    if (const char *v = std::getenv("BLR_WAIT_LIMIT_NS")) {
        const long long ns = std::atoll(v);
        if (ns >= 1000 && ns <= 10000000000ll) b.wait_ns = (unsigned long long)ns;
    }
    if (fault_injected("grid_barrier")) b.extra = 1;
    return b;
}

// Multi-path passes run grouped: one launch per stage of the pass for up to
// kMaxGroupPaths paths (the prologues and the reduction with a block row per
// path, the GEMMs with the paths in their tile sequence; y and dx receive the
// paths' contributions in path order), unless BLR_PATHS=loop asks for the
// paths' single-path passes in turn, or an option without a grouped form is
// on (fused small-M kernels, sign planes, token-major wide products, split-K).
bool paths_grouped() {
    const char *v = std::getenv("BLR_PATHS");
    if (v && std::strcmp(v, "loop") == 0) return false;
    const char *k = std::getenv("BLR_SPLITK");
    if (k && std::strcmp(k, "1") == 0) return false;
    return !plane_mode() && !wide_token_major() && !fused_small_enabled();
}

// Forward of paths [0, n) of a multi-path layer (n <= kMaxGroupPaths), path
// p on the workspace slice at ws0 + p * one: one prologue (x staged n times,
// with each path's g; for x of 64 MB or more only the re-layouts, the a-product
// staging every path's x itself), one a-product, one c-product.
int forward_grouped(const float *x, int n, const uint32_t *const *bits_u, const uint32_t *const *bits_v,
                    const float *const *g, const float *const *l, const float *const *h, float *y, int accumulate_y,
                    int M, int d_in, int d_out, int r, char *ws0, size_t one, int sms, cudaStream_t s) {
    const Layout L = make_layout(M, d_in, d_out, r);
    const GemmPlan p1 = plan_gemm(M, r, sms, 32, 0, n);
    const GemmPlan p2 = plan_gemm(M, d_out, sms, 64, kWideTileCost);
    const long long ps = (long long)one;
    GemmMaps m1{}, m2{};
    if (!make_gmap_act(&m1.act, ws0 + L.x16, M, d_in, p1.pair ? p1.bt / 2 : p1.bt, n, ps) ||
        !make_gmap_chunk(&m1.out32, ws0 + L.a32, M, r, false, n, ps) ||
        !make_gmap_chunk(&m1.out16, ws0 + L.al16, M, r, true, n, ps) ||
        !make_gmap_act(&m2.act, ws0 + L.al16, M, r, p2.pair ? p2.bt / 2 : p2.bt, n, ps) ||
        !make_gmap_chunk(&m2.in32, y, M, d_out, false) || !make_gmap_chunk(&m2.out32, y, M, d_out, false) ||
        !make_gmap_chunk(&m2.out16, ws0 + L.c16, M, d_out, true, n, ps))
        return BLR_ERR_CUDA;
    FwdGroup grp{};
    grp.n = n;
    GemmArgs f1{}, f2{};
    for (int p = 0; p < n; ++p) {
        char *w = ws0 + (size_t)p * one;
        grp.e[p] = FwdPathArgs{SignPrep{bits_v[p], reinterpret_cast<uint32_t *>(w + L.bp_f1), r, d_in, 1, sign_rows(r)},
                               SignPrep{bits_u[p], reinterpret_cast<uint32_t *>(w + L.bp_f2), d_out, r, 0,
                                        sign_rows(d_out)},
                               g[p], reinterpret_cast<uint16_t *>(w + L.x16), reinterpret_cast<uint32_t *>(w + L.header)};
        f1.colv_p[p] = l[p];
        f2.colv_p[p] = h[p];
    }
    uint32_t *status = reinterpret_cast<uint32_t *>(ws0 + L.header);
    f1.M = M;
    f1.N = r;
    f1.K = d_in;
    f1.Ns = sign_rows(r);
    f1.bsign = reinterpret_cast<const uint32_t *>(ws0 + L.bp_f1);
    f1.out32 = reinterpret_cast<float *>(ws0 + L.a32);
    f1.out16 = reinterpret_cast<uint16_t *>(ws0 + L.al16);
    f1.colv = l[0];
    f1.status = status;
    f1.paths = n;
    f1.pstride = ps;
    f2.M = M;
    f2.N = d_out;
    f2.K = r;
    f2.Ns = sign_rows(d_out);
    f2.bsign = reinterpret_cast<const uint32_t *>(ws0 + L.bp_f2);
    f2.out32 = y;
    f2.out16 = reinterpret_cast<uint16_t *>(ws0 + L.c16);
    f2.colv = h[0];
    f2.accumulate = accumulate_y;
    f2.status = status;
    f2.paths = n;
    f2.pstride = ps;
    {
        std::lock_guard<std::mutex> lk(g_tape_mu);
        for (int p = 0; p < n; ++p) g_tapes.erase(ws0 + (size_t)p * one);
    }
    const bool stg = p1.split <= 1 && stage_in_kernel((long long)M * d_in * 4) &&
                     stage_fits(M, p1.bt, d_in, (r + (p1.pair ? 255 : 127)) / (p1.pair ? 256 : 128), n);
    if (stg) {
        // every path's x16 staged inside the a-product, path-major like its tiles
        unsigned int *cnt0 = reinterpret_cast<unsigned int *>(ws0 + L.stg_cnt);
        f1.stg.src = x;
        f1.stg.col = g[0];
        f1.stg.dst = reinterpret_cast<uint16_t *>(ws0 + L.x16);
        f1.stg.cnt = cnt0;
        f1.stg.paths = n;
        f1.stg.pstride = ps;
        for (int p = 0; p < n; ++p) f1.stg.col_p[p] = g[p];
        GemmPlan pst = p1;
        pst.stg = 1;
        if (!make_tmap_x_stage(&m1.in32, x, M, d_in, 16) || !make_tmap_x_stage(&m1.sgn, x, M, d_in, 64))
            return BLR_ERR_CUDA;
        if (launch_prep_group(grp, cnt0, ps, stage_counters(M, p1.bt, d_in), "fwd_prep", s) != cudaSuccess)
            return BLR_ERR_CUDA;
        if (launch_gemm(kEpiFwd1, pst, m1, f1, s) != cudaSuccess) return BLR_ERR_CUDA;
    } else {
        if (launch_fwd_prologue(grp, x, M, d_in, s) != cudaSuccess) return BLR_ERR_CUDA;
        if (launch_gemm(kEpiFwd1, p1, m1, f1, s) != cudaSuccess) return BLR_ERR_CUDA;
    }
    if (launch_gemm(kEpiFwd2, p2, m2, f2, s) != cudaSuccess) return BLR_ERR_CUDA;
    for (int p = 0; p < n; ++p)
        record_tape(ws0 + (size_t)p * one, Tape{M, d_in, d_out, r, x, bits_u[p], bits_v[p], g[p], l[p], h[p], 0, false,
                                                0.0f, 0});
    return BLR_OK;
}

// Backward of paths [0, n) (tapes checked by the caller): one prologue (dy
// staged n times, with each path's h, scales and dh partials), one
// db-product, one dx'-product, one reduction of every path's partial sums.
int backward_grouped(const float *x, const float *dy, int n, const uint32_t *const *bits_u,
                     const uint32_t *const *bits_v, const float *const *g, const float *const *l,
                     const float *const *h, float *dx, int accumulate_dx, float *const *dg, float *const *dl,
                     float *const *dh, float gscale, int M, int d_in, int d_out, int r, char *ws0, size_t one, int sms,
                     cudaStream_t s) {
    const Layout L = make_layout(M, d_in, d_out, r);
    const GemmPlan p1 = plan_gemm(M, r, sms, 32, 0, n);
    const GemmPlan p2 = plan_gemm(M, d_in, sms, 64);
    const long long ps = (long long)one;
    GemmMaps m1{}, m2{};
    if (!make_gmap_act(&m1.act, ws0 + L.dy16, M, d_out, p1.pair ? p1.bt / 2 : p1.bt, n, ps) ||
        !make_gmap_chunk(&m1.in32, ws0 + L.a32, M, r, false, n, ps) ||
        !make_gmap_chunk(&m1.out16, ws0 + L.db16, M, r, true, n, ps) ||
        !make_gmap_act(&m2.act, ws0 + L.db16, M, r, p2.pair ? p2.bt / 2 : p2.bt, n, ps) ||
        !make_gmap_chunk(&m2.in32, x, M, d_in, false) || !make_gmap_chunk(&m2.out32, dx, M, d_in, false))
        return BLR_ERR_CUDA;
    int rows_dh = 0;
    BwdGroup grp{};
    grp.n = n;
    GemmArgs b1{}, b2{};
    for (int p = 0; p < n; ++p) {
        char *w = ws0 + (size_t)p * one;
        BwdPathArgs &e = grp.e[p];
        e.p0 = SignPrep{bits_u[p], reinterpret_cast<uint32_t *>(w + L.bp_b1), r, d_out, 1, sign_rows(r)};
        e.p1 = SignPrep{bits_v[p], reinterpret_cast<uint32_t *>(w + L.bp_b2), d_in, r, 0, sign_rows(d_in)};
        StageDyArgs &sa = e.sd;
        sa.dy = dy;
        sa.h = h[p];
        sa.c16 = reinterpret_cast<const uint16_t *>(w + L.c16);
        sa.l = l[p];
        sa.dy16 = reinterpret_cast<uint16_t *>(w + L.dy16);
        sa.s_inv = reinterpret_cast<float *>(w + L.s_inv);
        sa.sig = reinterpret_cast<float *>(w + L.sig);
        sa.sig_inv = reinterpret_cast<float *>(w + L.sig_inv);
        sa.part_dh = reinterpret_cast<float *>(w + L.part_dh);
        sa.blkmax = reinterpret_cast<float2 *>(w + L.blkmax);
        sa.gscale = gscale;
        sa.M = M;
        sa.d_out = d_out;
        sa.r = r;
        sa.rows_used = p == 0 ? &rows_dh : nullptr;
        sa.status = reinterpret_cast<uint32_t *>(w + L.header);
        sa.red_cnt = nullptr;
        b1.colv_p[p] = l[p];
        b2.colv_p[p] = g[p];
    }
    uint32_t *status = reinterpret_cast<uint32_t *>(ws0 + L.header);
    b1.M = M;
    b1.N = r;
    b1.K = d_out;
    b1.Ns = sign_rows(r);
    b1.bsign = reinterpret_cast<const uint32_t *>(ws0 + L.bp_b1);
    b1.out16 = reinterpret_cast<uint16_t *>(ws0 + L.db16);
    b1.colv = l[0];
    b1.row_inv = reinterpret_cast<const float *>(ws0 + L.s_inv);
    b1.row_scale = reinterpret_cast<const float *>(ws0 + L.sig);
    b1.part = reinterpret_cast<float *>(ws0 + L.part_dl);
    b1.status = status;
    b1.paths = n;
    b1.pstride = ps;
    b2.M = M;
    b2.N = d_in;
    b2.K = r;
    b2.Ns = sign_rows(d_in);
    b2.bsign = reinterpret_cast<const uint32_t *>(ws0 + L.bp_b2);
    b2.out32 = dx;
    b2.colv = g[0];
    b2.row_inv = reinterpret_cast<const float *>(ws0 + L.sig_inv);
    b2.part = reinterpret_cast<float *>(ws0 + L.part_dg);
    b2.accumulate = accumulate_dx;
    b2.status = status;
    b2.paths = n;
    b2.pstride = ps;
    const bool fold = reduce_folded();
    if (fold) grp.e[0].sd.red_cnt = reinterpret_cast<unsigned int *>(ws0 + L.header + kRedCntOffset);
    if (launch_bwd_prologue(grp, s) != cudaSuccess) return BLR_ERR_CUDA;
    if (launch_gemm(kEpiBwd1, p1, m1, b1, s) != cudaSuccess) return BLR_ERR_CUDA;
    if (fold) {
        // every path's dh, dl and dg reduced in the dx'-product's tail
        b2.fold = 1;
        b2.red = grid_barrier(grp.e[0].sd.red_cnt);
        b2.red_part_h = reinterpret_cast<const float *>(ws0 + L.part_dh);
        b2.red_part_l = reinterpret_cast<const float *>(ws0 + L.part_dl);
        b2.red_rows_h = rows_dh;
        b2.red_rows_l = p1.part_rows * epi_part_rows_per_tile(kEpiBwd1);
        b2.red_rows_g = p2.part_rows * epi_part_rows_per_tile(kEpiBwd2);
        b2.red_n_h = d_out;
        b2.red_n_l = r;
        for (int p = 0; p < n; ++p) {
            b2.red_out_h[p] = dh[p];
            b2.red_out_l[p] = dl[p];
            b2.red_out_g[p] = dg[p];
        }
    }
    if (launch_gemm(kEpiBwd2, p2, m2, b2, s) != cudaSuccess) return BLR_ERR_CUDA;
    if (fold) {
        for (int p = 0; p < n; ++p) mark_backward_done(ws0 + (size_t)p * one, gscale, rows_dh);
        return BLR_OK;
    }
    ReduceGroup rg{};
    rg.n = n;
    for (int p = 0; p < n; ++p) {
        char *w = ws0 + (size_t)p * one;
        rg.a[p] = ReduceSeg{reinterpret_cast<const float *>(w + L.part_dh), dh[p], rows_dh, d_out};
        rg.b[p] = ReduceSeg{reinterpret_cast<const float *>(w + L.part_dl), dl[p],
                            p1.part_rows * epi_part_rows_per_tile(kEpiBwd1), r};
        rg.c[p] = ReduceSeg{reinterpret_cast<const float *>(w + L.part_dg), dg[p],
                            p2.part_rows * epi_part_rows_per_tile(kEpiBwd2), d_in};
    }
    if (launch_reduce_partials(rg, s) != cudaSuccess) return BLR_ERR_CUDA;
    for (int p = 0; p < n; ++p) mark_backward_done(ws0 + (size_t)p * one, gscale, rows_dh);
    return BLR_OK;
}

// The per-path pointers of a multi-path call: every array present, every entry
// non-null and 16-byte aligned.
template <typename T>
bool path_ptrs_ok(T *const *a, int P, int *status) {
    if (!a) {
        *status = BLR_ERR_ARG;
        return false;
    }
    for (int p = 0; p < P; ++p) {
        if (!a[p]) {
            *status = BLR_ERR_ARG;
            return false;
        }
        if (!aligned16(a[p])) {
            *status = BLR_ERR_ALIGN;
            return false;
        }
    }
    return true;
}

}  // namespace blr

using namespace blr;

extern "C" {

size_t blr_workspace_bytes(int M, int d_in, int d_out, int r) {
    if (!shape_ok(M, d_in, d_out, r)) return 0;
    return make_layout(M, d_in, d_out, r).total;
}

int blr_workspace_release(const void *ws) {
    if (!ws) return BLR_ERR_ARG;
    std::lock_guard<std::mutex> lk(g_tape_mu);
    g_tapes.erase(ws);
    return BLR_OK;
}

int blr_pack_signs(const float *src, uint32_t *bits, int rows, int r, blr_stream_t stream) {
    if (!src || !bits) return BLR_ERR_ARG;
    if (rows < 1 || r < 1) return BLR_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(bits)) return BLR_ERR_ALIGN;
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("pack")) return BLR_ERR_CUDA;
    return launch_pack_signs(src, bits, rows, r, (cudaStream_t)stream) == cudaSuccess ? BLR_OK : BLR_ERR_CUDA;
}

int blr_unpack_signs(const uint32_t *bits, uint16_t *dst, int rows, int r, blr_stream_t stream) {
    if (!bits || !dst) return BLR_ERR_ARG;
    if (rows < 1 || r < 1) return BLR_ERR_SHAPE;
    if (!aligned16(bits) || !aligned16(dst)) return BLR_ERR_ALIGN;
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("unpack")) return BLR_ERR_CUDA;
    return launch_unpack_signs(bits, dst, rows, r, (cudaStream_t)stream) == cudaSuccess ? BLR_OK : BLR_ERR_CUDA;
}

int blr_forward(const float *x, const uint32_t *bits_u, const uint32_t *bits_v, const float *g, const float *l,
                const float *h, float *y, int accumulate_y, int M, int d_in, int d_out, int r, void *ws,
                size_t ws_bytes, blr_stream_t stream) {
    if (!x || !bits_u || !bits_v || !g || !l || !h || !y || !ws) return BLR_ERR_ARG;
    if (accumulate_y != 0 && accumulate_y != 1) return BLR_ERR_ARG;
    if (!shape_ok(M, d_in, d_out, r)) return BLR_ERR_SHAPE;
    const void *ptrs[] = {x, bits_u, bits_v, g, l, h, y, ws};
    for (const void *p : ptrs)
        if (!aligned16(p)) return BLR_ERR_ALIGN;
    const Layout L = make_layout(M, d_in, d_out, r);
    if (ws_bytes < L.total) return BLR_ERR_WORKSPACE;
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("forward")) return BLR_ERR_CUDA;

    cudaStream_t s = (cudaStream_t)stream;
    char *w = static_cast<char *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + L.header);
    uint32_t *bp_f1 = reinterpret_cast<uint32_t *>(w + L.bp_f1);
    uint32_t *bp_f2 = reinterpret_cast<uint32_t *>(w + L.bp_f2);
    uint16_t *x16 = reinterpret_cast<uint16_t *>(w + L.x16);
    float *a32 = reinterpret_cast<float *>(w + L.a32);
    uint16_t *al16 = reinterpret_cast<uint16_t *>(w + L.al16);
    uint16_t *c16 = reinterpret_cast<uint16_t *>(w + L.c16);

    uint16_t *plane_u = reinterpret_cast<uint16_t *>(w + L.plane_u);
    uint16_t *plane_v = reinterpret_cast<uint16_t *>(w + L.plane_v);
    // the TMEM-expansion tiles decide what counts as a small problem (fused path)
    const bool fused = !plan_gemm(M, r, sms).pair && !plan_gemm(M, d_out, sms).pair && fused_small_enabled();
    const GemmPlan q1 = plan_gemm(M, r, sms, fused ? 128 : 32);
    const GemmPlan q2 = plan_gemm(M, d_out, sms, fused ? 128 : 64, kWideTileCost);
    const bool planes = !fused && plane_mode();
    const bool dense2 = !fused && wide_token_major();
    const GemmPlan p1 = planes ? plan_gemm_plane(M, r, sms) : (fused ? q1 : plan_split(q1, M, r, d_in, sms));
    const GemmPlan p2 = planes ? plan_gemm_plane(M, d_out, sms) : q2;
    GemmMaps m1{}, m2{};
    DenseGemmLaunch d2{};
    if (dense2) {
        // c-product token-major: al16 [M][r] x S_U plane [d_out][r], both K-major
        d2.F[0] = M;
        d2.R = d_out;
        d2.K = r;
        d2.scale[0] = 1.0f;
        d2.accumulate = accumulate_y;
        d2.status = status;
        d2.sms = sms;
        d2.epm = 1;
        d2.colv = h;
        if (!make_tmap_act16(&d2.maps.a[0], al16, M, r, 128) || !make_tmap_act16(&d2.maps.b[0], plane_u, d_out, r, 256) ||
            !make_tmap_out_sw128(&d2.maps.o[0], y, M, d_out) || !make_tmap_out16_sw64(&d2.maps.o16, c16, M, d_out))
            return BLR_ERR_CUDA;
    }
    // a-product: S_V [d_in][r] read MN-major; c-product: S_U [d_out][r] read K-major
    if (planes && (!make_tmap_act16(&m1.sgn, plane_v, d_in, r, 64) || !make_tmap_act16(&m2.sgn, plane_u, d_out, r, 128)))
        return BLR_ERR_CUDA;
    if (!make_gmap_act(&m1.act, x16, M, d_in, p1.pair ? p1.bt / 2 : p1.bt) ||
        !make_gmap_chunk(&m1.out32, a32, M, r, false) || !make_gmap_chunk(&m1.out16, al16, M, r, true) ||
        !make_gmap_act(&m2.act, al16, M, r, p2.pair ? p2.bt / 2 : p2.bt) ||
        !make_gmap_chunk(&m2.in32, y, M, d_out, false) || !make_gmap_chunk(&m2.out32, y, M, d_out, false) ||
        !make_gmap_chunk(&m2.out16, c16, M, d_out, true))
        return BLR_ERR_CUDA;

    // a new forward starts a new tape: forget the old one first
    {
        std::lock_guard<std::mutex> lk(g_tape_mu);
        g_tapes.erase(ws);
    }
    // S_V [d_in][r/32] has its bits along r: the first product needs them along d_in
    SignPrep pv{bits_v, bp_f1, r, d_in, 1, sign_rows(r)};
    SignPrep pu{bits_u, bp_f2, d_out, r, 0, sign_rows(d_out)};
    if (planes) {
        // both products read +-1 f16 planes in the bitmaps' own order
        pv = SignPrep{bits_v, reinterpret_cast<uint32_t *>(plane_v), d_in, r, 2, 0};
        pu = SignPrep{bits_u, reinterpret_cast<uint32_t *>(plane_u), d_out, r, 2, 0};
    } else if (dense2) {
        pu = SignPrep{bits_u, reinterpret_cast<uint32_t *>(plane_u), d_out, r, 2, 0};
    }

    GemmArgs f1{};
    f1.M = M;
    f1.N = r;
    f1.K = d_in;
    f1.Ns = sign_rows(r);
    f1.bsign = bp_f1;
    f1.out32 = a32;
    f1.out16 = al16;
    f1.colv = l;
    f1.status = status;

    GemmArgs f2{};
    f2.M = M;
    f2.N = d_out;
    f2.K = r;
    f2.Ns = sign_rows(d_out);
    f2.bsign = bp_f2;
    f2.out32 = y;
    f2.out16 = c16;
    f2.colv = h;
    f2.accumulate = accumulate_y;
    f2.status = status;

    // x staged inside the a-product (not with sign planes or split-K tiles)
    const bool stg = !fused && !planes && p1.split <= 1 && stage_in_kernel((long long)M * d_in * 4) &&
                     stage_fits(M, p1.bt, d_in, (r + (p1.pair ? 255 : 127)) / (p1.pair ? 256 : 128));
    if (fused) {
        // small problem: the whole pass as one fused cooperative kernel
        SmallFwdArgs fa{pv, pu, x, g, x16, M, d_in, status,
                        grid_barrier(reinterpret_cast<unsigned int *>(w + L.header + kGridBarOffset)), f1, f2};
        if (launch_small_fwd(m1, m2, fa, small_grid(p1, r, p2, d_out, M, sms), s) != cudaSuccess)
            return BLR_ERR_CUDA;
    } else if (stg) {
        unsigned int *cnt = reinterpret_cast<unsigned int *>(w + L.stg_cnt);
        f1.stg.src = x;
        f1.stg.col = g;
        f1.stg.dst = x16;
        f1.stg.cnt = cnt;
        GemmPlan ps = p1;
        ps.stg = 1;
        // the a-product uses neither its input map nor a sign plane: they carry x
        if (!make_tmap_x_stage(&m1.in32, x, M, d_in, 16) || !make_tmap_x_stage(&m1.sgn, x, M, d_in, 64))
            return BLR_ERR_CUDA;
        const int ncnt = stage_counters(M, p1.bt, d_in);
        if (launch_prep(pv, pu, status, cnt, ncnt, "fwd_prep", s) != cudaSuccess) return BLR_ERR_CUDA;
        if (launch_gemm(kEpiFwd1, ps, m1, f1, s) != cudaSuccess) return BLR_ERR_CUDA;
        if (dense2) {
            if (launch_dense_gemm(d2, "gemm_fwd2", s) != cudaSuccess) return BLR_ERR_CUDA;
        } else if (launch_gemm(kEpiFwd2, p2, m2, f2, s) != cudaSuccess) {
            return BLR_ERR_CUDA;
        }
    } else {
        if (launch_fwd_prologue(pv, pu, x, g, x16, M, d_in, status, s) != cudaSuccess) return BLR_ERR_CUDA;
        if (launch_gemm(kEpiFwd1, p1, m1, f1, s) != cudaSuccess) return BLR_ERR_CUDA;
        if (dense2) {
            if (launch_dense_gemm(d2, "gemm_fwd2", s) != cudaSuccess) return BLR_ERR_CUDA;
        } else if (launch_gemm(kEpiFwd2, p2, m2, f2, s) != cudaSuccess) {
            return BLR_ERR_CUDA;
        }
    }

    record_tape(ws, Tape{M, d_in, d_out, r, x, bits_u, bits_v, g, l, h, 0, false, 0.0f, 0});
    return BLR_OK;
}

int blr_backward(const float *x, const float *dy, const uint32_t *bits_u, const uint32_t *bits_v, const float *g,
                 const float *l, const float *h, float *dx, int accumulate_dx, float *dg, float *dl, float *dh,
                 float gscale, int M, int d_in, int d_out, int r, void *ws, size_t ws_bytes, blr_stream_t stream) {
    if (!x || !dy || !bits_u || !bits_v || !g || !l || !h || !dx || !dg || !dl || !dh || !ws) return BLR_ERR_ARG;
    if (accumulate_dx != 0 && accumulate_dx != 1) return BLR_ERR_ARG;
    if (std::isnan(gscale) || (gscale > 0.0f && !pow2_positive(gscale))) return BLR_ERR_ARG;
    if (!shape_ok(M, d_in, d_out, r)) return BLR_ERR_SHAPE;
    const void *ptrs[] = {x, dy, bits_u, bits_v, g, l, h, dx, dg, dl, dh, ws};
    for (const void *p : ptrs)
        if (!aligned16(p)) return BLR_ERR_ALIGN;
    const Layout L = make_layout(M, d_in, d_out, r);
    if (ws_bytes < L.total) return BLR_ERR_WORKSPACE;
    if (!tape_matches(ws, M, d_in, d_out, r, x, bits_u, bits_v, g, l, h)) return BLR_ERR_STATE;
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("backward")) return BLR_ERR_CUDA;

    cudaStream_t s = (cudaStream_t)stream;
    char *w = static_cast<char *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + L.header);
    uint32_t *bp_b1 = reinterpret_cast<uint32_t *>(w + L.bp_b1);
    uint32_t *bp_b2 = reinterpret_cast<uint32_t *>(w + L.bp_b2);
    uint16_t *dy16 = reinterpret_cast<uint16_t *>(w + L.dy16);
    const float *a32 = reinterpret_cast<const float *>(w + L.a32);
    uint16_t *db16 = reinterpret_cast<uint16_t *>(w + L.db16);
    const uint16_t *c16 = reinterpret_cast<const uint16_t *>(w + L.c16);
    float *s_inv = reinterpret_cast<float *>(w + L.s_inv);
    float *sig = reinterpret_cast<float *>(w + L.sig);
    float *sig_inv = reinterpret_cast<float *>(w + L.sig_inv);
    float *part_dh = reinterpret_cast<float *>(w + L.part_dh);
    float *part_dl = reinterpret_cast<float *>(w + L.part_dl);
    float *part_dg = reinterpret_cast<float *>(w + L.part_dg);

    uint16_t *plane_u = reinterpret_cast<uint16_t *>(w + L.plane_u);
    uint16_t *plane_v = reinterpret_cast<uint16_t *>(w + L.plane_v);
    const bool fused =
        !plan_gemm(M, r, sms).pair && !plan_gemm(M, d_in, sms).pair && small_bwd_fits(d_out) && fused_small_enabled();
    const GemmPlan q1 = plan_gemm(M, r, sms, fused ? 128 : 32);
    const GemmPlan q2 = plan_gemm(M, d_in, sms, fused ? 128 : 64);
    const bool planes = !fused && plane_mode();
    const bool dense2 = !fused && wide_token_major();
    const GemmPlan p1 = planes ? plan_gemm_plane(M, r, sms) : (fused ? q1 : plan_split(q1, M, r, d_out, sms));
    const GemmPlan p2 = planes ? plan_gemm_plane(M, d_in, sms) : q2;
    GemmMaps m1{}, m2{};
    DenseGemmLaunch d2{};
    if (dense2) {
        // dx'-product token-major: db16 [M][r] x S_V plane [d_in][r], both K-major
        d2.F[0] = M;
        d2.R = d_in;
        d2.K = r;
        d2.scale[0] = 1.0f;
        d2.accumulate = accumulate_dx;
        d2.status = status;
        d2.sms = sms;
        d2.epm = 2;
        d2.colv = g;
        d2.row_inv = sig_inv;
        d2.xin = x;
        d2.part = part_dg;
        if (!make_tmap_act16(&d2.maps.a[0], db16, M, r, 128) || !make_tmap_act16(&d2.maps.b[0], plane_v, d_in, r, 256) ||
            !make_tmap_out_sw128(&d2.maps.o[0], dx, M, d_in))
            return BLR_ERR_CUDA;
    }
    // db-product: S_U [d_out][r] read MN-major; dx'-product: S_V [d_in][r] read K-major
    if (planes && (!make_tmap_act16(&m1.sgn, plane_u, d_out, r, 64) || !make_tmap_act16(&m2.sgn, plane_v, d_in, r, 128)))
        return BLR_ERR_CUDA;
    if (!make_gmap_act(&m1.act, dy16, M, d_out, p1.pair ? p1.bt / 2 : p1.bt) ||
        !make_gmap_chunk(&m1.in32, a32, M, r, false) || !make_gmap_chunk(&m1.out16, db16, M, r, true) ||
        !make_gmap_act(&m2.act, db16, M, r, p2.pair ? p2.bt / 2 : p2.bt) ||
        !make_gmap_chunk(&m2.in32, x, M, d_in, false) || !make_gmap_chunk(&m2.out32, dx, M, d_in, false))
        return BLR_ERR_CUDA;

    // S_U [d_out][r/32] has its bits along r: the first product needs them along d_out
    SignPrep pu{bits_u, bp_b1, r, d_out, 1, sign_rows(r)};
    SignPrep pv{bits_v, bp_b2, d_in, r, 0, sign_rows(d_in)};
    if (planes) {
        pu = SignPrep{bits_u, reinterpret_cast<uint32_t *>(plane_u), d_out, r, 2, 0};
        pv = SignPrep{bits_v, reinterpret_cast<uint32_t *>(plane_v), d_in, r, 2, 0};
    } else if (dense2) {
        pv = SignPrep{bits_v, reinterpret_cast<uint32_t *>(plane_v), d_in, r, 2, 0};
    }
    StageDyArgs sa{};
    sa.dy = dy;
    sa.h = h;
    sa.c16 = c16;
    sa.l = l;
    sa.dy16 = dy16;
    sa.s_inv = s_inv;
    sa.sig = sig;
    sa.sig_inv = sig_inv;
    sa.part_dh = part_dh;
    sa.blkmax = reinterpret_cast<float2 *>(w + L.blkmax);
    sa.gscale = gscale;
    sa.M = M;
    sa.d_out = d_out;
    sa.r = r;
    int rows_dh = 0;
    sa.rows_used = &rows_dh;
    sa.status = status;

    GemmArgs b1{};
    b1.M = M;
    b1.N = r;
    b1.K = d_out;
    b1.Ns = sign_rows(r);
    b1.bsign = bp_b1;
    b1.out16 = db16;
    b1.colv = l;
    b1.row_inv = s_inv;
    b1.row_scale = sig;
    b1.part = part_dl;
    b1.status = status;

    GemmArgs b2{};
    b2.M = M;
    b2.N = d_in;
    b2.K = r;
    b2.Ns = sign_rows(d_in);
    b2.bsign = bp_b2;
    b2.out32 = dx;
    b2.colv = g;
    b2.row_inv = sig_inv;
    b2.part = part_dg;
    b2.accumulate = accumulate_dx;
    b2.status = status;

    ReduceSeg sl{part_dl, dl, p1.part_rows * (p1.split == 4 ? 4 : epi_part_rows_per_tile(kEpiBwd1)), r};
    ReduceSeg sg{part_dg, dg, dense2 ? (M + 127) / 128 * 4 : p2.part_rows * epi_part_rows_per_tile(kEpiBwd2), d_in};
    if (fused) {
        // small problem: the whole pass as one fused cooperative kernel
        SmallBwdArgs ba{};
        ba.pu = pu;
        ba.pv = pv;
        ba.sd = sa;
        ba.gb = grid_barrier(reinterpret_cast<unsigned int *>(w + L.header + kGridBarOffset));
        ba.b1 = b1;
        ba.b2 = b2;
        ba.rh = ReduceSeg{part_dh, dh, 0, d_out};
        ba.rl = sl;
        ba.rg = sg;
        if (launch_small_bwd(m1, m2, ba, small_grid(p1, r, p2, d_in, M, sms), stage_dy_blocks(M, d_out), s) !=
            cudaSuccess)
            return BLR_ERR_CUDA;
        mark_backward_done(ws, gscale, rows_dh);
        return BLR_OK;
    }
    const bool fold = !dense2 && reduce_folded();
    if (fold) sa.red_cnt = reinterpret_cast<unsigned int *>(w + L.header + kRedCntOffset);
    // dy staged inside the db-product (large dy, CTA-pair tiles of one
    // path, no split-K or sign planes): a scale pass first, then the product
    // stages dy16 and adds the dh sums into kDyPartRowsPerCta rows per CTA
    const bool dstg = !planes && p1.pair && p1.split <= 1 && dy_stage_in_kernel() &&
                      stage_fits(M, p1.bt, d_out, (r + 255) / 256) && p1.grid <= kDyStageMaxCtas;
    int dh_rows = 0;
    if (dstg) {
        unsigned int *cnt = reinterpret_cast<unsigned int *>(w + L.stg_cnt);
        sa.zero_cnt = cnt;
        sa.n_cnt = stage_counters(M, p1.bt, d_out);
        sa.zero_part = part_dh;
        sa.n_part = (long long)p1.grid * kDyPartRowsPerCta * d_out;
        b1.stg.src = dy;
        b1.stg.col = h;
        b1.stg.dst = dy16;
        b1.stg.cnt = cnt;
        b1.stg.row_sinv = s_inv;
        b1.stg.part = part_dh;
        GemmPlan ps = p1;
        ps.stg = 2;
        // the db-product has no f32 output and no sign plane: those maps carry
        // dy (256 x 16 boxes for the ring, 256 x 64 for the L2 prefetches)
        if (!make_tmap_x_stage(&m1.out32, dy, M, d_out, 16) || !make_tmap_x_stage(&m1.sgn, dy, M, d_out, 64) ||
            !make_tmap_c_stage(&m1.aux, c16, M, d_out, 16))
            return BLR_ERR_CUDA;
        if (launch_bwd_scales(pu, pv, sa, s) != cudaSuccess) return BLR_ERR_CUDA;
        if (launch_gemm(kEpiBwd1, ps, m1, b1, s) != cudaSuccess) return BLR_ERR_CUDA;
        dh_rows = p1.grid * kDyPartRowsPerCta;
    } else {
        if (launch_bwd_prologue(pu, pv, sa, s) != cudaSuccess) return BLR_ERR_CUDA;
        if (launch_gemm(kEpiBwd1, p1, m1, b1, s) != cudaSuccess) return BLR_ERR_CUDA;
        dh_rows = rows_dh;
    }
    if (fold) {
        // dh, dl and dg reduced in the dx'-product's tail (the dh rows are known now)
        b2.fold = 1;
        b2.red = grid_barrier(sa.red_cnt);
        b2.red_part_h = part_dh;
        b2.red_part_l = part_dl;
        b2.red_rows_h = dh_rows;
        b2.red_rows_l = sl.rows;
        b2.red_rows_g = sg.rows;
        b2.red_n_h = d_out;
        b2.red_n_l = r;
        b2.red_out_h[0] = dh;
        b2.red_out_l[0] = dl;
        b2.red_out_g[0] = dg;
    }
    if (dense2) {
        if (launch_dense_gemm(d2, "gemm_bwd2", s) != cudaSuccess) return BLR_ERR_CUDA;
    } else if (launch_gemm(kEpiBwd2, p2, m2, b2, s) != cudaSuccess) {
        return BLR_ERR_CUDA;
    }
    if (!fold) {
        ReduceSeg sh{part_dh, dh, dh_rows, d_out};
        if (launch_reduce_partials(sh, sl, sg, s) != cudaSuccess) return BLR_ERR_CUDA;
    }
    mark_backward_done(ws, gscale, rows_dh);
    return BLR_OK;
}

size_t blr_paths_workspace_bytes(int P, int M, int d_in, int d_out, int r) {
    if (P < 1 || P > 64 || !shape_ok(M, d_in, d_out, r)) return 0;
    return (size_t)P * make_layout(M, d_in, d_out, r).total;
}


int blr_forward_paths(const float *x, int P, const uint32_t *const *bits_u, const uint32_t *const *bits_v,
                      const float *const *g, const float *const *l, const float *const *h, float *y,
                      int accumulate_y, int M, int d_in, int d_out, int r, void *ws, size_t ws_bytes,
                      blr_stream_t stream) {
    if (P < 1 || P > 64 || !x || !y || !ws) return BLR_ERR_ARG;
    if (accumulate_y != 0 && accumulate_y != 1) return BLR_ERR_ARG;
    if (!shape_ok(M, d_in, d_out, r)) return BLR_ERR_SHAPE;
    int st = BLR_OK;
    if (!path_ptrs_ok(bits_u, P, &st) || !path_ptrs_ok(bits_v, P, &st) || !path_ptrs_ok(g, P, &st) ||
        !path_ptrs_ok(l, P, &st) || !path_ptrs_ok(h, P, &st))
        return st;
    const size_t one = make_layout(M, d_in, d_out, r).total;
    if (ws_bytes < (size_t)P * one) return BLR_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(y) || !aligned16(ws)) return BLR_ERR_ALIGN;
    if (P > 1 && paths_grouped()) {
        int sms;
        st = device_info(&sms);
        if (st != BLR_OK) return st;
        if (fault_injected("forward")) return BLR_ERR_CUDA;
        // groups of up to kMaxGroupPaths paths; later groups add into y
        for (int p0 = 0; p0 < P; p0 += kMaxGroupPaths) {
            const int n = P - p0 < kMaxGroupPaths ? P - p0 : kMaxGroupPaths;
            st = forward_grouped(x, n, bits_u + p0, bits_v + p0, g + p0, l + p0, h + p0, y,
                                 (p0 > 0 || accumulate_y) ? 1 : 0, M, d_in, d_out, r,
                                 static_cast<char *>(ws) + (size_t)p0 * one, one, sms, (cudaStream_t)stream);
            if (st != BLR_OK) return st;
        }
        return BLR_OK;
    }
    for (int p = 0; p < P; ++p) {
        st = blr_forward(x, bits_u[p], bits_v[p], g[p], l[p], h[p], y, (p > 0 || accumulate_y) ? 1 : 0, M, d_in,
                         d_out, r, static_cast<char *>(ws) + (size_t)p * one, one, stream);
        if (st != BLR_OK) return st;
    }
    return BLR_OK;
}

int blr_backward_paths(const float *x, const float *dy, int P, const uint32_t *const *bits_u,
                       const uint32_t *const *bits_v, const float *const *g, const float *const *l,
                       const float *const *h, float *dx, int accumulate_dx, float *const *dg, float *const *dl,
                       float *const *dh, float gscale, int M, int d_in, int d_out, int r, void *ws,
                       size_t ws_bytes, blr_stream_t stream) {
    if (P < 1 || P > 64 || !x || !dy || !dx || !ws) return BLR_ERR_ARG;
    if (accumulate_dx != 0 && accumulate_dx != 1) return BLR_ERR_ARG;
    if (std::isnan(gscale) || (gscale > 0.0f && !pow2_positive(gscale))) return BLR_ERR_ARG;
    if (!shape_ok(M, d_in, d_out, r)) return BLR_ERR_SHAPE;
    int st = BLR_OK;
    if (!path_ptrs_ok(bits_u, P, &st) || !path_ptrs_ok(bits_v, P, &st) || !path_ptrs_ok(g, P, &st) ||
        !path_ptrs_ok(l, P, &st) || !path_ptrs_ok(h, P, &st) || !path_ptrs_ok(dg, P, &st) ||
        !path_ptrs_ok(dl, P, &st) || !path_ptrs_ok(dh, P, &st))
        return st;
    const size_t one = make_layout(M, d_in, d_out, r).total;
    if (ws_bytes < (size_t)P * one) return BLR_ERR_WORKSPACE;
    // every path's tape must be there before any path's backward is queued
    for (int p = 0; p < P; ++p)
        if (!tape_matches(static_cast<char *>(ws) + (size_t)p * one, M, d_in, d_out, r, x, bits_u[p], bits_v[p], g[p],
                          l[p], h[p]))
            return BLR_ERR_STATE;
    if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(ws)) return BLR_ERR_ALIGN;
    if (P > 1 && paths_grouped()) {
        int sms;
        st = device_info(&sms);
        if (st != BLR_OK) return st;
        if (fault_injected("backward")) return BLR_ERR_CUDA;
        for (int p0 = 0; p0 < P; p0 += kMaxGroupPaths) {
            const int n = P - p0 < kMaxGroupPaths ? P - p0 : kMaxGroupPaths;
            st = backward_grouped(x, dy, n, bits_u + p0, bits_v + p0, g + p0, l + p0, h + p0, dx,
                                  (p0 > 0 || accumulate_dx) ? 1 : 0, dg + p0, dl + p0, dh + p0, gscale, M, d_in, d_out,
                                  r, static_cast<char *>(ws) + (size_t)p0 * one, one, sms, (cudaStream_t)stream);
            if (st != BLR_OK) return st;
        }
        return BLR_OK;
    }
    for (int p = 0; p < P; ++p) {
        st = blr_backward(x, dy, bits_u[p], bits_v[p], g[p], l[p], h[p], dx, (p > 0 || accumulate_dx) ? 1 : 0, dg[p],
                          dl[p], dh[p], gscale, M, d_in, d_out, r, static_cast<char *>(ws) + (size_t)p * one, one,
                          stream);
        if (st != BLR_OK) return st;
    }
    return BLR_OK;
}

size_t blr_sign_workspace_bytes(int M, int d_in, int d_out, int r) {
    if (!shape_ok(M, d_in, d_out, r)) return 0;
    return make_sign_layout(M, r).total;
}

int blr_sign_grads(const float *x, const float *g, const float *l, float *gu, float *gv, int accumulate, int M, int d_in,
                   int d_out, int r, const void *ws, size_t ws_bytes, void *sws, size_t sws_bytes,
                   blr_stream_t stream) {
    if (!x || !g || !l || !gu || !gv || !ws || !sws) return BLR_ERR_ARG;
    if (accumulate != 0 && accumulate != 1) return BLR_ERR_ARG;
    if (!shape_ok(M, d_in, d_out, r)) return BLR_ERR_SHAPE;
    const void *ptrs[] = {x, g, l, gu, gv, ws, sws};
    for (const void *p : ptrs)
        if (!aligned16(p)) return BLR_ERR_ALIGN;
    const Layout L = make_layout(M, d_in, d_out, r);
    const SignLayout SL = make_sign_layout(M, r);
    if (ws_bytes < L.total || sws_bytes < SL.total) return BLR_ERR_WORKSPACE;
    // the products read only the pass's own staging in `ws` (x.g, dy.h, a.l,
    // db.l), so the record's shape and backward are what must match here
    Tape tape{};
    {
        std::lock_guard<std::mutex> lk(g_tape_mu);
        auto it = g_tapes.find(ws);
        if (it == g_tapes.end() || !it->second.backward_done || it->second.M != M || it->second.d_in != d_in ||
            it->second.d_out != d_out || it->second.r != r)
            return BLR_ERR_STATE;
        tape = it->second;
    }
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("sign")) return BLR_ERR_CUDA;

    cudaStream_t s = (cudaStream_t)stream;
    char *w = static_cast<char *>(const_cast<void *>(ws));
    char *sw = static_cast<char *>(sws);
    const uint16_t *x16 = reinterpret_cast<const uint16_t *>(w + L.x16);
    const uint16_t *dy16 = reinterpret_cast<const uint16_t *>(w + L.dy16);
    const uint16_t *al16 = reinterpret_cast<const uint16_t *>(w + L.al16);
    const uint16_t *db16 = reinterpret_cast<const uint16_t *>(w + L.db16);

    DenseGemmLaunch gl{};
    gl.F[0] = d_out;
    gl.F[1] = d_in;
    gl.R = r;
    gl.K = M;  // the products sum over tokens
    gl.a_mn = gl.b_mn = true;
    gl.accumulate = accumulate;
    gl.status = reinterpret_cast<uint32_t *>(w + L.header);
    gl.sms = sms;
    const uint16_t *bu = al16, *bv = db16;
    if (tape.gscale > 0.0f) {
        // one scale for every token: the staged a.l and db.l serve as they are
        gl.scale[0] = gl.scale[1] = 1.0f / tape.gscale;
    } else {
        SignRescaleArgs ra{};
        ra.al16 = al16;
        ra.db16 = db16;
        ra.s_inv = reinterpret_cast<const float *>(w + L.s_inv);
        ra.sig_inv = reinterpret_cast<const float *>(w + L.sig_inv);
        ra.blkmax = reinterpret_cast<const float2 *>(w + L.blkmax);
        ra.nblk = tape.stage_blocks;
        ra.M = M;
        ra.r = r;
        ra.bu = reinterpret_cast<uint16_t *>(sw + SL.bu);
        ra.bv = reinterpret_cast<uint16_t *>(sw + SL.bv);
        ra.gmax = reinterpret_cast<float *>(sw + SL.header);
        if (launch_sign_rescale(ra, sms, s) != cudaSuccess) return BLR_ERR_CUDA;
        bu = ra.bu;
        bv = ra.bv;
        gl.scale[0] = gl.scale[1] = 1.0f;
        gl.dscale[0] = ra.gmax;
        gl.dscale[1] = ra.gmax + 1;
    }
    if (!make_tmap_act16(&gl.maps.a[0], dy16, M, d_out, 64) || !make_tmap_act16(&gl.maps.b[0], bu, M, r, 64) ||
        !make_tmap_act16(&gl.maps.a[1], x16, M, d_in, 64) || !make_tmap_act16(&gl.maps.b[1], bv, M, r, 64) ||
        !make_tmap_out_sw128(&gl.maps.o[0], gu, d_out, r) || !make_tmap_out_sw128(&gl.maps.o[1], gv, d_in, r))
        return BLR_ERR_CUDA;
    return launch_dense_gemm(gl, "sign_gemm", s) == cudaSuccess ? BLR_OK : BLR_ERR_CUDA;
}

size_t blr_plane_workspace_bytes(int ntok, int n, int k) {
    if (!plane_shape_ok(ntok, n, k)) return 0;
    return 256 + align_up((size_t)ntok * (size_t)(n > k ? n : k) * 2, 256);
}

int blr_plane_linear(const float *x, const uint16_t *plane, float *y, int transpose, int accumulate, float scale,
                     int ntok, int n, int k, void *ws, size_t ws_bytes, blr_stream_t stream) {
    if (!x || !plane || !y || !ws) return BLR_ERR_ARG;
    if ((transpose != 0 && transpose != 1) || (accumulate != 0 && accumulate != 1)) return BLR_ERR_ARG;
    if (!pow2_positive(scale)) return BLR_ERR_ARG;
    if (!plane_shape_ok(ntok, n, k)) return BLR_ERR_SHAPE;
    const void *ptrs[] = {x, plane, y, ws};
    for (const void *p : ptrs)
        if (!aligned16(p)) return BLR_ERR_ALIGN;
    if (ws_bytes < blr_plane_workspace_bytes(ntok, n, k)) return BLR_ERR_WORKSPACE;
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("plane")) return BLR_ERR_CUDA;

    cudaStream_t s = (cudaStream_t)stream;
    char *w = static_cast<char *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(w);
    uint16_t *act16 = reinterpret_cast<uint16_t *>(w + 256);
    // forward: x [ntok][k] -> y [ntok][n] = x plane^T; transpose: x [ntok][n] -> y [ntok][k] = x plane
    const int kin = transpose ? n : k, nout = transpose ? k : n;
    if (launch_plane_stage(x, act16, (long long)ntok * kin, scale, status, sms, s) != cudaSuccess) return BLR_ERR_CUDA;
    DenseGemmLaunch gl{};
    gl.F[0] = ntok;
    gl.F[1] = 0;
    gl.scale[0] = 1.0f / scale;
    gl.R = nout;
    gl.K = kin;
    gl.accumulate = accumulate;
    gl.a_mn = false;           // act16 rows are K-vectors
    gl.b_mn = transpose != 0;  // plane rows are K-vectors (forward) or N-vectors (transpose)
    gl.status = status;
    gl.sms = sms;
    const bool ok = make_tmap_act16(&gl.maps.a[0], act16, ntok, kin, 128) &&
                    (transpose ? make_tmap_act16(&gl.maps.b[0], plane, n, k, 64)
                               : make_tmap_act16(&gl.maps.b[0], plane, n, k, dense_bn(nout))) &&
                    make_tmap_out_sw128(&gl.maps.o[0], y, ntok, nout);
    if (!ok) return BLR_ERR_CUDA;
    return launch_dense_gemm(gl, "plane_gemm", s) == cudaSuccess ? BLR_OK : BLR_ERR_CUDA;
}

int blr_adam(float *w, const float *grad, float *m1, float *m2, const float *mask, int n, int step, float lr,
             float b1, float b2, float eps, float gmul, float rel, blr_stream_t stream) {
    if (!w || !grad || !m1 || !m2) return BLR_ERR_ARG;
    if (n < 0) return BLR_ERR_SHAPE;
    if (step < 1 || !std::isfinite(lr) || !std::isfinite(gmul) || std::isnan(rel) || !std::isfinite(eps) ||
        eps < 0.0f || !(b1 >= 0.0f && b1 < 1.0f) || !(b2 >= 0.0f && b2 < 1.0f))
        return BLR_ERR_ARG;
    const void *ptrs[] = {w, grad, m1, m2, mask};
    for (const void *p : ptrs)
        if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return BLR_ERR_ALIGN;
    if (n == 0) return BLR_OK;
    int sms;
    int st = device_info(&sms);
    if (st != BLR_OK) return st;
    if (fault_injected("adam")) return BLR_ERR_CUDA;
    AdamArgs a{};
    a.w = w;
    a.grad = grad;
    a.m1 = m1;
    a.m2 = m2;
    a.mask = mask;
    a.n = n;
    a.lr = lr;
    a.b1 = b1;
    a.b2 = b2;
    a.eps = eps;
    a.gmul = gmul;
    a.rel = rel;
    a.bc1 = (float)(1.0 - std::pow((double)b1, (double)step));
    a.bc2 = (float)(1.0 - std::pow((double)b2, (double)step));
    if (!(a.bc1 > 0.0f) || !(a.bc2 > 0.0f)) return BLR_ERR_ARG;
    return launch_adam(a, sms, (cudaStream_t)stream) == cudaSuccess ? BLR_OK : BLR_ERR_CUDA;
}

int blr_check_status(const void *ws, size_t ws_bytes, blr_stream_t stream, uint32_t *device_code) {
    if (!ws || ws_bytes < 256) return BLR_ERR_ARG;
    uint32_t code = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&code, ws, sizeof(code), cudaMemcpyDeviceToHost, s) != cudaSuccess) return BLR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BLR_ERR_CUDA;
    if (device_code) *device_code = code;
    return code ? BLR_ERR_DEVICE_CHECK : BLR_OK;
}

const char *blr_status_string(int status) {
    switch (status) {
        case BLR_OK: return "ok";
        case BLR_ERR_ARG: return "invalid argument";
        case BLR_ERR_SHAPE: return "shape rule violated (M >= 1; d_in, d_out, r multiples of 32, >= 64; d_out <= 32768, d_in, r <= 65536)";
        case BLR_ERR_ALIGN: return "pointer not 16-byte aligned";
        case BLR_ERR_WORKSPACE: return "workspace too small";
        case BLR_ERR_STATE: return "backward without a matching forward on this workspace";
        case BLR_ERR_CUDA: return "CUDA call or kernel launch failed";
        case BLR_ERR_DEVICE_CHECK: return "a kernel recorded a failure in the workspace status word";
        case BLR_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3";
        default: return "unknown status";
    }
}

int blr_trace_begin(int capacity) {
    if (capacity < 1) return BLR_ERR_ARG;
    TraceState &t = g_trace;
    while ((int)t.ev.size() < 2 * capacity) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return BLR_ERR_CUDA;
        t.ev.push_back(e);
    }
    t.names.assign(capacity, nullptr);
    t.cap = capacity;
    t.n = 0;
    t.on = true;
    return BLR_OK;
}

int blr_trace_end(void) {
    g_trace.on = false;
    return BLR_OK;
}

int blr_trace_count(void) { return g_trace.n; }

const char *blr_trace_read(int i, float *ms) {
    TraceState &t = g_trace;
    if (i < 0 || i >= t.n) return nullptr;
    if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess) return nullptr;
    float v = 0.0f;
    if (cudaEventElapsedTime(&v, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess) return nullptr;
    if (ms) *ms = v;
    return t.names[i];
}

}  // extern "C"
