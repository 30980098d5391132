// blr_forward_noalloc: the blr forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or any allocator: a plugin running inside
// a host application that owns every device allocation and forbids raw
// allocations, or a real-time inference loop with a fixed memory budget that
// must never enter an allocator. They cannot provide the caller-owned
// workspace that blr_forward needs. This entry point takes the same inputs and
// output and uses a fixed scratch array in the library's own device memory
// instead (BLR_NOALLOC_SCRATCH_BYTES; every GPU that loads the library keeps it
// until the process exits).
//
// It runs the same kernels as blr_forward, with their workspace pointers taken
// from that array. The host needs the array's device address: the first call
// on each device looks it up with cudaGetSymbolAddress (with that device
// current) and caches it, so that first call should be made before any stream
// capture. All calls share the one array and it keeps the last call's
// contents; the kernels clear what must start at zero (the status word), and
// calls that overlap on the GPU race on the array. Its layout is the forward
// part of blr_forward's workspace layout (blr_layout.h), so both entry points
// carve the same regions for the same shape.
#include <mutex>

#include "../../include/blr.h"
#include "blr_kernels.h"
#include "blr_layout.h"

namespace blr {
namespace {

// The scratch array. Host code must not take its address with `&`: on the
// host the name is a stand-in, not a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BLR_NOALLOC_SCRATCH_BYTES];

std::mutex g_na_mu;
void *g_na_ptr[64];
int g_na_sms[64];
bool g_na_ran[64];  // a forward has been queued on this device's array

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn na_encode_fn() {
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

bool na_tmap(CUtensorMap *m, const void *base, int rows, int cols, int box_cols, int box_rows, bool f16,
             CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = na_encode_fn();
    if (!fn) return false;
    // the layer GEMMs read 3-D maps (a plane per path); one plane here
    const cuuint64_t esz = f16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)cols * esz, ((cuuint64_t)rows * cols * esz + 15) / 16 * 16};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device (looked up once
// per device), its SM count, and whether the device is supported.
int na_setup(void **ptr, int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BLR_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!g_na_ptr[dev]) {
        int maj = 0, min = 0, n = 0;
        if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BLR_ERR_CUDA;
        if (maj != 10 || min != 3) return BLR_ERR_UNSUPPORTED_DEVICE;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return BLR_ERR_CUDA;
        g_na_ptr[dev] = p;
        g_na_sms[dev] = n;
    }
    *ptr = g_na_ptr[dev];
    *sms = g_na_sms[dev];
    return BLR_OK;
}

}  // namespace
}  // namespace blr

using namespace blr;

extern "C" int blr_forward_noalloc(const float *x, const uint32_t *bits_u, const uint32_t *bits_v, const float *g,
                                   const float *l, const float *h, float *y, int accumulate_y, int M, int d_in,
                                   int d_out, int r, blr_stream_t stream) {
    if (!x || !bits_u || !bits_v || !g || !l || !h || !y) return BLR_ERR_ARG;
    if (accumulate_y != 0 && accumulate_y != 1) return BLR_ERR_ARG;
    if (!shape_ok(M, d_in, d_out, r)) return BLR_ERR_SHAPE;
    const void *ptrs[] = {x, bits_u, bits_v, g, l, h, y};
    for (const void *p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return BLR_ERR_ALIGN;
    // the forward regions of the workspace layout must fit the fixed scratch
    // array: no allocation happens here
    const Layout L = make_layout(M, d_in, d_out, r);
    if (L.fwd_total > (size_t)BLR_NOALLOC_SCRATCH_BYTES) return BLR_ERR_WORKSPACE;

    void *base = nullptr;
    int sms = 0;
    int st = na_setup(&base, &sms);
    if (st != BLR_OK) return st;
    if (fault_injected("noalloc")) return BLR_ERR_CUDA;

    char *w = static_cast<char *>(base);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + L.header);
    uint32_t *bp_f1 = reinterpret_cast<uint32_t *>(w + L.bp_f1);
    uint32_t *bp_f2 = reinterpret_cast<uint32_t *>(w + L.bp_f2);
    uint16_t *x16 = reinterpret_cast<uint16_t *>(w + L.x16);
    float *a32 = reinterpret_cast<float *>(w + L.a32);
    uint16_t *al16 = reinterpret_cast<uint16_t *>(w + L.al16);
    uint16_t *c16 = reinterpret_cast<uint16_t *>(w + L.c16);

    // the same tile plans as blr_forward
    const GemmPlan p1 = plan_gemm(M, r, sms, 32);
    const GemmPlan p2 = plan_gemm(M, d_out, sms, 64, kWideTileCost);
    GemmMaps m1{}, m2{};
    const auto none = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (!na_tmap(&m1.act, x16, M, d_in, 64, p1.pair ? p1.bt / 2 : p1.bt, true, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !na_tmap(&m1.out32, a32, M, r, 32, 32, false, none) || !na_tmap(&m1.out16, al16, M, r, 32, 32, true, none) ||
        !na_tmap(&m2.act, al16, M, r, 64, p2.pair ? p2.bt / 2 : p2.bt, true, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !na_tmap(&m2.in32, y, M, d_out, 32, 32, false, none) || !na_tmap(&m2.out32, y, M, d_out, 32, 32, false, none) ||
        !na_tmap(&m2.out16, c16, M, d_out, 32, 32, true, none))
        return BLR_ERR_CUDA;

    cudaStream_t s = (cudaStream_t)stream;
    SignPrep pv{bits_v, bp_f1, r, d_in, 1, sign_rows(r)};
    SignPrep pu{bits_u, bp_f2, d_out, r, 0, sign_rows(d_out)};
    if (launch_fwd_prologue(pv, pu, x, g, x16, M, d_in, status, s) != cudaSuccess) return BLR_ERR_CUDA;

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
    if (launch_gemm(kEpiFwd1, p1, m1, f1, s) != cudaSuccess) return BLR_ERR_CUDA;

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
    if (launch_gemm(kEpiFwd2, p2, m2, f2, s) != cudaSuccess) return BLR_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lk(g_na_mu);
        g_na_ran[dev] = true;
    }
    return BLR_OK;
}

extern "C" int blr_noalloc_check_status(blr_stream_t stream, uint32_t *device_code) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BLR_ERR_CUDA;
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_na_mu);
        if (!g_na_ran[dev]) return BLR_ERR_STATE;
        base = g_na_ptr[dev];
    }
    // word 0 of the array (the layout's header) is the status word
    uint32_t code = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&code, base, sizeof(code), cudaMemcpyDeviceToHost, s) != cudaSuccess) return BLR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BLR_ERR_CUDA;
    if (device_code) *device_code = code;
    return code ? BLR_ERR_DEVICE_CHECK : BLR_OK;
}
