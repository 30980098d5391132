// plane_linear's staging (train_mm.rs, plane_linear: `cvt` of x under the
// caller's scale into the f16 activation buffer): act16 = f16(x * scale),
// round to nearest even, 8 values per thread step (two 16-byte loads, one
// 16-byte store). Block 0 also clears the workspace status word, which the
// product that follows reports into.
#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

__global__ void __launch_bounds__(256) plane_stage_kernel(const float *x, uint16_t *act16, long long n8, float scale,
                                                          uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    uint4 *o = reinterpret_cast<uint4 *>(act16);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (long long)gridDim.x * blockDim.x) {
        const float4 a = __ldcs(x4 + 2 * i), b = __ldcs(x4 + 2 * i + 1);
        uint4 w;
        w.x = pack_half2(a.x * scale, a.y * scale);
        w.y = pack_half2(a.z * scale, a.w * scale);
        w.z = pack_half2(b.x * scale, b.y * scale);
        w.w = pack_half2(b.z * scale, b.w * scale);
        o[i] = w;
    }
}

cudaError_t launch_plane_stage(const float *x, uint16_t *act16, long long n, float scale, uint32_t *status, int sms,
                               cudaStream_t s) {
    const long long n8 = n / 8;
    long long blocks = (n8 + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    if (blocks < 1) blocks = 1;
    trace_before("plane_stage", s);
    const cudaError_t e = launch_k(plane_stage_kernel, dim3((unsigned)blocks), dim3(256), 0, s, x, act16, n8, scale,
                                   status);
    trace_after(s);
    return e;
}

}  // namespace blr
