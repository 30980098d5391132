// One Adam step over the layer's vectors (train_mm.rs, WGSL adam kernel and
// its wrapper adam): elementwise, f32 as on the page, no weight decay.
//   gr = grad * gmul;  m1 = b1 m1 + (1 - b1) gr;  m2 = b2 m2 + (1 - b2) gr^2
//   st = lr (m1 / (1 - b1^t)) / (sqrt(m2 / (1 - b2^t)) + eps)
//   w -= st * max(|w|, rel)  (rel > 0: relative steps)   or   w -= st
// Entries whose mask value is exactly 0 are left untouched. The two bias
// corrections 1 - b^t are formed once on the host (in double), not per element.
#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

__global__ void __launch_bounds__(256) adam_kernel(const AdamArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < a.n;
         i += (long long)gridDim.x * blockDim.x) {
        if (a.mask && a.mask[i] == 0.0f) continue;
        const float gr = a.grad[i] * a.gmul;
        const float m1 = a.b1 * a.m1[i] + (1.0f - a.b1) * gr;
        const float m2 = a.b2 * a.m2[i] + (1.0f - a.b2) * gr * gr;
        a.m1[i] = m1;
        a.m2[i] = m2;
        const float st = a.lr * (m1 / a.bc1) / (sqrtf(m2 / a.bc2) + a.eps);
        const float w = a.w[i];
        a.w[i] = a.rel > 0.0f ? w - st * fmaxf(fabsf(w), a.rel) : w - st;
    }
}

cudaError_t launch_adam(const AdamArgs &a, int sms, cudaStream_t s) {
    long long blocks = (a.n + 255) / 256;
    if (blocks > 4LL * sms) blocks = 4LL * sms;
    if (blocks < 1) blocks = 1;
    trace_before("adam", s);
    const cudaError_t e = launch_k(adam_kernel, dim3((unsigned)blocks), dim3(256), 0, s, a);
    trace_after(s);
    return e;
}

}  // namespace blr
