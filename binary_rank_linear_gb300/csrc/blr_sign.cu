// Sign gradients of the blr layer (train_mm.rs, blr_backward documentation
// and its test helper host_sign_grads):
//
//     G_U[i][k] = h_i l_k sum_t dy[t][i] a[t][k]        [d_out][r]
//     G_V[j][k] = g_j l_k sum_t x[t][j]  b[t][k]        [d_in][r],  b = db
//
// Two dense products with the tokens as the reduction dimension. The pass
// already holds every factor in f16, token-major: dy16 = dy.h.s_t,
// x16 = x.g, al16 = a.l, db16 = db.l.sigma_t. The pages transpose their
// operands into token-contiguous copies first (`cvt_t`); here the MMAs read
// the token-major arrays as they are, as MN-major operands (the feature or
// rank index contiguous, K = tokens strided), so no transposed copy exists.
//
// A product over tokens needs one gradient scale. With a fixed scale the
// staged arrays serve directly. With per-token powers of two, the rank-side
// operands are rescaled first: bu = al16 (1/s_t)/max(1/s_t) and
// bv = db16 (1/sigma_t)/max(1/sigma_t), powers of two <= 1 (exact unless a
// value falls into the f16 subnormals); the maxima multiply the products back.
// The two products themselves run on the dense tensor-core GEMM of
// blr_dense.cu (both operands MN-major).
#include "blr_device.cuh"
#include "blr_kernels.h"

namespace blr {

// ------------------------------------------------------------ rescale -----
// 8 f16 per thread step (16-byte accesses); every block first reduces the
// staging's per-block maxima (a few hundred pairs, from L2).
__global__ void __launch_bounds__(256) sign_rescale_kernel(const SignRescaleArgs a) {
    __shared__ float2 mx_s;
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x < 32) {
        float2 m = make_float2(0.0f, 0.0f);
        for (int i = threadIdx.x; i < a.nblk; i += 32) {
            const float2 v = a.blkmax[i];
            m.x = fmaxf(m.x, v.x);
            m.y = fmaxf(m.y, v.y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m.x = fmaxf(m.x, __shfl_xor_sync(0xFFFFFFFFu, m.x, o));
            m.y = fmaxf(m.y, __shfl_xor_sync(0xFFFFFFFFu, m.y, o));
        }
        if (threadIdx.x == 0) {
            // no row with a nonzero gradient: every operand row is zero, any scale will do
            if (!(m.x > 0.0f)) m.x = 1.0f;
            if (!(m.y > 0.0f)) m.y = 1.0f;
            mx_s = m;
            if (blockIdx.x == 0) {
                a.gmax[0] = m.x;
                a.gmax[1] = m.y;
            }
        }
    }
    __syncthreads();
    const float inv_u = 1.0f / mx_s.x, inv_v = 1.0f / mx_s.y;  // powers of two
    const int vpr = a.r / 8;                                      // 16-byte groups per row
    const long long n = (long long)a.M * vpr;
    const uint4 *al = reinterpret_cast<const uint4 *>(a.al16);
    const uint4 *db = reinterpret_cast<const uint4 *>(a.db16);
    uint4 *bu = reinterpret_cast<uint4 *>(a.bu);
    uint4 *bv = reinterpret_cast<uint4 *>(a.bv);
    auto scale8 = [](uint4 w, float f) {
        uint32_t *p = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&p[i]));
            p[i] = pack_half2(v.x * f, v.y * f);
        }
        return w;
    };
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / vpr);
        const float fu = __ldg(a.s_inv + t) * inv_u;
        const float fv = __ldg(a.sig_inv + t) * inv_v;
        bu[i] = scale8(al[i], fu);
        bv[i] = scale8(db[i], fv);
    }
}

// ------------------------------------------------------------ launcher ---
cudaError_t launch_sign_rescale(const SignRescaleArgs &a, int sms, cudaStream_t s) {
    const long long n = (long long)a.M * (a.r / 8);
    long long blocks = (n + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    trace_before("sign_rescale", s);
    const cudaError_t e = launch_k(sign_rescale_kernel, dim3((unsigned)blocks), dim3(256), 0, s, a);
    trace_after(s);
    return e;
}

}  // namespace blr
