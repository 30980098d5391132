// Fused small-M path of the blr layer: the whole forward, and the whole
// backward, each as one cooperative persistent kernel (one CTA per SM) whose
// phases are separated by grid barriers:
//
//   forward:  re-layouts + x staging | a = x16 S_V (a, a.l) | c = (a.l) S_U^T (y, c)
//   backward: re-layouts + dy staging (s_t, sigma_t, dh partials) | db (dl
//             partials, db.l) | dx' (dx, dg partials) | reduction of dh, dl, dg
//
// For small token counts the stand-alone kernels of the general path spend
// most of their time in per-launch costs (launch, TMEM allocation, pipeline
// fill and drain); here TMEM is allocated once, every phase uses every SM,
// and intermediate tensors stay in L2 between phases. The GEMM phases are the
// general path's warp roles (blr_gemm.cuh) with single-CTA 128-token tiles,
// each phase with freshly initialised barriers.
#include "blr_gemm.cuh"
#include "blr_stage.cuh"

namespace blr {

constexpr int kSmallBT = 128;
static_assert(GemmShape<kEpiFwd1, false, kSmallBT>::kThreads <= kGemmThreads &&
                  GemmShape<kEpiFwd2, false, kSmallBT>::kThreads <= kGemmThreads &&
                  GemmShape<kEpiBwd1, false, kSmallBT>::kThreads <= kGemmThreads &&
                  GemmShape<kEpiBwd2, false, kSmallBT>::kThreads <= kGemmThreads,
              "every phase's warp roles fit the fused kernels' block");

// Grid barrier: one arrival per CTA on a counter in global memory that only
// grows during a launch (zeroed before it); barrier k completes at k * grid
// (+ gb.extra). Bounded like every other wait, by gb.wait_ns: on timeout the
// CTA records it and carries on with its abort flag set, so that its
// remaining waits end early.
__device__ __forceinline__ void grid_sync(const GridBarrier &gb, unsigned int k, volatile int *abort_flag,
                                          uint32_t *status) {
    unsigned int *gbar = gb.gbar;
    const unsigned int target = k * gridDim.x + gb.extra;
    __syncthreads();
    if (threadIdx.x == 0) {
        // this CTA's TMA stores and generic writes are complete and visible
        // before its arrival, and the next phase's TMA loads follow the wait
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        atomicAdd(gbar, 1u);
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(gbar) : "memory");
            if (v >= target) break;
            if (globaltimer_ns() - t0 > gb.wait_ns) {
                *abort_flag = 1;
                atomicOr(status, kStTimeoutGrid);
                break;
            }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncthreads();
}

// One GEMM phase over all tiles, every CTA a tile worker.
template <int EPI>
__device__ __forceinline__ void small_gemm_phase(uint8_t *smem, const GemmMaps &m, const GemmArgs &args,
                                                 uint32_t tmem_base, volatile int *abort_flag) {
    const GemmLayout<EPI, false, kSmallBT> L(smem + kCtlBytes);
    if (threadIdx.x == 0) {
        L.init_barriers();
        fence_mbar_init();
    }
    gemm_prefetch_maps<EPI, false, kSmallBT>(m.act, m.in32, m.out32, m.out16);
    __syncthreads();
    gemm_roles<EPI, false, kSmallBT>(L, m.act, m.in32, m.out32, m.out16, args, tmem_base, abort_flag,
                                     (int)blockIdx.x, (int)gridDim.x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) L.inval_barriers();
}

__device__ __forceinline__ uint32_t small_setup(GemmCtl *ctl) {
    if (threadIdx.x == 0) ctl->abort_flag = 0;
    if (threadIdx.x / 32 == kWarpMma) {
        tmem_alloc(&ctl->tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return ctl->tmem_slot;
}

__device__ __forceinline__ void small_teardown(uint32_t tmem_base) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x / 32 == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    blr_small_fwd_kernel(const __grid_constant__ GemmMaps m1, const __grid_constant__ GemmMaps m2,
                         const SmallFwdArgs a) {
    uint8_t *smem = smem_base_1024();
    GemmCtl *ctl = reinterpret_cast<GemmCtl *>(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(&ctl->abort_flag);
    const uint32_t tmem_base = small_setup(ctl);
    // phase 1: status word, bitmap re-layouts, x16 = f16(x.g)
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    prep_share(a.pv, a.pu, (int)blockIdx.x, (int)gridDim.x);
    stage_x_run(a.x, a.g, a.x16, a.M, a.d_in, (int)blockIdx.x, (int)gridDim.x);
    grid_sync(a.gb, 1, abort_flag, a.status);
    // phase 2: a = x16 S_V; a (f32 tape) and a.l (f16)
    small_gemm_phase<kEpiFwd1>(smem, m1, a.f1, tmem_base, abort_flag);
    grid_sync(a.gb, 2, abort_flag, a.status);
    // phase 3: c = (a.l) S_U^T; y (+)= h.c, c (f16)
    small_gemm_phase<kEpiFwd2>(smem, m2, a.f2, tmem_base, abort_flag);
    small_teardown(tmem_base);
}

template <int GPT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    blr_small_bwd_kernel(const __grid_constant__ GemmMaps m1, const __grid_constant__ GemmMaps m2,
                         const SmallBwdArgs a) {
    uint8_t *smem = smem_base_1024();
    GemmCtl *ctl = reinterpret_cast<GemmCtl *>(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(&ctl->abort_flag);
    const uint32_t tmem_base = small_setup(ctl);
    // phase 1: bitmap re-layouts; dy16 = f16(dy.h.s_t), s_t, sigma_t, dh partials
    prep_share(a.pu, a.pv, (int)blockIdx.x, (int)gridDim.x);
    if ((int)blockIdx.x < a.stage_blocks)
        stage_dy_run<GPT>(a.sd, (int)blockIdx.x, a.stage_blocks, reinterpret_cast<float *>(smem + kCtlBytes),
                          a.stage_tpr, a.stage_nthr);
    grid_sync(a.gb, 1, abort_flag, a.b1.status);
    // phase 2: db = dy16 S_U / s_t; dl partials; db.l (f16) under sigma_t
    small_gemm_phase<kEpiBwd1>(smem, m1, a.b1, tmem_base, abort_flag);
    grid_sync(a.gb, 2, abort_flag, a.b1.status);
    // phase 3: dx' = (db.l) S_V^T / sigma_t; dx (+)= g.dx'; dg partials
    small_gemm_phase<kEpiBwd2>(smem, m2, a.b2, tmem_base, abort_flag);
    grid_sync(a.gb, 3, abort_flag, a.b1.status);
    // phase 4: dh, dl, dg += fixed-order sums of the partials
    reduce_partials_run(a.rh, a.rl, a.rg, (int)blockIdx.x, (int)gridDim.x, reinterpret_cast<float *>(smem + kCtlBytes));
    small_teardown(tmem_base);
}

template <typename Args>
static cudaError_t launch_coop(void (*kernel)(GemmMaps, GemmMaps, Args), int grid, size_t smem, cudaStream_t s,
                               const GemmMaps &m1, const GemmMaps &m2, const Args &args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, m1, m2, args);
}

size_t small_fwd_smem() {
    const size_t a = GemmShape<kEpiFwd1, false, kSmallBT>::kSmemBytes;
    const size_t b = GemmShape<kEpiFwd2, false, kSmallBT>::kSmemBytes;
    return a > b ? a : b;
}

size_t small_bwd_smem(size_t stage_bytes) {
    size_t m = GemmShape<kEpiBwd1, false, kSmallBT>::kSmemBytes;
    const size_t b = GemmShape<kEpiBwd2, false, kSmallBT>::kSmemBytes;
    if (b > m) m = b;
    if (1024 + kCtlBytes + stage_bytes > m) m = 1024 + kCtlBytes + stage_bytes;
    return m;
}

cudaError_t launch_small_fwd(const GemmMaps &m1, const GemmMaps &m2, const SmallFwdArgs &a, int grid,
                             cudaStream_t s) {
    const size_t smem = small_fwd_smem();
    cudaError_t pe = prepare_kernel_once(blr_small_fwd_kernel, (int)smem);
    if (pe != cudaSuccess) return pe;
    trace_before("small_fwd", s);
    cudaError_t e = cudaMemsetAsync(a.gb.gbar, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = launch_coop(blr_small_fwd_kernel, grid, smem, s, m1, m2, a);
    trace_after(s);
    return e;
}

template <int GPT>
static cudaError_t launch_small_bwd_t(const GemmMaps &m1, const GemmMaps &m2, const SmallBwdArgs &a, int grid,
                                      cudaStream_t s) {
    const size_t smem = small_bwd_smem(stage_dy_smem_bytes(a.sd.d_out, a.stage_tpr, a.stage_nthr));
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t pe = prepare_kernel_once(blr_small_bwd_kernel<GPT>, 227 * 1024);
    if (pe != cudaSuccess) return pe;
    trace_before("small_bwd", s);
    cudaError_t e = cudaMemsetAsync(a.gb.gbar, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = launch_coop(blr_small_bwd_kernel<GPT>, grid, smem, s, m1, m2, a);
    trace_after(s);
    return e;
}

// Staging geometry of the fused backward: threads per token row (a power of
// two, at most 256 so that one row fits the CTA's 448 threads) and float4
// groups per thread.
static int small_stage_tpr(int d_out) {
    const int t = stage_tpr(d_out);
    return t > 256 ? 256 : t;
}

bool small_bwd_fits(int d_out) {
    const int tpr = small_stage_tpr(d_out);
    return (d_out / 4 + tpr - 1) / tpr <= 8;
}

cudaError_t launch_small_bwd(const GemmMaps &m1, const GemmMaps &m2, SmallBwdArgs a, int grid, int rows_dh_reserved,
                             cudaStream_t s) {
    a.stage_tpr = small_stage_tpr(a.sd.d_out);
    a.stage_nthr = (kGemmThreads / a.stage_tpr) * a.stage_tpr;
    a.stage_blocks = grid < rows_dh_reserved ? grid : rows_dh_reserved;
    a.rh.rows = a.stage_blocks;
    if (a.sd.rows_used) *a.sd.rows_used = a.stage_blocks;
    const int gpt = (a.sd.d_out / 4 + a.stage_tpr - 1) / a.stage_tpr;
    if (gpt <= 2) return launch_small_bwd_t<2>(m1, m2, a, grid, s);
    if (gpt <= 8) return launch_small_bwd_t<8>(m1, m2, a, grid, s);
    return cudaErrorInvalidValue;
}

}  // namespace blr
