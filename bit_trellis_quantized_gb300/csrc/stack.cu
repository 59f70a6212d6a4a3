// Residual stream of a stack of MoE blocks: h += add, then the next block's
// fp16 input x = f16_rne(h / sqrt(mean(h^2) + eps)) (a weightless RMSNorm: the
// real model normalises before every MoE block; with random weights and no
// norm the block outputs would leave the fp16 range after a few layers).
//
// The fp16 rounding decides the next router's input, so the arithmetic is
// fixed: per row, thread t of 256 adds h[i]*h[i] (an f32 multiply, then an f32
// add) over i = t, t + 256, ... in ascending order; the 32 lanes of a warp are
// combined by the xor butterfly (offsets 16, 8, 4, 2, 1) and the 8 warp sums
// in warp order; mean = sum / hidden, r = sqrt(mean + eps), inv = 1 / r (IEEE
// division and square root, round to nearest even), x[i] = f16_rne(h[i] * inv).
#include <cuda_fp16.h>

#include "kernels.h"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kNormThreads = 256;
constexpr int kNormMaxPer = 8192 / kNormThreads;

__global__ void __launch_bounds__(kNormThreads) residual_rmsnorm_kernel(float* __restrict__ h,
                                                                         const float* __restrict__ add, int hidden,
                                                                         float eps, uint16_t* __restrict__ x) {
    __shared__ float wsum[kNormThreads / 32];
    __shared__ float inv_s;
    pdl_wait();
    pdl_trigger();
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    float* hr = h + (long long)blockIdx.x * hidden;
    const float* ar = add ? add + (long long)blockIdx.x * hidden : nullptr;
    float v[kNormMaxPer];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kNormMaxPer; ++j) {
        const int i = j * kNormThreads + t;
        if (i < hidden) {
            float hv = hr[i];
            if (ar) {
                hv = __fadd_rn(hv, ar[i]);
                hr[i] = hv;
            }
            v[j] = hv;
            s = __fadd_rn(__fmul_rn(hv, hv), s);
        }
    }
    if (!x) return;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, m));
    if (lane == 0) wsum[warp] = s;
    __syncthreads();
    if (t == 0) {
        float tot = wsum[0];
        for (int w = 1; w < kNormThreads / 32; ++w) tot = __fadd_rn(tot, wsum[w]);
        const float mean = __fdiv_rn(tot, static_cast<float>(hidden));
        inv_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    }
    __syncthreads();
    const float inv = inv_s;
    uint16_t* xr = x + (long long)blockIdx.x * hidden;
#pragma unroll
    for (int j = 0; j < kNormMaxPer; ++j) {
        const int i = j * kNormThreads + t;
        if (i < hidden) xr[i] = __half_as_ushort(__float2half_rn(__fmul_rn(v[j], inv)));
    }
}

}  // namespace

cudaError_t launch_residual_rmsnorm(float* h, const float* add, int T, int hidden, float eps, uint16_t* x,
                                    cudaStream_t s) {
    void* args[] = {&h, const_cast<float**>(&add), &hidden, &eps, &x};
    // programmatic launch: the CTAs wait (griddepcontrol.wait) for the block
    // that wrote `add` instead of waiting to be launched
    return launch_kernel(reinterpret_cast<const void*>(residual_rmsnorm_kernel), dim3(T), dim3(kNormThreads), 0, true,
                         s, args);
}

}  // namespace escha
