// MoE router: f16-rounded logits, top-k with ties to the lower expert id, and
// the softmax over the selected logits (= softmax over all experts
// renormalised over the top-k).
//
// Logits are rounded to f16 before top-k (hipfire PR #694, commit "Executed
// the moeblk golden against real shipped layer-0 weights"), so the f32
// summation order decides which logits tie. The order used here is fixed:
// each fp16*fp16 product is exact in f32; lane l of a warp adds, one at a
// time in ascending index order, the products whose index i has
// floor(i/8) mod 32 == l; the 32 partials are combined by the xor butterfly
// with offsets 16, 8, 4, 2, 1; the result is rounded to f16 (RNE).
#include "common.cuh"
#include "kernels.h"

namespace escha {

namespace {

// One warp per expert; every warp loops over the tokens.
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ Wg, int T, int H, int E,
                                                            uint16_t* __restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    const uint16_t* wrow = Wg + (long long)e * H;
    const int passes = H >> 8;
    for (int t = 0; t < T; ++t) {
        const uint16_t* xrow = x + (long long)t * H;
        float acc = 0.f;
        for (int p = 0; p < passes; ++p) {
            const int i0 = p * 256 + lane * 8;
            const uint4 xv = *reinterpret_cast<const uint4*>(xrow + i0);
            const uint4 wv = *reinterpret_cast<const uint4*>(wrow + i0);
            const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc = fmaf(h2f_bits(static_cast<uint16_t>(xs[k] & 0xFFFFu)),
                           h2f_bits(static_cast<uint16_t>(ws[k] & 0xFFFFu)), acc);
                acc = fmaf(h2f_bits(static_cast<uint16_t>(xs[k] >> 16)), h2f_bits(static_cast<uint16_t>(ws[k] >> 16)),
                           acc);
            }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, m);
        if (lane == 0) logits[(long long)t * E + e] = __half_as_ushort(__float2half_rn(acc));
    }
}

// One warp per token: top-k by (logit desc, id asc), softmax over the k.
__global__ void __launch_bounds__(256) router_topk_kernel(const uint16_t* __restrict__ logits, int T, int E, int topk,
                                                          int32_t* __restrict__ ids, float* __restrict__ w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    constexpr int kPer = 8;  // E <= 256
    float v[kPer];
    bool live[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        live[i] = e < E;
        v[i] = live[i] ? h2f_bits(logits[(long long)t * E + e]) : 0.f;
    }
    float sel_v[8];
    int sel_e[8];
    for (int k = 0; k < topk; ++k) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane + 32 * i;
            if (live[i] && (v[i] > bv || (v[i] == bv && e < be))) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, m);
            const int oe = __shfl_xor_sync(0xffffffffu, be, m);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if (lane + 32 * i == be) live[i] = false;
        sel_v[k] = bv;
        sel_e[k] = be;
    }
    if (lane == 0) {
        float den = 0.f;
        for (int k = 0; k < topk; ++k) den += expf(sel_v[k] - sel_v[0]);
        for (int k = 0; k < topk; ++k) {
            ids[(long long)t * topk + k] = sel_e[k];
            w[(long long)t * topk + k] = expf(sel_v[k] - sel_v[0]) / den;
        }
    }
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, const uint16_t* Wg, int T, int hidden, int E, int topk,
                          uint16_t* logits, int32_t* ids, float* w, unsigned int* counter, cudaStream_t s) {
    (void)counter;
    router_logits_kernel<<<(E + 7) / 8, 256, 0, s>>>(x, Wg, T, hidden, E, logits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    router_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, topk, ids, w);
    return cudaGetLastError();
}

}  // namespace escha
