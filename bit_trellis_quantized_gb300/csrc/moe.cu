// MoE combine: out[t] = sum_j w[t][j] * d[t*topk + j] + sigmoid(g . x[t]) * sh[t]
// with the routed terms summed in slot order and the shared expert gated by
// a sigmoid of an unrounded f32 dot product (MLX model card, "Router gates
// (mlp.gate, shared_expert_gate) fp16"; the combine itself is the standard
// Qwen MoE block the pages serve).
#include "common.cuh"
#include "kernels.h"

namespace escha {

namespace {

__global__ void __launch_bounds__(256) moe_combine_kernel(const float* __restrict__ d, const float* __restrict__ w,
                                                          int topk, int hidden, const float* __restrict__ sh,
                                                          const uint16_t* __restrict__ sh_gate,
                                                          const uint16_t* __restrict__ x, float* __restrict__ out) {
    const int t = blockIdx.y;
    __shared__ float red[8];
    __shared__ float gate_s;
    float gate = 0.f;
    if (sh) {
        const uint16_t* xr = x + (long long)t * hidden;
        float acc = 0.f;
        for (int i = threadIdx.x; i < hidden; i += 256) acc = fmaf(h2f_bits(sh_gate[i]), h2f_bits(xr[i]), acc);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s = 0.f;
            for (int i = 0; i < 8; ++i) s += red[i];
            gate_s = sigmoid_f(s);
        }
        __syncthreads();
        gate = gate_s;
    }
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= hidden) return;
    float acc = 0.f;
    for (int j = 0; j < topk; ++j) acc = fmaf(w[(long long)t * topk + j], d[((long long)t * topk + j) * hidden + i], acc);
    if (sh) acc = fmaf(gate, sh[(long long)t * hidden + i], acc);
    out[(long long)t * hidden + i] = acc;
}

}  // namespace

cudaError_t launch_moe_combine(const float* d, const float* w, int T, int topk, int hidden, const float* sh,
                               const uint16_t* sh_gate, const uint16_t* x, float* out, cudaStream_t s) {
    dim3 grid((hidden + 255) / 256, T);
    moe_combine_kernel<<<grid, 256, 0, s>>>(d, w, topk, hidden, sh, sh_gate, x, out);
    return cudaGetLastError();
}

}  // namespace escha
