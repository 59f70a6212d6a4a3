// Internal launch interfaces between the C-ABI layer (escha_api.cu) and the
// kernels. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace escha {

// Input modes of the trellis GEMV prologue.
constexpr int kXmF16 = 0;     // x is fp16 [rows][in]
constexpr int kXmF32 = 1;     // x is f32 [rows][in]
constexpr int kXmSwiglu = 2;  // x is a gate_up output f32 [rows][2*in]; input = silu(gate) * up

struct GemvArgs {
    const uint16_t* codes;  // expert 0's code tensor [in/16][out/16][16K]
    long long code_stride;  // words between consecutive experts' code tensors
    int in, out;
    int kt_per_cta;  // filled by the launcher
    int x_mode;
    const void* x;
    long long x_stride;  // elements between x rows
    const uint16_t* rin;
    long long rin_stride;  // elements between experts
    const uint16_t* rout;
    long long rout_stride;
    float* y;
    long long y_stride;
    // items: slot mode (one token per item, expert ids[item], x row item/x_div)
    // or plain mode (tokens item*NB .. item*NB+NB-1 of `batch`, expert 0)
    const int32_t* ids;
    int x_div;
    int batch;
    int slot_mode;
};

// Trellis GEMV. nb = tokens per item in plain mode (1, 2 or 4); items = grid z.
cudaError_t launch_trellis_gemv(const GemvArgs& a, int K, int nb, int items, int num_sms, cudaStream_t s);

// Dense decode of a code tensor to fp16 bit patterns W[in][out].
cudaError_t launch_trellis_decode(const uint16_t* codes, int in, int out, int K, uint16_t* W, cudaStream_t s);

// Router: logits (f16 bits) [T][E], then top-k + softmax. `counter` is a
// zeroed int in device memory used to elect the CTA that runs the top-k.
cudaError_t launch_router(const uint16_t* x, const uint16_t* Wg, int T, int hidden, int E, int topk,
                          uint16_t* logits, int32_t* ids, float* w, unsigned int* counter, cudaStream_t s);

// int8 w8a16 matvec / small-M GEMV: y[m][o] = sum_i (scale[o]*W[o][i]) * x[m][i].
// x_dtype: 1 = f16, 2 = bf16, 3 = f32; act = 0 plain, 1 SwiGLU of a
// [M][2*Kin] f32 input (gate first).
cudaError_t launch_int8_gemv(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                             long long x_stride, int act, int M, float* y, long long y_stride, int num_sms,
                             cudaStream_t s);

cudaError_t launch_int8_dequant(const int8_t* W, const float* scales, int N, int Kin, float* out, cudaStream_t s);

// MoE combine: out[t][i] = sum_j w[t][j] * d[t*topk + j][i] + sigmoid(g . x[t]) * sh[t][i]
// (sh may be null: no shared expert).
cudaError_t launch_moe_combine(const float* d, const float* w, int T, int topk, int hidden, const float* sh,
                               const uint16_t* sh_gate, const uint16_t* x, float* out, cudaStream_t s);

}  // namespace escha
