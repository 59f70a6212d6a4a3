// Device helpers shared by the kernels of the trellis MoE library (sm_103a).
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace escha {

namespace cg = cooperative_groups;

// ---------------------------------------------------------------------------
// Trellis codebook "cbA" (hipfire PR #694 summary, "What it is"; MLX model
// card table "Exactness of every tensor"): a 16-bit state s hashes to
//   r = ((s * 0xCBAC1FED) & 0x8FFF8FFF) ^ 0x3B603B60
// whose two fp16 halves are summed with round-to-nearest-even. __hadd is the
// IEEE fp16 add (RNE); both halves have exponent fields 12..15, so neither
// operand nor result is ever subnormal.
// ---------------------------------------------------------------------------
constexpr uint32_t kCbMul = 0xCBAC1FEDu;
constexpr uint32_t kCbMask = 0x8FFF8FFFu;
constexpr uint32_t kCbXor = 0x3B603B60u;

__device__ __forceinline__ __half cb_decode_h(uint32_t s) {
    const uint32_t u = s * kCbMul;
    const uint32_t r = (u & kCbMask) ^ kCbXor;
    const __half2 h = *reinterpret_cast<const __half2*>(&r);
    return __hadd(__low2half(h), __high2half(h));
}

__device__ __forceinline__ float cb_decode_f(uint32_t s) { return __half2float(cb_decode_h(s)); }

// Two decodes packed as one half2 (a in .x, b in .y).
// Each state's two halves are added by their own fp16 add (round to nearest
// even, like the pairwise form) and the sums packed: measured faster on GB300
// than gathering the low and the high halves first (fewer byte permutes on
// the integer pipe, which the decode saturates).
__device__ __forceinline__ __half2 cb_decode_h2(uint32_t sa, uint32_t sb) {
    const uint32_t ra = ((sa * kCbMul) & kCbMask) ^ kCbXor;
    const uint32_t rb = ((sb * kCbMul) & kCbMask) ^ kCbXor;
    const __half2 a2 = *reinterpret_cast<const __half2*>(&ra), b2 = *reinterpret_cast<const __half2*>(&rb);
    return __halves2half2(__hadd(__low2half(a2), __high2half(a2)), __hadd(__low2half(b2), __high2half(b2)));
}

// K = 2 pair decode. Weights t and t + 8 of a lane's stream (16 bits apart)
// share one 32-bit window P = s_t << 16 | s_{t+8}: one funnel shift extracts
// both states, and s_{t+8} * m = P * m - (s_t * m) << 16 (mod 2^32) costs a
// multiply-add instead of two integer-pipe instructions.
// Word pair p = w[2i] | w[2i+1] << 16 in stream order: (w[2i] << 16) | w[2i+1].
__device__ __forceinline__ uint32_t stream_pair(uint32_t p) { return __byte_perm(p, 0u, 0x1032); }
// 32 stream bits starting at bit O of q0 (q1 follows q0)
template <int O>
__device__ __forceinline__ uint32_t bits32(uint32_t q0, uint32_t q1) {
    if constexpr (O == 0) {
        return q0;
    } else {
        return __funnelshift_l(q1, q0, O);
    }
}
// codebook value from the product u = s * kCbMul
__device__ __forceinline__ __half cb_finish(uint32_t u) {
    const uint32_t r = (u & kCbMask) ^ kCbXor;
    const __half2 h = *reinterpret_cast<const __half2*>(&r);
    return __hadd(__low2half(h), __high2half(h));
}
// the two codebook values of the window P (states P >> 16 and P & 0xFFFF)
__device__ __forceinline__ void cb_decode_window(uint32_t P, __half& wa, __half& wb) {
    const uint32_t ua = (P >> 16) * kCbMul;
    const uint32_t ub = ua * 0xFFFF0000u + P * kCbMul;
    wa = cb_finish(ua);
    wb = cb_finish(ub);
}

// ---------------------------------------------------------------------------
// Bit-stream windows. A lane holds consecutive 16-bit code words w[0..n) as
// little-endian pairs p[i] = w[2i] | w[2i+1] << 16 (what a vector load of the
// words gives). window(a) = (w[a] << 16) | w[a+1]: 32 stream bits starting at
// word a, most significant bit first. The state at bit offset o (0..15) of
// word a is (window(a) >> (16 - o)) & 0xffff.
// ---------------------------------------------------------------------------
template <int A>
__device__ __forceinline__ uint32_t stream_window(const uint32_t* p) {
    if constexpr (A % 2 == 0) {
        return __byte_perm(p[A / 2], 0u, 0x1032);
    } else {
        return __byte_perm(p[A / 2], p[A / 2 + 1], 0x3254);
    }
}

template <int O>
__device__ __forceinline__ uint32_t window_state(uint32_t win) {
    if constexpr (O == 0) {
        return win >> 16;
    } else if constexpr (O == 8) {
        return __byte_perm(win, 0u, 0x4421);
    } else {
        return (win >> (16 - O)) & 0xFFFFu;
    }
}

// ---------------------------------------------------------------------------
// Warp-level Sylvester Hadamard-128 (unscaled) of 128 values held as 4
// consecutive values per lane: v[j] is element 4*lane + j. Index bits 0-1
// live inside the lane, bits 2-6 across lanes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void h128_warp(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float p = __shfl_xor_sync(0xffffffffu, v[j], m);
            v[j] = upper ? (p - v[j]) : (v[j] + p);
        }
    }
}

// ---------------------------------------------------------------------------
// Loads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ldg_stream_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// Router dot products: acc += x.lo * w.lo, then acc += x.hi * w.hi, fp16
// operands and an f32 accumulator, one rounding per step (the product of two
// fp16 values is exact in f32, so this equals an f32 fma of the converted
// operands). dot8_f16 takes 8 consecutive columns in order.
__device__ __forceinline__ void fma2_f16(uint32_t x2, uint32_t w2, float& acc) {
    asm("{\n\t.reg .f16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.f16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.f16 %0, xh, wh, %0;\n\t}"
        : "+f"(acc)
        : "r"(x2), "r"(w2));
}

__device__ __forceinline__ void dot8_f16(const uint4& xv, const uint4& wv, float& acc) {
    fma2_f16(xv.x, wv.x, acc);
    fma2_f16(xv.y, wv.y, acc);
    fma2_f16(xv.z, wv.z, acc);
    fma2_f16(xv.w, wv.w, acc);
}

__device__ __forceinline__ float h2f_bits(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ float bf2f_bits(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float g) { return 1.0f / (1.0f + expf(-g)); }

// Activation element load by dtype tag (1 = f16, 2 = bf16, 3 = f32).
__device__ __forceinline__ float load_act(const void* base, long long idx, int dtype) {
    if (dtype == 3) return static_cast<const float*>(base)[idx];
    const uint16_t b = static_cast<const uint16_t*>(base)[idx];
    return dtype == 1 ? h2f_bits(b) : bf2f_bits(b);
}

}  // namespace escha

#include <utility>

namespace escha {

// Compile-time loop: f(std::integral_constant<int, i>) for i = 0..N-1.
template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    static_for_impl(f, std::make_integer_sequence<int, N>{});
}

}  // namespace escha
