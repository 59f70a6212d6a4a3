// One MoE block of an Escha-W2 Qwen3.6-35B-A3B-style layer in three kernels
// chained by programmatic dependent launch:
//
//  1. router logits: f16-rounded logits in a fixed summation order (hipfire
//     PR #694, commit "Executed the moeblk golden against real shipped
//     layer-0 weights": logits are rounded to f16 before top-k), one warp per
//     expert spread over many SMs so the 1 MB router matrix streams in one
//     memory round trip. Extra CTAs of the same grid compute the int8 shared
//     expert's gate_up rows and its sigmoid gate.
//  2. gate_up: each routed CTA selects its token's top-k (ties to the lower
//     expert id) and softmax weights with one warp, then runs the expert's
//     gate_up projection (fused trellis decode GEMV with the input/output
//     Hadamard transforms and rout); a cluster splits the input rows and
//     pushes its partial sums into rank 0.
//  3. down + combine: one cluster per (token, 128-wide output block), rank
//     j*ks + h = routed expert j, input split h; every rank also computes an
//     equal share of the shared expert's down rows of the block. Ranks push
//     partials into rank 0, which finishes each expert (output transform,
//     routing weight), sums the experts in slot order and adds the shared
//     expert (SwiGLU with gate = first half: hipfire PR #694, commit "The
//     accumulation loop treated a zero activation as a no-op").
#include "kernels.h"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kK0Threads = 128;
constexpr int kK0Warps = kK0Threads / 32;
constexpr int kLgTG = 8;            // tokens per logits CTA
constexpr int kShMT = 4;            // tokens per pass of the shared-expert rows
constexpr int kShRowsPerWarp = 2;   // shared-expert rows per warp
constexpr int kGuThreads = 256;
constexpr int kGuWarps = kGuThreads / 32;
constexpr int kDnThreads = 256;
constexpr int kDnWarps = kDnThreads / 32;
constexpr int kMaxCluster = 16;
// SM count the input splits are sized for (GB300). A constant rather than the
// device's count, so a split, and with it the order of the partial sums, is a
// fixed function of the shape.
constexpr int kWaveSms = 152;

// ---------------------------------------------------------------------------
// 1. Router logits + shared expert gate_up.
// Summation order of a logit (its f16 rounding depends on it): lane l of the
// expert's warp adds, one at a time in ascending index order, the exact f32
// products x[i] * Wg[e][i] whose index has floor(i/8) mod 32 == l; the 32
// partials are combined by the xor butterfly (offsets 16, 8, 4, 2, 1) and
// rounded to f16 (RNE).
// ---------------------------------------------------------------------------
// Residual norm of tokens t0 .. t0+nt-1 (nt <= NT) by one CTA of 128 threads,
// hidden <= 2048: x = f16_rne(v * inv) with v = h + add, into xh (fp16,
// [nt][hidden], shared memory), in exactly the arithmetic of
// residual_rmsnorm_kernel: that kernel's thread u of 256 sums v_i^2 over
// i = u, u+256, ...; here thread r plays u = 2r and u = 2r+1 (one float2
// per step), so a warp holds two of the 256-thread kernel's warps (lanes 0-15
// and 16-31); its xor butterfly over offsets 16, 8, 4, 2, 1 becomes lane
// offsets 8, 4, 2, 1 and the add of the thread's two sums. Ends with the CTA
// synchronised.
template <int NT>
__device__ void resid_norm_cta(const MoeArgs& a, int t0, int nt, uint16_t* xh) {
    constexpr int J = 2048 / 256;
    __shared__ float wsum[NT][8];
    const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
    float2 v[NT][J];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int i = 2 * r + 256 * j;
            v[t][j] = make_float2(0.f, 0.f);
            if (t < nt && i < a.hidden) {
                const long long o = (long long)(t0 + t) * a.hidden + i;
                const float2 hv = __ldg(reinterpret_cast<const float2*>(a.rs_h + o));
                if (a.rs_add) {
                    const float2 av = __ldg(reinterpret_cast<const float2*>(a.rs_add + o));
                    v[t][j] = make_float2(__fadd_rn(hv.x, av.x), __fadd_rn(hv.y, av.y));
                } else {
                    v[t][j] = hv;
                }
            }
        }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            if (2 * r + 256 * j < a.hidden) {
                s0 = __fadd_rn(__fmul_rn(v[t][j].x, v[t][j].x), s0);
                s1 = __fadd_rn(__fmul_rn(v[t][j].y, v[t][j].y), s1);
            }
        }
#pragma unroll
        for (int m = 8; m >= 1; m >>= 1) {
            s0 = __fadd_rn(s0, __shfl_xor_sync(0xffffffffu, s0, m));
            s1 = __fadd_rn(s1, __shfl_xor_sync(0xffffffffu, s1, m));
        }
        s0 = __fadd_rn(s0, s1);
        if ((lane & 15) == 0) wsum[t][2 * warp + (lane >> 4)] = s0;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t >= nt) break;
        float tot = wsum[t][0];
#pragma unroll
        for (int w = 1; w < 8; ++w) tot = __fadd_rn(tot, wsum[t][w]);
        const float mean = __fdiv_rn(tot, static_cast<float>(a.hidden));
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.rs_eps)));
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int i = 2 * r + 256 * j;
            if (i < a.hidden) {
                const uint32_t lo = __half_as_ushort(__float2half_rn(__fmul_rn(v[t][j].x, inv)));
                const uint32_t hi = __half_as_ushort(__float2half_rn(__fmul_rn(v[t][j].y, inv)));
                *reinterpret_cast<uint32_t*>(xh + t * a.hidden + i) = lo | (hi << 16);
            }
        }
    }
    __syncthreads();
}

// FUSED (residual block, <= kFusedNormMaxT tokens, hidden <= 2048): x is
// computed by resid_norm_cta into xh (shared memory) after the wait, and CTA
// x = 0 also stores it as the block's x for the later kernels.
// t0: the CTA's first token (of a.T); tab (multi-layer launch): the table
// CTA (0, 0) stores at a.lay once the preceding kernel has finished.
template <bool FUSED>
__device__ void router_logits(const MoeArgs& a, int warp, int lane, uint16_t* xh, int t0, const MlTable* tab) {
    const int e = blockIdx.x * kK0Warps + warp;
    const int nt = min(kLgTG, a.T - t0);
    const uint16_t* wrow = a.router_w + (long long)(e < a.E ? e : 0) * a.hidden;
    const int passes = a.hidden >> 8;
    float acc[kLgTG];
#pragma unroll
    for (int t = 0; t < kLgTG; ++t) acc[t] = 0.f;
    for (int pg = 0; pg < passes; pg += 8) {
        uint4 wv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (pg + q < passes) wv[q] = ldg_stream_v4(wrow + (pg + q) * 256 + lane * 8);
        if (pg == 0) {
            // the first weights are in flight; x (and the workspace, which the
            // previous call's kernels may still read) only after the wait
            pdl_wait();
            if (blockIdx.x == 0 && blockIdx.y == 0) {  // the previous call has finished
                if (threadIdx.x == 0) *a.err = 0;
                if (tab)
                    for (int i = threadIdx.x; i < a.lay_n * static_cast<int>(sizeof(MoeLayerPtrs) / 8); i += kK0Threads)
                        reinterpret_cast<unsigned long long*>(a.lay)[i] = reinterpret_cast<const unsigned long long*>(tab->l)[i];
                // one token on the fused path: the expert kernel's counters start at zero
                if (a.fz_ctr)
                    for (int i = threadIdx.x; i < kFzCtrWords; i += kK0Threads) a.fz_ctr[i] = 0u;
            }
            if constexpr (FUSED) {
                resid_norm_cta<kFusedNormMaxT>(a, t0, nt, xh);
                if (blockIdx.x == 0) {
                    const int n16 = nt * a.hidden / 8;
                    for (int u = threadIdx.x; u < n16; u += kK0Threads)
                        reinterpret_cast<uint4*>(a.x_norm + (long long)t0 * a.hidden)[u] = reinterpret_cast<const uint4*>(xh)[u];
                }
            }
            if (e >= a.E) return;
        }
#pragma unroll
        for (int t = 0; t < kLgTG; ++t) {
            if (t < nt) {
                uint4 xv[8];
                if constexpr (FUSED) {
                    const uint16_t* xrow = xh + t * a.hidden;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (pg + q < passes) xv[q] = *reinterpret_cast<const uint4*>(xrow + (pg + q) * 256 + lane * 8);
                } else {
                    const uint16_t* xrow = a.x + (long long)(t0 + t) * a.hidden;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (pg + q < passes) xv[q] = __ldg(reinterpret_cast<const uint4*>(xrow + (pg + q) * 256 + lane * 8));
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (pg + q < passes) dot8_f16(xv[q], wv[q], acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kLgTG; ++t) {
        if (t < nt) {
            float v = acc[t];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, m);
            if (lane == 0) a.logits[(long long)(t0 + t) * a.E + e] = __half_as_ushort(__float2half_rn(v));
        }
    }
}

// x rows tb .. tb+mt-1 as f32 at xs[xs_swz(t*hidden + i)] (zeros for rows
// t >= mt up to MT), by the CTA's NW warps; each thread issues its loads in
// batches of 8 before storing any, so staging costs one L2 round trip per
// batch instead of one per load.
template <int NW, int MT>
__device__ __forceinline__ void stage_x_f32(const MoeArgs& a, int tb, int mt, float* xs) {
    constexpr int kB = 8, kStride = NW * 32;
    const int n = MT * a.hidden;
    for (int u0 = threadIdx.x; u0 * 8 < n; u0 += kB * kStride) {
        uint4 v[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int i = (u0 + b * kStride) * 8, t = i / a.hidden;
            v[b] = (i < n && t < mt) ? __ldg(reinterpret_cast<const uint4*>(a.x + (long long)(tb + t) * a.hidden + i % a.hidden))
                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int i = (u0 + b * kStride) * 8;
            if (i >= n) break;
            *reinterpret_cast<float4*>(xs + xs_swz(i)) =
                make_float4(h2f_bits(v[b].x & 0xFFFFu), h2f_bits(v[b].x >> 16), h2f_bits(v[b].y & 0xFFFFu), h2f_bits(v[b].y >> 16));
            *reinterpret_cast<float4*>(xs + xs_swz(i + 4)) =
                make_float4(h2f_bits(v[b].z & 0xFFFFu), h2f_bits(v[b].z >> 16), h2f_bits(v[b].w & 0xFFFFu), h2f_bits(v[b].w >> 16));
        }
    }
}

// Shared expert gate_up rows (kShRowsPerWarp per warp of NW) for every
// token, MT tokens per pass, and in warp NW-1 of CTA 0 the sigmoid gate (an
// f32 dot product of the fp16 gate vector with x, not rounded). Every sum
// runs in one order, whichever variant computes it: lane l adds, per row and
// token, the products of its 16 columns c*512 + 16l .. +15 for c = 0, 1, ...
// in column order (int8 rows), or of its 8 columns 256k + 8l .. +7 for k = 0,
// 1, ... (gate), and the 32 lanes are combined by the xor butterfly.
//
// Large hidden sizes: rows and gate vector are fetched into L2 before the wait
// for the preceding kernel and read with int8_rows_dot.
template <int NW, int MT>
__device__ void shared_gate_up_staged(const MoeArgs& a, int cta, float* xs, int warp, int lane) {
    constexpr int R = kShRowsPerWarp;
    const int rows = 2 * a.sh_inter;
    const int r0 = (cta * NW + warp) * R;
    const int nrows = min(R, rows - r0);  // <= 0: no rows in this warp
    const bool gate = cta == 0 && warp == NW - 1;
    const long long nb = nrows > 0 ? (long long)nrows * a.hidden : 0;  // bytes of this warp's rows
    for (long long off = lane * 128LL; off < nb; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.sh_gu_w8 + (long long)r0 * a.hidden + off));
    if (gate)
        for (int off = lane * 128; off < 2 * a.hidden; off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(a.sh_gate) + off));
    pdl_wait();  // x, and the workspace the previous call's kernels may still read
    for (int tb = 0; tb < a.T; tb += MT) {
        const int mt = min(MT, a.T - tb);
        __syncthreads();
        stage_x_f32<NW, MT>(a, tb, mt, xs);
        __syncthreads();
        if (nrows > 0) {
            float dots[R][MT];
            int8_rows_dot<R, MT>(a.sh_gu_w8 + (long long)r0 * a.hidden, a.hidden, nrows, a.hidden, xs, a.hidden, lane,
                                 dots);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= nrows) break;
                    const float sc = a.sh_gu_scale[r0 + r];
                    for (int t = 0; t < mt; ++t) a.shgu[(long long)(tb + t) * rows + r0 + r] = sc * dots[r][t];
                }
            }
        }
        if (gate) {
#pragma unroll 1
            for (int t = 0; t < mt; ++t) {
                float acc = 0.f;
#pragma unroll 1
                for (int i0 = lane * 8; i0 < a.hidden; i0 += 256) {
                    const uint4 g4 = __ldg(reinterpret_cast<const uint4*>(a.sh_gate + i0));
                    const float4 xa = *reinterpret_cast<const float4*>(xs + xs_swz(t * a.hidden + i0));
                    const float4 xb = *reinterpret_cast<const float4*>(xs + xs_swz(t * a.hidden + i0 + 4));
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.x & 0xFFFFu)), xa.x, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.x >> 16)), xa.y, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.y & 0xFFFFu)), xa.z, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.y >> 16)), xa.w, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.z & 0xFFFFu)), xb.x, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.z >> 16)), xb.y, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.w & 0xFFFFu)), xb.z, acc);
                    acc = fmaf(h2f_bits(static_cast<uint16_t>(g4.w >> 16)), xb.w, acc);
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
                if (lane == 0) a.shgate[tb + t] = sigmoid_f(acc);
            }
        }
    }
}

// hidden <= 2048: a warp's int8 rows and the gate vector are loaded into
// registers before the wait; after it the rows are converted to f32 once and
// each token is a short loop over shared-memory x (code executed once per warp
// is kept small: straight-line code of this size is bound by instruction
// fetch).
template <int NW, int MT>
__device__ void shared_gate_up_regs(const MoeArgs& a, int cta, float* xs, int warp, int lane) {
    constexpr int R = kShRowsPerWarp;
    const int rows = 2 * a.sh_inter;
    const int r0 = (cta * NW + warp) * R;
    const int nrows = min(R, rows - r0);
    const bool gate = cta == 0 && warp == NW - 1;
    uint4 wv[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            wv[r][c] = (r < nrows && c * 512 + lane * 16 < a.hidden)
                           ? ldg_stream_v4(a.sh_gu_w8 + (long long)(r0 + r) * a.hidden + c * 512 + lane * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
    uint4 gv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        gv[k] = (gate && lane * 8 + 256 * k < a.hidden)
                    ? __ldg(reinterpret_cast<const uint4*>(a.sh_gate + lane * 8 + 256 * k))
                    : make_uint4(0u, 0u, 0u, 0u);
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sc[r] = r < nrows ? a.sh_gu_scale[r0 + r] : 0.f;
    pdl_wait();  // x, and the workspace the previous call's kernels may still read
    float wf[R][64];  // (c, q, k): column c*512 + 16*lane + 4q + k
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float f[4];
            i8x4_to_f32(wv[r][c].x, f);
#pragma unroll
            for (int k = 0; k < 4; ++k) wf[r][16 * c + k] = f[k];
            i8x4_to_f32(wv[r][c].y, f);
#pragma unroll
            for (int k = 0; k < 4; ++k) wf[r][16 * c + 4 + k] = f[k];
            i8x4_to_f32(wv[r][c].z, f);
#pragma unroll
            for (int k = 0; k < 4; ++k) wf[r][16 * c + 8 + k] = f[k];
            i8x4_to_f32(wv[r][c].w, f);
#pragma unroll
            for (int k = 0; k < 4; ++k) wf[r][16 * c + 12 + k] = f[k];
        }
    for (int tb = 0; tb < a.T; tb += MT) {
        const int mt = min(MT, a.T - tb);
        __syncthreads();
        stage_x_f32<NW, MT>(a, tb, mt, xs);
        __syncthreads();
        if (nrows > 0) {
            // two tokens at a time (rows t >= mt are staged as zeros), so that
            // four independent sums hide the fma latency
#pragma unroll 1
            for (int t = 0; t < mt; t += 2) {
                float acc[R][2];
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int i0 = c * 512 + lane * 16;
                    if (i0 >= a.hidden) break;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float4 xv[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            xv[u] = *reinterpret_cast<const float4*>(xs + xs_swz((t + u) * a.hidden + i0 + 4 * q));
#pragma unroll
                        for (int r = 0; r < R; ++r)
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                acc[r][u] = fmaf(wf[r][16 * c + 4 * q], xv[u].x, acc[r][u]);
                                acc[r][u] = fmaf(wf[r][16 * c + 4 * q + 1], xv[u].y, acc[r][u]);
                                acc[r][u] = fmaf(wf[r][16 * c + 4 * q + 2], xv[u].z, acc[r][u]);
                                acc[r][u] = fmaf(wf[r][16 * c + 4 * q + 3], xv[u].w, acc[r][u]);
                            }
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        float v = acc[r][u];
#pragma unroll
                        for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                        if (lane == 0 && r < nrows && t + u < mt) a.shgu[(long long)(tb + t + u) * rows + r0 + r] = sc[r] * v;
                    }
            }
        }
        if (gate) {
#pragma unroll 1
            for (int t = 0; t < mt; t += 2) {
                float acc[2] = {0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int i0 = lane * 8 + 256 * k;
                    if (i0 >= a.hidden) break;
                    const float g[8] = {h2f_bits(static_cast<uint16_t>(gv[k].x & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(gv[k].x >> 16)),
                                        h2f_bits(static_cast<uint16_t>(gv[k].y & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(gv[k].y >> 16)),
                                        h2f_bits(static_cast<uint16_t>(gv[k].z & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(gv[k].z >> 16)),
                                        h2f_bits(static_cast<uint16_t>(gv[k].w & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(gv[k].w >> 16))};
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float4 xa = *reinterpret_cast<const float4*>(xs + xs_swz((t + u) * a.hidden + i0));
                        const float4 xb = *reinterpret_cast<const float4*>(xs + xs_swz((t + u) * a.hidden + i0 + 4));
                        acc[u] = fmaf(g[0], xa.x, acc[u]);
                        acc[u] = fmaf(g[1], xa.y, acc[u]);
                        acc[u] = fmaf(g[2], xa.z, acc[u]);
                        acc[u] = fmaf(g[3], xa.w, acc[u]);
                        acc[u] = fmaf(g[4], xb.x, acc[u]);
                        acc[u] = fmaf(g[5], xb.y, acc[u]);
                        acc[u] = fmaf(g[6], xb.z, acc[u]);
                        acc[u] = fmaf(g[7], xb.w, acc[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float v = acc[u];
#pragma unroll
                    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                    if (lane == 0 && t + u < mt) a.shgate[tb + t + u] = sigmoid_f(v);
                }
            }
        }
    }
}

// NT = 1 or 2 tokens, hidden <= 2048: the shared-expert rows of one warp
// (and, in warp 3 of CTA 0, the gate vector) are loaded into registers before
// the wait for the preceding kernel; after it only x is read, straight into
// registers (one L2 round trip, no staging). Sums in the order stated above.
// FUSED: x is computed by resid_norm_cta into xh after the wait and read
// from there.
template <int NT, bool FUSED>
__device__ void shared_gate_up_direct(const MoeArgs& a, int cta, int warp, int lane, uint16_t* xh) {
    constexpr int R = kShRowsPerWarp;
    const int rows = 2 * a.sh_inter;
    const int r0 = (cta * kK0Warps + warp) * R;
    const int nrows = min(R, rows - r0);
    const bool gate = cta == 0 && warp == kK0Warps - 1;
    // chunk c (512 columns) holds this lane's 16 columns when c*512 + 16*lane < hidden
    uint4 wv[R][4];
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        sc[r] = r < nrows ? a.sh_gu_scale[r0 + r] : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            wv[r][c] = (r < nrows && c * 512 + lane * 16 < a.hidden)
                           ? ldg_stream_v4(a.sh_gu_w8 + (long long)(r0 + r) * a.hidden + c * 512 + lane * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
    }
    uint4 gv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        gv[k] = (gate && lane * 8 + 256 * k < a.hidden)
                    ? __ldg(reinterpret_cast<const uint4*>(a.sh_gate + lane * 8 + 256 * k))
                    : make_uint4(0u, 0u, 0u, 0u);
    // the rows in f32 while the preceding kernel finishes: after the wait
    // only x is converted
    float wf[R][64];  // (c, q, k): column c*512 + 16*lane + 4q + k
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t words[4] = {wv[r][c].x, wv[r][c].y, wv[r][c].z, wv[r][c].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[4];
                i8x4_to_f32(words[q], f);
#pragma unroll
                for (int k = 0; k < 4; ++k) wf[r][16 * c + 4 * q + k] = f[k];
            }
        }
    pdl_wait();  // x, and the workspace the previous call's kernels may still read
    if constexpr (FUSED) resid_norm_cta<NT>(a, 0, a.T, xh);
    auto ldx = [&](long long off) -> uint4 {
        if constexpr (FUSED) return *reinterpret_cast<const uint4*>(xh + off);
        else return __ldg(reinterpret_cast<const uint4*>(a.x + off));
    };
    if (nrows > 0) {
        uint4 xv[NT][4][2];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    xv[t][c][h] = (t < a.T && c * 512 + lane * 16 < a.hidden)
                                      ? ldx((long long)t * a.hidden + c * 512 + lane * 16 + 8 * h)
                                      : make_uint4(0u, 0u, 0u, 0u);
        float acc[R][NT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c * 512 + lane * 16 >= a.hidden) break;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float xq[NT][4];
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint32_t x01 = q == 0 ? xv[t][c][0].x : q == 1 ? xv[t][c][0].z : q == 2 ? xv[t][c][1].x : xv[t][c][1].z;
                    const uint32_t x23 = q == 0 ? xv[t][c][0].y : q == 1 ? xv[t][c][0].w : q == 2 ? xv[t][c][1].y : xv[t][c][1].w;
                    xq[t][0] = h2f_bits(static_cast<uint16_t>(x01 & 0xFFFFu));
                    xq[t][1] = h2f_bits(static_cast<uint16_t>(x01 >> 16));
                    xq[t][2] = h2f_bits(static_cast<uint16_t>(x23 & 0xFFFFu));
                    xq[t][3] = h2f_bits(static_cast<uint16_t>(x23 >> 16));
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float* f = &wf[r][16 * c + 4 * q];
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        acc[r][t] = fmaf(f[0], xq[t][0], acc[r][t]);
                        acc[r][t] = fmaf(f[1], xq[t][1], acc[r][t]);
                        acc[r][t] = fmaf(f[2], xq[t][2], acc[r][t]);
                        acc[r][t] = fmaf(f[3], xq[t][3], acc[r][t]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float v = acc[r][t];
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                if (lane == 0 && r < nrows && t < a.T) a.shgu[(long long)t * rows + r0 + r] = sc[r] * v;
            }
    }
    if (gate) {
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i0 = lane * 8 + 256 * k;
            if (i0 >= a.hidden) break;
            const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4 xg = t < a.T ? ldx((long long)t * a.hidden + i0) : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t xw[4] = {xg.x, xg.y, xg.z, xg.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[t] = fmaf(h2f_bits(static_cast<uint16_t>(gw[q] & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(xw[q] & 0xFFFFu)), acc[t]);
                    acc[t] = fmaf(h2f_bits(static_cast<uint16_t>(gw[q] >> 16)), h2f_bits(static_cast<uint16_t>(xw[q] >> 16)), acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[t];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            if (lane == 0 && t < a.T) a.shgate[t] = sigmoid_f(v);
        }
    }
}

// Per-slot path: CTAs x < n_lg compute router logits; with a shared expert,
// the CTAs after them in row y = 0 compute its gate_up rows and its gate
// (4 warps each, MT tokens per pass), so that the gate_up kernel is routed
// experts only and the shared rows run while the logits are computed.
template <int MT, bool FUSED>
__global__ void __launch_bounds__(kK0Threads) moe_router_kernel(const MoeArgs a, int n_lg) {
    // The gate_up kernel can be scheduled at once, while the kernel before
    // this one may still run: every gate_up CTA waits for this grid (and so
    // for that kernel) before it touches x, the logits or the workspace.
    pdl_trigger();
    extern __shared__ __align__(16) float xs_sh[];
    uint16_t* xh = reinterpret_cast<uint16_t*>(xs_sh);  // residual block: normalised x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    static_assert(!FUSED || MT <= kFusedNormMaxT, "the residual norm runs in the router grid for few tokens only");
    if (static_cast<int>(blockIdx.x) < n_lg) {
        // waits for the preceding kernel after its first weight loads
        router_logits<FUSED>(a, warp, lane, xh, static_cast<int>(blockIdx.y) * kLgTG, nullptr);
        return;
    }
    if (blockIdx.y != 0) return;
    const int cta = static_cast<int>(blockIdx.x) - n_lg;
    if (a.hidden <= 2048) {
        if constexpr (MT <= 2) {
            shared_gate_up_direct<MT, FUSED>(a, cta, warp, lane, xh);
        } else {
            shared_gate_up_regs<kK0Warps, MT>(a, cta, xs_sh, warp, lane);
        }
    } else {
        shared_gate_up_staged<kK0Warps, MT>(a, cta, xs_sh, warp, lane);
    }
}

// One token, hidden <= 2048, few registers: shared_gate_up_direct<1> with
// the int8 rows kept packed until after the wait and converted as they are
// used (the same values, the same order of every sum), so that the router
// grid of a multi-layer launch, one row of CTAs per token, keeps many CTAs
// per SM.
__device__ void shared_gate_up_light(const MoeArgs& a, int cta, int warp, int lane) {
    constexpr int R = kShRowsPerWarp;
    const int rows = 2 * a.sh_inter;
    const int r0 = (cta * kK0Warps + warp) * R;
    const int nrows = min(R, rows - r0);
    const bool gate = cta == 0 && warp == kK0Warps - 1;
    uint4 wv[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            wv[r][c] = (r < nrows && c * 512 + lane * 16 < a.hidden)
                           ? ldg_stream_v4(a.sh_gu_w8 + (long long)(r0 + r) * a.hidden + c * 512 + lane * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
    pdl_wait();  // x, and the workspace the previous call's kernels may still read
    if (nrows > 0) {
        float acc[R] = {0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c * 512 + lane * 16 >= a.hidden) break;
            const uint4 x0 = __ldg(reinterpret_cast<const uint4*>(a.x + c * 512 + lane * 16));
            const uint4 x1 = __ldg(reinterpret_cast<const uint4*>(a.x + c * 512 + lane * 16 + 8));
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xq[4] = {h2f_bits(static_cast<uint16_t>(xw[2 * q] & 0xFFFFu)),
                                     h2f_bits(static_cast<uint16_t>(xw[2 * q] >> 16)),
                                     h2f_bits(static_cast<uint16_t>(xw[2 * q + 1] & 0xFFFFu)),
                                     h2f_bits(static_cast<uint16_t>(xw[2 * q + 1] >> 16))};
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t word = q == 0 ? wv[r][c].x : q == 1 ? wv[r][c].y : q == 2 ? wv[r][c].z : wv[r][c].w;
                    float f[4];
                    i8x4_to_f32(word, f);
                    acc[r] = fmaf(f[0], xq[0], acc[r]);
                    acc[r] = fmaf(f[1], xq[1], acc[r]);
                    acc[r] = fmaf(f[2], xq[2], acc[r]);
                    acc[r] = fmaf(f[3], xq[3], acc[r]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float v = acc[r];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            if (lane == 0 && r < nrows) a.shgu[r0 + r] = a.sh_gu_scale[r0 + r] * v;
        }
    }
    if (gate) {
        float acc = 0.f;
#pragma unroll 1
        for (int k = 0; k < 8; ++k) {
            const int i0 = lane * 8 + 256 * k;
            if (i0 >= a.hidden) break;
            const uint4 g4 = __ldg(reinterpret_cast<const uint4*>(a.sh_gate + i0));
            const uint4 xg = __ldg(reinterpret_cast<const uint4*>(a.x + i0));
            const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, xw[4] = {xg.x, xg.y, xg.z, xg.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fmaf(h2f_bits(static_cast<uint16_t>(gw[q] & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(xw[q] & 0xFFFFu)), acc);
                acc = fmaf(h2f_bits(static_cast<uint16_t>(gw[q] >> 16)), h2f_bits(static_cast<uint16_t>(xw[q] >> 16)), acc);
            }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (lane == 0) *a.shgate = sigmoid_f(acc);
    }
}

// Multi-layer per-slot launch: row y of the grid is token y, with its own
// layer. Its CTAs run the one-token code on a view of the arguments that
// holds that layer's weights and input and that token's outputs, so every
// logit, shared-expert row and gate has the one-token (and the one-layer
// multi-token) summation order.
__global__ void __launch_bounds__(kK0Threads) moe_router_ml_kernel(const MoeArgs a, int n_lg,
                                                                   const __grid_constant__ MlTable tab) {
    pdl_trigger();
    const int t = static_cast<int>(blockIdx.y);
    const MoeLayerPtrs& L = tab.l[t];
    MoeArgs la = a;
    la.T = 1;
    la.x = L.x;
    la.router_w = L.router_w;
    la.sh_gu_w8 = L.sh_gu_w8;
    la.sh_gu_scale = L.sh_gu_scale;
    la.sh_gate = L.sh_gate;
    la.logits = a.logits + (long long)t * a.E;
    la.shgu = a.shgu + (long long)t * 2 * a.sh_inter;
    la.shgate = a.shgate + t;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (static_cast<int>(blockIdx.x) < n_lg) {
        router_logits<false>(la, warp, lane, nullptr, 0, &tab);
        return;
    }
    shared_gate_up_light(la, static_cast<int>(blockIdx.x) - n_lg, warp, lane);
}

// Router logits for many tokens: a CTA stages 16 tokens of x in shared memory
// (1024 columns at a time) and each of its 8 warps computes 2 experts x 16
// tokens, so x is read from L2 once per 16 experts instead of once per
// expert. Each logit keeps the summation order stated above.
constexpr int kRtTok = 16, kRtExpW = 2, kRtExp = 8 * kRtExpW, kRtCols = 1024;

__global__ void __launch_bounds__(256) moe_router_tiled_kernel(const MoeArgs a) {
    __shared__ __align__(16) uint16_t xs[kRtTok][kRtCols];
    pdl_trigger();
    pdl_wait();  // x and the workspace (the previous call's kernels may still read it)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *a.err = 0;  // the previous call has finished
    const int e0 = blockIdx.x * kRtExp + warp * kRtExpW;
    const int t0 = blockIdx.y * kRtTok;
    const int nt = min(kRtTok, a.T - t0);
    float acc[kRtExpW][kRtTok];
#pragma unroll
    for (int j = 0; j < kRtExpW; ++j)
#pragma unroll
        for (int t = 0; t < kRtTok; ++t) acc[j][t] = 0.f;
    for (int c0 = 0; c0 < a.hidden; c0 += kRtCols) {
        const int ncols = min(kRtCols, a.hidden - c0);  // a multiple of 256
        __syncthreads();
        for (int i = tid; i < kRtTok * (kRtCols / 8); i += 256) {
            const int t = i / (kRtCols / 8), c = (i % (kRtCols / 8)) * 8;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t < nt && c < ncols) v = __ldg(reinterpret_cast<const uint4*>(a.x + (long long)(t0 + t) * a.hidden + c0 + c));
            *reinterpret_cast<uint4*>(&xs[t][c]) = v;
        }
        __syncthreads();
        uint4 wv[kRtExpW][kRtCols / 256];
#pragma unroll
        for (int j = 0; j < kRtExpW; ++j)
#pragma unroll
            for (int p = 0; p < kRtCols / 256; ++p)
                wv[j][p] = (e0 + j < a.E && p * 256 < ncols)
                               ? ldg_stream_v4(a.router_w + (long long)(e0 + j) * a.hidden + c0 + p * 256 + lane * 8)
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int p = 0; p < kRtCols / 256; ++p) {
            if (p * 256 >= ncols) break;
#pragma unroll
            for (int t = 0; t < kRtTok; ++t) {
                const uint4 xv = *reinterpret_cast<const uint4*>(&xs[t][p * 256 + lane * 8]);
#pragma unroll
                for (int j = 0; j < kRtExpW; ++j) dot8_f16(xv, wv[j][p], acc[j][t]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kRtExpW; ++j)
#pragma unroll
        for (int t = 0; t < kRtTok; ++t) {
            float v = acc[j][t];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, m);
            if (lane == 0 && t < nt && e0 + j < a.E)
                a.logits[(long long)(t0 + t) * a.E + e0 + j] = __half_as_ushort(__float2half_rn(v));
        }
}

// ---------------------------------------------------------------------------
// 2. gate_up of the routed experts.
// ---------------------------------------------------------------------------
template <int K>
__device__ void gate_up_routed(const MoeArgs& a, float* smem) {
    const int crank = static_cast<int>(cg::this_cluster().block_rank());
    const int csize = static_cast<int>(cg::this_cluster().num_blocks());
    const int ob = blockIdx.y;
    const int slot = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_out = 2 * a.inter;
    const int KT = a.hidden >> 4, NT = n_out >> 4;
    const int kt0 = crank * a.gu_kt_per_cta;
    const int kt1 = min(KT, kt0 + a.gu_kt_per_cta);
    const int nk = (kt1 - kt0) * 16;
    float* slots = smem;                     // [csize][128] partials, on rank 0
    float* xt = slots + kMaxCluster * 128;   // [gu_kt_per_cta * 16]
    float* red = xt + a.gu_kt_per_cta * 16;  // [kGuWarps][128] (+128: partial of ranks != 0)
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int e_s[8];
    __shared__ float w_s[8];

    if (crank == 0 && threadIdx.x == 0 && csize > 1) mbar_init(smem_u32(&bar), 32 * (csize - 1));
    cluster_arrive();  // rank 0's barrier is initialised before anyone arrives on it

    const int t = slot / a.topk;
    const int j = slot % a.topk;
    // x may still be written by the kernel before the router (this grid can
    // start while it runs): its loads go out right after the wait, beside
    // the logits' (only rin depends on the routing)
    pdl_wait();     // router logits (and, in a multi-layer launch, the layer table)
    pdl_trigger();  // logits complete: the down kernel may read them early
    const MoeLayerPtrs* ly = a.lay ? a.lay + t : nullptr;  // token t's layer (multi-layer launch)
    const uint16_t* xrow = ly ? ly->x : a.x + (long long)t * a.hidden;
    uint2 x_pre = make_uint2(0u, 0u);
    if (warp < nk / 128) x_pre = *reinterpret_cast<const uint2*>(xrow + kt0 * 16 + warp * 128 + 4 * lane);
    if (warp == 0) {
        int e_l;
        float w_l;
        topk_softmax_warp(a.logits + (long long)t * a.E, a.E, a.topk, lane, &e_l, &w_l);
        if (lane < a.topk) {
            e_s[lane] = e_l;
            w_s[lane] = w_l;
            if (crank == 0 && ob == 0 && j == 0) {  // one CTA per token publishes the routing
                int32_t* ids = ly && ly->ids ? ly->ids : a.ids + (long long)t * a.topk;
                float* ws = ly && ly->w ? ly->w : a.w + (long long)t * a.topk;
                ids[lane] = e_l;
                ws[lane] = w_l;
            }
        }
    } else if (a.rs_h && a.rs_add && crank == 0 && ob == 0 && j == 0) {
        // residual block: the same CTA stores h += add for its token (the
        // router grid, which read h, has finished)
        float* hr = a.rs_h + (long long)t * a.hidden;
        const float* ar = a.rs_add + (long long)t * a.hidden;
        for (int i = (threadIdx.x - 32) * 4; i < a.hidden; i += (kGuThreads - 32) * 4) {
            const float4 hv = *reinterpret_cast<const float4*>(hr + i);
            const float4 av = *reinterpret_cast<const float4*>(ar + i);
            *reinterpret_cast<float4*>(hr + i) =
                make_float4(__fadd_rn(hv.x, av.x), __fadd_rn(hv.y, av.y), __fadd_rn(hv.z, av.z), __fadd_rn(hv.w, av.w));
        }
    }
    __syncthreads();
    const int e = e_s[j];
    const uint16_t* codes = (ly ? ly->gu_codes : a.gu_codes) + (long long)e * KT * NT * (16 * K);
    LaneCodes<K> cur;
    const TileStrides grid{NT, 1};  // experts are stored kt-major
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);

    // xt = H128(rin_e * x[t]) over this CTA's inputs
    const uint16_t* rin = (ly ? ly->gu_rin : a.gu_rin) + (long long)e * a.hidden;
    for (int blk = warp; blk < nk / 128; blk += kGuWarps) {
        const int ib = kt0 * 16 + blk * 128 + 4 * lane;
        const uint2 rb = *reinterpret_cast<const uint2*>(rin + ib);
        const uint2 xb = blk == warp ? x_pre : *reinterpret_cast<const uint2*>(xrow + ib);
        float v[4];
        v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * h2f_bits(static_cast<uint16_t>(xb.x & 0xFFFFu));
        v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * h2f_bits(static_cast<uint16_t>(xb.x >> 16));
        v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * h2f_bits(static_cast<uint16_t>(xb.y & 0xFFFFu));
        v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * h2f_bits(static_cast<uint16_t>(xb.y >> 16));
        h128_warp(v, lane);
        *reinterpret_cast<float4*>(xt + blk * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    uint2 rout_pre = make_uint2(0u, 0u);  // rank 0's output scales, fetched while the loop runs
    if (crank == 0 && warp == 0)
        rout_pre = *reinterpret_cast<const uint2*>((ly ? ly->gu_rout : a.gu_rout) + (long long)e * n_out + ob * 128 +
                                                   4 * lane);
    float* zp = crank == 0 ? slots : red + kGuWarps * 128;  // rank 0 keeps its partial in slot 0
    cta_gemv_partial<K, 1, kGuWarps>(codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);

    cluster_wait();
    if (crank != 0) {
        if (warp == 0 && !a.skip_cluster_arrive) {
            const uint32_t dst = cluster_map(smem_u32(slots + crank * 128 + 4 * lane), 0);
            st_cluster_v4(dst, *reinterpret_cast<const float4*>(zp + 4 * lane));
            mbar_arrive_cluster(cluster_map(smem_u32(&bar), 0));
        }
        return;
    }
    if (warp == 0) {
        if (csize > 1) mbar_wait_bounded(smem_u32(&bar), a.err, 1, 1ll << a.mbar_limit_log2);
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < csize; ++r) {
            const float4 z4 = *reinterpret_cast<const float4*>(slots + r * 128 + 4 * lane);
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        output_transform_regs(v, rout_pre, lane);
        *reinterpret_cast<float4*>(a.ygu + (long long)slot * n_out + ob * 128 + 4 * lane) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

template <int K>
// Four CTAs per SM (64 registers): with the shared expert's rows in the
// router grid this kernel holds only the routed decode.
__global__ void __launch_bounds__(kGuThreads, 4) moe_gate_up_kernel(const MoeArgs a) {
    extern __shared__ __align__(16) float smem[];
    gate_up_routed<K>(a, smem);
}

// ---------------------------------------------------------------------------
// 3. down + combine.
// ---------------------------------------------------------------------------
// MINB CTAs per SM: 4 (64 registers) when the grid needs more than one wave
// of 3, else 3 (80 registers, faster per CTA).
template <int K, int MINB>
__global__ void __launch_bounds__(kDnThreads, MINB) moe_down_kernel(const MoeArgs a) {
    const int rank = static_cast<int>(cg::this_cluster().block_rank());
    const int csz = static_cast<int>(cg::this_cluster().num_blocks());
    const int ks = a.dn_ksplit;
    const int j = rank / ks, h = rank % ks;
    const int ob = blockIdx.y;
    const int t = blockIdx.z;
    // token t's layer in a multi-layer launch (the table was stored by the
    // router kernel, which finished before this grid was scheduled, as the
    // logits read below)
    const MoeLayerPtrs* ly = a.lay ? a.lay + t : nullptr;
    const int8_t* sh_dn_w8 = ly ? ly->sh_dn_w8 : a.sh_dn_w8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ __align__(16) float smem[];
    float* slots = smem;                      // [csz][128] partials, on rank 0
    float* shres = slots + kMaxCluster * 128; // [128] shared-expert rows of the block, on rank 0
    float* dres = shres + 128;                // [topk][128] finished experts, on rank 0
    float* red = dres + 8 * 128;              // [kDnWarps][128] (+128: partial of ranks != 0)
    float* xt = red + (kDnWarps + 1) * 128;   // [inter / ks] (rounded up to 32)
    float* xsh = xt + a.dn_xt_floats;          // [sh_inter] (rounded up to 32): SwiGLU(shgu[t]), swizzled
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int e_s[8];
    __shared__ float w_s[8];

    if (rank == 0 && threadIdx.x == 0 && csz > 1) mbar_init(smem_u32(&bar), 32 * (csz - 1));
    cluster_arrive();

    // This rank's share of the shared expert's 128 down rows of the block:
    // rows rank*sh_per + warp + 8*i; with sh_inter <= 512 a warp's first two
    // rows are prefetched now.
    const int sh_per = (128 + csz - 1) / csz;
    uint4 shw[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int rr = warp + kDnWarps * i, row = rank * sh_per + rr;
        if (a.sh_inter > 0 && a.sh_inter <= 512 && rr < sh_per && row < 128 && lane * 16 < a.sh_inter)
            shw[i] = ldg_stream_v4(sh_dn_w8 + (long long)(ob * 128 + row) * a.sh_inter + lane * 16);
    }

    const int slot = t * a.topk + j;
    // The logits kernel finished before this grid was scheduled (every
    // gate_up CTA waited for it before triggering this launch).
    if (warp == 0) {
        int e_l;
        float w_l;
        topk_softmax_warp(a.logits + (long long)t * a.E, a.E, a.topk, lane, &e_l, &w_l);
        if (lane < a.topk) {
            e_s[lane] = e_l;
            w_s[lane] = w_l;
        }
    }
    __syncthreads();
    const int e = e_s[j];
    const int KT = a.inter >> 4, NT = a.hidden >> 4;
    const int rows_h = KT / ks;  // whole Hadamard blocks per input split
    const int kt0 = h * rows_h, kt1 = kt0 + rows_h;
    const int nk = rows_h * 16;
    const uint16_t* codes = (ly ? ly->dn_codes : a.dn_codes) + (long long)e * KT * NT * (16 * K);
    LaneCodes<K> cur;
    const TileStrides grid{NT, 1};  // experts are stored kt-major
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);
    const uint16_t* rin = (ly ? ly->dn_rin : a.dn_rin) + (long long)e * a.inter;
    uint2 rin_pre = make_uint2(0u, 0u);
    if (warp < nk / 128) rin_pre = *reinterpret_cast<const uint2*>(rin + kt0 * 16 + warp * 128 + 4 * lane);
    pdl_wait();  // gate_up outputs and the shared expert's gate_up
    pdl_trigger();  // a dependent (the next residual norm) waits for this grid before reading

    // the shared expert's down input, SwiGLU(shgu[t]): its loads (two per
    // thread for sh_inter <= 512) go out together with the routed input
    // transform's, and the shared rows after the main loop then only need
    // their dot products
    const int n_sh = a.sh_inter;
    const float* gu = a.shgu + (long long)t * 2 * n_sh;
    float shg[2] = {0.f, 0.f}, shu[2] = {0.f, 0.f};
    if (n_sh > 0 && n_sh <= 2 * kDnThreads) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = threadIdx.x + q * kDnThreads;
            if (i < n_sh) {
                shg[q] = gu[i];
                shu[q] = gu[n_sh + i];
            }
        }
    }

    // xt = H128(rin_e * SwiGLU(ygu[slot])) over this rank's inputs
    const float* yr = a.ygu + (long long)slot * 2 * a.inter;
    for (int blk = warp; blk < nk / 128; blk += kDnWarps) {
        const int ib = kt0 * 16 + blk * 128 + 4 * lane;
        const float4 g = *reinterpret_cast<const float4*>(yr + ib);
        const float4 u = *reinterpret_cast<const float4*>(yr + a.inter + ib);
        const uint2 rb = blk == warp ? rin_pre : *reinterpret_cast<const uint2*>(rin + ib);
        float v[4];
        v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * (silu_f(g.x) * u.x);
        v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * (silu_f(g.y) * u.y);
        v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * (silu_f(g.z) * u.z);
        v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * (silu_f(g.w) * u.w);
        h128_warp(v, lane);
        *reinterpret_cast<float4*>(xt + blk * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (n_sh > 0 && n_sh <= 2 * kDnThreads) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = threadIdx.x + q * kDnThreads;
            if (i < n_sh) xsh[xs_swz(i)] = silu_f(shg[q]) * shu[q];
        }
    } else {
        for (int i = threadIdx.x; i < n_sh; i += kDnThreads) xsh[xs_swz(i)] = silu_f(gu[i]) * gu[n_sh + i];
    }
    __syncthreads();
    uint2 rout_pre = make_uint2(0u, 0u);  // rank 0: every expert's output scales, fetched while the loop runs
    if (rank == 0 && warp < a.topk)
        rout_pre = *reinterpret_cast<const uint2*>((ly ? ly->dn_rout : a.dn_rout) + (long long)e_s[warp] * a.hidden +
                                                   ob * 128 + 4 * lane);
    float* zp = rank == 0 ? slots : red + kDnWarps * 128;
    cta_gemv_partial<K, 1, kDnWarps>(codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);

    // shared expert rows: xt <- SwiGLU(shgu[t]); the values go to rank 0's
    // shres (directly on rank 0, through distributed shared memory elsewhere)
    if (a.sh_inter > 0) {
        cluster_wait();  // rank 0's shared memory may be written from here on (xsh is complete: the main
                         // loop ended with a CTA barrier)
        const float gate = a.shgate[t];
        for (int rr = warp, i = 0; rr < sh_per; rr += kDnWarps, ++i) {
            const int sh_row = rank * sh_per + rr;
            if (sh_row >= 128) break;
            float dot;
            if (n_sh <= 512 && i < 2) {
                float acc = 0.f;
                if (lane * 16 < n_sh) {
                    const uint4 wv = i == 0 ? shw[0] : shw[1];
                    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float f[4];
                        i8x4_to_f32(words[q], f);
                        const float4 xv = *reinterpret_cast<const float4*>(xsh + xs_swz(lane * 16 + 4 * q));
                        acc = fmaf(f[0], xv.x, acc);
                        acc = fmaf(f[1], xv.y, acc);
                        acc = fmaf(f[2], xv.z, acc);
                        acc = fmaf(f[3], xv.w, acc);
                    }
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
                dot = acc;
            } else {
                float d1[1][1];
                int8_rows_dot<1, 1, 4>(sh_dn_w8 + (long long)(ob * 128 + sh_row) * n_sh, n_sh, 1, n_sh, xsh, n_sh, lane,
                                       d1);
                dot = d1[0][0];
            }
            const float sh_val = gate * ((ly ? ly->sh_dn_scale : a.sh_dn_scale)[ob * 128 + sh_row] * dot);
            if (lane == 0) {
                if (rank == 0) {
                    shres[sh_row] = sh_val;
                } else if (!a.skip_cluster_arrive) {
                    const uint32_t dst = cluster_map(smem_u32(shres + sh_row), 0);
                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(sh_val) : "memory");
                }
            }
        }
    } else {
        cluster_wait();
    }

    if (rank != 0) {
        __syncthreads();
        if (warp == 0 && !a.skip_cluster_arrive) {
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            const uint32_t dst = cluster_map(smem_u32(slots + rank * 128 + 4 * lane), 0);
            st_cluster_v4(dst, *reinterpret_cast<const float4*>(zp + 4 * lane));
            mbar_arrive_cluster(cluster_map(smem_u32(&bar), 0));
        }
        return;
    }
    if (csz > 1) {
        if (warp == 0) mbar_wait_bounded(smem_u32(&bar), a.err, 2, 1ll << a.mbar_limit_log2);
    }
    __syncthreads();
    if (warp < a.topk) {  // warp q finishes expert q: its splits in order, output transform, routing weight
        const int q = warp;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sp = 0; sp < ks; ++sp) {
            const float4 z4 = *reinterpret_cast<const float4*>(slots + (q * ks + sp) * 128 + 4 * lane);
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        output_transform_regs(v, rout_pre, lane);
        const float wq = w_s[q];
        *reinterpret_cast<float4*>(dres + q * 128 + 4 * lane) = make_float4(wq * v[0], wq * v[1], wq * v[2], wq * v[3]);
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int i = threadIdx.x;
        float sum = 0.f;
        for (int q = 0; q < a.topk; ++q) sum += dres[q * 128 + i];
        if (a.sh_inter > 0) sum += shres[i];
        (ly ? ly->out : a.out + (long long)t * a.hidden)[ob * 128 + i] = sum;
    }
}

cudaError_t launch_ex(const void* func, dim3 grid, dim3 block, int smem, int cluster_x, bool pdl, cudaStream_t s,
                      const MoeArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster_x > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    void* args[] = {const_cast<MoeArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, func, args);
}

template <int K>
cudaError_t launch_gate_up(MoeArgs a, int num_sms, cudaStream_t s) {
    (void)num_sms;  // splits are sized for kWaveSms
    const int oblks = 2 * a.inter / 128;
    const int slots = a.T * a.topk;
    const SlotPlan sp = slot_plan(a.T, a.hidden, a.inter, a.topk);
    const int csize = sp.gu_csize;
    a.gu_kt_per_cta = sp.gu_kt_per_cta;
    const int smem = (kMaxCluster * 128 + a.gu_kt_per_cta * 16 + (kGuWarps + 1) * 128) * 4;
    const void* f = reinterpret_cast<const void*>(moe_gate_up_kernel<K>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_ex(f, dim3(csize, oblks, slots), dim3(kGuThreads), smem, csize, true, s, a);
}

template <int K>
cudaError_t launch_down(MoeArgs a, int num_sms, cudaStream_t s) {
    (void)num_sms;  // splits are sized for kWaveSms
    a.dn_ksplit = slot_plan(a.T, a.hidden, a.inter, a.topk).dn_ksplit;
    const int csz = a.topk * a.dn_ksplit;
    a.dn_xt_floats = (a.inter / a.dn_ksplit + 31) / 32 * 32;
    // routed inputs of one rank, then the shared expert's inputs (swizzled
    // staging works on groups of 32 floats)
    const int nsh = (a.sh_inter + 31) / 32 * 32;
    const int smem = (kMaxCluster * 128 + 128 + 8 * 128 + (kDnWarps + 1) * 128 + a.dn_xt_floats + nsh) * 4;
    // More than one wave of 3 CTAs per SM: the 64-register build, 4 per SM
    // (measured on GB300 for the 35B layer: 4 tokens 52.3 -> 46.9 us per
    // block, 8 tokens 88.9 -> 85.0, 16 tokens 155.9 -> 148.2; with one
    // wave, 1-2 tokens, it was slower: 1 token 21.0 -> 21.6 us).
    const long long ctas = (long long)csz * (a.hidden / 128) * a.T;
    const void* f = ctas > 3LL * kWaveSms ? reinterpret_cast<const void*>(moe_down_kernel<K, 4>)
                                          : reinterpret_cast<const void*>(moe_down_kernel<K, 3>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (csz > 8) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return launch_ex(f, dim3(csz, a.hidden / 128, a.T), dim3(kDnThreads), smem, csz, true, s, a);
}

}  // namespace

SlotPlan slot_plan(int T, int hidden, int inter, int topk) {
    SlotPlan p{};
    const int oblks = 2 * inter / 128;
    const int slots = T * topk;
    const int kblks = hidden / 128;
    // gate_up: the largest input split (CTAs per cluster, <= 8) for which the
    // routed CTAs fit in one wave of 4 CTAs per SM; when only an unsplit grid
    // fits, a split of two is still taken while it needs at most 1.8 waves:
    // an unsplit grid that fills a wave only partly leaves SMs with 3 CTAs
    // beside SMs with 4 (measured on GB300 for the 35B layer: 8 one-token
    // blocks of distinct layers in one launch 11.05 -> 10.68 us per block
    // with the split; 1.3 waves was the limit before, set with 3 CTAs per
    // SM). Four CTAs per SM instead of three: 1 token 23.7 -> 21.5 us per
    // block, 2 tokens 35.8 -> 31.1 us, 4 to 16 tokens unchanged.
    auto ctas = [&](int cs) { return (long long)cs * oblks * slots; };
    int csize = 1;
    for (int c = 1; c <= 8 && c <= kblks; ++c) {
        const int per = (kblks + c - 1) / c;
        const int cs = (kblks + per - 1) / per;
        if (ctas(cs) <= 4LL * kWaveSms) csize = cs;
    }
    if (csize == 1 && kblks >= 2 && 10 * ctas(2) <= 18LL * 4 * kWaveSms) csize = 2;
    const int per = (kblks + csize - 1) / csize;
    p.gu_csize = (kblks + per - 1) / per;
    p.gu_kt_per_cta = per * 8;
    // down: each expert's input split in two when it spans an even number
    // (>= 2) of Hadamard blocks, the cluster stays within 16 CTAs and the
    // split grid still fits one wave of 3 CTAs per SM (one token for the 35B
    // layer; from 2 tokens on the unsplit grid was measured faster on GB300,
    // e.g. 8 tokens 109 -> 92 us per block).
    const long long split_ctas = 2LL * topk * (hidden / 128) * T;
    p.dn_ksplit = ((inter / 128) % 2 == 0 && 2 * topk <= kMaxCluster && split_ctas <= 3LL * kWaveSms) ? 2 : 1;
    return p;
}

cudaError_t launch_moe_router(const MoeArgs& a, bool with_shared, cudaStream_t s) {
    if (!with_shared && a.T >= kRtTok) {
        void* args[] = {const_cast<MoeArgs*>(&a)};
        return launch_kernel(reinterpret_cast<const void*>(moe_router_tiled_kernel),
                             dim3((a.E + kRtExp - 1) / kRtExp, (a.T + kRtTok - 1) / kRtTok), dim3(256), 0, true, s,
                             args);
    }
    int n_lg = (a.E + kK0Warps - 1) / kK0Warps;
    const int rows_per_cta = kK0Warps * kShRowsPerWarp;
    const int n_sh = with_shared && a.sh_inter > 0 ? (2 * a.sh_inter + rows_per_cta - 1) / rows_per_cta : 0;
    // tokens per pass of the shared rows: 1 or 2 read x straight into
    // registers (hidden <= 2048), otherwise x is staged in shared memory
    const int mt = a.T <= 2 ? a.T : kShMT;
    int smem = n_sh > 0 && !(mt <= 2 && a.hidden <= 2048) ? mt * a.hidden * 4 : 0;
    if (a.x_norm) smem = max(smem, kFusedNormMaxT * a.hidden * 2);  // residual block: normalised x (fp16)
    const bool fused = a.x_norm != nullptr;  // set by the caller for <= kFusedNormMaxT tokens only
    static_assert(kFusedNormMaxT == 1, "fused router instantiations cover one token");
    const void* f = mt == 1   ? (fused ? reinterpret_cast<const void*>(moe_router_kernel<1, true>)
                                       : reinterpret_cast<const void*>(moe_router_kernel<1, false>))
                    : mt == 2 ? reinterpret_cast<const void*>(moe_router_kernel<2, false>)
                              : reinterpret_cast<const void*>(moe_router_kernel<kShMT, false>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_lg + n_sh, (a.T + kLgTG - 1) / kLgTG);
    cfg.blockDim = dim3(kK0Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<MoeArgs*>(&a), &n_lg};
    return cudaLaunchKernelExC(&cfg, f, args);
}

cudaError_t launch_moe_router_ml(const MoeArgs& a, const MlTable& tab, cudaStream_t s) {
    int n_lg = (a.E + kK0Warps - 1) / kK0Warps;
    const int rows_per_cta = kK0Warps * kShRowsPerWarp;
    const int n_sh = a.sh_inter > 0 ? (2 * a.sh_inter + rows_per_cta - 1) / rows_per_cta : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_lg + n_sh, a.T);
    cfg.blockDim = dim3(kK0Threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<MoeArgs*>(&a), &n_lg, const_cast<MlTable*>(&tab)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(moe_router_ml_kernel), args);
}

cudaError_t launch_moe_gate_up(const MoeArgs& a, int num_sms, cudaStream_t s) {
    return a.gu_K == 2 ? launch_gate_up<2>(a, num_sms, s) : launch_gate_up<3>(a, num_sms, s);
}

cudaError_t launch_moe_down(const MoeArgs& a, int num_sms, cudaStream_t s) {
    return a.dn_K == 2 ? launch_down<2>(a, num_sms, s) : launch_down<3>(a, num_sms, s);
}

}  // namespace escha
