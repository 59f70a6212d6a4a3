// One MoE block of an Escha-W2 Qwen3.6-35B-A3B-style layer in three kernels
// chained by programmatic dependent launch:
//
//  1. router logits: f16-rounded logits in a fixed summation order (hipfire
//     PR #694, commit "Executed the moeblk golden against real shipped
//     layer-0 weights": logits are rounded to f16 before top-k), one warp per
//     expert spread over many SMs so the 1 MB router matrix streams in one
//     memory round trip.
//  2. gate_up: each routed CTA selects its token's top-k (ties to the lower
//     expert id) and softmax weights with one warp, then runs the expert's
//     gate_up projection (fused trellis decode GEMV with the input/output
//     Hadamard transforms and rout); a cluster splits the input rows and
//     pushes its partial sums into rank 0. Extra CTAs, which do not wait for
//     the router, compute the int8 shared expert's gate_up rows and its
//     sigmoid gate.
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
// acc += x.lo * w.lo, then acc += x.hi * w.hi: fp16 operands, f32 accumulator,
// one rounding per step (the product of two fp16 values is exact in f32, so
// this equals an f32 fma of the converted operands).
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

__device__ void router_logits(const MoeArgs& a, int warp, int lane) {
    const int e = blockIdx.x * kK0Warps + warp;
    const int t0 = blockIdx.y * kLgTG;
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
            if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.err = 0;  // the previous call has finished
            if (e >= a.E) return;
        }
#pragma unroll
        for (int t = 0; t < kLgTG; ++t) {
            if (t < nt) {
                const uint16_t* xrow = a.x + (long long)(t0 + t) * a.hidden;
                uint4 xv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (pg + q < passes) xv[q] = __ldg(reinterpret_cast<const uint4*>(xrow + (pg + q) * 256 + lane * 8));
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

// Shared expert gate_up rows (kShRowsPerWarp per warp) for every token, and
// in CTA 0 the sigmoid gate (an f32 dot product of the fp16 gate vector with
// x, not rounded).
__device__ void shared_gate_up(const MoeArgs& a, int cta, float* xs, int warp, int lane) {
    const int rows = 2 * a.sh_inter;
    const int r0 = (cta * kGuWarps + warp) * kShRowsPerWarp;
    for (int tb = 0; tb < a.T; tb += kShMT) {
        const int mt = min(kShMT, a.T - tb);
        __syncthreads();
        for (int i = threadIdx.x * 8; i < kShMT * a.hidden; i += kGuThreads * 8) {
            const int t = i / a.hidden, c = i % a.hidden;
            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
            if (t < mt) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + (long long)(tb + t) * a.hidden + c));
                lo = make_float4(h2f_bits(v.x & 0xFFFFu), h2f_bits(v.x >> 16), h2f_bits(v.y & 0xFFFFu), h2f_bits(v.y >> 16));
                hi = make_float4(h2f_bits(v.z & 0xFFFFu), h2f_bits(v.z >> 16), h2f_bits(v.w & 0xFFFFu), h2f_bits(v.w >> 16));
            }
            *reinterpret_cast<float4*>(xs + xs_swz(i)) = lo;
            *reinterpret_cast<float4*>(xs + xs_swz(i + 4)) = hi;
        }
        __syncthreads();
        if (r0 < rows) {
            float dots[kShRowsPerWarp][kShMT];
            int8_rows_dot<kShRowsPerWarp, kShMT>(a.sh_gu_w8 + (long long)r0 * a.hidden, a.hidden, rows - r0, a.hidden,
                                                 xs, a.hidden, lane, dots);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < kShRowsPerWarp; ++r) {
                    if (r0 + r >= rows) break;
                    const float sc = a.sh_gu_scale[r0 + r];
                    for (int t = 0; t < mt; ++t) a.shgu[(long long)(tb + t) * rows + r0 + r] = sc * dots[r][t];
                }
            }
        }
        if (cta == 0 && warp == kGuWarps - 1) {
            float acc[kShMT] = {};
#pragma unroll 8
            for (int i0 = lane * 8; i0 < a.hidden; i0 += 256) {
                const uint4 gv = __ldg(reinterpret_cast<const uint4*>(a.sh_gate + i0));
                const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int t = 0; t < kShMT; ++t) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        acc[t] = fmaf(h2f_bits(static_cast<uint16_t>(gw[k] & 0xFFFFu)), xs[xs_swz(t * a.hidden + i0 + 2 * k)],
                                      acc[t]);
                        acc[t] = fmaf(h2f_bits(static_cast<uint16_t>(gw[k] >> 16)), xs[xs_swz(t * a.hidden + i0 + 2 * k + 1)],
                                      acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kShMT; ++t) {
                float v = acc[t];
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                if (lane == 0 && t < mt) a.shgate[tb + t] = sigmoid_f(v);
            }
        }
    }
}

__global__ void __launch_bounds__(kK0Threads) moe_router_kernel(const MoeArgs a) {
    // The gate_up kernel can be scheduled at once; its routed CTAs wait for
    // this grid before reading the logits.
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    router_logits(a, warp, lane);  // waits for the preceding kernel after its first weight loads
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
// 2. gate_up (routed) + shared expert down rows.
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
    // x is this call's input: its loads for the input transform go out before
    // the wait for the router (only rin depends on the routing)
    const uint16_t* xrow = a.x + (long long)t * a.hidden;
    uint2 x_pre = make_uint2(0u, 0u);
    if (warp < nk / 128) x_pre = *reinterpret_cast<const uint2*>(xrow + kt0 * 16 + warp * 128 + 4 * lane);
    pdl_wait();     // router logits
    pdl_trigger();  // logits complete: the down kernel may read them early
    if (warp == 0) {
        int e_l;
        float w_l;
        topk_softmax_warp(a.logits + (long long)t * a.E, a.E, a.topk, lane, &e_l, &w_l);
        if (lane < a.topk) {
            e_s[lane] = e_l;
            w_s[lane] = w_l;
            if (crank == 0 && ob == 0 && j == 0) {  // one CTA per token publishes the routing
                a.ids[(long long)t * a.topk + lane] = e_l;
                a.w[(long long)t * a.topk + lane] = w_l;
            }
        }
    }
    __syncthreads();
    const int e = e_s[j];
    const uint16_t* codes = a.gu_codes + (long long)e * KT * NT * (16 * K);
    LaneCodes<K> cur;
    const TileStrides grid{NT, 1};  // experts are stored kt-major
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);

    // xt = H128(rin_e * x[t]) over this CTA's inputs
    const uint16_t* rin = a.gu_rin + (long long)e * a.hidden;
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
        rout_pre = *reinterpret_cast<const uint2*>(a.gu_rout + (long long)e * n_out + ob * 128 + 4 * lane);
    float* zp = crank == 0 ? slots : red + kGuWarps * 128;  // rank 0 keeps its partial in slot 0
    cta_gemv_partial<K, 1, kGuWarps>(codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);

    cluster_wait();
    if (crank != 0) {
        if (warp == 0) {
            const uint32_t dst = cluster_map(smem_u32(slots + crank * 128 + 4 * lane), 0);
            st_cluster_v4(dst, *reinterpret_cast<const float4*>(zp + 4 * lane));
            mbar_arrive_cluster(cluster_map(smem_u32(&bar), 0));
        }
        return;
    }
    if (warp == 0) {
        if (csize > 1) mbar_wait_bounded(smem_u32(&bar), a.err, 1);
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
__global__ void __launch_bounds__(kGuThreads, 3) moe_gate_up_kernel(const MoeArgs a) {
    extern __shared__ __align__(16) float smem[];
    if (static_cast<int>(blockIdx.z) < a.T * a.topk) {
        gate_up_routed<K>(a, smem);
    } else {
        pdl_trigger();  // needs nothing from the router
        const int cta = ((blockIdx.z - a.T * a.topk) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        shared_gate_up(a, cta, smem, threadIdx.x >> 5, threadIdx.x & 31);
    }
}

// ---------------------------------------------------------------------------
// 3. down + combine.
// ---------------------------------------------------------------------------
template <int K>
__global__ void __launch_bounds__(kDnThreads, 3) moe_down_kernel(const MoeArgs a) {
    const int rank = static_cast<int>(cg::this_cluster().block_rank());
    const int csz = static_cast<int>(cg::this_cluster().num_blocks());
    const int ks = a.dn_ksplit;
    const int j = rank / ks, h = rank % ks;
    const int ob = blockIdx.y;
    const int t = blockIdx.z;
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
            shw[i] = ldg_stream_v4(a.sh_dn_w8 + (long long)(ob * 128 + row) * a.sh_inter + lane * 16);
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
    const uint16_t* codes = a.dn_codes + (long long)e * KT * NT * (16 * K);
    LaneCodes<K> cur;
    const TileStrides grid{NT, 1};  // experts are stored kt-major
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);
    const uint16_t* rin = a.dn_rin + (long long)e * a.inter;
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
        rout_pre = *reinterpret_cast<const uint2*>(a.dn_rout + (long long)e_s[warp] * a.hidden + ob * 128 + 4 * lane);
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
                int8_rows_dot<1, 1, 4>(a.sh_dn_w8 + (long long)(ob * 128 + sh_row) * n_sh, n_sh, 1, n_sh, xsh, n_sh, lane,
                                       d1);
                dot = d1[0][0];
            }
            const float sh_val = gate * (a.sh_dn_scale[ob * 128 + sh_row] * dot);
            if (lane == 0) {
                if (rank == 0) {
                    shres[sh_row] = sh_val;
                } else {
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
        if (warp == 0) {
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            const uint32_t dst = cluster_map(smem_u32(slots + rank * 128 + 4 * lane), 0);
            st_cluster_v4(dst, *reinterpret_cast<const float4*>(zp + 4 * lane));
            mbar_arrive_cluster(cluster_map(smem_u32(&bar), 0));
        }
        return;
    }
    if (csz > 1) {
        if (warp == 0) mbar_wait_bounded(smem_u32(&bar), a.err, 2);
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
        a.out[(long long)t * a.hidden + ob * 128 + i] = sum;
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
    const int kblks = a.hidden / 128;
    // Largest input split (CTAs per cluster, <= 8) for which the routed CTAs
    // plus the shared gate_up CTAs fit in one wave of 3 CTAs per SM; when only
    // an unsplit grid fits, a split of two is still taken while it needs at
    // most 1.3 waves (measured on GB300 for the 35B layer: 4 tokens 61 -> 56
    // us per block; 5 tokens, 1.5 waves, is slower split).
    const int rows_per_cta = kGuWarps * kShRowsPerWarp;
    auto shared_z = [&](int per_z) {
        return a.sh_inter > 0 ? (2 * a.sh_inter + per_z * rows_per_cta - 1) / (per_z * rows_per_cta) : 0;
    };
    auto ctas = [&](int cs) { return (long long)cs * oblks * (slots + shared_z(cs * oblks)); };
    int csize = 1;
    for (int c = 1; c <= 8 && c <= kblks; ++c) {
        const int per = (kblks + c - 1) / c;
        const int cs = (kblks + per - 1) / per;
        if (ctas(cs) <= 3LL * kWaveSms) csize = cs;
    }
    if (csize == 1 && kblks >= 2 && 10 * ctas(2) <= 13LL * 3 * kWaveSms) csize = 2;
    const int per = (kblks + csize - 1) / csize;
    csize = (kblks + per - 1) / per;
    a.gu_kt_per_cta = per * 8;
    const int sh_z = shared_z(csize * oblks);
    const int smem_routed = (kMaxCluster * 128 + a.gu_kt_per_cta * 16 + (kGuWarps + 1) * 128) * 4;
    const int smem_shared = a.sh_inter > 0 ? kShMT * a.hidden * 4 : 0;
    const int smem = smem_routed > smem_shared ? smem_routed : smem_shared;
    const void* f = reinterpret_cast<const void*>(moe_gate_up_kernel<K>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_ex(f, dim3(csize, oblks, slots + sh_z), dim3(kGuThreads), smem, csize, true, s, a);
}

template <int K>
cudaError_t launch_down(MoeArgs a, int num_sms, cudaStream_t s) {
    (void)num_sms;  // splits are sized for kWaveSms
    // Split each expert's input in two when it spans an even number (>= 2)
    // of Hadamard blocks, the cluster stays within 16 CTAs and the split grid
    // still fits one wave of 3 CTAs per SM (one token for the 35B layer;
    // from 2 tokens on the unsplit grid was measured faster on GB300, e.g. 8
    // tokens 109 -> 92 us per block).
    const long long split_ctas = 2LL * a.topk * (a.hidden / 128) * a.T;
    a.dn_ksplit = ((a.inter / 128) % 2 == 0 && 2 * a.topk <= kMaxCluster && split_ctas <= 3LL * kWaveSms) ? 2 : 1;
    const int csz = a.topk * a.dn_ksplit;
    a.dn_xt_floats = (a.inter / a.dn_ksplit + 31) / 32 * 32;
    // routed inputs of one rank, then the shared expert's inputs (swizzled
    // staging works on groups of 32 floats)
    const int nsh = (a.sh_inter + 31) / 32 * 32;
    const int smem = (kMaxCluster * 128 + 128 + 8 * 128 + (kDnWarps + 1) * 128 + a.dn_xt_floats + nsh) * 4;
    const void* f = reinterpret_cast<const void*>(moe_down_kernel<K>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (csz > 8) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return launch_ex(f, dim3(csz, a.hidden / 128, a.T), dim3(kDnThreads), smem, csz, true, s, a);
}

}  // namespace

cudaError_t launch_moe_router(const MoeArgs& a, cudaStream_t s) {
    if (a.T >= kRtTok) {
        void* args[] = {const_cast<MoeArgs*>(&a)};
        return launch_kernel(reinterpret_cast<const void*>(moe_router_tiled_kernel),
                             dim3((a.E + kRtExp - 1) / kRtExp, (a.T + kRtTok - 1) / kRtTok), dim3(256), 0, true, s,
                             args);
    }
    const int n_lg = (a.E + kK0Warps - 1) / kK0Warps;
    return launch_ex(reinterpret_cast<const void*>(moe_router_kernel), dim3(n_lg, (a.T + kLgTG - 1) / kLgTG),
                     dim3(kK0Threads), 0, 0, true, s, a);
}

cudaError_t launch_moe_gate_up(const MoeArgs& a, int num_sms, cudaStream_t s) {
    return a.gu_K == 2 ? launch_gate_up<2>(a, num_sms, s) : launch_gate_up<3>(a, num_sms, s);
}

cudaError_t launch_moe_down(const MoeArgs& a, int num_sms, cudaStream_t s) {
    return a.dn_K == 2 ? launch_down<2>(a, num_sms, s) : launch_down<3>(a, num_sms, s);
}

}  // namespace escha
