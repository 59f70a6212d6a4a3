// Fused trellis decode GEMV for sm_103a:
//   y = rout * H128(W^T H128(rin * x))   (both H128 unscaled, one exact 2^-7)
// with W decoded from the packed trellis codes inside the inner loop and never
// written anywhere (hipfire PR #694, summary "What it is", and the commit
// introducing the native expert-indexed GEMV: "trellis code stays verbatim and
// is decoded INSIDE the GEMV").
//
// Work decomposition. A CTA owns one 128-wide output block (8 tiles of 16
// output columns) of one projection item and a slice of the input tiles.
// The CTAs covering one output block form a thread-block cluster; their
// partial sums are reduced through distributed shared memory in a fixed
// rank order (deterministic, no atomics), then cluster rank 0 applies the
// output Hadamard, the 2^-7 scale and rout.
//
// Inner loop. Warp w walks the input-tile rows kt = kt0 + w, kt0 + w + 8, ...
// One warp load covers one tile row of the output block: 8 tiles x 16K words
// (512 B at K=2, 768 B at K=3), coalesced. Lane l takes tile l/4, quarter
// c = l%4 of its words: half-rows 8c..8c+7, i.e. input rows 4c..4c+3 of the
// tile, all 16 output columns. The word that follows the lane's last one (the
// end of a tail-biting window) comes from the neighbouring lane by shuffle.
#include "common.cuh"
#include "kernels.h"

namespace escha {

namespace {

constexpr int kThreads = 256;

// Loads the lane's 4K words of tile row `kt` (plus nothing else).
template <int K>
struct LaneCodes {
    uint32_t p[2 * K + 1];  // p[2K] low half receives the neighbour's first word
};

template <int K>
__device__ __forceinline__ void load_lane_codes(LaneCodes<K>& lc, const uint16_t* row_base, int lane) {
    if constexpr (K == 2) {
        const uint4 v = ldg_stream_v4(row_base + lane * 8);
        lc.p[0] = v.x;
        lc.p[1] = v.y;
        lc.p[2] = v.z;
        lc.p[3] = v.w;
    } else {
        const uint16_t* b = row_base + lane * 12;
        const uint2 v0 = ldg_stream_v2(b);
        const uint2 v1 = ldg_stream_v2(b + 4);
        const uint2 v2 = ldg_stream_v2(b + 8);
        lc.p[0] = v0.x;
        lc.p[1] = v0.y;
        lc.p[2] = v1.x;
        lc.p[3] = v1.y;
        lc.p[4] = v2.x;
        lc.p[5] = v2.y;
    }
}

// Decode the lane's 64 weights and accumulate acc[t][q] += W[r][q] * xt[t][r]
// for its 4 input rows r (xr[t][0..3]). Half-row j (input row j/2, output
// columns 8*(j%2)..+7) starts at bit 8*K*j of the lane's words; its weight m
// at bit 8*K*j + K*m. All offsets are compile-time constants.
template <int K, int NB>
__device__ __forceinline__ void decode_fma(const LaneCodes<K>& lc, const float (&xr)[NB][4], float (&acc)[NB][16]) {
    static_for<64>([&](auto I) {
        constexpr int j = decltype(I)::value / 8;
        constexpr int m = decltype(I)::value % 8;
        constexpr int b = 8 * K * j + K * m;
        const uint32_t s = window_state<(b & 15)>(stream_window<(b >> 4)>(lc.p));
        const float wv = cb_decode_f(s);
#pragma unroll
        for (int t = 0; t < NB; ++t) acc[t][8 * (j & 1) + m] = fmaf(wv, xr[t][j >> 1], acc[t][8 * (j & 1) + m]);
    });
}

// Input transform for this CTA's input slice: xt[t][i] = H128(rin * x[t])
// (unscaled), block by block, one warp per (token, 128-block).
template <int NB, int XM>
__device__ void input_transform(const GemvArgs& a, int xrow0, int ntok, int i0, int nk, float* xt, int warp, int lane,
                                int expert) {
    const int nblk = nk / 128;
    const uint16_t* rin = a.rin + (long long)expert * a.rin_stride;
    for (int wb = warp; wb < NB * nblk; wb += kThreads / 32) {
        const int t = wb / nblk;
        const int blk = wb % nblk;
        const int ib = i0 + blk * 128 + 4 * lane;  // first of this lane's 4 inputs
        float v[4];
        if (t < ntok) {
            const long long row = (long long)(xrow0 + t) * a.x_stride;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float xv;
                if constexpr (XM == kXmF16) {
                    xv = h2f_bits(static_cast<const uint16_t*>(a.x)[row + ib + j]);
                } else if constexpr (XM == kXmF32) {
                    xv = static_cast<const float*>(a.x)[row + ib + j];
                } else {  // SwiGLU of a gate_up output row: gate first, then up
                    const float* yr = static_cast<const float*>(a.x) + row;
                    xv = silu_f(yr[ib + j]) * yr[a.in + ib + j];
                }
                v[j] = h2f_bits(rin[ib + j]) * xv;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = 0.f;
        }
        h128_warp(v, lane);
        float4* dst = reinterpret_cast<float4*>(xt + t * nk + blk * 128 + 4 * lane);
        *dst = make_float4(v[0], v[1], v[2], v[3]);
    }
}

template <int K, int NB, int XM>
__global__ void __launch_bounds__(kThreads, 2) trellis_gemv_kernel(const GemvArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = static_cast<int>(cluster.block_rank());
    const int csize = static_cast<int>(cluster.num_blocks());
    const int ob = blockIdx.y;
    const int item = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int expert, xrow0, yrow0, ntok;
    if (a.slot_mode) {
        expert = a.ids ? a.ids[item] : 0;
        xrow0 = item / a.x_div;
        yrow0 = item;
        ntok = 1;
    } else {
        expert = 0;
        xrow0 = yrow0 = item * NB;
        ntok = min(NB, a.batch - item * NB);
    }

    const int KT = a.in >> 4;
    const int NT = a.out >> 4;
    const int kt0 = crank * a.kt_per_cta;
    const int kt1 = min(KT, kt0 + a.kt_per_cta);
    const int nk = (kt1 - kt0) * 16;  // a multiple of 128

    extern __shared__ __align__(16) float smem[];
    float* xt = smem;                       // [NB][nk]
    float* red = smem + NB * a.kt_per_cta * 16;  // [8 warps][NB][128]
    float* zp = red + 8 * NB * 128;         // [NB][128] this CTA's partial

    const uint16_t* codes = a.codes + (long long)expert * a.code_stride;
    // this warp's first tile row, this output block
    const int nit = (kt1 - kt0) >> 3;  // rows per warp (kt1 - kt0 is a multiple of 8)
    auto row_ptr = [&](int it) {
        const int kt = kt0 + warp + 8 * it;
        return codes + ((long long)kt * NT + ob * 8) * (16 * K);
    };

    LaneCodes<K> cur;
    if (nit > 0) load_lane_codes<K>(cur, row_ptr(0), lane);

    input_transform<NB, XM>(a, xrow0, ntok, kt0 * 16, nk, xt, warp, lane, expert);
    __syncthreads();

    float acc[NB][16];
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[t][q] = 0.f;

    const int c = lane & 3;
    const int nbr = (lane & ~3) | ((lane + 1) & 3);
    for (int it = 0; it < nit; ++it) {
        LaneCodes<K> nxt;
        if (it + 1 < nit) load_lane_codes<K>(nxt, row_ptr(it + 1), lane);
        // neighbour's first word closes this lane's last window
        cur.p[2 * K] = __shfl_sync(0xffffffffu, cur.p[0], nbr) & 0xFFFFu;
        const int kt = kt0 + warp + 8 * it;
        float xr[NB][4];
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const float4 xv = *reinterpret_cast<const float4*>(xt + t * nk + (kt - kt0) * 16 + 4 * c);
            xr[t][0] = xv.x;
            xr[t][1] = xv.y;
            xr[t][2] = xv.z;
            xr[t][3] = xv.w;
        }
        decode_fma<K, NB>(cur, xr, acc);
        if (it + 1 < nit) cur = nxt;
    }

    // Reduce-scatter over the 4 lanes of a tile: lane c ends up owning output
    // columns 4c..4c+3 of tile lane/4.
#pragma unroll
    for (int t = 0; t < NB; ++t) {
        float h8[8];
        const bool hi2 = (c & 2) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float send = hi2 ? acc[t][i] : acc[t][8 + i];
            const float keep = hi2 ? acc[t][8 + i] : acc[t][i];
            h8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        const bool hi1 = (c & 1) != 0;
        float h4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float send = hi1 ? h8[i] : h8[4 + i];
            const float keep = hi1 ? h8[4 + i] : h8[i];
            h4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        float4* dst = reinterpret_cast<float4*>(red + (warp * NB + t) * 128 + (lane >> 2) * 16 + 4 * c);
        *dst = make_float4(h4[0], h4[1], h4[2], h4[3]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < NB * 128; i += kThreads) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w * NB * 128 + i];
        zp[i] = s;
    }

    // Cluster reduction in rank order, then the output transform on rank 0.
    cluster.sync();
    if (crank == 0 && warp < NB && warp < ntok) {
        const int t = warp;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = 0.f;
        for (int r = 0; r < csize; ++r) {
            const float* rz = cluster.map_shared_rank(zp, r);
            const float4 z4 = *reinterpret_cast<const float4*>(rz + t * 128 + 4 * lane);
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        h128_warp(v, lane);
        const uint16_t* rout = a.rout + (long long)expert * a.rout_stride + ob * 128 + 4 * lane;
        float* y = a.y + (long long)(yrow0 + t) * a.y_stride + ob * 128 + 4 * lane;
        float4 o;
        o.x = h2f_bits(rout[0]) * (v[0] * 0.0078125f);
        o.y = h2f_bits(rout[1]) * (v[1] * 0.0078125f);
        o.z = h2f_bits(rout[2]) * (v[2] * 0.0078125f);
        o.w = h2f_bits(rout[3]) * (v[3] * 0.0078125f);
        *reinterpret_cast<float4*>(y) = o;
    }
    cluster.sync();  // keep every rank's shared memory alive until rank 0 has read it
}

template <int K, int NB, int XM>
cudaError_t launch_t(const GemvArgs& a, int csize, int items, cudaStream_t s) {
    const int smem = (NB * a.kt_per_cta * 16 + 8 * NB * 128 + NB * 128) * (int)sizeof(float);
    auto kern = trellis_gemv_kernel<K, NB, XM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, a.out / 128, items);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int K, int NB>
cudaError_t launch_xm(const GemvArgs& a, int csize, int items, cudaStream_t s) {
    switch (a.x_mode) {
        case kXmF16: return launch_t<K, NB, kXmF16>(a, csize, items, s);
        case kXmF32: return launch_t<K, NB, kXmF32>(a, csize, items, s);
        default: return launch_t<K, NB, kXmSwiglu>(a, csize, items, s);
    }
}

template <int K>
cudaError_t launch_nb(const GemvArgs& a, int nb, int csize, int items, cudaStream_t s) {
    switch (nb) {
        case 1: return launch_xm<K, 1>(a, csize, items, s);
        case 2: return launch_xm<K, 2>(a, csize, items, s);
        default: return launch_xm<K, 4>(a, csize, items, s);
    }
}

}  // namespace

void gemv_plan(int in, int items_times_oblk, int num_sms, int* kt_per_cta, int* csize) {
    const int kblks = in / 128;
    // Aim for about 3 CTAs per SM in total; at most 8 CTAs per cluster.
    const int target = 3 * num_sms;
    int per = 1;
    while (true) {
        const int cs = (kblks + per - 1) / per;
        if (cs <= 8 && (long long)cs * items_times_oblk <= target) break;
        if (per >= kblks) break;
        ++per;
    }
    int cs = (kblks + per - 1) / per;
    while (cs > 8) {
        ++per;
        cs = (kblks + per - 1) / per;
    }
    *kt_per_cta = per * 8;
    *csize = cs;
}

cudaError_t launch_trellis_gemv(const GemvArgs& a, int K, int nb, int items, int num_sms, cudaStream_t s) {
    GemvArgs b = a;
    int csize;
    gemv_plan(a.in, items * (a.out / 128), num_sms, &b.kt_per_cta, &csize);
    return K == 2 ? launch_nb<2>(b, nb, csize, items, s) : launch_nb<3>(b, nb, csize, items, s);
}

}  // namespace escha
