// One trellis-coded projection, y[b] = rout * H128(W^T H128(rin * x[b])),
// for a batch of tokens sharing the weight (hipfire PR #694, commit
// "EschaProj holds what a trellis weight needs": H128-in -> trellis GEMV ->
// H128-out).
//
// Grid: x = CTAs splitting the input rows (one thread-block cluster per
// output block), y = 128-wide output blocks, z = groups of NB tokens. Each
// CTA transforms its slice of the input (rin * x, then the blockwise
// Hadamard), runs the fused decode GEMV over its rows, and the cluster sums
// the partials through distributed shared memory in rank order
// (deterministic, no atomics); rank 0 applies the output transform.
#include "kernels.h"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// xt[t][i] = H128(rin * x[t]) (unscaled) for this CTA's inputs i0..i0+nk-1,
// one warp per (token, 128-block).
template <int NB, int XM>
__device__ void gemv_input_transform(const GemvArgs& a, int xrow0, int ntok, int i0, int nk, float* xt, int warp,
                                     int lane) {
    const int nblk = nk / 128;
    for (int wb = warp; wb < NB * nblk; wb += kWarps) {
        const int t = wb / nblk;
        const int blk = wb % nblk;
        const int ib = i0 + blk * 128 + 4 * lane;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (t < ntok) {
            const long long row = (long long)(xrow0 + t) * a.x_stride;
            const uint2 rb = *reinterpret_cast<const uint2*>(a.rin + ib);
            const float r4[4] = {h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(rb.x >> 16)),
                                 h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)), h2f_bits(static_cast<uint16_t>(rb.y >> 16))};
            if constexpr (XM == kXmF16) {
                const uint2 xb = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + row + ib);
                v[0] = r4[0] * h2f_bits(static_cast<uint16_t>(xb.x & 0xFFFFu));
                v[1] = r4[1] * h2f_bits(static_cast<uint16_t>(xb.x >> 16));
                v[2] = r4[2] * h2f_bits(static_cast<uint16_t>(xb.y & 0xFFFFu));
                v[3] = r4[3] * h2f_bits(static_cast<uint16_t>(xb.y >> 16));
            } else {
                const float4 xv = *reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + row + ib);
                v[0] = r4[0] * xv.x;
                v[1] = r4[1] * xv.y;
                v[2] = r4[2] * xv.z;
                v[3] = r4[3] * xv.w;
            }
        }
        h128_warp(v, lane);
        *reinterpret_cast<float4*>(xt + t * nk + blk * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// One token per CTA: 64 registers, 4 CTAs per SM; 2 or 4 tokens: 2 per SM.
template <int K, int NB, int XM>
__global__ void __launch_bounds__(kThreads, NB == 1 ? 4 : 2) trellis_gemv_kernel(const GemvArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = static_cast<int>(cluster.block_rank());
    const int csize = static_cast<int>(cluster.num_blocks());
    const int ob = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row0 = blockIdx.z * NB;
    const int ntok = min(NB, a.batch - row0);

    const int KT = a.in >> 4;
    const int kt0 = crank * a.kt_per_cta;
    const int kt1 = min(KT, kt0 + a.kt_per_cta);
    const int nk = (kt1 - kt0) * 16;

    extern __shared__ __align__(16) float smem[];
    float* xt = smem;                            // [NB][kt_per_cta*16]
    float* red = xt + NB * a.kt_per_cta * 16;    // [kWarps][NB][128]
    float* zp = red + kWarps * NB * 128;         // [NB][128]
    float* slots = zp + NB * 128;                // [16][NB][128] the ranks' partials, on rank 0
    // [kWarps][4 KB] weights decoded ahead of the wait (one row per warp)
    uint32_t* wd = reinterpret_cast<uint32_t*>(slots + 16 * NB * 128);

    // One token and one tile row per warp (kt_per_cta comes in multiples of
    // 8, so the CTA's inputs are one Hadamard block): everything but x is a
    // weight, so the decode and the loads of rin, rout and the bias run
    // before the wait, while the preceding kernel finishes. The next launch
    // may then be scheduled at once, to decode its own weights meanwhile
    // (1024 x 2048, one token, 1024 calls in a graph: 3.80 -> 3.12 us per
    // call with the decode ahead, 3.01 with the early trigger).
    const bool ahead = NB == 1 && a.kt_per_cta <= kWarps;
    if (ahead) pdl_trigger();

    const TileStrides grid = tile_strides(a.in, a.out, a.nt_major != 0);
    LaneCodes<K> cur;
    const bool has_row = kt0 + warp < kt1;
    if (has_row) load_lane_codes<K>(cur, a.codes, grid, kt0 + warp, ob * 8, lane);
    uint2 rin_pre = make_uint2(0u, 0u), rout_pre = make_uint2(0u, 0u);
    float4 bias_pre = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ahead) {
        if (warp == 0) rin_pre = *reinterpret_cast<const uint2*>(a.rin + kt0 * 16 + 4 * lane);
        if (crank == 0 && warp == 0) {
            rout_pre = *reinterpret_cast<const uint2*>(a.rout + ob * 128 + 4 * lane);
            if (a.bias) bias_pre = *reinterpret_cast<const float4*>(a.bias + ob * 128 + 4 * lane);
        }
        if (has_row) {
            cur.p[2 * K] = __shfl_sync(0xffffffffu, cur.p[0], (lane & ~3) | ((lane + 1) & 3)) & 0xFFFFu;
            decode_store<K>(cur, wd + warp * 1024, lane);
        }
    }
    pdl_wait();  // x may be the previous launch's output
    if (ahead) {
        if (warp == 0) {  // xt = H128(rin * x) of the CTA's one input block
            const long long row = (long long)row0 * a.x_stride + kt0 * 16 + 4 * lane;
            float v[4];
            const float r4[4] = {h2f_bits(static_cast<uint16_t>(rin_pre.x & 0xFFFFu)),
                                 h2f_bits(static_cast<uint16_t>(rin_pre.x >> 16)),
                                 h2f_bits(static_cast<uint16_t>(rin_pre.y & 0xFFFFu)),
                                 h2f_bits(static_cast<uint16_t>(rin_pre.y >> 16))};
            if constexpr (XM == kXmF16) {
                const uint2 xb = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + row);
                v[0] = r4[0] * h2f_bits(static_cast<uint16_t>(xb.x & 0xFFFFu));
                v[1] = r4[1] * h2f_bits(static_cast<uint16_t>(xb.x >> 16));
                v[2] = r4[2] * h2f_bits(static_cast<uint16_t>(xb.y & 0xFFFFu));
                v[3] = r4[3] * h2f_bits(static_cast<uint16_t>(xb.y >> 16));
            } else {
                const float4 xv = *reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + row);
                v[0] = r4[0] * xv.x;
                v[1] = r4[1] * xv.y;
                v[2] = r4[2] * xv.z;
                v[3] = r4[3] * xv.w;
            }
            h128_warp(v, lane);
            *reinterpret_cast<float4*>(xt + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
        }
        __syncthreads();
        float2 acc2[1][8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc2[0][i] = make_float2(0.f, 0.f);
        if (has_row) {
            const float4 xv = *reinterpret_cast<const float4*>(xt + warp * 16 + 4 * (lane & 3));
            const float xr[4] = {xv.x, xv.y, xv.z, xv.w};
            fma_decoded<K>(wd + warp * 1024, lane, xr, acc2[0]);
        }
        cta_partial_reduce<K, 1, kWarps>(acc2, red, zp);
    } else {
        gemv_input_transform<NB, XM>(a, row0, ntok, kt0 * 16, nk, xt, warp, lane);
        __syncthreads();
        cta_gemv_partial<K, NB, kWarps>(a.codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);
    }
    // The next launch on the stream may start now; it prefetches its own codes
    // and waits for this grid before it reads activations or writes outputs.
    if (!ahead) pdl_trigger();

    // Ranks != 0 push their partials into rank 0's slots and one cluster
    // barrier (release / acquire) publishes them; rank 0 then reads only its
    // own shared memory and the other ranks are done (3.01 -> 2.78 us per
    // call above, against rank 0 reading every rank's shared memory between
    // two barriers).
    if (crank != 0) {
        for (int i = threadIdx.x; i < NB * 32; i += kThreads)
            st_cluster_v4(cluster_map(smem_u32(slots + crank * NB * 128 + 4 * i), 0),
                          *reinterpret_cast<const float4*>(zp + 4 * i));
    }
    cluster.sync();
    if (crank != 0) return;
    if (warp < ntok) {
        const int t = warp;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < csize; ++r) {
            const float4 z4 = *reinterpret_cast<const float4*>((r == 0 ? zp : slots + r * NB * 128) + t * 128 + 4 * lane);
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        if (ahead) {
            output_transform_regs(v, rout_pre, lane);
        } else {
            output_transform_warp(v, a.rout + ob * 128, lane);
            if (a.bias) bias_pre = *reinterpret_cast<const float4*>(a.bias + ob * 128 + 4 * lane);
        }
        if (a.bias) {  // additive output bias, after the output transform
            v[0] += bias_pre.x;
            v[1] += bias_pre.y;
            v[2] += bias_pre.z;
            v[3] += bias_pre.w;
        }
        *reinterpret_cast<float4*>(a.y + (long long)(row0 + t) * a.y_stride + ob * 128 + 4 * lane) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

template <int K, int NB, int XM>
cudaError_t launch_t(const GemvArgs& a, int csize, int items, cudaStream_t s) {
    const int ahead = NB == 1 && a.kt_per_cta <= kWarps ? kWarps * 4096 : 0;  // weights decoded ahead
    const int smem = (NB * a.kt_per_cta * 16 + kWarps * NB * 128 + NB * 128 + 16 * NB * 128) * (int)sizeof(float) + ahead;
    auto kern = trellis_gemv_kernel<K, NB, XM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (csize > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, a.out / 128, items);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int K, int NB>
cudaError_t launch_xm(const GemvArgs& a, int csize, int items, cudaStream_t s) {
    return a.x_mode == kXmF16 ? launch_t<K, NB, kXmF16>(a, csize, items, s) : launch_t<K, NB, kXmF32>(a, csize, items, s);
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

namespace {

void gemv_plan_clusters(int in, int blocks_per_split, int num_sms, int ctas_per_sm, int max_cluster,
                        int* kt_per_cta, int* csize) {
    // Most input-row splits (at most max_cluster CTAs per cluster) whose grid
    // still fits in one wave of resident CTAs, but at most 16 Hadamard blocks
    // (2048 inputs) per CTA so the transformed input stays small in shared
    // memory.
    const int kblks = in / 128;
    const long long slots = (long long)num_sms * ctas_per_sm;
    int cs = 1;
    for (int c = 1; c <= max_cluster && c <= kblks; ++c) {
        if ((long long)c * blocks_per_split <= slots) cs = c;
    }
    const int cs_min = (kblks + 15) / 16;
    if (cs < cs_min) cs = cs_min < 8 ? cs_min : 8;
    const int per = (kblks + cs - 1) / cs;
    *kt_per_cta = per * 8;
    *csize = (kblks + per - 1) / per;
}

}  // namespace

void gemv_plan(int in, int blocks_per_split, int num_sms, int ctas_per_sm, int* kt_per_cta, int* csize) {
    gemv_plan_clusters(in, blocks_per_split, num_sms, ctas_per_sm, 8, kt_per_cta, csize);
}

cudaError_t launch_trellis_gemv(const GemvArgs& a, int K, int nb, int items, int num_sms, cudaStream_t s) {
    GemvArgs b = a;
    int csize;
    // clusters of up to 16 CTAs for one token per CTA (a short, latency-bound
    // projection: 1024 x 2048 went from 3.88 to 3.73 us); with 2 or 4 tokens
    // per CTA the larger cluster reduction costs more than it saves. One
    // token per CTA plans for 4 resident CTAs per SM (5120 -> 6144 at one
    // token 20.4 -> 16.7 us; other shapes within 1%).
    // The split is sized for GB300's 152 SMs whatever the device reports, so
    // the order of the partial sums (and the result's bits) is a fixed
    // function of the shape.
    (void)num_sms;
    gemv_plan_clusters(a.in, items * (a.out / 128), 152, nb == 1 ? 4 : 2, nb == 1 ? 16 : 8, &b.kt_per_cta, &csize);
    return K == 2 ? launch_nb<2>(b, nb, csize, items, s) : launch_nb<3>(b, nb, csize, items, s);
}

}  // namespace escha
