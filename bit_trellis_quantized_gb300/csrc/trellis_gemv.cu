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

    const TileStrides grid = tile_strides(a.in, a.out, a.nt_major != 0);
    LaneCodes<K> cur;
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, a.codes, grid, kt0 + warp, ob * 8, lane);
    pdl_wait();  // x may be the previous launch's output
    gemv_input_transform<NB, XM>(a, row0, ntok, kt0 * 16, nk, xt, warp, lane);
    __syncthreads();
    cta_gemv_partial<K, NB, kWarps>(a.codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);
    // The next launch on the stream may start now; it prefetches its own codes
    // and waits for this grid before it reads activations or writes outputs.
    pdl_trigger();

    cluster.sync();
    if (crank == 0 && warp < ntok) {
        const int t = warp;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < csize; ++r) {
            const float4 z4 = *reinterpret_cast<const float4*>(cluster.map_shared_rank(zp, r) + t * 128 + 4 * lane);
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        output_transform_warp(v, a.rout + ob * 128, lane);
        if (a.bias) {  // additive output bias, after the output transform
            const float4 b4 = *reinterpret_cast<const float4*>(a.bias + ob * 128 + 4 * lane);
            v[0] += b4.x;
            v[1] += b4.y;
            v[2] += b4.z;
            v[3] += b4.w;
        }
        *reinterpret_cast<float4*>(a.y + (long long)(row0 + t) * a.y_stride + ob * 128 + 4 * lane) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
    cluster.sync();  // every rank's shared memory stays alive until rank 0 has read it
}

template <int K, int NB, int XM>
cudaError_t launch_t(const GemvArgs& a, int csize, int items, cudaStream_t s) {
    const int smem = (NB * a.kt_per_cta * 16 + kWarps * NB * 128 + NB * 128) * (int)sizeof(float);
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
