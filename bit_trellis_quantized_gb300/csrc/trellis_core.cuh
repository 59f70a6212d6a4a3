// Device building blocks of the fused trellis decode GEMV (sm_103a).
//
// A CTA accumulates, for one 128-wide output block (8 tiles of 16 output
// columns), the partial sums z[t][o] = sum_i W[i][o] * xt[t][i] over a range
// of input-tile rows kt, with W decoded from the packed trellis codes in
// registers and never stored (hipfire PR #694 "Escha-W2 port: 2-bit trellis
// decoded in the GEMV", summary "What it is": the packed codes stay resident
// and each weight is decoded where the matvec consumes it).
//
// Inner loop. Warp w walks the tile rows kt0 + w, kt0 + w + NW, ... One warp
// load covers one tile row of the output block: 8 tiles x 16K words (512 B at
// K=2, 768 B at K=3), fully coalesced. Lane l takes tile l/4 and quarter
// c = l%4 of its words: half-rows 8c..8c+7, i.e. input rows 4c..4c+3 of the
// tile with all 16 output columns. The word after the lane's last one (the
// end of its last 16-bit window, wrapping to word 0 for c = 3: tail-biting)
// comes from the neighbouring lane by shuffle.
#pragma once

#include "common.cuh"

namespace escha {

// Programmatic dependent launch: wait until the preceding kernel on the
// stream has completed and its writes are visible (no-op without PDL), and
// allow the next kernel to be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int K>
struct LaneCodes {
    uint32_t p[2 * K + 1];  // word pairs; p[2K] low half receives the neighbour's first word
};

// Tile grid of a code tensor: tile (kt, nt) starts at codes + (kt * s_kt +
// nt * s_nt) * 16K words. kt-major (as checkpoints store it, [in/16][out/16]):
// s_kt = out/16, s_nt = 1. nt-major (the load-time transpose that puts a tile
// column's tiles next to each other, [out/16][in/16]): s_kt = 1, s_nt = in/16.
struct TileStrides {
    long long s_kt, s_nt;
};

__host__ __device__ inline TileStrides tile_strides(int in, int out, bool nt_major) {
    return nt_major ? TileStrides{1, in / 16} : TileStrides{out / 16, 1};
}

// The lane's 4K words of tile row kt of the output block whose first tile
// column is nt0: tile nt0 + lane/4, input rows 4*(lane%4) .. +3.
template <int K>
__device__ __forceinline__ void load_lane_codes(LaneCodes<K>& lc, const uint16_t* codes, const TileStrides& g, int kt,
                                                int nt0, int lane) {
    const uint16_t* tile = codes + ((long long)kt * g.s_kt + (long long)(nt0 + (lane >> 2)) * g.s_nt) * (16 * K);
    if constexpr (K == 2) {
        const uint4 v = ldg_stream_v4(tile + (lane & 3) * 8);
        lc.p[0] = v.x;
        lc.p[1] = v.y;
        lc.p[2] = v.z;
        lc.p[3] = v.w;
    } else {
        const uint16_t* b = tile + (lane & 3) * 12;
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

// Decode the lane's 64 weights and accumulate into its 16 column sums per
// token over its 4 input rows. Half-row j (input row j/2, output columns
// 8*(j%2)..+7) starts at bit 8*K*j of the lane's words and its weight m at
// bit 8*K*j + K*m; all offsets are compile-time constants.
// K = 3 decodes weights in pairs (m, m+1); K = 2 takes columns m and m + 8 of
// one input row from a single 32-bit stream window (cb_decode_window). Both
// were measured faster on GB300 than one weight at a time (fewer
// integer-pipe instructions). Each pair of weights meets the same input, so
// for one token one packed fma.rn.f32x2 (__ffma2_rn: two independent f32
// fmas, each rounded to nearest even) updates both column sums: acc2[t][i]
// holds the sums of columns acc2_col<K>(i, 0) and acc2_col<K>(i, 1). Every
// sum still receives its weights in the same order, with the same roundings.
template <int K>
__host__ __device__ constexpr int acc2_col(int i, int half) {
    return K == 2 ? i + 8 * half : 2 * i + half;
}

// acc += w * (x, x): one packed fma for one token; for several tokens two
// scalar fmas (the register pairs the packed form needs spill the 2- and
// 4-token GEMV builds). Same results either way.
template <int NB>
__device__ __forceinline__ float2 fma_pair(float2 w, float x, float2 acc) {
    if constexpr (NB == 1) {
        return __ffma2_rn(w, make_float2(x, x), acc);
    } else {
        return make_float2(fmaf(w.x, x, acc.x), fmaf(w.y, x, acc.y));
    }
}

template <int K, int NB>
__device__ __forceinline__ void decode_fma(const LaneCodes<K>& lc, const float (&xr)[NB][4], float2 (&acc2)[NB][8]) {
    if constexpr (K == 2) {  // weights (row r, col m) and (row r, col m + 8) share a window
        uint32_t q[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) q[i] = stream_pair(lc.p[i]);
        static_for<32>([&](auto I) {
            constexpr int r = decltype(I)::value / 8, m = decltype(I)::value % 8;
            __half ha, hb;
            cb_decode_window(bits32<2 * m>(q[r], q[r + 1]), ha, hb);
            const float2 w = make_float2(__half2float(ha), __half2float(hb));
#pragma unroll
            for (int t = 0; t < NB; ++t) acc2[t][m] = fma_pair<NB>(w, xr[t][r], acc2[t][m]);
        });
        return;
    }
    static_for<32>([&](auto I) {
        constexpr int j = (2 * decltype(I)::value) / 8;
        constexpr int m = (2 * decltype(I)::value) % 8;
        constexpr int b0 = 8 * K * j + K * m, b1 = b0 + K;
        const uint32_t s0 = window_state<(b0 & 15)>(stream_window<(b0 >> 4)>(lc.p));
        const uint32_t s1 = window_state<(b1 & 15)>(stream_window<(b1 >> 4)>(lc.p));
        const float2 w = __half22float2(cb_decode_h2(s0, s1));
        constexpr int i = (8 * (j & 1) + m) / 2;  // columns 2i, 2i + 1
#pragma unroll
        for (int t = 0; t < NB; ++t) acc2[t][i] = fma_pair<NB>(w, xr[t][j >> 1], acc2[t][i]);
    });
}

// Decode ahead of the activations. decode_store writes the lane's 64
// weights of one tile row as 32 half2 pairs, in the order decode_fma
// consumes them, to the warp's 4 KB of shared memory `wd` (layout
// [8][32 lanes][4 words]: a warp's 16-byte accesses are conflict-free).
// fma_decoded later runs decode_fma's multiply-adds on them for one token:
// the same weights in the same order, so the same results.
template <int K>
__device__ __forceinline__ void decode_store(const LaneCodes<K>& lc, uint32_t* wd, int lane) {
    uint32_t h[4];
    auto put = [&](auto I, __half2 w) {
        constexpr int i = decltype(I)::value;
        h[i % 4] = *reinterpret_cast<const uint32_t*>(&w);
        if constexpr (i % 4 == 3)
            *reinterpret_cast<uint4*>(wd + ((i / 4) * 32 + lane) * 4) = make_uint4(h[0], h[1], h[2], h[3]);
    };
    if constexpr (K == 2) {
        uint32_t q[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) q[i] = stream_pair(lc.p[i]);
        static_for<32>([&](auto I) {
            constexpr int r = decltype(I)::value / 8, m = decltype(I)::value % 8;
            __half ha, hb;
            cb_decode_window(bits32<2 * m>(q[r], q[r + 1]), ha, hb);
            put(I, __halves2half2(ha, hb));
        });
    } else {
        static_for<32>([&](auto I) {
            constexpr int j = (2 * decltype(I)::value) / 8;
            constexpr int m = (2 * decltype(I)::value) % 8;
            constexpr int b0 = 8 * K * j + K * m, b1 = b0 + K;
            const uint32_t s0 = window_state<(b0 & 15)>(stream_window<(b0 >> 4)>(lc.p));
            const uint32_t s1 = window_state<(b1 & 15)>(stream_window<(b1 >> 4)>(lc.p));
            put(I, cb_decode_h2(s0, s1));
        });
    }
}

template <int K>
__device__ __forceinline__ void fma_decoded(const uint32_t* wd, int lane, const float (&xr)[4], float2 (&acc2)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(wd + (q * 32 + lane) * 4);
        const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int I = 4 * q + u;
            const float2 w = __half22float2(*reinterpret_cast<const __half2*>(&h[u]));
            if constexpr (K == 2) {
                acc2[I % 8] = fma_pair<1>(w, xr[I / 8], acc2[I % 8]);
            } else {
                const int j = (2 * I) / 8, m = (2 * I) % 8;
                const int i = (8 * (j & 1) + m) / 2;
                acc2[i] = fma_pair<1>(w, xr[j >> 1], acc2[i]);
            }
        }
    }
}

// The warp's column sums (acc2 as decode_fma leaves them) reduce-scattered
// over the 4 lanes of each tile and stored as the warp's row of `red`
// ([NW][NB][128] floats, smem).
template <int K, int NB>
__device__ __forceinline__ void warp_partial_store(const float2 (&acc2)[NB][8], float* red) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = lane & 3;
    // column sums in column order
    float acc[NB][16];
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc[t][acc2_col<K>(i, 0)] = acc2[t][i].x;
            acc[t][acc2_col<K>(i, 1)] = acc2[t][i].y;
        }
    // Reduce-scatter over the 4 lanes of a tile: lane c keeps output columns
    // 4c..4c+3 of tile lane/4.
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
        *reinterpret_cast<float4*>(red + (warp * NB + t) * 128 + (lane >> 2) * 16 + 4 * c) =
            make_float4(h4[0], h4[1], h4[2], h4[3]);
    }
}

// zp[i] = the warps' rows of red summed in warp order (i < n), by the CTA's
// NW warps. No barrier.
template <int NW>
__device__ __forceinline__ void cta_sum_rows(const float* red, int n, float* zp) {
    for (int i = threadIdx.x; i < n; i += NW * 32) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += red[w * n + i];
        zp[i] = s;
    }
}

// In-CTA reduction of the warps' column sums into zp[NB][128] (smem); `red`
// is smem scratch of NW*NB*128 floats. Ends with __syncthreads().
template <int K, int NB, int NW>
__device__ __forceinline__ void cta_partial_reduce(const float2 (&acc2)[NB][8], float* red, float* zp) {
    warp_partial_store<K, NB>(acc2, red);
    __syncthreads();
    cta_sum_rows<NW>(red, NB * 128, zp);
    __syncthreads();
}

// Main loop and in-CTA reduction. `codes` is the expert's code tensor, `g`
// its tile grid, `ob` the output block, rows kt0..kt1-1,
// `xt` the transformed inputs [NB][nk] of those rows (smem), `first` the
// lane's codes of its first row (already loaded). Writes the CTA's partial
// sums zp[NB][128] (smem). `red` is smem scratch of NW*NB*128 floats.
// Ends with __syncthreads().
template <int K, int NB, int NW>
__device__ __forceinline__ void cta_gemv_partial(const uint16_t* codes, const TileStrides& g, int ob, int kt0, int kt1,
                                                 const float* xt, int nk, LaneCodes<K>& cur, float* red,
                                                 float* zp) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = lane & 3;
    const int nbr = (lane & ~3) | ((lane + 1) & 3);
    float2 acc2[NB][8];
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc2[t][i] = make_float2(0.f, 0.f);

    auto step = [&](LaneCodes<K>& lc, int kt) {
        lc.p[2 * K] = __shfl_sync(0xffffffffu, lc.p[0], nbr) & 0xFFFFu;
        float xr[NB][4];
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const float4 xv = *reinterpret_cast<const float4*>(xt + t * nk + (kt - kt0) * 16 + 4 * c);
            xr[t][0] = xv.x;
            xr[t][1] = xv.y;
            xr[t][2] = xv.z;
            xr[t][3] = xv.w;
        }
        decode_fma<K, NB>(lc, xr, acc2);
    };
    // rows kt0 + warp + i*NW, two per iteration: `cur` and `nxt` take turns, so
    // the codes of the next row load while a row is decoded and are never
    // copied (a register copy would wait for the load)
    LaneCodes<K> nxt;
    for (int kt = kt0 + warp; kt < kt1; kt += 2 * NW) {
        const bool more1 = kt + NW < kt1;
        if (more1) load_lane_codes<K>(nxt, codes, g, kt + NW, ob * 8, lane);
        step(cur, kt);
        if (!more1) break;
        if (kt + 2 * NW < kt1) load_lane_codes<K>(cur, codes, g, kt + 2 * NW, ob * 8, lane);
        step(nxt, kt + NW);
    }

    cta_partial_reduce<K, NB, NW>(acc2, red, zp);
}

// cta_gemv_partial<K, 1, NW> for one token whose transformed inputs xg[nk]
// (rows kt0..kt1-1) lie in global memory, written by another CTA of the
// running grid (read through L2): each warp loads the 4 inputs of a tile
// row together with that row's codes, so no CTA barrier precedes the
// decode. Same arithmetic and order as cta_gemv_partial<K, 1, NW>.
template <int K, int NW>
__device__ __forceinline__ void cta_gemv_partial_gx(const uint16_t* codes, const TileStrides& g, int ob, int kt0, int kt1,
                                                    const float* xg, LaneCodes<K>& cur, float* red, float* zp) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = lane & 3;
    const int nbr = (lane & ~3) | ((lane + 1) & 3);
    float2 acc2[1][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[0][i] = make_float2(0.f, 0.f);
    auto load_x = [&](int kt) { return __ldcg(reinterpret_cast<const float4*>(xg + (kt - kt0) * 16 + 4 * c)); };
    auto step = [&](LaneCodes<K>& lc, const float4& xv) {
        lc.p[2 * K] = __shfl_sync(0xffffffffu, lc.p[0], nbr) & 0xFFFFu;
        const float xr[1][4] = {{xv.x, xv.y, xv.z, xv.w}};
        decode_fma<K, 1>(lc, xr, acc2);
    };
    LaneCodes<K> nxt;
    float4 xc = make_float4(0.f, 0.f, 0.f, 0.f), xn = xc;
    if (kt0 + warp < kt1) xc = load_x(kt0 + warp);
    for (int kt = kt0 + warp; kt < kt1; kt += 2 * NW) {
        const bool more1 = kt + NW < kt1;
        if (more1) {
            load_lane_codes<K>(nxt, codes, g, kt + NW, ob * 8, lane);
            xn = load_x(kt + NW);
        }
        step(cur, xc);
        if (!more1) break;
        if (kt + 2 * NW < kt1) {
            load_lane_codes<K>(cur, codes, g, kt + 2 * NW, ob * 8, lane);
            xc = load_x(kt + 2 * NW);
        }
        step(nxt, xn);
    }
    cta_partial_reduce<K, 1, NW>(acc2, red, zp);
}

// Output transform of one 128-block by one warp: v holds 4 consecutive
// values per lane (element 4*lane + j); returns rout * (2^-7 * H128(v)) in v.
// (Both Hadamards run unscaled; their two 1/sqrt(128) factors make the exact
// 2^-7, applied before rout so that rout stays the final multiply.)
// rb: the lane's 4 rout values (fp16 bits), already loaded.
__device__ __forceinline__ void output_transform_regs(float (&v)[4], uint2 rb, int lane) {
    h128_warp(v, lane);
    v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * (v[0] * 0.0078125f);
    v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * (v[1] * 0.0078125f);
    v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * (v[2] * 0.0078125f);
    v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * (v[3] * 0.0078125f);
}

__device__ __forceinline__ void output_transform_warp(float (&v)[4], const uint16_t* rout_blk, int lane) {
    output_transform_regs(v, *reinterpret_cast<const uint2*>(rout_blk + 4 * lane), lane);
}

// int8 weights -> exact floats without a conversion instruction: each byte,
// biased to b + 128, is placed in the mantissa of 2^23 and 2^23 + 128 is
// subtracted.
__device__ __forceinline__ void i8x4_to_f32(uint32_t v, float (&f)[4]) {
    const uint32_t u = v ^ 0x80808080u;
    const float bias = 8388736.0f;  // 2^23 + 128
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
}

// Position of activation element i in a staged activation buffer. Lane l of
// an int8 row dot reads the float4s 4l + q (q = 0..3) of each 512-column
// chunk; unswizzled, the 8 lanes of a shared-memory wavefront would hit only
// 2 of the 8 16-byte bank groups. XOR-ing the float4 index with bits 3..5 of
// itself spreads them over all 8.
__device__ __forceinline__ int xs_swz(int i) {
    const int f = i >> 2;
    return ((f ^ ((f >> 3) & 7)) << 2) | (i & 3);
}

// One warp: dot products of R int8 rows (row r at w + r*ld, n columns,
// n % 16 == 0) with MT f32 vectors in shared memory, element i of vector t
// at xs[xs_swz(t*xstride + i)] (xstride % 32 == 0). All
// 16-byte loads of a group of NCH chunks of 512 columns are issued before any
// arithmetic, so a warp waits for memory once per group, not once per row.
// Rows r >= nrows are skipped. Lane 0 holds the sums.
template <int R, int MT, int NCH = 4>
__device__ __forceinline__ void int8_rows_dot(const int8_t* w, long long ld, int nrows, int n, const float* xs,
                                              int xstride, int lane, float (&out)[R][MT]) {
    float acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = 0.f;
    for (int g0 = 0; g0 < n; g0 += NCH * 512) {
        uint4 wv[R][NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = g0 + c * 512 + lane * 16;
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (r < nrows && i0 < n) wv[r][c] = ldg_stream_v4(w + r * ld + i0);
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = g0 + c * 512 + lane * 16;
            if (i0 >= n) break;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float xq[MT][4];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const float4 xv = *reinterpret_cast<const float4*>(xs + xs_swz(t * xstride + i0 + 4 * q));
                    xq[t][0] = xv.x;
                    xq[t][1] = xv.y;
                    xq[t][2] = xv.z;
                    xq[t][3] = xv.w;
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= nrows) break;
                    const uint32_t word = q == 0 ? wv[r][c].x : q == 1 ? wv[r][c].y : q == 2 ? wv[r][c].z : wv[r][c].w;
                    float f[4];
                    i8x4_to_f32(word, f);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        acc[r][t] = fmaf(f[0], xq[t][0], acc[r][t]);
                        acc[r][t] = fmaf(f[1], xq[t][1], acc[r][t]);
                        acc[r][t] = fmaf(f[2], xq[t][2], acc[r][t]);
                        acc[r][t] = fmaf(f[3], xq[t][3], acc[r][t]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float v = acc[r][t];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            out[r][t] = v;
        }
}

// Top-k of one token's f16 logits by one warp: ids ordered by (logit desc,
// id asc), ties to the lower expert id, and the softmax over the k selected
// logits. E <= 256, k <= 8. Each logit becomes a unique 32-bit key whose
// order is (value, then lower id): the f16 bit pattern mapped to an
// order-preserving unsigned 16-bit value (with -0 folded into +0, since the
// two compare equal), above 0xFFFF - id. k rounds of a warp-wide max
// (__reduce_max_sync) pick the keys. Lane j < k returns expert j and weight j.
// bits[i] holds the f16 logit of expert lane + 32 i (ignored for experts >= E).
__device__ __forceinline__ void topk_softmax_warp_bits(const uint16_t (&bits)[8], int E, int topk, int lane,
                                                       int* e_out, float* w_out) {
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        uint32_t b = e < E ? bits[i] : 0u;
        if (b == 0x8000u) b = 0u;
        const uint32_t ord = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
        key[i] = e < E ? ((ord << 16) | (0xFFFFu - static_cast<uint32_t>(e))) : 0u;
    }
    uint32_t mine = 0u;
    for (int k = 0; k < topk; ++k) {
        uint32_t m = key[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) m = max(m, key[i]);
        const uint32_t g = __reduce_max_sync(0xffffffffu, m);
#pragma unroll
        for (int i = 0; i < 8; ++i) key[i] = key[i] == g ? 0u : key[i];
        if (lane == k) mine = g;
    }
    const uint32_t ord = mine >> 16;
    const uint32_t lbits = (ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu);
    const float lv = h2f_bits(static_cast<uint16_t>(lbits));
    const float top = __shfl_sync(0xffffffffu, lv, 0);
    float ex = lane < topk ? expf(lv - top) : 0.f;
    float den = ex;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) den += __shfl_xor_sync(0xffffffffu, den, m);
    *e_out = static_cast<int>(0xFFFFu - (mine & 0xFFFFu));
    *w_out = ex / den;
}

__device__ __forceinline__ void topk_softmax_warp(const uint16_t* logits, int E, int topk, int lane, int* e_out,
                                                  float* w_out) {
    uint16_t bits[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) bits[i] = lane + 32 * i < E ? logits[lane + 32 * i] : 0;
    topk_softmax_warp_bits(bits, E, topk, lane, e_out, w_out);
}

// ---------------------------------------------------------------------------
// One-way cluster reduction: ranks push 128-float partials into rank 0's
// shared memory and arrive on an mbarrier there; rank 0 waits with an
// iteration limit (a flag is raised instead of hanging if arrivals never
// come). Shared-memory addresses are 32-bit shared-window addresses.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Waits for phase 0 of the mbarrier; gives up after `limit` polls (each poll
// may suspend for a while inside try_wait) and sets *err.
__device__ __forceinline__ void mbar_wait_bounded(uint32_t bar, int* err, int code, long long limit = 1ll << 24) {
    for (long long it = 0; !mbar_try_wait(bar, 0); ++it) {
        if (it > limit) {
            if (err) atomicExch(err, code);
            break;
        }
    }
}

}  // namespace escha
