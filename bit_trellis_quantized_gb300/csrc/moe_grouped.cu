// Batched / prefill MoE block: tokens grouped by expert, each expert's packed
// trellis codes decoded once per work item (up to `cap` of its tokens) and fed
// to the 5th-generation tensor cores (tcgen05) as a dense contraction (hipfire
// PR #694, commits on the grouped prefill GEMM: decode each expert's weights
// once and share them across its tokens instead of re-reading them per slot).
//
// Kernels, after the router-logits kernel shared with the batch-1 path:
//  1. top-k: one warp per token (ids ordered by (logit desc, id asc), softmax
//     over the k selected logits).
//  2. grouping: one CTA; stable counting sort of the slots t*k + j by expert
//     -> counts, offsets, perm (grouped position -> slot), each slot's padded
//     position (every expert's run padded to a multiple of 4 tokens) and the
//     work items (expert, first position) of at most `cap` tokens.
//  3. prep (gate_up, later down): for every (slot, 128-input block) writes
//     x~ = H128(rin_e * input) * 2^-8, split into fp16 hi and lo, as rows 2P
//     and 2P+1 (P = padded position) of the B image, in the layout the MMA
//     reads. The input is x[token] for gate_up, SwiGLU(gate_up output) for
//     down.
//  4. grouped GEMM: one CTA per (work item, 128-wide output block). The 8
//     warps decode one tile row each per 128-input block into an MN-major A
//     operand; the item's B rows arrive by bulk copy; one thread issues the
//     MMAs (M = 128 outputs, N = 2 x tokens) into TMEM. The epilogue adds the
//     hi and lo columns and applies 2^8, the output Hadamard, 2^-7 and rout.
//  5. combine: out[t] = sum_j w[t][j] * down(slot t*k + j) + sigmoid(g . x[t])
//     * shared(x[t]) in slot order (the shared expert runs on the int8 GEMM).
#include "kernels.h"
#include "tc_mainloop.cuh"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr float kPrescale = 0.00390625f;  // 2^-8: keeps x~ inside the fp16 range, undone in the epilogue

// ---------------------------------------------------------------------------
// 1. top-k
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_topk_kernel(const MoeArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    pdl_wait();
    pdl_trigger();
    if (t >= a.T) return;
    int e;
    float w;
    topk_softmax_warp(a.logits + (long long)t * a.E, a.E, a.topk, lane, &e, &w);
    if (lane < a.topk) {
        a.ids[(long long)t * a.topk + lane] = e;
        a.w[(long long)t * a.topk + lane] = w;
    }
}

// Lanes whose 9-bit value v equals this lane's (the mask match_any would give),
// from one ballot per bit.
__device__ __forceinline__ unsigned match_any_9bit(int v) {
    unsigned m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 9; ++b) {
        const bool bit = (v >> b) & 1;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

// ---------------------------------------------------------------------------
// 2. grouping (one CTA of 32 warps). Warp w owns the slots of segment w (in
// slot order) and walks them 32 at a time; lanes holding the same expert
// find each other with ballots, so ranks inside a round follow lane order and
// the sort is stable without atomics.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024, 1) moe_group_kernel(const MoeArgs a) {
    __shared__ int hist[32][256];  // per-warp counts, then per-warp running starts within each expert
    __shared__ int off_s[257], poff_s[257], ibase_s[257];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.T * a.topk, E = a.E, cap = a.grp_cap;
    const int seg = (S + 31) / 32;
    const int s_begin = warp * seg, s_end = min(S, s_begin + seg);
    const unsigned lt = (1u << lane) - 1u;
    pdl_wait();
    pdl_trigger();
    for (int i = tid; i < 32 * 256; i += 1024) (&hist[0][0])[i] = 0;
    __syncthreads();
    // pass 1: per-warp counts (the ids of 8 rounds are loaded before any is used)
    for (int s0 = s_begin; s0 < s_end; s0 += 256) {
        int ev[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int s = s0 + 32 * r + lane;
            ev[r] = s < s_end ? a.ids[s] : 256 + lane;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if (s0 + 32 * r >= s_end) break;  // warp-uniform
            const bool valid = s0 + 32 * r + lane < s_end;
            const unsigned m = match_any_9bit(ev[r]);
            if (valid && (m & lt) == 0) hist[warp][ev[r]] += __popc(m);
            __syncwarp();
        }
    }
    __syncthreads();
    int cnt = 0;
    if (tid < E) {  // per-expert: each warp's start inside the expert's run
        for (int w = 0; w < 32; ++w) {
            const int c = hist[w][tid];
            hist[w][tid] = cnt;
            cnt += c;
        }
        a.grp_counts[tid] = cnt;
    }
    // exclusive scans over experts (warps 0..7 hold experts 32*warp + lane)
    __shared__ int wsum[3][8];
    int c4 = 0, ni = 0;
    if (tid < 256) {
        c4 = tid < E ? (cnt + 3) & ~3 : 0;
        ni = tid < E ? (cnt + cap - 1) / cap : 0;
        if (tid >= E) cnt = 0;
        int v0 = cnt, v1 = c4, v2 = ni;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u0 = __shfl_up_sync(0xffffffffu, v0, d);
            const int u1 = __shfl_up_sync(0xffffffffu, v1, d);
            const int u2 = __shfl_up_sync(0xffffffffu, v2, d);
            if (lane >= d) {
                v0 += u0;
                v1 += u1;
                v2 += u2;
            }
        }
        if (lane == 31) {
            wsum[0][warp] = v0;
            wsum[1][warp] = v1;
            wsum[2][warp] = v2;
        }
        off_s[tid] = v0 - cnt;  // warp-local exclusive, completed below
        poff_s[tid] = v1 - c4;
        ibase_s[tid] = v2 - ni;
    }
    __syncthreads();
    if (tid < 256) {
        int b0 = 0, b1 = 0, b2 = 0;
        for (int w = 0; w < warp; ++w) {
            b0 += wsum[0][w];
            b1 += wsum[1][w];
            b2 += wsum[2][w];
        }
        off_s[tid] += b0;
        poff_s[tid] += b1;
        ibase_s[tid] += b2;
        if (tid == 255) {
            off_s[256] = off_s[255] + cnt;
            poff_s[256] = poff_s[255] + c4;
            ibase_s[256] = ibase_s[255] + ni;
        }
    }
    __syncthreads();
    if (tid < E) {
        a.grp_offsets[tid] = off_s[tid];
        a.grp_poff[tid] = poff_s[tid];
        for (int j = 0; j < ni; ++j)
            a.grp_items[ibase_s[tid] + j] =
                make_int4(tid, min(cap, cnt - j * cap), 2 * (poff_s[tid] + j * cap), off_s[tid] + j * cap);
    }
    if (tid == 0) {
        a.grp_offsets[E] = off_s[256];
        *a.grp_nitems = ibase_s[256];
    }
    // pass 2: stable scatter
    for (int s0 = s_begin; s0 < s_end; s0 += 256) {
        int ev[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int s = s0 + 32 * r + lane;
            ev[r] = s < s_end ? a.ids[s] : 256 + lane;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if (s0 + 32 * r >= s_end) break;  // warp-uniform
            const int s = s0 + 32 * r + lane;
            const bool valid = s < s_end;
            const int e = ev[r];
            const unsigned m = match_any_9bit(e);
            const int start = valid ? hist[warp][e] : 0;
            __syncwarp();
            if (valid) {
                const int rk = start + __popc(m & lt);
                a.grp_perm[off_s[e] + rk] = s;
                a.grp_ppos[s] = poff_s[e] + rk;
                if ((m & lt) == 0) hist[warp][e] = start + __popc(m);
            }
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------------------
// 3. prep: the B image of one projection
// ---------------------------------------------------------------------------
struct GroupedProj {
    const uint16_t* codes;  // [E] x tile grid of [in/16][out/16] (kt-major) or [out/16][in/16] tiles of 16K words
    const uint16_t* rin;    // [E][in]
    const uint16_t* rout;   // [E][out]
    int in, out;
    int mode;               // 0: input = x[token] (fp16); 1: input = SwiGLU(ygu[slot]); 2: input = xf[token] (f32)
    float* y;               // [slots][out]
    TileStrides grid;       // tile grid of one expert's codes
    const float* bias;      // f32 [out] added after the output transform, or null
    const float* xf;        // mode 2: f32 input [T][in]
    int kblk_per_split;     // 64-input blocks per K split (blockIdx.z); in/64 without a split
    float* part;            // with K splits: f32 partial sums [splits][slots][out], else null
};

// One warp per (slot, 4 consecutive 128-input blocks): 8 lanes per block, 16
// consecutive values per lane, so the blockwise Hadamard runs its first four
// butterfly stages in registers and only the last three across lanes
// (shuffles within the 8 lanes). Loads and image stores are 16-byte vectors.
__global__ void __launch_bounds__(256) moe_prep_kernel(const MoeArgs a, const GroupedProj p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int nblk = p.in >> 7;
    const int ngrp = (nblk + 3) / 4;
    const long long task = (long long)blockIdx.x * 8 + warp;
    if (task >= (long long)a.T * a.topk * ngrp) return;  // warp-uniform
    const int s = static_cast<int>(task / ngrp);
    const int b = static_cast<int>(task % ngrp) * 4 + (lane >> 3);
    const int l8 = lane & 7;
    const bool live = b < nblk;  // lanes of a block past the input still join the shuffles
    // a dense linear (no ids) is one expert with the tokens in order
    const int e = a.ids ? a.ids[s] : 0;
    const int P = a.grp_ppos ? a.grp_ppos[s] : s;
    const int ib = b * 128 + 16 * l8;
    float v[16];
    if (live) {
        const uint4* rp = reinterpret_cast<const uint4*>(p.rin + (long long)e * p.in + ib);
        const uint4 r0 = rp[0], r1 = rp[1];
        const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        if (p.mode == 2) {
            const float4* xp = reinterpret_cast<const float4*>(p.xf + (long long)(s / a.topk) * p.in + ib);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = xp[q];
                v[4 * q] = f.x;
                v[4 * q + 1] = f.y;
                v[4 * q + 2] = f.z;
                v[4 * q + 3] = f.w;
            }
        } else if (p.mode == 0) {
            const uint4* xp = reinterpret_cast<const uint4*>(a.x + (long long)(s / a.topk) * a.hidden + ib);
            const uint4 x0 = xp[0], x1 = xp[1];
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                v[2 * q] = h2f_bits(static_cast<uint16_t>(xw[q] & 0xFFFFu));
                v[2 * q + 1] = h2f_bits(static_cast<uint16_t>(xw[q] >> 16));
            }
        } else {
            const float4* gp = reinterpret_cast<const float4*>(a.ygu + (long long)s * 2 * a.inter + ib);
            const float4* up = reinterpret_cast<const float4*>(a.ygu + (long long)s * 2 * a.inter + a.inter + ib);
            float4 g4[4], u4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                g4[q] = gp[q];
                u4[q] = up[q];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[4 * q] = silu_f(g4[q].x) * u4[q].x;
                v[4 * q + 1] = silu_f(g4[q].y) * u4[q].y;
                v[4 * q + 2] = silu_f(g4[q].z) * u4[q].z;
                v[4 * q + 3] = silu_f(g4[q].w) * u4[q].w;
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            v[2 * q] *= h2f_bits(static_cast<uint16_t>(rw[q] & 0xFFFFu));
            v[2 * q + 1] *= h2f_bits(static_cast<uint16_t>(rw[q] >> 16));
        }
    } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = 0.f;
    }
    // unscaled Sylvester butterflies: index bits 0-3 in registers, 4-6 across lanes
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j & m) continue;
            const float x0 = v[j], x1 = v[j | m];
            v[j] = x0 + x1;
            v[j | m] = x0 - x1;
        }
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        const float sgn = (l8 & m) ? -1.f : 1.f;  // upper element: partner - own; lower: own + partner
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float pv = __shfl_xor_sync(0xffffffffu, v[j], m);
            v[j] = fmaf(sgn, v[j], pv);
        }
    }
    if (!live) return;
    uint32_t hv[8], lv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float s0 = v[2 * q] * kPrescale, s1 = v[2 * q + 1] * kPrescale;
        const __half h0 = __float2half_rn(s0), h1 = __float2half_rn(s1);
        const __half q0 = __float2half_rn(s0 - __half2float(h0)), q1 = __float2half_rn(s1 - __half2float(h1));
        hv[q] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
        lv[q] = static_cast<uint32_t>(__half_as_ushort(q0)) | (static_cast<uint32_t>(__half_as_ushort(q1)) << 16);
    }
    const int chunk = 2 * b + (l8 >> 2);
    const uint32_t k_in = static_cast<uint32_t>((16 * l8) & 63);
    uint8_t* base = a.grp_img + (long long)chunk * a.grp_img_rows * 128;
    *reinterpret_cast<uint4*>(base + tc::kmajor_off(2u * P, k_in)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(base + tc::kmajor_off(2u * P, k_in + 8u)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
    *reinterpret_cast<uint4*>(base + tc::kmajor_off(2u * P + 1u, k_in)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    *reinterpret_cast<uint4*>(base + tc::kmajor_off(2u * P + 1u, k_in + 8u)) = make_uint4(lv[4], lv[5], lv[6], lv[7]);
}

// ---------------------------------------------------------------------------
// 4. grouped GEMM
// ---------------------------------------------------------------------------
// Half tile rows. A warp decodes 4 of the 8 tiles of one tile row of the
// output block (16 inputs x 64 outputs): lane = 8 * tile + c, c = 0..7, owns
// input rows 2c and 2c+1 of its tile, i.e. bits [32 K c, 32 K (c+1)) of the
// tile's stream = K 32-bit words, plus the first 16-bit word of the next lane
// of the tile (tail-biting: lane 0 after lane 7) for the windows that cross
// the end.
template <int K>
struct HalfRowCodes {
    uint32_t p[K + 1];
};

// The lane's K 32-bit words at b: words (lane % 8) * 2K .. of its tile
// (64 B per tile at K = 2, 8-byte aligned per lane; 96 B at K = 3, 4-byte
// aligned).
template <int K>
__device__ __forceinline__ void load_half_row_at(HalfRowCodes<K>& lc, const uint16_t* b) {
    if constexpr (K == 2) {
        const uint2 v = ldg_stream_v2(b);
        lc.p[0] = v.x;
        lc.p[1] = v.y;
    } else {
        lc.p[0] = ldg_stream_u32(b);
        lc.p[1] = ldg_stream_u32(b + 2);
        lc.p[2] = ldg_stream_u32(b + 4);
    }
}

// Byte offsets, inside a tile row's A slice, of the lane's four 16-byte
// stores: index 2 * rr + h = input row 2c + rr, columns 8h .. 8h + 7 of the
// lane's tile (tile0 + lane / 8); element (m, k) sits at
// mnmajor_off(m, k, 2048, 1024).
__device__ __forceinline__ void half_row_store_offsets(uint32_t (&off)[4], int lane, int tile0) {
    const uint32_t c = static_cast<uint32_t>(lane & 7);
    const uint32_t m0 = 16u * static_cast<uint32_t>(tile0 + (lane >> 3));
#pragma unroll
    for (int i = 0; i < 4; ++i) off[i] = tc::mnmajor_off(m0 + 8u * (i & 1), 2u * c + (i >> 1), 2048u, 1024u);
}

// The lane's 32 weights (input rows 2c, 2c+1; 16 output columns of its
// tile) into the MN-major A slice of the tile row at the offsets above.
// Needs lc.p[K] = the next lane's first word.
template <int K>
__device__ __forceinline__ void decode_half_row_to_smem(const HalfRowCodes<K>& lc, uint8_t* slice,
                                                        const uint32_t (&off)[4]) {
    if constexpr (K == 2) {  // weights (row rr, col m) and (row rr, col m + 8) share a window
        const uint32_t q[3] = {stream_pair(lc.p[0]), stream_pair(lc.p[1]), stream_pair(lc.p[2])};
        static_for<2>([&](auto R) {
            constexpr int rr = decltype(R)::value;
            __half w[16];
            static_for<8>([&](auto M) {
                constexpr int m = decltype(M)::value;
                cb_decode_window(bits32<2 * m>(q[rr], q[rr + 1]), w[m], w[m + 8]);
            });
            static_for<2>([&](auto H) {  // columns 8h .. 8h + 7
                constexpr int h = decltype(H)::value;
                uint32_t packed[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const __half2 w2 = __halves2half2(w[8 * h + 2 * p], w[8 * h + 2 * p + 1]);
                    packed[p] = *reinterpret_cast<const uint32_t*>(&w2);
                }
                *reinterpret_cast<uint4*>(slice + off[2 * rr + h]) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            });
        });
        return;
    }
    static_for<4>([&](auto J) {  // quarter j: input row 2c + j/2, columns 8*(j%2)..+7
        constexpr int j = decltype(J)::value;
        uint32_t packed[4];
        static_for<4>([&](auto P) {
            constexpr int p = decltype(P)::value;
            constexpr int b0 = 8 * K * j + K * (2 * p);
            constexpr int b1 = b0 + K;
            const uint32_t s0 = window_state<(b0 & 15)>(stream_window<(b0 >> 4)>(lc.p));
            const uint32_t s1 = window_state<(b1 & 15)>(stream_window<(b1 >> 4)>(lc.p));
            const __half2 w2 = cb_decode_h2(s0, s1);
            packed[p] = *reinterpret_cast<const uint32_t*>(&w2);
        });
        *reinterpret_cast<uint4*>(slice + off[j]) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    });
}

// One CTA per (work item, 128-wide output block), K blocks of 64 inputs, 8
// decode warps + 1 issuer warp: per block decode warp w writes half tile row
// w%2 of tile row 4b + w/2 into one of two A stages (16 KB) and arrives on an
// mbarrier, without waiting for the other warps; the issuer waits for the
// stage and the item's bulk-copied B rows, issues the MMAs and copies the
// next block's B. Shared memory (2 x 16 KB A + 2 x 2 cap x 128 B B) stays
// under 100 KB for every item size, so two CTAs share an SM and one's
// prologue and epilogue overlap the other's decode.
template <int K, int STAGES>
__global__ void __launch_bounds__(tc::kMlThreads + 32, 2)
    moe_grouped_gemm_kernel(const MoeArgs a, const GroupedProj p) {
    constexpr int kThreads = tc::kMlThreads + 32, kDecodeWarps = tc::kMlThreads / 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int cap = a.grp_cap;
    const uint32_t b_chunk = 256u * static_cast<uint32_t>(cap);  // 2*cap rows x 128 B
    uint8_t* Abuf = smem;                                         // [STAGES][16 KB]
    uint8_t* Bbuf = smem + STAGES * 16384;                        // [STAGES][b_chunk]
    float* zs = reinterpret_cast<float*>(smem);                   // epilogue: [cap][128] f32 over A and B
    __shared__ tc::WsBars bars;
    __shared__ uint32_t tmem_base;
    __shared__ int slot_s[kGrpCapMax];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ob = blockIdx.x;
    const int item = blockIdx.y;

    pdl_wait();  // the B image (and the grouping) are complete
    pdl_trigger();
    // the item's descriptor is loaded together with the item count (entries
    // past the count are never used), so one round trip gives everything the
    // CTA needs to start its other loads
    int nitems;
    int4 desc;
    if (a.grp_items) {
        nitems = *a.grp_nitems;
        desc = a.grp_items[item];
    } else {  // dense linear: one expert, items of cap tokens in token order
        nitems = (a.T + cap - 1) / cap;
        desc = make_int4(0, min(cap, a.T - item * cap), 2 * item * cap, item * cap);
    }
    if (item >= nitems) return;
    const int e = desc.x, nt = desc.y;
    const uint2 rb = *reinterpret_cast<const uint2*>(p.rout + (long long)e * p.out + ob * 128 + 4 * lane);
    const int npad = (2 * nt + 15) & ~15;  // MMA N: hi/lo rows of nt tokens, multiple of 16
    const int nt4 = (nt + 3) & ~3;          // rows copied: whole 8-row atoms
    for (int i = tid; i < nt; i += kThreads) slot_s[i] = a.grp_perm ? a.grp_perm[desc.w + i] : desc.w + i;
    const uint32_t tcols = 2u * static_cast<uint32_t>(cap) < 32u ? 32u : 2u * static_cast<uint32_t>(cap);
    if (tid == 0) tc::ws_bars_init(bars);
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, tcols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = tc::idesc_f16(128, npad, true, false, false);

    const int KT = p.in >> 4, NT = p.out >> 4;
    const uint16_t* codes = p.codes + (long long)e * KT * NT * (16 * K);
    const int kb0 = blockIdx.z * p.kblk_per_split;                // first 64-input block of this K split
    const int nblk = min((p.in >> 6) - kb0, p.kblk_per_split);  // blocks of 64 inputs = 4 tile rows
    const int hr = warp >> 1, half = warp & 1;
    // two register sets by chunk parity: chunk b + 1's codes load into one
    // while chunk b is decoded from the other (no set is ever copied: a copy
    // would wait for the load). The lane's code pointer advances by one
    // 64-input block (4 tile rows) per chunk.
    HalfRowCodes<K> c0, c1;
    const long long blk_step = 4 * p.grid.s_kt * (16 * K);
    const uint16_t* cp = codes + ((long long)(4 * kb0 + hr) * p.grid.s_kt +
                                  (long long)(ob * 8 + 4 * half + (lane >> 3)) * p.grid.s_nt) * (16 * K) +
                         (lane & 7) * (2 * K);
    uint32_t soff[4];
    half_row_store_offsets(soff, lane, 4 * half);
    if (warp < kDecodeWarps) load_half_row_at<K>(c0, cp);
    const int nbr = (lane & ~7) | ((lane + 1) & 7);
    const uint8_t* img = a.grp_img + (long long)desc.z * 128 + (long long)kb0 * a.grp_img_rows * 128;

    const bool ok = tc::mma_mainloop_ws<STAGES, true>(
        Abuf, Bbuf, b_chunk, img, (long long)a.grp_img_rows * 128, 256u * static_cast<uint32_t>(nt4), nblk, tmem,
        idesc, bars, [&](int b, uint8_t* A) {
            const bool more = b + 1 < nblk;
            uint8_t* slice = A + hr * 4096;
            cp += blk_step;
            if ((b & 1) == 0) {
                if (more) load_half_row_at<K>(c1, cp);
                c0.p[K] = __shfl_sync(0xffffffffu, c0.p[0], nbr) & 0xFFFFu;
                decode_half_row_to_smem<K>(c0, slice, soff);
            } else {
                if (more) load_half_row_at<K>(c0, cp);
                c1.p[K] = __shfl_sync(0xffffffffu, c1.p[0], nbr) & 0xFFFFu;
                decode_half_row_to_smem<K>(c1, slice, soff);
            }
        });
    if (!ok && tid == 0) atomicExch(a.err, 3);

    // epilogue: TMEM lane m holds columns 2i (hi) and 2i + 1 (lo) of token i;
    // warps w and w + 4 share lane quarter w % 4 and split the columns
    if (ok && warp < kDecodeWarps) {
        const int q = warp & 3, m = 32 * q + lane;
        for (int c0c = 16 * (warp >> 2); c0c < npad; c0c += 32) {
            float v[16];
            tc::tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + c0c, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int qq = 0; qq < 8; ++qq) {
                const int i = c0c / 2 + qq;
                if (i < nt) zs[i * 128 + m] = v[2 * qq] + v[2 * qq + 1];
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, tcols);
    if (!ok) return;
    if (p.part) {  // K split: the partial sums go out, the reduction applies the output transform
        float* dst = p.part + ((long long)blockIdx.z * a.T * a.topk) * p.out + ob * 128 + 4 * lane;
        for (int i = warp; i < nt; i += kThreads / 32) {
            const float4 z4 = *reinterpret_cast<const float4*>(zs + i * 128 + 4 * lane);
            *reinterpret_cast<float4*>(dst + (long long)slot_s[i] * p.out) = z4;
        }
        return;
    }
    for (int i = warp; i < nt; i += kThreads / 32) {
        const float4 z4 = *reinterpret_cast<const float4*>(zs + i * 128 + 4 * lane);
        float v[4] = {z4.x * 256.f, z4.y * 256.f, z4.z * 256.f, z4.w * 256.f};  // undo the 2^-8 prescale (exact)
        output_transform_regs(v, rb, lane);
        if (p.bias) {  // additive output bias, after the output transform
            const float4 b4 = *reinterpret_cast<const float4*>(p.bias + ob * 128 + 4 * lane);
            v[0] += b4.x;
            v[1] += b4.y;
            v[2] += b4.z;
            v[3] += b4.w;
        }
        *reinterpret_cast<float4*>(p.y + (long long)slot_s[i] * p.out + ob * 128 + 4 * lane) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

// K-split reduction of a dense projection: one warp per (token, 128-output
// block) adds the splits' partial sums in split order, undoes the 2^-8
// prescale, applies the output transform and the bias.
__global__ void __launch_bounds__(256) dense_split_reduce_kernel(const GroupedProj p, int M, int splits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    const int nob = p.out >> 7;
    const long long task = (long long)blockIdx.x * 8 + warp;
    if (task >= (long long)M * nob) return;
    const int t = static_cast<int>(task / nob), ob = static_cast<int>(task % nob);
    const uint2 rb = *reinterpret_cast<const uint2*>(p.rout + ob * 128 + 4 * lane);
    const float* src = p.part + (long long)t * p.out + ob * 128 + 4 * lane;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int z = 0; z < splits; ++z) {
        const float4 z4 = *reinterpret_cast<const float4*>(src + (long long)z * M * p.out);
        v[0] += z4.x;
        v[1] += z4.y;
        v[2] += z4.z;
        v[3] += z4.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] *= 256.f;
    output_transform_regs(v, rb, lane);
    if (p.bias) {
        const float4 b4 = *reinterpret_cast<const float4*>(p.bias + ob * 128 + 4 * lane);
        v[0] += b4.x;
        v[1] += b4.y;
        v[2] += b4.z;
        v[3] += b4.w;
    }
    *reinterpret_cast<float4*>(p.y + (long long)t * p.out + ob * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
}

// ---------------------------------------------------------------------------
// 5. combine: out[t] = sum_j w[t][j] * d[t*k + j] + sigmoid(g . x[t]) * sh[t]
// ---------------------------------------------------------------------------
// One CTA per token. For hidden <= 2048 every load of a thread (its two
// float4 columns of the k down outputs and of the shared output, and its
// part of the gate's dot product) is issued before any arithmetic, so the
// CTA waits for memory once; larger hidden sizes loop.
constexpr int kCombineMaxK = 8;

__global__ void __launch_bounds__(256) moe_combine_kernel(const MoeArgs a, const float* d) {
    const int t = blockIdx.x;
    __shared__ float red[8];
    __shared__ float gate_s;
    pdl_wait();
    pdl_trigger();  // a dependent (the next residual norm) waits for this grid before reading
    const float* wt = a.w + (long long)t * a.topk;
    const uint16_t* xr = a.x + (long long)t * a.hidden;
    const bool two = a.hidden <= 2 * 4 * 256 && a.topk <= kCombineMaxK;
    float4 dv[2][kCombineMaxK], sv[2];
    float wj[kCombineMaxK];
    if (two) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = 4 * threadIdx.x + q * 4 * 256;
            if (i >= a.hidden) continue;
#pragma unroll
            for (int j = 0; j < kCombineMaxK; ++j)
                if (j < a.topk) dv[q][j] = *reinterpret_cast<const float4*>(d + ((long long)t * a.topk + j) * a.hidden + i);
            if (a.sh_inter > 0) sv[q] = *reinterpret_cast<const float4*>(a.sh + (long long)t * a.hidden + i);
        }
#pragma unroll
        for (int j = 0; j < kCombineMaxK; ++j)
            if (j < a.topk) wj[j] = wt[j];
    }
    float gate = 0.f;
    if (a.sh_inter > 0) {
        float acc = 0.f;
        for (int i = threadIdx.x; i < a.hidden; i += 256) acc = fmaf(h2f_bits(a.sh_gate[i]), h2f_bits(xr[i]), acc);
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
    if (two) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = 4 * threadIdx.x + q * 4 * 256;
            if (i >= a.hidden) continue;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kCombineMaxK; ++j) {
                if (j >= a.topk) break;
                acc.x = fmaf(wj[j], dv[q][j].x, acc.x);
                acc.y = fmaf(wj[j], dv[q][j].y, acc.y);
                acc.z = fmaf(wj[j], dv[q][j].z, acc.z);
                acc.w = fmaf(wj[j], dv[q][j].w, acc.w);
            }
            if (a.sh_inter > 0) {
                acc.x = fmaf(gate, sv[q].x, acc.x);
                acc.y = fmaf(gate, sv[q].y, acc.y);
                acc.z = fmaf(gate, sv[q].z, acc.z);
                acc.w = fmaf(gate, sv[q].w, acc.w);
            }
            *reinterpret_cast<float4*>(a.out + (long long)t * a.hidden + i) = acc;
        }
        return;
    }
    for (int i = 4 * threadIdx.x; i < a.hidden; i += 4 * 256) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.topk; ++j) {
            const float w = wt[j];
            const float4 v = *reinterpret_cast<const float4*>(d + ((long long)t * a.topk + j) * a.hidden + i);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        if (a.sh_inter > 0) {
            const float4 v = *reinterpret_cast<const float4*>(a.sh + (long long)t * a.hidden + i);
            acc.x = fmaf(gate, v.x, acc.x);
            acc.y = fmaf(gate, v.y, acc.y);
            acc.z = fmaf(gate, v.z, acc.z);
            acc.w = fmaf(gate, v.w, acc.w);
        }
        *reinterpret_cast<float4*>(a.out + (long long)t * a.hidden + i) = acc;
    }
}

// stages: 2 or 3 shared-memory stages (A and B). Fewer stages let more
// CTAs share an SM when items are small.
template <int K>
cudaError_t launch_grouped(const MoeArgs& a, const GroupedProj& p, int stages, cudaStream_t s) {
    const int smem = stages * (16384 + 256 * a.grp_cap) + 1024;
    const void* f = stages == 3 ? reinterpret_cast<const void*>(moe_grouped_gemm_kernel<K, 3>)
                                : reinterpret_cast<const void*>(moe_grouped_gemm_kernel<K, 2>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<MoeArgs*>(&a), const_cast<GroupedProj*>(&p)};
    const int splits = ((p.in >> 6) + p.kblk_per_split - 1) / p.kblk_per_split;
    return launch_kernel(f, dim3(p.out / 128, a.grp_max_items, splits), dim3(tc::kMlThreads + 32), smem, true, s,
                         args);
}

cudaError_t launch_prep(const MoeArgs& a, const GroupedProj& p, cudaStream_t s) {
    const long long tasks = (long long)a.T * a.topk * ((p.in / 128 + 3) / 4);
    void* args[] = {const_cast<MoeArgs*>(&a), const_cast<GroupedProj*>(&p)};
    return launch_kernel(reinterpret_cast<const void*>(moe_prep_kernel), dim3(static_cast<unsigned>((tasks + 7) / 8)),
                         dim3(256), 0, true, s, args);
}

}  // namespace

cudaError_t launch_kernel(const void* f, dim3 grid, dim3 block, int smem, bool pdl, cudaStream_t s, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, f, args);
}

GroupPlan group_plan(int T, int topk, int E, int hidden, int inter, int sh_inter) {
    GroupPlan g{};
    const long long S = (long long)T * topk;
    const long long want = 2 * S / E + 8;  // twice the mean run per expert, plus slack
    g.cap = 16;
    while (g.cap < kGrpCapMax && g.cap < want) g.cap *= 2;
    g.max_items = static_cast<int>(S / g.cap) + E;  // full items plus at most one partial per expert
    g.pos_cap = static_cast<int>((S + 3 * E + 3) & ~3ll);
    // items[max_items] (16 B each), counts[E], offsets[E+1], poff[E], nitems, perm[S], ppos[S]
    g.int_bytes = (size_t)g.max_items * 16 + (size_t)(E + (E + 1) + E + 1 + 2 * S) * 4;
    const size_t trellis_img = (size_t)(hidden > inter ? hidden : inter) * 2 * g.pos_cap * 2;
    size_t shared_img = 0;
    if (sh_inter > 0) {
        const size_t gu = int8_gemm_ws_bytes(2 * sh_inter, hidden, T), dn = int8_gemm_ws_bytes(hidden, sh_inter, T);
        shared_img = gu > dn ? gu : dn;
    }
    g.img_bytes = trellis_img;
    g.shared_img_bytes = shared_img;
    return g;
}

cudaError_t launch_moe_topk_group(const MoeArgs& a, cudaStream_t s) {
    void* args[] = {const_cast<MoeArgs*>(&a)};
    cudaError_t e = launch_kernel(reinterpret_cast<const void*>(moe_topk_kernel), dim3((a.T + 7) / 8), dim3(256), 0,
                                  true, s, args);
    if (e != cudaSuccess) return e;
    return launch_kernel(reinterpret_cast<const void*>(moe_group_kernel), dim3(1), dim3(1024), 0, true, s, args);
}

cudaError_t launch_moe_grouped(const MoeArgs& a, float* d, int num_sms, cudaStream_t s) {
    (void)num_sms;
    cudaError_t e = launch_moe_topk_group(a, s);
    if (e != cudaSuccess) return e;
    const GroupedProj gu{a.gu_codes, a.gu_rin, a.gu_rout, a.hidden, 2 * a.inter, 0, a.ygu,
                         tile_strides(a.hidden, 2 * a.inter, false), nullptr, nullptr, a.hidden >> 6, nullptr};
    if ((e = launch_prep(a, gu, s)) != cudaSuccess) return e;
    // MoE items: two stages, so that items of up to 32 tokens run 4 CTAs per
    // SM (3 with three stages; measured on GB300 for the 35B layer: 17 / 64 /
    // 256 tokens 165.7 / 290.4 / 346.2 -> 161.6 / 279.1 / 333.3 us per block;
    // 2048 tokens, items of 128 with two stages already, unchanged)
    e = a.gu_K == 2 ? launch_grouped<2>(a, gu, 2, s) : launch_grouped<3>(a, gu, 2, s);
    if (e != cudaSuccess) return e;
    const GroupedProj dn{a.dn_codes, a.dn_rin, a.dn_rout, a.inter, a.hidden, 1, d,
                         tile_strides(a.inter, a.hidden, false), nullptr, nullptr, a.inter >> 6, nullptr};
    if ((e = launch_prep(a, dn, s)) != cudaSuccess) return e;
    return a.dn_K == 2 ? launch_grouped<2>(a, dn, 2, s) : launch_grouped<3>(a, dn, 2, s);
}

cudaError_t launch_dense_grouped(const DenseArgs& d, cudaStream_t s) {
    MoeArgs a{};
    a.T = d.M;
    a.topk = 1;
    a.E = 1;
    a.hidden = d.in;
    a.x = static_cast<const uint16_t*>(d.x_f32 ? nullptr : d.x);
    a.grp_cap = d.cap;
    a.grp_img = d.img;
    a.grp_img_rows = d.img_rows;
    a.err = d.err;
    const int nblk = d.in >> 6;
    const int bps = (nblk + d.splits - 1) / d.splits;
    const int splits = (nblk + bps - 1) / bps;  // every split starts inside K
    const GroupedProj p{d.codes, d.rin, d.rout, d.in, d.out, d.x_f32 ? 2 : 0, d.y,
                        tile_strides(d.in, d.out, d.nt_major != 0), d.bias,
                        static_cast<const float*>(d.x_f32 ? d.x : nullptr), bps, splits > 1 ? d.part : nullptr};
    cudaError_t e = launch_prep(a, p, s);
    if (e != cudaSuccess) return e;
    a.grp_max_items = (d.M + d.cap - 1) / d.cap;
    // dense items: three stages up to 32 tokens, two from 64 (measured on
    // GB300: 64 tokens 5120 -> 17408 57.8 -> 49.6 us, 17408 -> 5120 72.6 ->
    // 69.8 us; with two stages 8-32 tokens were 1-4% slower)
    const int stages = d.cap <= 32 ? 3 : 2;
    e = d.K == 2 ? launch_grouped<2>(a, p, stages, s) : launch_grouped<3>(a, p, stages, s);
    if (e != cudaSuccess || splits == 1) return e;
    int M = d.M, sp = splits;
    void* rargs[] = {const_cast<GroupedProj*>(&p), &M, &sp};
    const long long tasks = (long long)d.M * (d.out >> 7);
    return launch_kernel(reinterpret_cast<const void*>(dense_split_reduce_kernel),
                         dim3(static_cast<unsigned>((tasks + 7) / 8)), dim3(256), 0, true, s, rargs);
}

int dense_ksplit(int in, int out, int M, int cap) {
    const long long base = (long long)(out >> 7) * ((M + cap - 1) / cap);  // CTAs without a split
    const int nblk = in >> 6;
    long long ks = (2 * 152 + base - 1) / base;  // about one wave of two CTAs per SM
    if (ks > nblk / 4) ks = nblk / 4;            // at least 4 blocks of 64 inputs per split
    if (ks > 16) ks = 16;
    return ks < 1 ? 1 : static_cast<int>(ks);
}

cudaError_t launch_moe_combine(const MoeArgs& a, const float* d, cudaStream_t s) {
    void* args[] = {const_cast<MoeArgs*>(&a), const_cast<float**>(&d)};
    return launch_kernel(reinterpret_cast<const void*>(moe_combine_kernel), dim3(a.T),
                         dim3(256), 0, true, s, args);
}

}  // namespace escha
