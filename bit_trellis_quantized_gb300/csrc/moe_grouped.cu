// Batched / prefill MoE block: tokens grouped by expert, each expert's packed
// trellis codes decoded once per group of up to kGrpTok tokens and fed to the
// 5th-generation tensor cores (tcgen05) as a dense contraction (hipfire PR
// #694, commits on the grouped prefill GEMM: decode each expert's weights once
// and share them across its tokens instead of re-reading them per slot).
//
// Kernels, after the router-logits kernel shared with the batch-1 path:
//  1. top-k: one warp per token (ids ordered by (logit desc, id asc), softmax
//     over the k selected logits).
//  2. grouping: one CTA; stable counting sort of the (token, slot) pairs by
//     expert -> counts, offsets, perm, and a list of work items
//     (expert, first group position) of at most kGrpTok tokens each.
//  3. grouped GEMM (gate_up, then down): one CTA per (work item, 128-wide
//     output block). Per 128-input block: the 8 warps decode one tile row
//     each into an MN-major A operand in shared memory; the input transform
//     H128(rin * input) of the item's tokens, prescaled by 2^-8 and split into
//     fp16 hi + lo parts, fills the K-major B operand (rows 2i and 2i+1 for
//     token i); one thread issues the tcgen05 MMAs (M = 128 outputs, N = 2 x
//     tokens, K = 16 per instruction) into a TMEM accumulator, double-buffered
//     against the next block's decode. The epilogue adds the hi and lo
//     columns, applies the output Hadamard, 2^-7 * 2^8 and rout.
//  4. combine: out[t] = sum_j w[t][j] * down(slot t*k + j) + sigmoid(g . x[t])
//     * shared(x[t]) in slot order; the shared expert runs on the int8 GEMV.
#include "kernels.h"
#include "tcgen05.cuh"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kGrpThreads = 256;
constexpr int kGrpWarps = kGrpThreads / 32;
constexpr int kARowBytes = 4096;                  // one tile row: M = 128 outputs x K = 16 inputs, fp16
constexpr int kABufBytes = 8 * kARowBytes;        // one 128-input block
constexpr int kBRows = 2 * kGrpTok;               // hi and lo row per token
constexpr int kBChunkBytes = kBRows * 128;        // 64 inputs of every B row
constexpr int kBBufBytes = 2 * kBChunkBytes;      // one 128-input block
constexpr int kSmemOperands = 2 * kABufBytes + 2 * kBBufBytes;
constexpr float kPrescale = 0.00390625f;          // 2^-8: B operand range guard, undone in the epilogue

// ---------------------------------------------------------------------------
// 1. top-k
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_topk_kernel(const MoeArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    pdl_wait();
    if (t >= a.T) return;
    int e;
    float w;
    topk_softmax_warp(a.logits + (long long)t * a.E, a.E, a.topk, lane, &e, &w);
    if (lane < a.topk) {
        a.ids[(long long)t * a.topk + lane] = e;
        a.w[(long long)t * a.topk + lane] = w;
    }
}

// ---------------------------------------------------------------------------
// 2. grouping (one CTA of 1024 threads)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024, 1) moe_group_kernel(const MoeArgs a) {
    __shared__ int cnt[256];
    __shared__ int base[256];
    __shared__ int wcnt[32][256];  // per-warp counts of one 1024-slot chunk, then per-warp bases
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.T * a.topk;
    pdl_wait();
    for (int e = tid; e < 256; e += 1024) cnt[e] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += 1024) atomicAdd(&cnt[a.ids[s]], 1);
    __syncthreads();
    if (tid == 0) {  // exclusive scan, work items
        int off = 0, items = 0;
        for (int e = 0; e < a.E; ++e) {
            a.grp_counts[e] = cnt[e];
            a.grp_offsets[e] = off;
            base[e] = off;
            for (int g0 = 0; g0 < cnt[e]; g0 += kGrpTok) {
                a.grp_items[items] = (e << 16) | g0;
                ++items;
            }
            off += cnt[e];
        }
        a.grp_offsets[a.E] = off;
        *a.grp_nitems = items;
    }
    __syncthreads();
    // stable scatter, 1024 slots at a time in slot order
    const unsigned lt = (1u << lane) - 1u;
    for (int s0 = 0; s0 < S; s0 += 1024) {
        const int s = s0 + tid;
        const bool valid = s < S;
        const int e = valid ? a.ids[s] : 256 + lane;  // invalid lanes never match a real expert
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(m & lt);
        for (int i = tid; i < 32 * 256; i += 1024) (&wcnt[0][0])[i] = 0;
        __syncthreads();
        if (valid && rank == 0) wcnt[warp][e] = __popc(m);
        __syncthreads();
        for (int ee = tid; ee < 256; ee += 1024) {  // per-warp exclusive bases for expert ee
            int run = base[ee];
            for (int w = 0; w < 32; ++w) {
                const int c = wcnt[w][ee];
                wcnt[w][ee] = run;
                run += c;
            }
            base[ee] = run;
        }
        __syncthreads();
        if (valid) a.grp_perm[wcnt[warp][e] + rank] = s;
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// 3. grouped GEMM
// ---------------------------------------------------------------------------
struct GroupedProj {
    const uint16_t* codes;  // [E][in/16][out/16][16K]
    const uint16_t* rin;    // [E][in]
    const uint16_t* rout;   // [E][out]
    int in, out;
    int mode;               // 0: input = x[token] (fp16); 1: input = SwiGLU(ygu[slot])
    float* y;               // [slots][out]
};

// The lane's 64 decoded weights of one tile row (tile lane/4, input rows
// 4c..4c+3, 16 output columns each) written into the MN-major A slice of that
// row: element (m = 16*(lane/4) + q, k = r) at mnmajor_off(m, k, 2048, 1024).
template <int K>
__device__ __forceinline__ void decode_row_to_smem(const LaneCodes<K>& lc, uint8_t* slice, int lane) {
    const int tile = lane >> 2, c = lane & 3;
    const uint32_t m0 = 16u * tile;
    static_for<8>([&](auto J) {  // half-row j: input row 4c + j/2, columns 8*(j%2)..+7
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
        const uint32_t k = 4u * c + (j >> 1);
        const uint32_t m = m0 + 8u * (j & 1);
        *reinterpret_cast<uint4*>(slice + tc::mnmajor_off(m, k, 2048u, 1024u)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
    });
}

template <int K>
__global__ void __launch_bounds__(kGrpThreads, 1) moe_grouped_gemm_kernel(const MoeArgs a, const GroupedProj p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* Abuf = smem;                       // [2][8 rows][4 KB]
    uint8_t* Bbuf = smem + 2 * kABufBytes;      // [2][2 chunks][kBRows x 128 B]
    float* zs = reinterpret_cast<float*>(smem); // epilogue: [kGrpTok][128] f32, reuses the A buffers
    __shared__ __align__(8) unsigned long long mma_done[2];
    __shared__ uint32_t tmem_base;
    __shared__ int slot_s[kGrpTok];
    __shared__ int row_s[kGrpTok];  // x row (token) for mode 0, slot for mode 1
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ob = blockIdx.x;
    const int item = blockIdx.y;

    pdl_wait();  // grouping (and for down, the gate_up outputs) complete
    pdl_trigger();
    if (item >= *a.grp_nitems) return;
    const int packed = a.grp_items[item];
    const int e = packed >> 16, g0 = packed & 0xFFFF;
    const int nt = min(kGrpTok, a.grp_counts[e] - g0);
    const int npad = (2 * nt + 15) & ~15;  // MMA N: hi/lo rows of nt tokens, multiple of 16
    for (int i = tid; i < kGrpTok; i += kGrpThreads) {
        const int s = i < nt ? a.grp_perm[a.grp_offsets[e] + g0 + i] : 0;
        slot_s[i] = s;
        row_s[i] = p.mode == 0 ? s / a.topk : s;
    }
    if (tid == 0) {
        tc::mbar_init_cta(tc::smem_addr(&mma_done[0]), 1);
        tc::mbar_init_cta(tc::smem_addr(&mma_done[1]), 1);
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 128);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = tc::idesc_f16(128, npad, true, false, false);

    const int KT = p.in >> 4, NT = p.out >> 4;
    const uint16_t* codes = p.codes + (long long)e * KT * NT * (16 * K);
    const uint16_t* rin = p.rin + (long long)e * p.in;
    const int nblk = p.in / 128;
    bool ok = true;
    LaneCodes<K> cur;
    load_lane_codes<K>(cur, codes + ((long long)warp * NT + ob * 8) * (16 * K), lane);
    const int nbr = (lane & ~3) | ((lane + 1) & 3);

    for (int b = 0; b < nblk; ++b) {
        const int buf = b & 1;
        uint8_t* A = Abuf + buf * kABufBytes;
        uint8_t* B = Bbuf + buf * kBBufBytes;
        if (b >= 2) {  // the MMAs of block b-2 have finished reading this buffer
            if (!tc::mbar_wait_parity_bounded(tc::smem_addr(&mma_done[buf]), ((b >> 1) - 1) & 1)) ok = false;
        }
        // prefetch the next block's row while this one is decoded
        LaneCodes<K> nxt;
        const bool more = b + 1 < nblk;
        if (more) load_lane_codes<K>(nxt, codes + ((long long)(8 * (b + 1) + warp) * NT + ob * 8) * (16 * K), lane);
        // B: x~ for every token of the item, hi/lo, this block's 128 inputs
        for (int i = warp; i < nt; i += kGrpWarps) {
            const int ib = b * 128 + 4 * lane;
            float v[4];
            const uint2 rb = *reinterpret_cast<const uint2*>(rin + ib);
            if (p.mode == 0) {
                const uint2 xb = *reinterpret_cast<const uint2*>(a.x + (long long)row_s[i] * a.hidden + ib);
                v[0] = h2f_bits(static_cast<uint16_t>(xb.x & 0xFFFFu));
                v[1] = h2f_bits(static_cast<uint16_t>(xb.x >> 16));
                v[2] = h2f_bits(static_cast<uint16_t>(xb.y & 0xFFFFu));
                v[3] = h2f_bits(static_cast<uint16_t>(xb.y >> 16));
            } else {
                const float* yr = a.ygu + (long long)row_s[i] * 2 * a.inter;
                const float4 g = *reinterpret_cast<const float4*>(yr + ib);
                const float4 u = *reinterpret_cast<const float4*>(yr + a.inter + ib);
                v[0] = silu_f(g.x) * u.x;
                v[1] = silu_f(g.y) * u.y;
                v[2] = silu_f(g.z) * u.z;
                v[3] = silu_f(g.w) * u.w;
            }
            v[0] *= h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu));
            v[1] *= h2f_bits(static_cast<uint16_t>(rb.x >> 16));
            v[2] *= h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu));
            v[3] *= h2f_bits(static_cast<uint16_t>(rb.y >> 16));
            h128_warp(v, lane);
            __half hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float sv = v[q] * kPrescale;
                hi[q] = __float2half_rn(sv);
                lo[q] = __float2half_rn(sv - __half2float(hi[q]));
            }
            // K index inside the block: 4*lane .. 4*lane + 3 -> chunk (4*lane)/64
            const int kk = 4 * lane;
            uint8_t* chunk = B + (kk >> 6) * kBChunkBytes;
            const uint32_t k_in = static_cast<uint32_t>(kk & 63);
            const uint2 hv = make_uint2(static_cast<uint32_t>(__half_as_ushort(hi[0])) | (static_cast<uint32_t>(__half_as_ushort(hi[1])) << 16),
                                        static_cast<uint32_t>(__half_as_ushort(hi[2])) | (static_cast<uint32_t>(__half_as_ushort(hi[3])) << 16));
            const uint2 lv = make_uint2(static_cast<uint32_t>(__half_as_ushort(lo[0])) | (static_cast<uint32_t>(__half_as_ushort(lo[1])) << 16),
                                        static_cast<uint32_t>(__half_as_ushort(lo[2])) | (static_cast<uint32_t>(__half_as_ushort(lo[3])) << 16));
            *reinterpret_cast<uint2*>(chunk + tc::kmajor_off(2u * i, k_in)) = hv;
            *reinterpret_cast<uint2*>(chunk + tc::kmajor_off(2u * i + 1u, k_in)) = lv;
        }
        // A: warp w decodes tile row 8b + w of output block ob
        cur.p[2 * K] = __shfl_sync(0xffffffffu, cur.p[0], nbr) & 0xFFFFu;
        decode_row_to_smem<K>(cur, A + warp * kARowBytes, lane);
        if (more) cur = nxt;
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad =
                    tc::smem_desc(tc::smem_addr(A + kk * kARowBytes), 2048u, 1024u, tc::kSwizzle128B);
                const uint64_t bd = tc::smem_desc(tc::smem_addr(B + (kk >> 2) * kBChunkBytes) + (kk & 3) * 32u, 16u,
                                                  1024u, tc::kSwizzle128B);
                tc::mma_f16(tmem, ad, bd, idesc, b > 0 || kk > 0);
            }
            tc::commit(tc::smem_addr(&mma_done[buf]));
        }
    }
    // the last commit covers every MMA issued before it
    const int last = nblk - 1;
    if (!tc::mbar_wait_parity_bounded(tc::smem_addr(&mma_done[last & 1]), (last >> 1) & 1)) ok = false;
    if (nblk >= 2) {  // and the other buffer's final phase has completed as well
        const int prev = nblk - 2;
        if (!tc::mbar_wait_parity_bounded(tc::smem_addr(&mma_done[prev & 1]), (prev >> 1) & 1)) ok = false;
    }
    tc::fence_after_sync();
    if (!ok && tid == 0) atomicExch(a.err, 3);

    // epilogue: TMEM lane m holds columns 2i (hi) and 2i + 1 (lo) of token i
    __syncthreads();  // every warp is done with the A buffers before zs overwrites them
    if (warp < 4 && ok) {
        const int m = 32 * warp + lane;
        for (int c0 = 0; c0 < npad; c0 += 16) {
            float v[16];
            tc::tmem_ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = c0 / 2 + q;
                if (i < nt) zs[i * 128 + m] = v[2 * q] + v[2 * q + 1];
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
    if (!ok) return;
    const uint16_t* rout = p.rout + (long long)e * p.out + ob * 128;
    const uint2 rb = *reinterpret_cast<const uint2*>(rout + 4 * lane);
    for (int i = warp; i < nt; i += kGrpWarps) {
        const float4 z4 = *reinterpret_cast<const float4*>(zs + i * 128 + 4 * lane);
        float v[4] = {z4.x * 256.f, z4.y * 256.f, z4.z * 256.f, z4.w * 256.f};  // undo the 2^-8 prescale (exact)
        output_transform_regs(v, rb, lane);
        *reinterpret_cast<float4*>(p.y + (long long)slot_s[i] * p.out + ob * 128 + 4 * lane) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

// ---------------------------------------------------------------------------
// 4. combine: out[t] = sum_j w[t][j] * d[t*k + j] + sigmoid(g . x[t]) * sh[t]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_combine_kernel(const MoeArgs a, const float* d) {
    const int t = blockIdx.y;
    __shared__ float red[8];
    __shared__ float gate_s;
    pdl_wait();
    float gate = 0.f;
    if (a.sh_inter > 0) {
        const uint16_t* xr = a.x + (long long)t * a.hidden;
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
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= a.hidden) return;
    float acc = 0.f;
    for (int j = 0; j < a.topk; ++j)
        acc = fmaf(a.w[(long long)t * a.topk + j], d[((long long)t * a.topk + j) * a.hidden + i], acc);
    if (a.sh_inter > 0) acc = fmaf(gate, a.sh[(long long)t * a.hidden + i], acc);
    a.out[(long long)t * a.hidden + i] = acc;
}

cudaError_t launch_plain(const void* f, dim3 grid, dim3 block, int smem, bool pdl, cudaStream_t s, void** args) {
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

template <int K>
cudaError_t launch_grouped(const MoeArgs& a, const GroupedProj& p, cudaStream_t s) {
    const int smem = kSmemOperands + 1024;
    const void* f = reinterpret_cast<const void*>(moe_grouped_gemm_kernel<K>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // at most one partial chunk per expert on top of the full ones
    const int max_items = (a.T * a.topk) / kGrpTok + a.E;
    void* args[] = {const_cast<MoeArgs*>(&a), const_cast<GroupedProj*>(&p)};
    return launch_plain(f, dim3(p.out / 128, max_items), dim3(kGrpThreads), smem, true, s, args);
}

}  // namespace

size_t grouped_extra_bytes(int T, int topk, int E) {
    // counts[E], offsets[E+1], items[T*topk/kGrpTok + E], nitems, perm[T*topk]
    return (size_t)(E + (E + 1) + (T * topk) / kGrpTok + E + 1 + T * topk) * 4;
}

cudaError_t launch_moe_grouped(const MoeArgs& a, float* d, int num_sms, cudaStream_t s) {
    (void)num_sms;
    void* args[] = {const_cast<MoeArgs*>(&a)};
    cudaError_t e = launch_plain(reinterpret_cast<const void*>(moe_topk_kernel), dim3((a.T + 7) / 8), dim3(256), 0,
                                 true, s, args);
    if (e != cudaSuccess) return e;
    e = launch_plain(reinterpret_cast<const void*>(moe_group_kernel), dim3(1), dim3(1024), 0, true, s, args);
    if (e != cudaSuccess) return e;
    GroupedProj gu{a.gu_codes, a.gu_rin, a.gu_rout, a.hidden, 2 * a.inter, 0, a.ygu};
    e = a.gu_K == 2 ? launch_grouped<2>(a, gu, s) : launch_grouped<3>(a, gu, s);
    if (e != cudaSuccess) return e;
    GroupedProj dn{a.dn_codes, a.dn_rin, a.dn_rout, a.inter, a.hidden, 1, d};
    e = a.dn_K == 2 ? launch_grouped<2>(a, dn, s) : launch_grouped<3>(a, dn, s);
    return e;
}

cudaError_t launch_moe_combine(const MoeArgs& a, const float* d, cudaStream_t s) {
    void* args[] = {const_cast<MoeArgs*>(&a), const_cast<float**>(&d)};
    return launch_plain(reinterpret_cast<const void*>(moe_combine_kernel), dim3((a.hidden + 255) / 256, a.T),
                        dim3(256), 0, false, s, args);
}

}  // namespace escha
