// A sequence of one-token MoE blocks in ONE cooperative launch.
//
// A decode step runs its MoE blocks one after the other, one token each. Run
// as separate launches, every block pays its grid boundaries (the router
// grid before gate_up, gate_up before down, the block before the next); at
// one token those waits, not the decode, are most of the time. Here all
// blocks of the sequence are one grid of resident CTAs (a cooperative
// launch) that take work units from one queue, in queue order:
//
//   R  router: 8 experts' logits (one warp each); in a residual stack the
//      unit first computes x = RMSNorm(h + previous output) itself
//   S  the int8 shared expert's gate_up: 2 rows per warp, and its gate
//   G  gate_up: one (slot, 128-wide output block, input split)
//   X  the shared expert's down rows (up to 3 per warp)
//   F  one slot's gate_up outputs: the G units' split partial sums added,
//      then the output transform
//   D  down: one (slot, output block, input split)
//   C  combine: one output block; finishes every expert's down outputs of
//      the block and adds them and the shared expert (hipfire PR #694,
//      commit "Executed the moeblk golden against real shipped layer-0
//      weights": the weighted sum of the routed experts' gate_up -> SwiGLU
//      -> down plus the sigmoid-gated shared expert).
// G and D units only publish their partial sums (a release add on a
// counter, with no answer to wait for); F and C add them.
//
// A unit waits (bounded) only for units earlier in the queue: G, F, D and C
// for their block's routing (the block's last R unit computes the top-k and
// publishes it), F for its slot's G units, D for its slot's F unit, X for
// its block's shared gate_up rows, C for its output block's D units and for
// X, and, in a stack, R for the previous block's output.
// Work is taken in queue order, so the earliest unfinished unit is always
// being run by some CTA: no deadlock while all CTAs are resident, which the
// cooperative launch guarantees. A residual stack is queued block after
// block (R S G X F D C). Independent blocks (each its own input) are queued
// as a software pipeline of depth 2: R S of blocks 0..2, G X of blocks 0 and
// 1, F of block 0, then per step b: R S of block b + 3, G X of block b + 2,
// F of block b + 1, D of block b, C of block b - 1. A unit is taken long
// after the units it waits for, so few CTAs sit idle waiting, and the
// blocks' routers, gate_ups and downs overlap.
//
// Each unit's arithmetic, the input splits and every summation order are
// those of the per-slot kernels at one token (slot_plan), so every block's
// outputs are bit for bit those of escha_moe_block / escha_moe_block_resid.
// Every wait gives up after wait_ns, sets the workspace status word and
// skips the unit's work, so the kernel always ends.
#include <atomic>
#include <mutex>

#include "coop.cuh"
#include "kernels.h"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kMbThreads = 256;
constexpr int kMbWarps = kMbThreads / 32;
constexpr int kMbMaxHidden = 2048;
constexpr int kMbMaxShInter = 512;
constexpr int kMbMaxOb = 32;

// Counter words of one block (unsigned, offsets in words).
constexpr int kMcLogit = 0;                    // R units done
constexpr int kMcShGu = 1;                     // S units done
constexpr int kMcShDn = 2;                     // X units done
constexpr int kMcDone = 3;                     // output blocks finished
constexpr int kMcGu = 4;                       // [8] gate_up partial sums arrived per slot
constexpr int kMcGuJ = kMcGu + 8;              // [8] the slot's gate_up outputs finished (F unit)
constexpr int kMcCmb = kMcGuJ + 8;             // [kMbMaxOb] down partial sums arrived per output block
// [8] 64-bit words, one per slot: routing weight bits << 32 | (expert + 1),
// published by the block's last R unit (0 until then)
constexpr int kMcRoute = kMcCmb + kMbMaxOb;
constexpr int kMcWords = kMcRoute + 16;
static_assert(kMcRoute % 2 == 0 && kMbCtrWords % 2 == 0, "64-bit routing words");
static_assert(kMcWords <= kMbCtrWords, "counter block");

constexpr int kErrLogit = 8, kErrShGu = 9, kErrGuJ = 10, kErrShDn = 11, kErrPrev = 12, kErrNotCoop = 13,
              kErrCmb = 14, kErrGu = 15;

// The block's routing (experts and weights of its slots, published by its
// last R unit) into the CTA's cache: thread j < topk reads slot j's word,
// which carries the expert, its weight and the publication at once.
__device__ __forceinline__ bool mb_routing(const MbHead& m, int b, int* tk_block, int* e_s, float* w_s) {
    if (*tk_block == b) return true;
    int ok = 1;
    if (threadIdx.x < m.topk) {
        const unsigned long long* rt =
            reinterpret_cast<const unsigned long long*>(m.ctr + (long long)b * kMbCtrWords + kMcRoute) + threadIdx.x;
        unsigned long long v = ld_acquire_u64(rt);
        if (static_cast<unsigned>(v) == 0u) {
            const unsigned long long t0 = global_ns();
            for (;;) {
                __nanosleep(200);
                v = ld_acquire_u64(rt);
                if (static_cast<unsigned>(v) != 0u) break;
                if (static_cast<long long>(global_ns() - t0) > m.wait_ns) {
                    atomicCAS(m.err, 0, kErrLogit);
                    ok = 0;
                    break;
                }
            }
        }
        e_s[threadIdx.x] = static_cast<int>(static_cast<unsigned>(v)) - 1;
        w_s[threadIdx.x] = __uint_as_float(static_cast<unsigned>(v >> 32));
    }
    if (!__syncthreads_and(ok)) return false;
    if (threadIdx.x == 0) *tk_block = b;
    return true;
}

// Residual norm of one token by one CTA of 256 threads, in the arithmetic of
// residual_rmsnorm_kernel (thread t sums v_i^2 over i = t, t + 256, ...; xor
// butterfly in each warp; the 8 warp sums in order): xh = f16_rne(v * inv),
// v = h + add. Ends with the CTA synchronised.
__device__ __forceinline__ void mb_norm(const MbHead& m, const float* add, uint16_t* xh) {
    __shared__ float wsum[kMbWarps];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    constexpr int J = kMbMaxHidden / kMbThreads;
    float v[J];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int i = j * kMbThreads + t;
        v[j] = 0.f;
        if (i < m.hidden) {
            float hv = __ldcg(m.res + i);
            if (add) hv = __fadd_rn(hv, __ldcg(add + i));
            v[j] = hv;
            s = __fadd_rn(__fmul_rn(hv, hv), s);
        }
    }
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, k));
    if (lane == 0) wsum[warp] = s;
    __syncthreads();
    float tot = wsum[0];
#pragma unroll
    for (int w = 1; w < kMbWarps; ++w) tot = __fadd_rn(tot, wsum[w]);
    const float mean = __fdiv_rn(tot, static_cast<float>(m.hidden));
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, m.eps)));
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int i = j * kMbThreads + t;
        if (i < m.hidden) xh[i] = __half_as_ushort(__float2half_rn(__fmul_rn(v[j], inv)));
    }
    __syncthreads();
}

// The token's input x (fp16 bits) of block b.
__device__ __forceinline__ const uint16_t* mb_x(const MbHead& m, const MbBlock& B) { return m.stack ? m.xbuf : B.x; }
static_assert(sizeof(MbBlock) % 8 == 0, "descriptor copied in 8-byte words");

// R unit r of block b: logits of experts 8 r .. 8 r + 7 (the per-slot
// router's order: lane l adds the products of columns 256 p + 8 l .. + 7 for
// p = 0, 1, ... in order, then the xor butterfly, then f16 rounding).
__device__ __forceinline__ void mb_router(const MbHead& m, const MbBlock& B, int b, int r, float* sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = r * kMbWarps + warp;
    const int passes = m.hidden >> 8;
    uint4 wv[kMbMaxHidden / 256];
    const uint16_t* wrow = B.router_w + (long long)(e < m.E ? e : 0) * m.hidden;
#pragma unroll
    for (int q = 0; q < kMbMaxHidden / 256; ++q)
        if (q < passes) wv[q] = ldg_stream_v4(wrow + q * 256 + lane * 8);
    unsigned* ctr = m.ctr + (long long)b * kMbCtrWords;
    const uint16_t* x;
    uint16_t* xh = reinterpret_cast<uint16_t*>(sm);
    if (m.stack) {
        if (b > 0) {  // the previous block's output is complete (and h holds its input's residual)
            const unsigned* pc = m.ctr + (long long)(b - 1) * kMbCtrWords;
            if (!cta_wait_geq(pc + kMcDone, static_cast<unsigned>(m.hidden / 128), m.wait_ns, m.err, kErrPrev)) return;
        }
        mb_norm(m, b > 0 ? m.outbuf : nullptr, xh);
        if (r == 0)
            for (int i = threadIdx.x; i < m.hidden / 8; i += kMbThreads)
                __stcg(reinterpret_cast<uint4*>(m.xbuf) + i, reinterpret_cast<const uint4*>(xh)[i]);
        x = xh;
    } else {
        x = B.x;
    }
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kMbMaxHidden / 256; ++q) {
        if (q < passes) {
            const int i = q * 256 + lane * 8;
            const uint4 xv = m.stack ? *reinterpret_cast<const uint4*>(x + i) : __ldg(reinterpret_cast<const uint4*>(x + i));
            dot8_f16(xv, wv[q], acc);
        }
    }
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, k);
    if (lane == 0 && e < m.E) __stcg(m.logits + (long long)b * m.E + e, __half_as_ushort(__float2half_rn(acc)));
    __syncthreads();
    __shared__ int last_s;
    if (threadIdx.x == 0) last_s = atom_add_acq_rel(ctr + kMcLogit, 1u) == static_cast<unsigned>(m.nR - 1);
    __syncthreads();
    if (!last_s || warp != 0) return;
    // the block's last R unit: the top-k once, published for every G and D unit
    const uint16_t* lg = m.logits + (long long)b * m.E;
    uint16_t bits[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) bits[i] = lane + 32 * i < m.E ? __ldcg(lg + lane + 32 * i) : 0;
    int e_l;
    float w_l;
    topk_softmax_warp_bits(bits, m.E, m.topk, lane, &e_l, &w_l);
    if (lane < m.topk) {
        __stcg(B.ids + lane, e_l);
        __stcg(B.w + lane, w_l);
        st_release_u64(reinterpret_cast<unsigned long long*>(ctr + kMcRoute) + lane,
                       (static_cast<unsigned long long>(__float_as_uint(w_l)) << 32) | static_cast<unsigned>(e_l + 1));
    }
}

// S unit s of block b: shared gate_up rows 16 s .. 16 s + 15 (2 per warp) and,
// in unit 0, the gate (warp 7); the per-slot router's orders.
__device__ __forceinline__ void mb_shared_gate_up(const MbHead& m, const MbBlock& B, int b, int s, float* xs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = 2 * m.sh_inter;
    const int r0 = (s * kMbWarps + warp) * 2;
    const int nrows = min(2, rows - r0);
    for (long long off = lane * 128LL; off < (long long)max(nrows, 0) * m.hidden; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(B.sh_gu_w8 + (long long)r0 * m.hidden + off));
    unsigned* ctr = m.ctr + (long long)b * kMbCtrWords;
    // in a stack, x is written by the block's first R unit
    if (m.stack && !cta_wait_geq(ctr + kMcLogit, static_cast<unsigned>(m.nR), m.wait_ns, m.err, kErrLogit)) return;
    const uint16_t* x = mb_x(m, B);
    for (int i = threadIdx.x * 8; i < m.hidden; i += kMbThreads * 8) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(x + i));
        *reinterpret_cast<float4*>(xs + xs_swz(i)) =
            make_float4(h2f_bits(v.x & 0xFFFFu), h2f_bits(v.x >> 16), h2f_bits(v.y & 0xFFFFu), h2f_bits(v.y >> 16));
        *reinterpret_cast<float4*>(xs + xs_swz(i + 4)) =
            make_float4(h2f_bits(v.z & 0xFFFFu), h2f_bits(v.z >> 16), h2f_bits(v.w & 0xFFFFu), h2f_bits(v.w >> 16));
    }
    __syncthreads();
    if (nrows > 0) {
        float dots[2][1];
        int8_rows_dot<2, 1>(B.sh_gu_w8 + (long long)r0 * m.hidden, m.hidden, nrows, m.hidden, xs, m.hidden, lane, dots);
        if (lane == 0)
            for (int k = 0; k < nrows; ++k)
                __stcg(m.shgu + (long long)b * rows + r0 + k, B.sh_gu_scale[r0 + k] * dots[k][0]);
    }
    if (s == 0 && warp == kMbWarps - 1) {
        float acc = 0.f;
        for (int i0 = lane * 8; i0 < m.hidden; i0 += 256) {
            const uint4 g4 = __ldg(reinterpret_cast<const uint4*>(B.sh_gate + i0));
            const float4 xa = *reinterpret_cast<const float4*>(xs + xs_swz(i0));
            const float4 xb = *reinterpret_cast<const float4*>(xs + xs_swz(i0 + 4));
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
        for (int k = 16; k >= 1; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
        if (lane == 0) __stcg(m.shgate + b, sigmoid_f(acc));
    }
    __syncthreads();
    if (threadIdx.x == 0) red_add_release(ctr + kMcShGu, 1u);
}

// G unit u of block b (slot j, output block ob, input split c), expert e:
// the split's partial sums, published on the slot for its F unit.
// In a stack, unit 0 also stores h += (previous output) before its partial
// sums go out: every reader of h for this block (its R units) has finished,
// and the next block's R units, and this block's output (written over the
// previous one), come after every G unit.
template <int K>
__device__ __forceinline__ void mb_gate_up(const MbHead& m, const MbBlock& B, int b, int u, int e, float* sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int oblks = 2 * m.inter / 128, cs = m.gu_csize;
    const int j = u / (oblks * cs), ob = (u / cs) % oblks, c = u % cs;
    const int n_out = 2 * m.inter;
    const int KT = m.hidden >> 4, NT = n_out >> 4;
    const int kt0 = c * m.gu_kt, kt1 = min(KT, kt0 + m.gu_kt), nk = (kt1 - kt0) * 16;
    const uint16_t* codes = B.gu_codes + (long long)e * KT * NT * (16 * K);
    const TileStrides grid{NT, 1};
    float* xt = sm;
    float* red = xt + m.xt_floats;
    LaneCodes<K> cur;
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);
    const uint16_t* rin = B.gu_rin + (long long)e * m.hidden;
    const uint16_t* x = mb_x(m, B);
    for (int blk = warp; blk < nk / 128; blk += kMbWarps) {
        const int ib = kt0 * 16 + blk * 128 + 4 * lane;
        const uint2 rb = *reinterpret_cast<const uint2*>(rin + ib);
        const uint2 xb = __ldcg(reinterpret_cast<const uint2*>(x + ib));
        float v[4];
        v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * h2f_bits(static_cast<uint16_t>(xb.x & 0xFFFFu));
        v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * h2f_bits(static_cast<uint16_t>(xb.x >> 16));
        v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * h2f_bits(static_cast<uint16_t>(xb.y & 0xFFFFu));
        v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * h2f_bits(static_cast<uint16_t>(xb.y >> 16));
        h128_warp(v, lane);
        *reinterpret_cast<float4*>(xt + blk * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (m.stack && u == 0 && b > 0)
        for (int i = threadIdx.x * 4; i < m.hidden; i += kMbThreads * 4) {
            const float4 hv = __ldcg(reinterpret_cast<const float4*>(m.res + i));
            const float4 av = __ldcg(reinterpret_cast<const float4*>(m.outbuf + i));
            __stcg(reinterpret_cast<float4*>(m.res + i),
                   make_float4(__fadd_rn(hv.x, av.x), __fadd_rn(hv.y, av.y), __fadd_rn(hv.z, av.z), __fadd_rn(hv.w, av.w)));
        }
    __syncthreads();
    float* zp = red + kMbWarps * 128;
    cta_gemv_partial<K, 1, kMbWarps>(codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);

    // warp 0 stores the split's partial sums and publishes them on the slot
    // (its lanes' stores are ordered before lane 0's release by the warp
    // barrier); the slot's F unit adds the splits
    if (warp == 0) {
        float* part = m.gu_part + ((long long)b * m.topk * oblks + (long long)j * oblks + ob) * cs * 128;
        __stcg(reinterpret_cast<float4*>(part + c * 128 + 4 * lane), *reinterpret_cast<const float4*>(zp + 4 * lane));
        __syncwarp();
        if (lane == 0) red_add_release(m.ctr + (long long)b * kMbCtrWords + kMcGu + j, 1u);
    }
}

// F unit j of block b: slot j's gate_up outputs, output block ob by warp
// ob % NW: the G units' split partial sums added in split order, then the
// output transform (the per-slot gate_up kernel's rank 0); then, from them,
// the slot's down inputs H128(rin * SwiGLU(gate, up)), 128-block i by warp i
// % NW (the per-slot down kernel's prologue), into the workspace for the
// slot's D units.
__device__ __forceinline__ void mb_gate_up_finish(const MbHead& m, const MbBlock& B, int b, int j, const int* e_s,
                                                  float* ys) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int oblks = 2 * m.inter / 128, cs = m.gu_csize, n_out = 2 * m.inter, nib = m.inter / 128;
    const int e = e_s[j];
    uint2 rout_pre = make_uint2(0u, 0u), rin_pre = make_uint2(0u, 0u);
    if (warp < oblks) rout_pre = *reinterpret_cast<const uint2*>(B.gu_rout + (long long)e * n_out + warp * 128 + 4 * lane);
    const uint16_t* rin = B.dn_rin + (long long)e * m.inter;
    if (warp < nib) rin_pre = *reinterpret_cast<const uint2*>(rin + warp * 128 + 4 * lane);
    unsigned* ctr = m.ctr + (long long)b * kMbCtrWords;
    if (!cta_wait_geq(ctr + kMcGu + j, static_cast<unsigned>(oblks * cs), m.wait_ns, m.err, kErrGu)) return;
    for (int ob = warp; ob < oblks; ob += kMbWarps) {
        const float* part = m.gu_part + ((long long)b * m.topk * oblks + (long long)j * oblks + ob) * cs * 128;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < cs; ++r) {
            const float4 z4 = __ldcg(reinterpret_cast<const float4*>(part + r * 128 + 4 * lane));
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        const uint2 rb = ob == warp ? rout_pre : *reinterpret_cast<const uint2*>(B.gu_rout + (long long)e * n_out + ob * 128 + 4 * lane);
        output_transform_regs(v, rb, lane);
        *reinterpret_cast<float4*>(ys + ob * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    float* xd = m.xdg + ((long long)b * m.topk + j) * m.inter;
    for (int i = warp; i < nib; i += kMbWarps) {
        const float4 gv = *reinterpret_cast<const float4*>(ys + i * 128 + 4 * lane);
        const float4 uv = *reinterpret_cast<const float4*>(ys + (nib + i) * 128 + 4 * lane);
        const uint2 rb = i == warp ? rin_pre : *reinterpret_cast<const uint2*>(rin + i * 128 + 4 * lane);
        float v[4];
        v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * (silu_f(gv.x) * uv.x);
        v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * (silu_f(gv.y) * uv.y);
        v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * (silu_f(gv.z) * uv.z);
        v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * (silu_f(gv.w) * uv.w);
        h128_warp(v, lane);
        __stcg(reinterpret_cast<float4*>(xd + i * 128 + 4 * lane), make_float4(v[0], v[1], v[2], v[3]));
    }
    __syncthreads();
    if (threadIdx.x == 0 && !m.skip_publish) red_add_release(ctr + kMcGuJ + j, 1u);
}

// X unit x of block b: shared down rows x * 8 + warp + k * 8 * nX (the
// per-slot down kernel's order for sh_inter <= 512).
__device__ __forceinline__ void mb_shared_down(const MbHead& m, const MbBlock& B, int b, int xu, float* xsh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_sh = m.sh_inter;
    const int nwarps = m.nX * kMbWarps;
    for (int row = xu * kMbWarps + warp; row < m.hidden; row += nwarps)
        for (int off = lane * 128; off < n_sh; off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(B.sh_dn_w8 + (long long)row * n_sh + off));
    unsigned* ctr = m.ctr + (long long)b * kMbCtrWords;
    if (!cta_wait_geq(ctr + kMcShGu, static_cast<unsigned>(m.nS), m.wait_ns, m.err, kErrShGu)) return;
    const float* gu = m.shgu + (long long)b * 2 * n_sh;
    for (int i = threadIdx.x; i < n_sh; i += kMbThreads) xsh[xs_swz(i)] = silu_f(__ldcg(gu + i)) * __ldcg(gu + n_sh + i);
    __syncthreads();
    const float gate = __ldcg(m.shgate + b);
    for (int row = xu * kMbWarps + warp; row < m.hidden; row += nwarps) {
        float acc = 0.f;
        if (lane * 16 < n_sh) {
            const uint4 wv = ldg_stream_v4(B.sh_dn_w8 + (long long)row * n_sh + lane * 16);
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
        for (int k = 16; k >= 1; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
        if (lane == 0) __stcg(m.sh + (long long)b * m.hidden + row, gate * (B.sh_dn_scale[row] * acc));
    }
    __syncthreads();
    if (threadIdx.x == 0) red_add_release(ctr + kMcShDn, 1u);
}

// D unit d of block b (slot j, output block ob, input split h): SwiGLU of
// the slot's finished gate_up outputs, rin and the input Hadamard, then the
// split's partial sums of the 128 outputs, published on ob for the C unit.
template <int K>
__device__ __forceinline__ void mb_down(const MbHead& m, const MbBlock& B, int b, int d, const int* e_s, const float* w_s,
                                        float* sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nob = m.hidden / 128, ks = m.dn_ks;
    const int j = d / (nob * ks), ob = (d / ks) % nob, h = d % ks;
    const int e = e_s[j];
    const int KT = m.inter >> 4, NT = m.hidden >> 4;
    const int rows_h = KT / ks;
    const int kt0 = h * rows_h, kt1 = kt0 + rows_h;
    const uint16_t* codes = B.dn_codes + (long long)e * KT * NT * (16 * K);
    const TileStrides grid{NT, 1};
    float* red = sm;
    LaneCodes<K> cur;
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);
    {
        constexpr int kLines = 16 * K * 2 * 8 / 128;  // 128-byte lines per tile row of the block
        for (int i = threadIdx.x; i < rows_h * kLines; i += kMbThreads) {
            const uint16_t* p = codes + ((long long)(kt0 + i / kLines) * NT + ob * 8) * (16 * K) + (i % kLines) * 64;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
    unsigned* ctr = m.ctr + (long long)b * kMbCtrWords;
    if (!cta_wait_geq(ctr + kMcGuJ + j, 1u, m.wait_ns, m.err, kErrGuJ)) return;
    float* zp = red + kMbWarps * 128;
    cta_gemv_partial_gx<K, kMbWarps>(codes, grid, ob, kt0, kt1,
                                     m.xdg + ((long long)b * m.topk + j) * m.inter + kt0 * 16, cur, red, zp);

    if (warp == 0) {
        float* part = m.dn_part + (((long long)b * nob + ob) * m.topk) * ks * 128;  // [topk][ks][128] of the block
        __stcg(reinterpret_cast<float4*>(part + (j * ks + h) * 128 + 4 * lane), *reinterpret_cast<const float4*>(zp + 4 * lane));
        __syncwarp();
        if (lane == 0) red_add_release(ctr + kMcCmb + ob, 1u);
    }
}

// C unit: output block ob of block b. Warp q adds expert q's down split
// partials in split order and applies its output transform and routing
// weight; the experts are added in slot order and the shared expert last
// (the per-slot down kernel's rank 0); in a stack the last block also adds
// its output to h.
__device__ __forceinline__ void mb_combine(const MbHead& m, const MbBlock& B, int b, int ob, const int* e_s,
                                           const float* w_s, float* sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nob = m.hidden / 128, ks = m.dn_ks;
    uint2 rout_pre = make_uint2(0u, 0u);
    if (warp < m.topk)
        rout_pre = *reinterpret_cast<const uint2*>(B.dn_rout + (long long)e_s[warp] * m.hidden + ob * 128 + 4 * lane);
    unsigned* ctr = m.ctr + (long long)b * kMbCtrWords;
    int ok = 1;
    if (threadIdx.x == 0) {
        ok = wait_geq(ctr + kMcCmb + ob, static_cast<unsigned>(m.topk * ks), m.wait_ns, m.err, kErrCmb);
        if (ok && m.sh_inter > 0) ok = wait_geq(ctr + kMcShDn, static_cast<unsigned>(m.nX), m.wait_ns, m.err, kErrShDn);
    }
    if (!__syncthreads_and(ok)) return;
    const float* part = m.dn_part + (((long long)b * nob + ob) * m.topk) * ks * 128;
    float* dres = sm;  // [topk][128]
    if (warp < m.topk) {
        const int q = warp;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sp = 0; sp < ks; ++sp) {
            const float4 z4 = __ldcg(reinterpret_cast<const float4*>(part + (q * ks + sp) * 128 + 4 * lane));
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
        for (int q = 0; q < m.topk; ++q) sum += dres[q * 128 + i];
        if (m.sh_inter > 0) sum += __ldcg(m.sh + (long long)b * m.hidden + ob * 128 + i);
        float* out = m.stack ? m.outbuf : B.out;
        __stcg(out + ob * 128 + i, sum);
        if (m.stack && b == m.n_blocks - 1) __stcg(m.res + ob * 128 + i, __fadd_rn(__ldcg(m.res + ob * 128 + i), sum));
    }
    __syncthreads();
    if (threadIdx.x == 0) red_add_release(ctr + kMcDone, 1u);
}

// Queue position q -> (block, unit index within the block): the segment
// holding q (the last one whose first position is <= q; binary search).
__device__ __forceinline__ void mb_unit_at(const MbSeg* seg, int n_segs, int q, int* b, int* l) {
    int lo = 0, hi = n_segs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg[mid].pos <= q) lo = mid;
        else hi = mid - 1;
    }
    *b = seg[lo].block;
    *l = seg[lo].first + (q - seg[lo].pos);
}

__global__ void __launch_bounds__(kMbThreads, 4) moe_multi_kernel(const __grid_constant__ MbArgs args) {
    extern __shared__ __align__(16) float sm[];
    // the launch's settings, the blocks' descriptors and the queue's segments
    // live in shared memory: units read them there (not through the
    // parameter space, and not held in registers across the work loop)
    __shared__ __align__(16) MbHead m;
    __shared__ __align__(16) MbBlock blk_s[kMbMaxBlocks];
    __shared__ __align__(16) MbSeg seg_s[kMbMaxSegs];
    __shared__ int tk_block;
    __shared__ int e_s[8];
    __shared__ float w_s[8];
    __shared__ int4 qbl_s[2];  // the next unit (queue position, block, unit in block), two slots used in turn
    static_assert(sizeof(MbHead) % 8 == 0 && sizeof(MbBlock) % 8 == 0 && sizeof(MbSeg) % 4 == 0, "copied in words");
    const int n_segs = args.n_segs;
    if (threadIdx.x < static_cast<int>(sizeof(MbHead) / 8))
        reinterpret_cast<unsigned long long*>(&m)[threadIdx.x] = reinterpret_cast<const unsigned long long*>(&args.h)[threadIdx.x];
    for (int i = threadIdx.x; i < args.h.n_blocks * static_cast<int>(sizeof(MbBlock) / 8); i += kMbThreads)
        reinterpret_cast<unsigned long long*>(blk_s)[i] = reinterpret_cast<const unsigned long long*>(args.blk)[i];
    for (int i = threadIdx.x; i < n_segs * static_cast<int>(sizeof(MbSeg) / 4); i += kMbThreads)
        reinterpret_cast<int*>(seg_s)[i] = reinterpret_cast<const int*>(args.seg)[i];
    __syncthreads();
    pdl_wait();
    cg::grid_group grid = cg::this_grid();
    if (!grid.is_valid()) {  // not launched cooperatively: nothing may wait on another CTA
        if (blockIdx.x == 0 && threadIdx.x == 0) *m.err = kErrNotCoop;
        return;
    }
    // zero the counters and the queue, once for the whole sequence
    const long long words = (long long)m.n_blocks * kMbCtrWords + 32;
    for (long long i = (long long)blockIdx.x * kMbThreads + threadIdx.x; i < words; i += (long long)gridDim.x * kMbThreads)
        m.ctr[i] = 0u;
    if (blockIdx.x == 0 && threadIdx.x == 0) *m.err = 0;
    if (threadIdx.x == 0) tk_block = -1;
    grid.sync();

    unsigned* queue = m.ctr + (long long)m.n_blocks * kMbCtrWords;
    const int total = m.n_blocks * m.U;
    // thread 0 takes the queue positions and looks them up; the next unit
    // reaches the CTA through qbl_s (one barrier per unit)
    if (threadIdx.x == 0) {
        const int q0 = static_cast<int>(atomicAdd(queue, 1u));
        int b0 = 0, l0 = 0;
        if (q0 < total) mb_unit_at(seg_s, n_segs, q0, &b0, &l0);
        qbl_s[0] = make_int4(q0, b0, l0, 0);
    }
    __syncthreads();
    for (int it = 0;; ++it) {
        const int4 cur = qbl_s[it & 1];
        if (cur.x >= total) break;
        const int b = cur.y, l = cur.z;
        int q_next = 0;
        if (threadIdx.x == 0) q_next = static_cast<int>(atomicAdd(queue, 1u));  // in flight while this unit runs
        const MbBlock& B = blk_s[b];
        if (l < m.nR) {
            mb_router(m, B, b, l, sm);
        } else if (l < m.nR + m.nS) {
            mb_shared_gate_up(m, B, b, l - m.nR, sm);
        } else if (l < m.nR + m.nS + m.nG) {
            const int u = l - m.nR - m.nS;
            if (mb_routing(m, b, &tk_block, e_s, w_s)) {
                const int e = e_s[u / (2 * m.inter / 128 * m.gu_csize)];
                if (B.gu_K == 2)
                    mb_gate_up<2>(m, B, b, u, e, sm);
                else
                    mb_gate_up<3>(m, B, b, u, e, sm);
            }
        } else if (l < m.nR + m.nS + m.nG + m.nX) {
            mb_shared_down(m, B, b, l - m.nR - m.nS - m.nG, sm);
        } else if (l < m.nR + m.nS + m.nG + m.nX + m.nF) {
            if (mb_routing(m, b, &tk_block, e_s, w_s)) mb_gate_up_finish(m, B, b, l - m.nR - m.nS - m.nG - m.nX, e_s, sm);
        } else if (l < m.nR + m.nS + m.nG + m.nX + m.nF + m.nD) {
            const int d = l - m.nR - m.nS - m.nG - m.nX - m.nF;
            if (mb_routing(m, b, &tk_block, e_s, w_s)) {
                if (B.dn_K == 2)
                    mb_down<2>(m, B, b, d, e_s, w_s, sm);
                else
                    mb_down<3>(m, B, b, d, e_s, w_s, sm);
            }
        } else {
            if (mb_routing(m, b, &tk_block, e_s, w_s))
                mb_combine(m, B, b, l - m.nR - m.nS - m.nG - m.nX - m.nF - m.nD, e_s, w_s, sm);
        }
        if (threadIdx.x == 0) {
            int bn = 0, ln = 0;
            if (q_next < total) mb_unit_at(seg_s, n_segs, q_next, &bn, &ln);
            qbl_s[(it + 1) & 1] = make_int4(q_next, bn, ln, 0);
        }
        __syncthreads();
    }
}

}  // namespace

bool multi_shape_ok(int hidden, int inter, int E, int topk, int sh_inter) {
    if (hidden > kMbMaxHidden || hidden % 256 || hidden / 128 > kMbMaxOb) return false;
    if (inter % 128 || 2 * inter / 128 > kMbMaxOb) return false;
    if (E < 1 || E > 256 || topk < 1 || topk > 8) return false;
    if (sh_inter > kMbMaxShInter || sh_inter % 16) return false;
    return true;
}

MbPlan multi_plan(int n_blocks, int hidden, int inter, int E, int topk, int sh_inter) {
    const SlotPlan sp = slot_plan(1, hidden, inter, topk);
    MbPlan p{};
    p.gu_csize = sp.gu_csize;
    p.gu_kt = sp.gu_kt_per_cta;
    p.dn_ks = sp.dn_ksplit;
    p.nR = (E + kMbWarps - 1) / kMbWarps;
    p.nS = sh_inter > 0 ? (2 * sh_inter + 2 * kMbWarps - 1) / (2 * kMbWarps) : 0;
    p.nG = topk * (2 * inter / 128) * sp.gu_csize;
    p.nX = sh_inter > 0 ? (hidden + 3 * kMbWarps - 1) / (3 * kMbWarps) : 0;
    p.nD = topk * (hidden / 128) * sp.dn_ksplit;
    p.nF = topk;
    p.nC = hidden / 128;
    p.U = p.nR + p.nS + p.nG + p.nX + p.nF + p.nD + p.nC;
    p.xt_floats = (sp.gu_kt_per_cta * 16 + 31) / 32 * 32;
    // G: xt, the reduction scratch, the partial sums; S: x as floats; X: the
    // shared SwiGLU; R in a stack: the normalised x; F: one slot's gate_up
    // outputs
    const int unit_floats =
        max(max(p.xt_floats + (kMbWarps + 1) * 128, hidden), max(max(sh_inter, hidden / 2), 2 * inter));
    p.smem = unit_floats * 4;
    const size_t n = n_blocks;
    p.ctr_bytes = (n * kMbCtrWords + 32) * 4;
    p.logits_bytes = n * E * 2;
    p.xdg_bytes = n * topk * inter * 4;
    p.shgu_bytes = n * 2 * sh_inter * 4;
    p.shgate_bytes = n * 4;
    p.sh_bytes = n * hidden * 4;
    p.gu_part_bytes = n * topk * (2 * inter / 128) * sp.gu_csize * 128 * 4;
    p.dn_part_bytes = n * (hidden / 128) * topk * sp.dn_ksplit * 128 * 4;
    p.ids_bytes = n * topk * 4;
    return p;
}

cudaError_t multi_grid(int num_sms, int smem, int* grid) {
    int per_sm = 0;
    *grid = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_multi_kernel, kMbThreads, smem);
    if (e != cudaSuccess) return e;
    *grid = per_sm * num_sms;
    return cudaSuccess;
}

cudaError_t launch_moe_multi(const MbArgs& m, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMbThreads);
    cfg.dynamicSmemBytes = m.h.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<MbArgs*>(&m)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(moe_multi_kernel), args);
}

}  // namespace escha
