// One MoE block for one token (batch-1 decode): the per-slot router kernel,
// then ONE cooperative kernel for the experts.
//
// The three per-slot kernels (moe_block.cu) meet at two grid boundaries:
// every gate_up CTA waits for the whole router grid and recomputes the
// token's top-k, and every down CTA waits for the whole gate_up grid. At one
// token those waits, not the decode, are most of the block's time. Here the
// router kernel (launched programmatically, so it loads its weights while
// the previous kernel finishes) is followed by one cooperative grid (all CTAs
// resident at once) whose CTAs hand work to each other through counters in
// the workspace, which the router kernel zeroes:
//
//   CTAs [0, n_gate_up)          one gate_up unit each: (slot j, 128-wide
//                                output block, input split c);
//   CTAs [n_gate_up, grid)       the int8 shared expert's down rows;
//   n_down down units            (slot j, output block, input split h), on
//                                the shared-expert CTAs first, then on
//                                gate_up CTAs after their gate_up unit.
//
// Every CTA computes the token's top-k from the router's logits. A gate_up
// unit pushes its partial sums to the workspace; the last of a block's input
// splits to arrive (an atomic count) adds them in split order and applies
// the output transform. A down unit starts when its expert's gate_up outputs
// are complete; the last of an output block's down units (all experts, all
// splits) finishes every expert of the block (splits in order, output
// transform, routing weight) and adds the experts in slot order and the
// shared expert (hipfire PR #694, commit "Executed the moeblk golden against
// real shipped layer-0 weights": the block is the weighted sum of the routed
// experts' gate_up -> SwiGLU -> down plus the sigmoid-gated shared expert).
//
// A cooperative grid is scheduled only when all of it fits, so it cannot
// start while the previous grid still holds SMs; the router kernel in front
// of it can, which is why it stays a separate launch.
//
// The input splits and every summation order are those of the per-slot
// kernels at one token (slot_plan), so the outputs are bit for bit the same.
// Every wait on another CTA is bounded (fz_wait_ns): a wait that runs out
// sets the workspace status word and the CTA skips the work that needed it,
// so the kernel always ends.
#include <atomic>
#include <mutex>

#include "coop.cuh"
#include "kernels.h"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kFzThreads = 256;
constexpr int kFzWarps = kFzThreads / 32;
constexpr int kFzMaxHidden = 2048;
constexpr int kFzMaxShInter = 512;
constexpr int kFzMaxOb = 32;  // gate_up output blocks (2 * inter / 128) and down output blocks (hidden / 128)

// Counter words in the workspace (unsigned, offsets in words; kFzCtrWords
// in all, zeroed by the router kernel of the same call).
constexpr int kCtShDn = 0;                     // shared-down CTAs finished
constexpr int kCtGu = 1;                       // [8][kFzMaxOb]: gate_up splits arrived per (slot, block)
constexpr int kCtGuJ = kCtGu + 8 * kFzMaxOb;   // [8]: gate_up blocks finished per slot
constexpr int kCtCmb = kCtGuJ + 8;             // [kFzMaxOb]: down units finished per output block
constexpr int kCtWords = kCtCmb + kFzMaxOb;
static_assert(kCtWords <= kFzCtrWords, "counter block");

// Status codes of waits that ran out (the workspace status word).
constexpr int kErrGuJ = 5, kErrShDn = 6, kErrNotCoop = 7;

struct FzGeo {
    int n_gate_up, n_extra, n_down;
    int gu_csize, gu_kt, dn_ks;
    int xt_floats;
};

// The token's routing, by warp 0 from the router's f16 logits: experts and
// weights of the slots into e_s / w_s (shared memory). Ends with the CTA
// synchronised.
__device__ void fz_topk(const MoeArgs& a, int* e_s, float* w_s) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        uint16_t bits[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) bits[i] = lane + 32 * i < a.E ? __ldcg(a.logits + lane + 32 * i) : 0;
        int e_l;
        float w_l;
        topk_softmax_warp_bits(bits, a.E, a.topk, lane, &e_l, &w_l);
        if (lane < a.topk) {
            e_s[lane] = e_l;
            w_s[lane] = w_l;
        }
    }
    __syncthreads();
}

// gate_up unit u: slot j, output block ob, input split c; expert e. The
// first unit also stores the residual stream's h += add (residual block),
// before its partial sums go out: every down unit, and so the block's output
// (which may be written over add), comes after that.
template <int K, bool FUSED>
__device__ void fz_gate_up(const MoeArgs& a, const FzGeo& g, int u, int e, float* xt, float* red) {
    __shared__ int last_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int oblks = 2 * a.inter / 128, cs = g.gu_csize;
    const int j = u / (oblks * cs), ob = (u / cs) % oblks, c = u % cs;
    const int n_out = 2 * a.inter;
    const int KT = a.hidden >> 4, NT = n_out >> 4;
    const int kt0 = c * g.gu_kt, kt1 = min(KT, kt0 + g.gu_kt), nk = (kt1 - kt0) * 16;
    const uint16_t* codes = a.gu_codes + (long long)e * KT * NT * (16 * K);
    const TileStrides grid{NT, 1};
    LaneCodes<K> cur;
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);
    uint2 rout_pre = make_uint2(0u, 0u);  // for the split that finishes the block
    if (warp == 0) rout_pre = *reinterpret_cast<const uint2*>(a.gu_rout + (long long)e * n_out + ob * 128 + 4 * lane);
    // xt = H128(rin_e * x) over this split's inputs
    const uint16_t* rin = a.gu_rin + (long long)e * a.hidden;
    const uint16_t* xrow = FUSED ? a.x_norm : a.x;
    for (int blk = warp; blk < nk / 128; blk += kFzWarps) {
        const int ib = kt0 * 16 + blk * 128 + 4 * lane;
        const uint2 rb = *reinterpret_cast<const uint2*>(rin + ib);
        const uint2 xb = __ldcg(reinterpret_cast<const uint2*>(xrow + ib));
        float v[4];
        v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * h2f_bits(static_cast<uint16_t>(xb.x & 0xFFFFu));
        v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * h2f_bits(static_cast<uint16_t>(xb.x >> 16));
        v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * h2f_bits(static_cast<uint16_t>(xb.y & 0xFFFFu));
        v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * h2f_bits(static_cast<uint16_t>(xb.y >> 16));
        h128_warp(v, lane);
        *reinterpret_cast<float4*>(xt + blk * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (FUSED && u == 0 && a.rs_add)  // the router grid, which read h and add, has finished
        for (int i = threadIdx.x * 4; i < a.hidden; i += kFzThreads * 4) {
            const float4 hv = __ldcg(reinterpret_cast<const float4*>(a.rs_h + i));
            const float4 av = __ldcg(reinterpret_cast<const float4*>(a.rs_add + i));
            *reinterpret_cast<float4*>(a.rs_h + i) =
                make_float4(__fadd_rn(hv.x, av.x), __fadd_rn(hv.y, av.y), __fadd_rn(hv.z, av.z), __fadd_rn(hv.w, av.w));
        }
    __syncthreads();
    float* zp = red + kFzWarps * 128;
    cta_gemv_partial<K, 1, kFzWarps>(codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);

    float* part = a.fz_gu_part + (long long)(j * oblks + ob) * cs * 128;
    if (warp == 0) __stcg(reinterpret_cast<float4*>(part + c * 128 + 4 * lane), *reinterpret_cast<const float4*>(zp + 4 * lane));
    __syncthreads();
    if (threadIdx.x == 0)
        last_s = atom_add_acq_rel(a.fz_ctr + kCtGu + j * kFzMaxOb + ob, 1u) == static_cast<unsigned>(cs - 1);
    __syncthreads();
    if (!last_s || warp != 0) return;
    // the last split: all splits' partials in split order, then the output transform
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < cs; ++r) {
        const float4 z4 = r == c ? *reinterpret_cast<const float4*>(zp + 4 * lane)
                                 : __ldcg(reinterpret_cast<const float4*>(part + r * 128 + 4 * lane));
        v[0] += z4.x;
        v[1] += z4.y;
        v[2] += z4.z;
        v[3] += z4.w;
    }
    output_transform_regs(v, rout_pre, lane);
    __stcg(reinterpret_cast<float4*>(a.ygu + (long long)j * n_out + ob * 128 + 4 * lane), make_float4(v[0], v[1], v[2], v[3]));
    __syncwarp();
    if (lane == 0 && !a.fz_skip_publish) red_add_release(a.fz_ctr + kCtGuJ + j, 1u);
}

// down unit d: slot j, output block ob, input split h. The last of the
// block's topk * ks units to arrive finishes the block: warp q adds expert
// q's split partials in split order, applies its output transform and
// routing weight; then the experts are added in slot order and the shared
// expert last (the order of the per-slot down kernel's rank 0).
template <int K>
__device__ void fz_down(const MoeArgs& a, const FzGeo& g, int d, const int* e_s, const float* w_s, float* xt,
                        float* red) {
    __shared__ int last_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nob = a.hidden / 128, ks = g.dn_ks;
    const int j = d / (nob * ks), ob = (d / ks) % nob, h = d % ks;
    const int e = e_s[j];
    const int KT = a.inter >> 4, NT = a.hidden >> 4;
    const int rows_h = KT / ks;
    const int kt0 = h * rows_h, kt1 = kt0 + rows_h, nk = rows_h * 16;
    const uint16_t* codes = a.dn_codes + (long long)e * KT * NT * (16 * K);
    const TileStrides grid{NT, 1};
    LaneCodes<K> cur;
    if (kt0 + warp < kt1) load_lane_codes<K>(cur, codes, grid, kt0 + warp, ob * 8, lane);
    {  // the unit's other code rows into L2 while its expert's gate_up runs
        constexpr int kLines = 16 * K * 2 * 8 / 128;  // 128-byte lines per tile row of the block
        for (int i = threadIdx.x; i < rows_h * kLines; i += kFzThreads) {
            const uint16_t* p = codes + ((long long)(kt0 + i / kLines) * NT + ob * 8) * (16 * K) + (i % kLines) * 64;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
    const uint16_t* rin = a.dn_rin + (long long)e * a.inter;
    uint2 rin_pre = make_uint2(0u, 0u);
    if (warp < nk / 128) rin_pre = *reinterpret_cast<const uint2*>(rin + kt0 * 16 + warp * 128 + 4 * lane);
    uint2 rout_pre = make_uint2(0u, 0u);  // warp q: expert q's output scales of the block, in case this unit finishes it
    if (warp < a.topk)
        rout_pre = *reinterpret_cast<const uint2*>(a.dn_rout + (long long)e_s[warp] * a.hidden + ob * 128 + 4 * lane);
    if (!cta_wait_geq(a.fz_ctr + kCtGuJ + j, static_cast<unsigned>(2 * a.inter / 128), a.fz_wait_ns, a.err, kErrGuJ)) return;

    // xt = H128(rin_e * SwiGLU(ygu[j])) over this split's inputs
    const float* yr = a.ygu + (long long)j * 2 * a.inter;
    for (int blk = warp; blk < nk / 128; blk += kFzWarps) {
        const int ib = kt0 * 16 + blk * 128 + 4 * lane;
        const float4 gv = __ldcg(reinterpret_cast<const float4*>(yr + ib));
        const float4 uv = __ldcg(reinterpret_cast<const float4*>(yr + a.inter + ib));
        const uint2 rb = blk == warp ? rin_pre : *reinterpret_cast<const uint2*>(rin + ib);
        float v[4];
        v[0] = h2f_bits(static_cast<uint16_t>(rb.x & 0xFFFFu)) * (silu_f(gv.x) * uv.x);
        v[1] = h2f_bits(static_cast<uint16_t>(rb.x >> 16)) * (silu_f(gv.y) * uv.y);
        v[2] = h2f_bits(static_cast<uint16_t>(rb.y & 0xFFFFu)) * (silu_f(gv.z) * uv.z);
        v[3] = h2f_bits(static_cast<uint16_t>(rb.y >> 16)) * (silu_f(gv.w) * uv.w);
        h128_warp(v, lane);
        *reinterpret_cast<float4*>(xt + blk * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    float* zp = red + kFzWarps * 128;
    cta_gemv_partial<K, 1, kFzWarps>(codes, grid, ob, kt0, kt1, xt, nk, cur, red, zp);

    // partials of the block: [topk][ks][128]
    float* part = a.fz_dn_part + (long long)ob * a.topk * ks * 128;
    if (warp == 0) __stcg(reinterpret_cast<float4*>(part + (j * ks + h) * 128 + 4 * lane), *reinterpret_cast<const float4*>(zp + 4 * lane));
    __syncthreads();
    if (threadIdx.x == 0)
        last_s = atom_add_acq_rel(a.fz_ctr + kCtCmb + ob, 1u) == static_cast<unsigned>(a.topk * ks - 1);
    __syncthreads();
    if (!last_s) return;
    float* dres = red;  // [topk][128], free again
    if (warp < a.topk) {
        const int q = warp;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sp = 0; sp < ks; ++sp) {
            const float4 z4 = (q == j && sp == h) ? *reinterpret_cast<const float4*>(zp + 4 * lane)
                                                  : __ldcg(reinterpret_cast<const float4*>(part + (q * ks + sp) * 128 + 4 * lane));
            v[0] += z4.x;
            v[1] += z4.y;
            v[2] += z4.z;
            v[3] += z4.w;
        }
        output_transform_regs(v, rout_pre, lane);
        const float wq = w_s[q];
        *reinterpret_cast<float4*>(dres + q * 128 + 4 * lane) = make_float4(wq * v[0], wq * v[1], wq * v[2], wq * v[3]);
    }
    int ok = 1;
    if (a.sh_inter > 0 && threadIdx.x == 0)
        ok = wait_geq(a.fz_ctr + kCtShDn, static_cast<unsigned>(g.n_extra), a.fz_wait_ns, a.err, kErrShDn);
    if (!__syncthreads_and(ok)) return;
    if (threadIdx.x < 128) {
        const int i = threadIdx.x;
        float sum = 0.f;
        for (int q = 0; q < a.topk; ++q) sum += dres[q * 128 + i];
        if (a.sh_inter > 0) sum += __ldcg(a.sh + ob * 128 + i);
        a.out[ob * 128 + i] = sum;
    }
}

// Shared expert down rows (the CTAs after the gate_up ones; its gate_up rows
// and gate came from the router kernel): row o = gate * (scale_o * sum_i
// w8[o][i] * SwiGLU(gu)_i); lane l takes columns 16 l .. 16 l + 15 in order,
// then the xor butterfly (the per-slot down kernel's order for sh_inter <=
// 512).
__device__ void fz_shared_down(const MoeArgs& a, const FzGeo& g, int xc, float* xsh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_sh = a.sh_inter;
    for (int i = threadIdx.x; i < n_sh; i += kFzThreads)
        xsh[xs_swz(i)] = silu_f(__ldcg(a.shgu + i)) * __ldcg(a.shgu + n_sh + i);
    __syncthreads();
    const float gate = __ldcg(a.shgate);
    const int nwarps = g.n_extra * kFzWarps;
    for (int row = xc * kFzWarps + warp; row < a.hidden; row += nwarps) {
        float acc = 0.f;
        if (lane * 16 < n_sh) {
            const uint4 wv = ldg_stream_v4(a.sh_dn_w8 + (long long)row * n_sh + lane * 16);
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
        if (lane == 0) __stcg(a.sh + row, gate * (a.sh_dn_scale[row] * acc));
    }
    __syncthreads();
    if (threadIdx.x == 0) red_add_release(a.fz_ctr + kCtShDn, 1u);
}

template <int GK, int DK, bool FUSED>
__global__ void __launch_bounds__(kFzThreads, 4) moe_fused_kernel(const MoeArgs a, const FzGeo g) {
    extern __shared__ __align__(16) float smem[];
    float* xt = smem;                        // routed transformed inputs of a unit
    float* red = xt + g.xt_floats;           // [kFzWarps + 1][128]
    float* xsh = red + (kFzWarps + 1) * 128; // shared expert's down input
    __shared__ int e_s[8];
    __shared__ float w_s[8];
    const int cta = static_cast<int>(blockIdx.x);
    const bool is_gu = cta < g.n_gate_up;
    const int xc = cta - g.n_gate_up;  // extra CTAs: shared down rows
    // down unit of this CTA: the extra CTAs take units 0.., then the gate_up CTAs
    const int d = !is_gu ? xc : g.n_extra + cta;
    const bool has_dn = d < g.n_down;

    if (!is_gu && a.sh_inter > 0) {  // this warp's shared down rows into L2
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int row = xc * kFzWarps + warp; row < a.hidden; row += g.n_extra * kFzWarps)
            for (int off = lane * 128; off < a.sh_inter; off += 32 * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.sh_dn_w8 + (long long)row * a.sh_inter + off));
    }
    pdl_wait();  // the router kernel: logits, shared gate_up rows, zeroed counters (and x_norm)
    cg::grid_group grid = cg::this_grid();
    if (!grid.is_valid()) {  // not launched cooperatively: nothing may wait on another CTA
        if (cta == 0 && threadIdx.x == 0) *a.err = kErrNotCoop;
        return;
    }
    fz_topk(a, e_s, w_s);
    if (cta == 0 && threadIdx.x < a.topk) {  // the routing outputs
        a.ids[threadIdx.x] = e_s[threadIdx.x];
        a.w[threadIdx.x] = w_s[threadIdx.x];
    }
    if (is_gu) {
        const int u = cta;
        const int j = u / (2 * a.inter / 128 * g.gu_csize);
        fz_gate_up<GK, FUSED>(a, g, u, e_s[j], xt, red);
    } else if (a.sh_inter > 0) {
        fz_shared_down(a, g, xc, xsh);
    }
    pdl_trigger();  // the next kernel may start loading its weights as SMs free up
    if (!has_dn) return;
    __syncthreads();  // the previous role's shared memory is free again
    fz_down<DK>(a, g, d, e_s, w_s, xt, red);
}

FzGeo fz_geo(const FusedPlan& p, int hidden, int inter, int topk) {
    const SlotPlan sp = slot_plan(1, hidden, inter, topk);
    FzGeo g{};
    g.n_gate_up = p.n_gate_up;
    g.n_extra = p.n_extra;
    g.n_down = p.n_down;
    g.gu_csize = sp.gu_csize;
    g.gu_kt = sp.gu_kt_per_cta;
    g.dn_ks = sp.dn_ksplit;
    g.xt_floats = (max(sp.gu_kt_per_cta * 16, inter / sp.dn_ksplit) + 31) / 32 * 32;
    return g;
}

const void* fused_kernel(int gu_K, int dn_K, bool fused_norm) {
#define ESCHA_FZ(G, D)                                                                                       \
    if (gu_K == G && dn_K == D)                                                                              \
        return fused_norm ? reinterpret_cast<const void*>(moe_fused_kernel<G, D, true>)                      \
                          : reinterpret_cast<const void*>(moe_fused_kernel<G, D, false>);
    ESCHA_FZ(2, 2)
    ESCHA_FZ(2, 3)
    ESCHA_FZ(3, 2)
    ESCHA_FZ(3, 3)
#undef ESCHA_FZ
    return nullptr;
}

}  // namespace

// CTAs after the gate_up ones: enough for at most 3 shared-down rows per
// warp, and at least every SM slot the gate_up CTAs leave (4 per SM on the
// 152-SM GB300), where the first down units then start at once.
int fz_extra(int hidden, int sh_inter, int n_gate_up, int n_down) {
    const int rows = sh_inter > 0 ? (hidden + 3 * kFzWarps - 1) / (3 * kFzWarps) : 0;
    const int free_slots = max(0, 4 * 152 - n_gate_up);
    return max(rows, min(n_down, free_slots));
}

bool fused_shape_ok(int hidden, int inter, int E, int topk, int sh_inter) {
    if (hidden > kFzMaxHidden || hidden % 256 || hidden / 128 > kFzMaxOb) return false;
    if (inter % 128 || 2 * inter / 128 > kFzMaxOb) return false;
    if (E < 1 || E > 256 || topk < 1 || topk > 8) return false;
    if (sh_inter > kFzMaxShInter || sh_inter % 16) return false;
    const FusedPlan p = fused_plan(hidden, inter, E, topk, sh_inter);
    return p.n_down <= p.grid;
}

FusedPlan fused_plan(int hidden, int inter, int E, int topk, int sh_inter) {
    (void)E;
    const SlotPlan sp = slot_plan(1, hidden, inter, topk);
    FusedPlan p{};
    p.n_gate_up = topk * (2 * inter / 128) * sp.gu_csize;
    p.n_down = topk * (hidden / 128) * sp.dn_ksplit;
    p.n_extra = fz_extra(hidden, sh_inter, p.n_gate_up, p.n_down);
    p.grid = p.n_gate_up + p.n_extra;
    const FzGeo g = fz_geo(p, hidden, inter, topk);
    p.smem = (g.xt_floats + (kFzWarps + 1) * 128 + kFzMaxShInter) * 4;
    p.ctr_bytes = kFzCtrWords * 4;
    p.gu_part_bytes = (size_t)topk * (2 * inter / 128) * sp.gu_csize * 128 * 4;
    p.dn_part_bytes = (size_t)topk * (hidden / 128) * sp.dn_ksplit * 128 * 4;
    p.dres_bytes = 0;
    return p;
}

cudaError_t fused_fits(const FusedPlan& p, int gu_K, int dn_K, int num_sms, bool* fits) {
    *fits = false;
    for (int fused = 0; fused < 2; ++fused) {
        const void* f = fused_kernel(gu_K, dn_K, fused != 0);
        if (!f) return cudaSuccess;
        int per_sm = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kFzThreads, p.smem);
        if (e != cudaSuccess) return e;
        if ((long long)per_sm * num_sms < p.grid) return cudaSuccess;
    }
    *fits = true;
    return cudaSuccess;
}

// Whether a cooperative launch may also be programmatic (start while the
// preceding kernel finishes) on a device: -1 not known yet, 0 no, 1 yes.
// Learnt from the first launch made outside a stream capture; until then the
// launch is cooperative only.
static std::atomic<int> g_coop_pdl[64];
static std::once_flag g_coop_pdl_init;

cudaError_t launch_moe_fused(const MoeArgs& a, const FusedPlan& p, cudaStream_t s) {
    std::call_once(g_coop_pdl_init, [] {
        for (auto& v : g_coop_pdl) v.store(-1);
    });
    const FzGeo g = fz_geo(p, a.hidden, a.inter, a.topk);
    const void* f = fused_kernel(a.gu_K, a.dn_K, a.x_norm != nullptr);
    if (!f) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kFzThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    void* args[] = {const_cast<MoeArgs*>(&a), const_cast<FzGeo*>(&g)};
    int pdl = g_coop_pdl[dev].load();
    if (pdl < 0) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
            cfg.numAttrs = 2;
            e = cudaLaunchKernelExC(&cfg, f, args);
            if (e == cudaSuccess) {
                g_coop_pdl[dev].store(1);
                return e;
            }
            cudaGetLastError();  // not supported together: cooperative launches only from now on
            g_coop_pdl[dev].store(0);
        }
        pdl = 0;
    }
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace escha
