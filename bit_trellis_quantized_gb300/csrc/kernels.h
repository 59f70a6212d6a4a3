// Internal launch interfaces between the C-ABI layer (escha_api.cu) and the
// kernels. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace escha {

// Input modes of the trellis GEMV prologue.
constexpr int kXmF16 = 0;  // x is fp16 [rows][in]
constexpr int kXmF32 = 1;  // x is f32 [rows][in]

struct GemvArgs {
    const uint16_t* codes;  // code tensor [in/16][out/16][16K]
    int in, out;
    int kt_per_cta;  // filled by the launcher
    int x_mode;      // kXmF16 or kXmF32
    const void* x;
    long long x_stride;  // elements between x rows
    const uint16_t* rin;
    const uint16_t* rout;
    float* y;
    long long y_stride;
    int batch;
    int nt_major;        // code tiles stored [out/16][in/16] (else [in/16][out/16])
    const float* bias;   // f32 [out] added after the output transform, or null
};

// Trellis GEMV of one projection for `batch` tokens, nb tokens per CTA
// (1, 2 or 4); items = ceil(batch / nb).
cudaError_t launch_trellis_gemv(const GemvArgs& a, int K, int nb, int items, int num_sms, cudaStream_t s);

// Input-row split of a trellis GEMV: CTAs per cluster and rows per CTA.
void gemv_plan(int in, int blocks_per_split, int num_sms, int ctas_per_sm, int* kt_per_cta, int* csize);

// Dense decode of a code tensor to fp16 bit patterns W[in][out].
cudaError_t launch_trellis_decode(const uint16_t* codes, int in, int out, int K, uint16_t* W, cudaStream_t s);

// int8 w8a16 GEMV: y[m][o] = sum_i (scale[o]*W[o][i]) * x[m][i]; x_dtype
// 1 = f16, 2 = bf16, 3 = f32.
cudaError_t launch_int8_gemv(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                             long long x_stride, int act, int M, float* y, long long y_stride, int num_sms,
                             cudaStream_t s);

cudaError_t launch_int8_dequant(const int8_t* W, const float* scales, int N, int Kin, float* out, cudaStream_t s);

// int8 w8a16 GEMM on the tensor cores (same result as the GEMV, for many
// tokens): a prep kernel writes x (or SwiGLU of x when act == 1) as the MMA's
// B image into the scratch `img` (int8_gemm_ws_bytes(N, Kin, M) bytes: the
// image, then the partial sums of the K splits), then one CTA per 128 outputs
// x 256 image rows x K split runs the MMAs; with several splits a last kernel
// adds the partials in split order. Needs Kin % 128 == 0.
size_t int8_gemm_image_bytes(int Kin, int M);
size_t int8_gemm_ws_bytes(int N, int Kin, int M);
int int8_gemm_ksplit(int N, int Kin, int M, int parts);
constexpr int kInt8GemmMinM = 16;  // smallest M that takes the GEMM
cudaError_t launch_int8_gemm(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                             long long x_stride, int act, int M, float* y, long long y_stride, void* img,
                             cudaStream_t s);

// Launch with cudaLaunchKernelExC; pdl = programmatic dependent launch (the
// kernel waits for its predecessor with griddepcontrol.wait).
cudaError_t launch_kernel(const void* f, dim3 grid, dim3 block, int smem, bool pdl, cudaStream_t s, void** args);

// One token's layer in a multi-layer per-slot launch: independent one-token
// blocks of one shape (and one K pair), token t running layer t, each with
// its own input and outputs.
struct MoeLayerPtrs {
    const uint16_t* router_w;
    const uint16_t* gu_codes;
    const uint16_t* gu_rin;
    const uint16_t* gu_rout;
    const uint16_t* dn_codes;
    const uint16_t* dn_rin;
    const uint16_t* dn_rout;
    const int8_t* sh_gu_w8;
    const float* sh_gu_scale;
    const int8_t* sh_dn_w8;
    const float* sh_dn_scale;
    const uint16_t* sh_gate;
    const uint16_t* x;  // fp16 [hidden]
    float* out;         // [hidden]
    int32_t* ids;       // [topk]
    float* w;           // [topk]
};
constexpr int kMlMaxT = 16;  // blocks of one multi-layer launch (the per-slot path's token limit)
struct MlTable {
    MoeLayerPtrs l[kMlMaxT];
};

// Everything the three MoE-block kernels read and write.
struct MoeArgs {
    int T, hidden, inter, E, topk, sh_inter;
    const uint16_t* x;         // fp16 [T][hidden]
    const uint16_t* router_w;  // fp16 [E][hidden]
    const uint16_t* gu_codes;
    int gu_K;
    const uint16_t* gu_rin;
    const uint16_t* gu_rout;
    const uint16_t* dn_codes;
    int dn_K;
    const uint16_t* dn_rin;
    const uint16_t* dn_rout;
    const int8_t* sh_gu_w8;
    const float* sh_gu_scale;
    const int8_t* sh_dn_w8;
    const float* sh_dn_scale;
    const uint16_t* sh_gate;
    uint16_t* logits;  // f16 [T][E]
    float* out;      // [T][hidden]
    int32_t* ids;    // [T][topk]
    float* w;        // [T][topk]
    float* ygu;      // [T*topk][2*inter]
    float* shgu;     // [T][2*sh_inter]
    float* shgate;   // [T]
    float* sh;       // [T][hidden] gated shared-expert output
    int* err;        // set non-zero if a bounded wait gave up (zeroed by the router kernel)
    // residual block on the per-slot path (kFusedNormMaxT tokens at most,
    // hidden <= 2048): the router grid computes x = x_norm from rs_h + rs_add
    // (weightless RMSNorm, the residual_rmsnorm arithmetic) and the gate_up
    // grid stores rs_h += rs_add. x_norm == nullptr: x is an input.
    float* rs_h;
    const float* rs_add;
    float rs_eps;
    uint16_t* x_norm;
    int gu_kt_per_cta;  // filled by the gate_up launcher
    int dn_ksplit;      // filled by the down launcher
    int dn_xt_floats;   // filled by the down launcher: routed input floats of one down rank (multiple of 32)
    // grouped path (T > kSlotModeMaxT): token grouping by expert
    int grp_cap;        // tokens per work item (16, 32, 64 or 128)
    int grp_max_items;  // T*topk/grp_cap + E
    int* grp_counts;    // [E]
    int* grp_offsets;   // [E+1]
    int* grp_poff;      // [E]: first padded position of each expert (runs padded to 4 tokens)
    int4* grp_items;    // [grp_max_items]: {expert, tokens, first B-image row, first index into perm}
    int* grp_nitems;    // [1]
    int* grp_perm;      // [T*topk]: slots t*topk + j sorted stably by expert
    int* grp_ppos;      // [T*topk]: padded position of each slot
    uint8_t* grp_img;   // B image: [in/64 chunks][grp_img_rows][128 B]
    int grp_img_rows;   // 2 * padded positions
    // single-token fused kernel (moe_fused.cu): counters (zeroed by the
    // kernel itself before a grid barrier), split-K partial sums and the
    // finished experts' down outputs, all in the workspace
    unsigned* fz_ctr;   // kFzCtrWords words, zeroed by the router kernel (null: not the fused path)
    float* fz_gu_part;  // [topk][2*inter/128][gu_csize][128]
    float* fz_dn_part;  // [hidden/128][topk][dn_ksplit][128]
    float* fz_dres;     // unused (the finishing CTA keeps the experts' outputs in shared memory)
    long long fz_wait_ns;   // a wait on another CTA gives up after this long
    int fz_skip_publish;    // test hook: the gate_up outputs are never published, so every wait on them gives up
    // per-slot cluster reductions (gate_up, down): rank 0's mbarrier wait
    // gives up after 2^mbar_limit_log2 polls; test hook skip_cluster_arrive:
    // ranks != 0 write nothing into rank 0's shared memory and never arrive,
    // so that wait runs out
    int mbar_limit_log2;
    int skip_cluster_arrive;
    // multi-layer per-slot launch: token t's layer, input and outputs (in the
    // workspace, written by the router kernel; null: one layer, x, out, ids
    // and w as above)
    MoeLayerPtrs* lay;
    int lay_n;  // entries of lay (the launch's tokens)
};

// Largest token count of a grouped work item, and the largest batch that
// runs the per-slot GEMV path instead.
constexpr int kGrpCapMax = 128;
constexpr int kSlotModeMaxT = 16;
// Largest batch whose residual norm runs inside the per-slot router grid
// (measured on GB300 in a 40-block stack: 1 token 25.3 -> 24.6 us per layer;
// 2 tokens were slower fused, 36.0 against 34.2 us, as every router CTA
// normalises every token).
constexpr int kFusedNormMaxT = 1;

// Scratch of the grouped path for T tokens.
struct GroupPlan {
    int cap, max_items, pos_cap;
    size_t int_bytes;  // items (16 B each, first), counts, offsets, poff, nitems, perm, ppos
    size_t img_bytes;         // B image (shared by the gate_up and down projections)
    size_t shared_img_bytes;  // scratch of the shared expert's int8 GEMMs (its own region)
};
GroupPlan group_plan(int T, int topk, int E, int hidden, int inter, int sh_inter);
// top-k (ids, w) and the grouping by expert.
cudaError_t launch_moe_topk_group(const MoeArgs& a, cudaStream_t s);
// top-k, grouping, grouped gate_up and down GEMMs (down output d [T*topk][hidden]).
cudaError_t launch_moe_grouped(const MoeArgs& a, float* d, int num_sms, cudaStream_t s);
// Dense trellis linear on the grouped tensor-core GEMM: one expert, tokens in
// order, items of `cap` tokens; the B image (img, img_rows rows per 64-input
// chunk, img_rows >= 2 * round_up(M, 4)) is written by the prep kernel.
struct DenseArgs {
    const uint16_t* codes;
    int in, out, K, nt_major;
    const void* x;  // [M][in] fp16 or f32
    int x_f32;
    int M, cap;
    const uint16_t* rin;
    const uint16_t* rout;
    const float* bias;  // [out] or null
    float* y;           // [M][out]
    uint8_t* img;
    int img_rows;
    int splits;   // K splits (dense_ksplit); > 1 needs part
    float* part;  // f32 [splits][M][out] partial sums
    int* err;
};
cudaError_t launch_dense_grouped(const DenseArgs& d, cudaStream_t s);
// K splits of the dense grouped GEMM: a fixed function of the shape.
int dense_ksplit(int in, int out, int M, int cap);

// Sets the message escha_last_error() returns on this host thread.
void set_last_error(const char* msg);

// Whole-tile transpose of a code tensor: [in/16][out/16] tiles -> [out/16][in/16].
cudaError_t launch_codes_to_nt_major(const uint16_t* src, int in, int out, int K, uint16_t* dst, cudaStream_t s);

// out = sum_j w * d + sigmoid(gate) * sh
cudaError_t launch_moe_combine(const MoeArgs& a, const float* d, cudaStream_t s);

// h[t] += add[t] (add nullable); then, when x is not null, x[t] = fp16 of the
// weightless RMSNorm of h[t] (summation order fixed in stack.cu).
cudaError_t launch_residual_rmsnorm(float* h, const float* add, int T, int hidden, float eps, uint16_t* x,
                                    cudaStream_t s);

// with_shared (per-slot path): the same grid also computes the shared
// expert's gate_up rows and gate
cudaError_t launch_moe_router(const MoeArgs& a, bool with_shared, cudaStream_t s);
// Multi-layer per-slot launch (a.lay set, a.T = blocks <= kMlMaxT, hidden <=
// 2048): token t's router logits and shared-expert gate_up rows with layer
// t's weights; CTA (0, 0) also stores the table at a.lay for the gate_up and
// down kernels.
cudaError_t launch_moe_router_ml(const MoeArgs& a, const MlTable& tab, cudaStream_t s);
cudaError_t launch_moe_gate_up(const MoeArgs& a, int num_sms, cudaStream_t s);

// One token, two kernels: the per-slot router kernel (logits, the shared
// expert's gate_up rows and gate; it also zeroes the counters below), then
// one cooperative grid for everything else (top-k, gate_up, down, shared
// expert down rows, combine) whose CTAs hand work to each other through
// counters in the workspace (bounded waits). Same splits and summation
// orders as the three per-slot kernels, so the same bits.
// fused_fits: the shape is one the kernel covers (hidden <= 2048, shared
// expert inter <= 512) and its grid fits on the device at once.
constexpr int kFzCtrWords = 320;
struct FusedPlan {
    int n_gate_up, n_extra, n_down, grid, smem;
    size_t ctr_bytes, gu_part_bytes, dn_part_bytes, dres_bytes;
};
bool fused_shape_ok(int hidden, int inter, int E, int topk, int sh_inter);
FusedPlan fused_plan(int hidden, int inter, int E, int topk, int sh_inter);
// cudaSuccess and *fits = false when the grid cannot be resident at once
cudaError_t fused_fits(const FusedPlan& p, int gu_K, int dn_K, int num_sms, bool* fits);
cudaError_t launch_moe_fused(const MoeArgs& a, const FusedPlan& p, cudaStream_t s);

// A sequence of one-token blocks in one cooperative launch (moe_multi.cu):
// independent blocks (each its own input and output) or a residual stack
// (h += previous output, x = RMSNorm(h), block; h += the last output).
constexpr int kMbMaxBlocks = 48;
constexpr int kMbCtrWords = 320;
struct MbBlock {
    const uint16_t* router_w;
    const uint16_t* gu_codes;
    const uint16_t* gu_rin;
    const uint16_t* gu_rout;
    const uint16_t* dn_codes;
    const uint16_t* dn_rin;
    const uint16_t* dn_rout;
    const int8_t* sh_gu_w8;
    const float* sh_gu_scale;
    const int8_t* sh_dn_w8;
    const float* sh_dn_scale;
    const uint16_t* sh_gate;
    int gu_K, dn_K;
    const uint16_t* x;  // independent blocks: the input token (fp16 [hidden])
    float* out;         // independent blocks: the output [hidden]
    int32_t* ids;       // [topk]
    float* w;           // [topk]
};
struct MbPlan {
    int gu_csize, gu_kt, dn_ks;
    // work units per block: router, shared gate_up, gate_up, shared down,
    // gate_up finish, down, combine
    int nR, nS, nG, nX, nF, nD, nC, U;
    int xt_floats, smem;
    size_t ctr_bytes, logits_bytes, xdg_bytes, shgu_bytes, shgate_bytes, sh_bytes, gu_part_bytes, dn_part_bytes, ids_bytes;
};
struct MbHead {
    int n_blocks, hidden, inter, E, topk, sh_inter;
    int stack;       // 1: residual stack on res, xbuf, outbuf
    float* res;      // [hidden] the residual stream h
    float eps;
    uint16_t* xbuf;  // [hidden] the current block's normalised input
    float* outbuf;   // [hidden] the current block's output
    unsigned* ctr;   // [n_blocks][kMbCtrWords], then the work queue
    uint16_t* logits;
    float* xdg;      // [n_blocks][topk][inter]: the slots' transformed down inputs
    float* shgu;
    float* shgate;
    float* sh;
    float* gu_part;
    float* dn_part;
    int* err;
    long long wait_ns;
    int skip_publish;
    int gu_csize, gu_kt, dn_ks;
    int nR, nS, nG, nX, nF, nD, nC, U;
    int xt_floats, smem;
};
// The work queue in segments: units [first, first + count) of block `block`,
// segment after segment; `pos` = the queue position of the segment's first
// unit.
constexpr int kMbMaxSegs = 5 * kMbMaxBlocks + 8;
struct MbSeg {
    short block;
    short first;
    short count;
    short pad;
    int pos;
};
struct MbArgs {
    MbHead h;
    int n_segs;
    MbSeg seg[kMbMaxSegs];
    MbBlock blk[kMbMaxBlocks];
};
bool multi_shape_ok(int hidden, int inter, int E, int topk, int sh_inter);
MbPlan multi_plan(int n_blocks, int hidden, int inter, int E, int topk, int sh_inter);
// CTAs of the cooperative grid: every CTA slot of the device (smem bytes per CTA)
cudaError_t multi_grid(int num_sms, int smem, int* grid);
cudaError_t launch_moe_multi(const MbArgs& m, int grid, cudaStream_t s);

// Input splits of the per-slot path for T tokens: gate_up CTAs per output
// block (gu_csize, each over gu_kt_per_cta tile rows) and down splits per
// expert (dn_ksplit). A fixed function of the shape, so a result does not
// depend on the device; the single-token fused kernel takes the same splits
// and so gives the same bits.
struct SlotPlan {
    int gu_csize, gu_kt_per_cta, dn_ksplit;
};
SlotPlan slot_plan(int T, int hidden, int inter, int topk);
cudaError_t launch_moe_down(const MoeArgs& a, int num_sms, cudaStream_t s);

}  // namespace escha
