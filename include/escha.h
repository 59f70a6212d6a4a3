/*
 * escha.h - C ABI of the GB300 (sm_103a) trellis MoE expert library.
 *
 * The library computes the MoE expert path of an Escha-W2 ("eschamoe")
 * 2/3-bit Qwen3.6-35B-A3B-style layer with the packed trellis codes decoded
 * inside the GEMV, never materialised as dense weights, plus the int8 w8a16
 * matvec/GEMM of the dense layers.
 *
 * Sources (by page):
 *   [PR694]  hipfire PR #694 "Escha-W2 port: 2-bit trellis decoded in the GEMV"
 *            (summary section "What it is" and the PR's commit messages);
 *   [MLX]    model card "dogfoodai/Qwen3.6-35B-A3B-Escha-W2-trellis-mlx",
 *            table "Exactness of every tensor";
 *   [CARD]   model card "EschaLabs/Qwen3.6-35B-A3B-Escha-W2", "Format notes".
 *
 * Conventions shared by every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them. fp16 / bf16 tensors are passed as their
 *     16-bit patterns (uint16_t). All tensors are dense row-major, contiguous.
 *   - Tensor pointers must be 16-byte aligned (ESCHA_E_ALIGN otherwise).
 *   - `stream` is a cudaStream_t (0 = the legacy default stream). Work is
 *     only enqueued on it; no call synchronises the host.
 *   - Scratch memory comes from the caller's workspace `ws` of `ws_bytes`
 *     bytes; each entry point has a *_workspace() query. A larger workspace
 *     is accepted. The library allocates no device memory.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the kernel enqueued before it on the stream is still
 *     running, and it reads weights (code tensors, rin / rout, int8
 *     matrices, scales, router weights) before waiting for that kernel.
 *     Activations and outputs are only touched after the wait. Some of the
 *     library's kernels release the kernel after them before their own wait
 *     (the routers, and the one-token GEMV that decodes its weights ahead),
 *     so a chain of library calls does not order weight writes: weights must
 *     be written by work that is ordered before the call by a stream point
 *     these launches cannot pass (a memory copy, an event record, a kernel
 *     launched without programmatic dependent launch, or host
 *     synchronisation) rather than by another call of this library.
 *   - Every argument is validated before anything is enqueued. On error the
 *     call returns a negative ESCHA_E_* code, enqueues nothing, and
 *     escha_last_error() describes the problem. Asynchronous device faults
 *     surface at the caller's next synchronisation, as for any CUDA work.
 *   - Trellis code tensors: uint16 [in/16][out/16][16*K] (tile grid stored
 *     with the input-tile index outermost), K = bits per weight in {2, 3},
 *     equal to the code tensor's last dimension / 16 [PR694 commit "Read
 *     Escha's test suite"; CARD "Format notes"]. Each 16x16 tile's 16*K words
 *     form one cyclic bit stream (most significant bit of each word first);
 *     weight t = 16*r + q of the tile (r = input row, q = output column)
 *     takes the 16-bit window starting at bit t*K as its trellis state, and
 *     the state decodes through the "cbA" hash
 *        r = ((s * 0xCBAC1FED) & 0x8FFF8FFF) ^ 0x3B603B60,
 *        w = fp16_rne(fp16(r & 0xffff) + fp16(r >> 16))
 *     [PR694 "What it is"; MLX "Exactness of every tensor"].
 *   - Rotations: each trellis projection computes
 *        y = rout * H(W^T H(rin * x))
 *     with H the blockwise Sylvester Hadamard-128 scaled by 1/sqrt(128) on
 *     both sides [PR694 "What it is"; MLX note on mx.hadamard_transform];
 *     rout is the final multiply, so channels whose rout is 0 (the per-expert
 *     prune mask of gate_up) come out exactly +-0 [PR694 commits "Second
 *     review pass" and "Naive one-thread-per-block butterfly"].
 */
#ifndef ESCHA_H
#define ESCHA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------- */
#define ESCHA_OK 0
#define ESCHA_E_ARG (-1)       /* null pointer, bad enum, non-positive count */
#define ESCHA_E_SHAPE (-2)     /* dimension not a multiple of 16 / 128, too large */
#define ESCHA_E_K (-3)         /* bits per weight not 2 or 3 */
#define ESCHA_E_WORKSPACE (-4) /* workspace smaller than *_workspace() */
#define ESCHA_E_ALIGN (-5)     /* pointer not 16-byte aligned */
#define ESCHA_E_CUDA (-6)      /* CUDA error while enqueueing (launch/config) */
#define ESCHA_E_DEVICE (-7)    /* current device is not an sm_103 GPU */
#define ESCHA_E_CKPT (-8)      /* checkpoint breaks the escha leaf contract */
#define ESCHA_E_IO (-9)        /* shard missing, unreadable or not safetensors */

/* ---- element types --------------------------------------------------- */
#define ESCHA_F16 1
#define ESCHA_BF16 2
#define ESCHA_F32 3

/* Message describing the last error returned on this host thread. */
const char* escha_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
int escha_version(void);

/* ---- trellis decode (diagnostic export) ----------------------------------
 * Decodes a whole code tensor to dense fp16 weights, W[in][out] (uint16 bit
 * patterns), for the bit-exact decode check [PR694 commit "Task 7 (G2): one-
 * shot decode of Escha-W2 packed trellis tiles"]. Not part of the hot path:
 * the GEMV entry points never materialise W.
 *   codes  uint16 [in/16][out/16][16*K]
 *   in,out multiples of 16;  K in {2, 3}
 *   W      uint16 [in][out] output
 * Errors: ESCHA_E_ARG (null), ESCHA_E_SHAPE, ESCHA_E_K, ESCHA_E_ALIGN. */
int escha_trellis_decode(const uint16_t* codes, int in, int out, int K, uint16_t* W, void* stream);

/* ---- one trellis-coded projection ----------------------------------------
 * y[b] = rout * H(W^T H(rin * x[b])) for b < batch, all tokens sharing the
 * one weight [PR694 commit "EschaProj holds what a trellis weight needs";
 * the projection as "H128-in -> trellis GEMV -> H128-out"]. Accumulation is
 * fp32; decoded weights are exact fp16.
 *   codes   uint16 [in/16][out/16][16*K], K in {2, 3}
 *   in,out  multiples of 128 (whole Hadamard blocks), in <= 65536
 *   x       [batch][in], x_dtype ESCHA_F16 or ESCHA_F32
 *   rin     fp16 [in];  rout fp16 [out]
 *   y       f32 [batch][out] output
 *   ws      escha_trellis_gemv_workspace(in, out, K, batch) bytes (may be 0)
 * Errors: ESCHA_E_ARG, ESCHA_E_SHAPE, ESCHA_E_K, ESCHA_E_ALIGN,
 *         ESCHA_E_WORKSPACE, ESCHA_E_CUDA, ESCHA_E_DEVICE. */
size_t escha_trellis_gemv_workspace(int in, int out, int K, int batch);
int escha_trellis_gemv(const uint16_t* codes, int in, int out, int K, const void* x, int x_dtype, int batch,
                       const uint16_t* rin, const uint16_t* rout, float* y, void* ws, size_t ws_bytes,
                       void* stream);

/* ---- tile-grid transpose (load time) --------------------------------------
 * Moves whole tiles of a code tensor from the stored kt-major grid
 * [in/16][out/16][16*K] to the nt-major grid [out/16][in/16][16*K], so the
 * tiles that one output tile column walks through sit next to each other
 * [PR694 commit on the nt-major tile grid: transposed at load, payload kept
 * verbatim, tile contents untouched, every decoded weight identical].
 *   codes  uint16 source, dst uint16 destination of the same size; the two
 *          must not overlap (ESCHA_E_ARG). Both caller-owned, 16-byte aligned.
 *   in,out multiples of 16;  K in {2, 3}
 * dst is a weight for the calls that read it: order the transpose before
 * them by a stream point that programmatic launches cannot pass (see the
 * conventions above), e.g. an event record or host synchronisation.
 * Errors: ESCHA_E_ARG, ESCHA_E_SHAPE, ESCHA_E_K, ESCHA_E_ALIGN, ESCHA_E_CUDA,
 *         ESCHA_E_DEVICE. */
int escha_codes_to_nt_major(const uint16_t* codes, int in, int out, int K, uint16_t* dst, void* stream);

/* ---- dense trellis linear ---------------------------------------------------
 * y[m] = rout * H(W^T H(rin * x[m])) + bias for m < M: one dense projection
 * served as the one-expert case of the expert kernels [PR694 commits
 * "EschaProj holds what a trellis weight needs" (one expert, ids all zero)
 * and on batched prefill grouping all slots of a dense linear into a single
 * group, so each weight is read once per batch rather than once per slot].
 * The bias is the dense export's additive per-projection output bias [PR694
 * commit adding the escha dense export's biases in decode and prefill]: it is
 * added after the output transform, so for gate/up it lands before any
 * activation the caller applies, and for down/o_proj it may equally be added
 * onto the residual afterwards.
 * M <= 2 (M <= 12 when in * out <= 2^23) runs the fused per-token decode
 * GEMV (weights decoded once per 1, 2 or 4 tokens); larger M writes an fp16
 * hi/lo image of H(rin * x) and runs the tcgen05 tensor-core GEMM with all
 * tokens in one group (weights decoded once per 16..128 tokens), its inputs
 * split over up to 16 CTAs when output blocks x items leave SMs idle (the
 * partial sums are added in a fixed order). Accumulation is fp32 on both
 * routes; the route and the split are fixed functions of (in, out, M).
 *   codes    uint16, kt-major [in/16][out/16][16*K] (nt_major = 0) or
 *            nt-major [out/16][in/16][16*K] (nt_major = 1, see
 *            escha_codes_to_nt_major); K in {2, 3}
 *   in,out   multiples of 128, in <= 65536
 *   x        [M][in], x_dtype ESCHA_F16 or ESCHA_F32;  1 <= M <= 65536
 *   rin      fp16 [in];  rout fp16 [out];  bias f32 [out] or NULL
 *   y        f32 [M][out] output
 *   ws       escha_dense_linear_workspace(in, out, K, M) bytes, caller-owned;
 *            its first 4 bytes are a status word, set to 0 by the call and
 *            non-zero if a kernel gave up a bounded wait (outputs invalid).
 * All pointers 16-byte aligned. Errors: ESCHA_E_ARG, ESCHA_E_SHAPE,
 * ESCHA_E_K, ESCHA_E_ALIGN, ESCHA_E_WORKSPACE, ESCHA_E_CUDA, ESCHA_E_DEVICE;
 * on error nothing is enqueued. */
size_t escha_dense_linear_workspace(int in, int out, int K, int M);
int escha_dense_linear(const uint16_t* codes, int in, int out, int K, int nt_major, const void* x, int x_dtype, int M,
                       const uint16_t* rin, const uint16_t* rout, const float* bias, float* y, void* ws,
                       size_t ws_bytes, void* stream);

/* ---- checkpoint loader (safetensors shards of an Escha-W2 export) ---------
 * A shard is an 8-byte little-endian header length N, N bytes of JSON
 * ({name: {"dtype", "shape", "data_offsets": [begin, end]}}, begin/end
 * relative to the data after the header) and the data. Opening checks the
 * escha leaf contract [PR694 commit reading Escha's test suite; model card
 * "EschaLabs/Qwen3.6-35B-A3B-Escha-W2", section "Format notes"]:
 *   - a coded projection <prefix> has the required leaves <prefix>.escha_code
 *     (I16/U16 [in/16][out/16][16*K], or [E][..] for stacked experts),
 *     .escha_rin (F16 [in] / [E][in]) and .escha_rout (F16 [out] / [E][out]);
 *     a missing one is ESCHA_E_CKPT naming it;
 *   - .escha_s_in, .escha_s_out (all ones as shipped: never applied) and
 *     .escha_config (int32[9], informational) are optional;
 *   - any other leaf escha_* (e.g. escha_rotation_theta, a rotation variant
 *     the format anticipates) is ESCHA_E_CKPT naming it;
 *   - K = (last dimension of escha_code) / 16, K in {2, 3};
 *   - <prefix>.bias (F32/F16/BF16 [out]) is the dense export's additive
 *     output bias [PR694 commit on the dense export's biases]; the dense
 *     coded projections of one layer ("...layers.<n>.") carry biases all
 *     together or not at all, else ESCHA_E_CKPT.
 * A tensor name present in two shards, offsets that disagree with the shape
 * or an unknown dtype are rejected too. The handle owns only host memory. */
typedef struct escha_ckpt escha_ckpt;

typedef struct escha_proj_info {
    char prefix[256];    /* tensor names without ".escha_code" etc. */
    int K;               /* bits per weight, from the code tensor's shape */
    int n_experts;       /* 0: one dense projection; E: E stacked experts */
    int in, out;
    int has_bias;        /* <prefix>.bias present (dense projections only) */
    int has_s_in, has_s_out, has_config;
    int scales_all_ones; /* s_in / s_out absent or all ones */
    int config_k;        /* escha_config[1] when present (reported, not trusted), else -1 */
} escha_proj_info;

typedef struct escha_tensor_info {
    char dtype[8];       /* safetensors dtype: "F16", "BF16", "F32", "I16", "U16", "I8", "I32", ... */
    int ndim;
    long long shape[8];
    size_t nbytes;
} escha_tensor_info;

/* Opens and validates n_paths shards; *out receives a handle to close with
 * escha_ckpt_close. Errors: ESCHA_E_ARG, ESCHA_E_IO, ESCHA_E_CKPT. */
int escha_ckpt_open(const char* const* paths, int n_paths, escha_ckpt** out);
void escha_ckpt_close(escha_ckpt* c);
/* Coded projections, in name order. */
int escha_ckpt_num_projections(const escha_ckpt* c);
int escha_ckpt_projection(const escha_ckpt* c, int i, escha_proj_info* info);
/* Any tensor by name (router weights, int8 matrices and their scales, ...). */
int escha_ckpt_tensor_info(const escha_ckpt* c, const char* name, escha_tensor_info* info);
/* Its bytes, as stored, into dst (dst_device 0: host memory, 1: device
 * memory through `stream`, synchronised before return). dst_bytes must be at
 * least info.nbytes. Errors: ESCHA_E_ARG, ESCHA_E_IO, ESCHA_E_CUDA. */
int escha_ckpt_read(const escha_ckpt* c, const char* name, void* dst, size_t dst_bytes, int dst_device, void* stream);
/* Projection i's leaves into caller-owned device buffers: codes (the code
 * tensor's size; nt_major = 1 moves a dense projection's tiles to the
 * nt-major grid at load, see escha_codes_to_nt_major; experts stay
 * kt-major), rin / rout fp16, and, when bias is not NULL, the bias widened
 * to f32 [out] (ESCHA_E_ARG if the projection has none). Synchronises
 * `stream` before returning. Errors: ESCHA_E_ARG, ESCHA_E_IO, ESCHA_E_CUDA. */
int escha_ckpt_load_projection(const escha_ckpt* c, int i, uint16_t* codes, uint16_t* rin, uint16_t* rout,
                               float* bias, int nt_major, void* stream);

/* ---- one MoE block ------------------------------------------------------
 * For each token b of x [T][hidden] (fp16):
 *   logits = f16(x[b] . Wg[e]) for every expert e (f32 sums in a fixed
 *            order, rounded to f16 before top-k [PR694 commit "Executed the
 *            moeblk golden against real shipped layer-0 weights"]);
 *   ids    = the topk largest logits, ties to the lower expert id, ordered
 *            by (logit desc, id asc); w = softmax over those topk logits;
 *   h_j    = SwiGLU(gate_up_j(x[b])) with the gate the FIRST half [PR694
 *            commit "The accumulation loop treated a zero activation"];
 *   out[b] = sum_j w_j * down_j(h_j) + sigmoid(g . x[b]) * shared(x[b]),
 *            the sum over j in slot order, the shared expert int8 w8a16.
 * K is uniform per projection across experts (one code tensor per layer and
 * projection [PR694 commit "Converted the real 12.30 GB checkpoint"]).
 * Pointers of an absent shared expert may be null when sh_inter == 0. */
typedef struct escha_moe_layer {
    int hidden;    /* multiple of 256, <= 8192 */
    int inter;     /* routed expert intermediate size, multiple of 128, <= 8192 */
    int n_experts; /* 1..256 */
    int topk;      /* 1..8, <= n_experts */
    const uint16_t* router_w; /* fp16 [E][hidden] */
    /* routed experts, gate_up: in = hidden, out = 2*inter */
    const uint16_t* gu_codes; /* [E][hidden/16][2*inter/16][16*gu_K] */
    int gu_K;
    const uint16_t* gu_rin;  /* fp16 [E][hidden] */
    const uint16_t* gu_rout; /* fp16 [E][2*inter] (prune mask as zeros) */
    /* routed experts, down: in = inter, out = hidden */
    const uint16_t* dn_codes; /* [E][inter/16][hidden/16][16*dn_K] */
    int dn_K;
    const uint16_t* dn_rin;  /* fp16 [E][inter] */
    const uint16_t* dn_rout; /* fp16 [E][hidden] */
    /* shared expert (int8 w8a16, dequant = f32 scale * w8 per row [MLX]) */
    int sh_inter; /* 0 = no shared expert; else multiple of 16, <= 8192 */
    const int8_t* sh_gu_w8; /* [2*sh_inter][hidden] */
    const float* sh_gu_scale; /* [2*sh_inter] */
    const int8_t* sh_dn_w8; /* [hidden][sh_inter] */
    const float* sh_dn_scale; /* [hidden] */
    const uint16_t* sh_gate;  /* fp16 [hidden], sigmoid gate of the shared expert */
} escha_moe_layer;

/* The first 4 bytes of the workspace hold a status word that the call sets
 * to 0 when its first kernel starts and to a non-zero value if a kernel had
 * to give up waiting on a cluster peer or, at one token, on another CTA of
 * the fused kernel (it then returns instead of hanging; the outputs of that
 * call are invalid). Read it after synchronising.
 * One token can also run (escha_debug_set_moe_route(2); the layer must have
 * hidden <= 2048 and shared-expert inter <= 512, and the grid must fit on the
 * device at once) as TWO kernels: the router kernel, then one cooperative
 * kernel in which top-k, gate_up, down, the shared expert's down rows and the
 * combine hand work to each other through counters kept in the workspace;
 * the router kernel zeroes them, so nothing in the workspace has to start at
 * zero. Its input splits and summation orders are those of the per-slot
 * kernels, so the results are bit for bit the same. It is not the default:
 * a cooperative grid is scheduled only when all of it fits, so it cannot
 * overlap the kernels around it, and on GB300 a single block took 22.05 us
 * this way against 21.4 us for the per-slot kernels. Calls that share a
 * workspace must not overlap on the GPU (as for every path).
 * Larger batches (the grouped path) run the int8 shared expert on a second
 * stream beside the routed kernels: a non-blocking stream and two events per
 * host thread and device, created by the first such call made outside a
 * stream capture and reused after (calls inside a capture fork and join
 * through them, and are captured as parallel branches); until they exist,
 * the shared expert runs on `stream` itself. Results are identical either way.
 * Batches of up to 16 tokens run fused decode GEMVs per (token, expert);
 * larger batches group the tokens by expert and decode each expert's codes
 * once per work item of up to 128 of its tokens, feeding tcgen05
 * tensor-core MMAs.
 *   x       fp16 [T][hidden];  1 <= T <= 8192
 *   out     f32 [T][hidden] output
 *   ids_out int32 [T][topk] output, may be null
 *   w_out   f32 [T][topk] output, may be null
 *   ws      escha_moe_block_workspace(L, T) bytes */
size_t escha_moe_block_workspace(const escha_moe_layer* L, int T);
int escha_moe_block(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out, float* w_out,
                    void* ws, size_t ws_bytes, void* stream);

/* Residual MoE block: h += add (add nullable), x = f16_rne(h * inv) with the
 * weightless RMSNorm of escha_residual_rmsnorm, then escha_moe_block on x:
 * bit for bit the same h, x, out, ids and weights as those two calls in a
 * row. On one token with hidden <= 2048 (batch-1 decode of the
 * Qwen3.6-35B-A3B layer) the norm runs inside the block's router grid: one
 * kernel boundary fewer per layer of a decode stack; otherwise the norm
 * kernel runs first.
 *   h    f32 [T][hidden], updated in place;  add f32 [T][hidden] or NULL
 *   eps  >= 0;  x fp16 bits [T][hidden], written (the block's input)
 *   out may be the same buffer as add (the previous block's output); x must
 *   not overlap h, add or out. Other arguments, workspace and errors as
 *   escha_moe_block. */
int escha_moe_block_resid(const escha_moe_layer* L, float* h, const float* add, float eps, uint16_t* x, int T,
                          float* out, int32_t* ids_out, float* w_out, void* ws, size_t ws_bytes, void* stream);

/* Measurement export: escha_moe_block that also records four caller-created
 * CUDA events (cudaEvent_t, any of them may be null) on `stream`: events[0]
 * before the router kernel (on up to 16 tokens it also computes the shared
 * expert's gate_up rows and gate), [1] after it, [2] after the routed gate_up
 * kernel, [3] after the down/combine kernel. Recording events between the kernels serialises them (no
 * programmatic overlap), so each interval is one kernel's duration. When one
 * token runs on the fused path, [0] is recorded before the router kernel,
 * [1] after it, and [2] and [3] after the cooperative expert kernel. Same
 * results and errors as escha_moe_block. */
int escha_moe_block_timed(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out,
                          float* w_out, void* ws, size_t ws_bytes, void* stream, void* const* events);

/* ---- many one-token blocks in few launches ----------------------------
 * The decode step of a model runs its MoE blocks one after another for one
 * token. Launched one block at a time, each block pays its kernels' grid
 * boundaries, which at one token cost more than the decode itself. The
 * layers must share hidden (a multiple of 256, <= 2048), inter (2*inter/128
 * <= 32), n_experts, topk and sh_inter (<= 512); ESCHA_E_SHAPE otherwise.
 *
 * escha_moe_blocks: independent blocks, block i on its own token:
 *   x[i] fp16 [hidden] -> out[i] f32 [hidden]; ids_out / w_out: arrays of
 *   per-block [topk] outputs, or NULL (either the array or an entry).
 *   Up to 16 blocks whose layers share gu_K and dn_K run on the per-slot
 *   kernels (ESCHA_PATH_SLOT): one launch each of the router, gate_up and
 *   down/combine kernels over every block's slots, token t with layer t,
 *   exactly as escha_moe_block runs n tokens of one layer (so n copies of
 *   one layer give bit for bit escha_moe_block's output for those n
 *   tokens); the input splits are those of n tokens, so the bits differ
 *   from n one-token calls (within the block's tolerance). Otherwise
 *   (more blocks, or K differing between layers) the blocks run in the
 *   sequence kernel below (ESCHA_PATH_SEQUENCE), where every block gives bit
 *   for bit escha_moe_block's one-token output; a block's router and
 *   gate_up work overlaps the previous block's down.
 *   escha_moe_blocks_path tells which (or a negative error code);
 *   escha_debug_set_blocks_route(0 by shape, 1 per-slot kernels (ESCHA_E_SHAPE
 *   when they do not cover the blocks), 2 sequence kernel) forces one, for
 *   tests (process-wide, read when a call is enqueued).
 *
 * The sequence kernel runs up to 48 blocks in ONE cooperative launch (every
 * CTA resident): the CTAs take work units (router rows, the shared expert's
 * rows, gate_up and down pieces of each routed expert) from one queue and
 * hand results to each other through counters in the workspace; every wait
 * is bounded (the status word reports a wait that ran out; see
 * escha_debug_set_fused_wait). gu_K / dn_K may differ per layer.
 *
 * escha_moe_stack: a residual stack, the blocks of one decode step, in the
 * sequence kernel:
 *   for each block i: h += out_buf (i > 0), x_buf = fp16 RMSNorm(h) (the
 *   weightless norm of escha_residual_rmsnorm, same arithmetic), out_buf =
 *   block_i(x_buf); at the end h += out_buf. The same h, x_buf and out_buf
 *   bits as escha_moe_block_resid per block followed by
 *   escha_residual_rmsnorm(h, out_buf, x_out = NULL).
 *   h f32 [hidden] (updated), x_buf fp16 [hidden], out_buf f32 [hidden]
 *   (written; h, x_buf, out_buf must not overlap); ids_out int32 and w_out
 *   f32 [n_blocks][topk] or NULL.
 * Workspace: escha_moe_seq_workspace(layers, n_blocks) bytes (independent of
 * the call's kind); nothing in it has to start at zero. */
size_t escha_moe_seq_workspace(const escha_moe_layer* const* layers, int n_blocks);
int escha_moe_blocks_path(const escha_moe_layer* const* layers, int n_blocks);
int escha_debug_set_blocks_route(int mode);
int escha_moe_blocks(const escha_moe_layer* const* layers, int n_blocks, const uint16_t* const* x, float* const* out,
                     int32_t* const* ids_out, float* const* w_out, void* ws, size_t ws_bytes, void* stream);
/* Measurement export: escha_moe_blocks that also records four caller-created
 * CUDA events (any may be null) on `stream`: on the per-slot route [0]
 * before the router kernel, [1] after it, [2] after the gate_up kernel, [3]
 * after the down/combine kernel (recording between the kernels serialises
 * them, so each interval is one kernel's duration); on the sequence route
 * [0] before its launch and [1]..[3] after it. Same results and errors as
 * escha_moe_blocks. */
int escha_moe_blocks_timed(const escha_moe_layer* const* layers, int n_blocks, const uint16_t* const* x,
                           float* const* out, int32_t* const* ids_out, float* const* w_out, void* ws, size_t ws_bytes,
                           void* stream, void* const* events);
int escha_moe_stack(const escha_moe_layer* const* layers, int n_blocks, float* h, float eps, uint16_t* x_buf,
                    float* out_buf, int32_t* ids_out, float* w_out, void* ws, size_t ws_bytes, void* stream);

/* Which kernels escha_moe_block(L, T) runs on the current device (with the
 * route setting below): ESCHA_PATH_FUSED (the router kernel and one
 * cooperative expert kernel, T = 1),
 * ESCHA_PATH_SLOT (router, gate_up and down/combine kernels per (token,
 * expert), T <= 16) or ESCHA_PATH_GROUPED (tokens grouped by expert on the
 * tensor cores, T > 16); a negative ESCHA_E_* code for an invalid layer. */
#define ESCHA_PATH_FUSED 1
#define ESCHA_PATH_SLOT 2
#define ESCHA_PATH_GROUPED 3
#define ESCHA_PATH_SEQUENCE 4
int escha_moe_block_path(const escha_moe_layer* L, int T);

/* Diagnostic exports (tests and measurements; not part of the hot path).
 * escha_debug_set_moe_route: how one-token blocks run in this process:
 *   0 (default) or 1 = the three per-slot kernels, 2 = the router kernel and
 *   the cooperative expert kernel (ESCHA_E_SHAPE when the layer or the device
 *   does not allow it). ESCHA_E_ARG for other modes.
 * escha_debug_set_fused_wait: the fused kernel's bound on each wait for
 *   another CTA (wait_ns in [1e3, 6e10], default 2e9) and, for tests, a hook
 *   (skip_publish = 1) that keeps every expert's gate_up outputs from being
 *   published, so every down unit's wait for them runs out: the kernel then
 *   ends with the status word set to 5 instead of hanging. Both settings are
 *   process-wide and read when a call is enqueued.
 * escha_debug_set_cluster_wait: the per-slot kernels' cluster reductions
 *   (gate_up, down/combine), where ranks != 0 store their partial sums into
 *   rank 0's shared memory and arrive on its mbarrier: rank 0's wait gives
 *   up after 2^poll_limit_log2 polls (poll_limit_log2 in [8, 30], default
 *   24), sets the status word (1: gate_up, 2: down) and goes on. For tests,
 *   skip_arrive = 1 makes ranks != 0 write nothing into rank 0's shared
 *   memory and never arrive, so every such wait runs out; the outputs are
 *   then invalid and the status word says so. Process-wide, read when a call
 *   is enqueued; ESCHA_E_ARG for values out of range. */
int escha_debug_set_cluster_wait(int poll_limit_log2, int skip_arrive);
int escha_debug_set_moe_route(int mode);
int escha_debug_set_fused_wait(long long wait_ns, int skip_publish);

/* ---- MoE block with built-in scratch (no allocation by the caller) -------
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory when they run the block (an operator
 * plugin in a framework that owns all device allocations, work issued while a
 * stream is captured into a CUDA graph in a mode that forbids cudaMalloc, a
 * process whose memory is fixed at start-up). Same computation, arguments,
 * outputs and errors as escha_moe_block, minus the workspace: the scratch is a
 * device buffer of ESCHA_NOALLOC_SCRATCH_BYTES built into the library, which
 * every GPU that loads the library holds until the process exits.
 *   - Calls whose escha_moe_block_workspace(L, T) exceeds the buffer are
 *     rejected with ESCHA_E_WORKSPACE before anything is enqueued: for a
 *     hidden-2048, inter-512, 256-expert, top-8 layer, T <= 16 fits (the
 *     per-slot path, 731 KB at T = 16); the grouped path of T >= 17 needs
 *     several MB (its B image) and is rejected.
 *   - The first call on a device looks the buffer's device address up
 *     (cudaGetSymbolAddress), and so does the first call after the device's
 *     context changed (cudaDeviceReset loads the library's module anew); make
 *     such a call before any stream capture.
 *   - All calls on a device share the one buffer, which keeps the last call's
 *     contents: calls that can overlap on the GPU (different streams without
 *     ordering between them) race and corrupt each other's results. Nothing
 *     in the buffer needs to be zero beforehand.
 *   - The library allocates nothing for this call. */
#define ESCHA_NOALLOC_SCRATCH_BYTES (2u << 20)
int escha_moe_block_noalloc(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out,
                            float* w_out, void* stream);

/* ---- residual stream between MoE blocks ----------------------------------
 * h[t][i] += add[t][i] (add nullable), then, when x_out is not null,
 * x_out[t][i] = f16_rne(h[t][i] * inv_t) with inv_t = 1 / sqrt(mean_i(h^2) +
 * eps): a weightless RMSNorm, the input of the next block. In the pages'
 * model every escha projection takes a plain RMS-normed input ([PR694],
 * commit on escha_run_proj / escha_run_resid); random weights without a norm
 * drive block outputs out of the fp16 range, so a stack of synthetic blocks
 * needs one. The fp16 rounding feeds the router, so
 * the arithmetic is fixed: f32 multiply then add of h^2 per thread t of 256
 * over i = t, t+256, ... ascending; xor butterfly 16..1 within each warp, the
 * 8 warp sums in order; mean = sum / hidden, IEEE sqrt and division.
 *   h      f32 [T][hidden], updated in place;  add f32 [T][hidden] or NULL
 *   x_out  fp16 bits [T][hidden] or NULL (then only the add is done)
 *   hidden 1..8192, eps >= 0 */
int escha_residual_rmsnorm(float* h, const float* add, int T, int hidden, float eps, uint16_t* x_out, void* stream);

/* ---- routing diagnostic -------------------------------------------------
 * Diagnostic export, not used by the hot path: the router, top-k and
 * grouping steps of escha_moe_block (the grouped path's kernels, run for any
 * T) with their intermediate results copied out, for bit-exact checks.
 *   logits_out  fp16 bits [T][E]: f16_rne of the router dot products, summed in
 *               the order stated for escha_moe_block (nullable)
 *   ids_out     int32 [T][topk], w_out f32 [T][topk] (required, 4-byte aligned)
 *   counts_out  int32 [E]: slots per expert (nullable)
 *   offsets_out int32 [E+1]: exclusive prefix sum of counts (nullable)
 *   perm_out    int32 [T*topk]: the slots t*topk + j in expert order, stable in
 *               slot order within an expert (nullable)
 * Workspace from escha_moe_route_workspace(L, T); layer checks and errors as
 * escha_moe_block. Grouping as in [PR694], commits on the grouped prefill GEMM
 * (per-expert offsets and a slot permutation feeding one GEMM per expert). */
size_t escha_moe_route_workspace(const escha_moe_layer* L, int T);
int escha_moe_route(const escha_moe_layer* L, const uint16_t* x, int T, uint16_t* logits_out, int32_t* ids_out,
                    float* w_out, int32_t* counts_out, int32_t* offsets_out, int32_t* perm_out, void* ws,
                    size_t ws_bytes, void* stream);

/* ---- int8 w8a16 ----------------------------------------------------------
 * y[m][o] = sum_i (scale[o] * W[o][i]) * x[m][i], f32 output, with the int8
 * weights used as stored (no dequantised copy) [MTPLX PR #242 "serve Qwen3.6-35B-A3B-Escha-W2 natively", table
 * "Improvements": int8 non-experts, fused matvec, no dequant at load; MLX
 * "Exactness of every tensor": dequant = f32 scale*w8]. M < 16 (or Kin not a
 * multiple of 128) runs the CUDA-core matvec; M >= 16 with Kin % 128 == 0 runs
 * the tensor-core GEMM (int8 converted exactly to the activation's 16-bit type;
 * f32 activations split into bf16 hi + lo), whose scratch (B image and K-split
 * partial sums) comes from the workspace: ws_bytes >= int8_w8a16_workspace(N,
 * Kin, M), else ESCHA_E_WORKSPACE.
 *   W      int8 [N][Kin];  scales f32 [N]
 *   N      >= 1;  Kin multiple of 16, <= 51200 (<= 51168 on the matvec path
 *          with M >= 2)
 *   x      [M][Kin], x_dtype ESCHA_BF16, ESCHA_F16 or ESCHA_F32
 *   y      f32 [M][N] output */
size_t int8_w8a16_workspace(int N, int Kin, int M);
int int8_w8a16_matvec(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype, int M,
                      float* y, void* ws, size_t ws_bytes, void* stream);

/* Diagnostic export: out[o][i] = fl32(scale[o] * W[o][i]) (one IEEE f32
 * multiply), for the bit-exact dequant check. Not used by the hot path. */
int int8_w8a16_dequant(const int8_t* W, const float* scales, int N, int Kin, float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ESCHA_H */
