// C ABI of the trellis MoE library: argument validation, workspace layout and
// kernel launches. Every check runs before anything is enqueued; errors are
// returned as ESCHA_E_* codes with a thread-local message.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "escha.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

void escha::set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

namespace {

struct DeviceInfo {
    int ok = -1;  // -1 unknown, 0 not sm_103, 1 fine
    int num_sms = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

// Current device must be an sm_103 part (the kernels are built for sm_103a only).
int device_check(int* num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(ESCHA_E_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.ok < 0) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        d.ok = (major == 10 && minor == 3) ? 1 : 0;
        d.num_sms = sms;
        if (!d.ok) {
            return fail(ESCHA_E_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                        minor);
        }
    }
    if (!d.ok) return fail(ESCHA_E_DEVICE, "device %d is not an sm_103 GPU", dev);
    *num_sms = d.num_sms;
    return ESCHA_OK;
}

int cuda_status(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ESCHA_OK;
}

size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

// Diagnostic settings (escha_debug_*): the route of one-token blocks (0 and
// 1 the three per-slot kernels, measured faster for a single block; 2 the
// router kernel plus the cooperative expert kernel, or an error where that
// path does not apply) and the cooperative kernel's wait limit and test hook.
std::atomic<int> g_moe_route_mode{0};
// escha_moe_blocks: 0 = by shape, 1 = the per-slot kernels over all blocks, 2 = the sequence kernel
std::atomic<int> g_blocks_route{0};
std::atomic<long long> g_fz_wait_ns{2000000000ll};
std::atomic<int> g_fz_skip_publish{0};
std::atomic<int> g_mbar_limit_log2{24};
std::atomic<int> g_skip_cluster_arrive{0};

int check_trellis(const uint16_t* codes, int in, int out, int K, int mult, const char* name) {
    if (!codes) return fail(ESCHA_E_ARG, "%s: codes is null", name);
    if (!aligned16(codes)) return fail(ESCHA_E_ALIGN, "%s: codes not 16-byte aligned", name);
    if (K != 2 && K != 3) return fail(ESCHA_E_K, "%s: K=%d, must be 2 or 3", name, K);
    if (in <= 0 || out <= 0 || in % mult || out % mult)
        return fail(ESCHA_E_SHAPE, "%s: in=%d out=%d must be positive multiples of %d", name, in, out, mult);
    return ESCHA_OK;
}

// Dense linear: the per-token fused GEMV decodes the weights once per 1, 2 or
// 4 tokens; the grouped tensor-core GEMM decodes them once per item of
// dense_cap(M) tokens but has a fixed cost of its own (the B image, a second
// launch, TMEM). Measured on GB300 (5120 x 6144 .. 17408 x 5120), the GEMV is
// faster up to 2 tokens, and up to 12 tokens for weights of at most 2^23
// values; the GEMM from there on.
constexpr int kDenseGemvMaxM = 12;
constexpr int kDenseMaxM = 65536;

bool dense_uses_gemv(int in, int out, int M) {
    return M <= 2 || (M <= kDenseGemvMaxM && (long long)in * out <= (1ll << 23));
}

int dense_cap(int M) {
    int cap = 16;
    while (cap < escha::kGrpCapMax && cap < M) cap *= 2;
    return cap;
}

struct DenseWs {
    size_t err, img, part, total;
    int img_rows, splits;
};

// Status word, then (grouped GEMM only) the B image, in/64 chunks of
// 2 * round_up(M, 4) rows of 128 bytes, and the K split partial sums.
DenseWs dense_ws_layout(int in, int out, int M) {
    DenseWs w{};
    w.err = 0;
    w.img = 256;
    const bool gemm = !dense_uses_gemv(in, out, M);
    w.img_rows = gemm ? 2 * ((M + 3) & ~3) : 0;
    w.splits = gemm ? escha::dense_ksplit(in, out, M, dense_cap(M)) : 1;
    w.part = w.img + align_up((size_t)(in / 64) * w.img_rows * 128);
    w.total = w.part + (w.splits > 1 ? align_up((size_t)w.splits * M * out * 4) : 0);
    return w;
}

// Workspace layout of escha_moe_block (256-byte aligned regions).
// int8 w8a16 product of M tokens: the tensor-core GEMM from kInt8GemmMinM
// tokens on (when Kin allows it and an image buffer is given), else the GEMV.
cudaError_t int8_matmul(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                        long long x_stride, int act, int M, float* y, long long y_stride, void* img, int sms,
                        cudaStream_t s) {
    if (M >= escha::kInt8GemmMinM && Kin % 128 == 0 && img)
        return escha::launch_int8_gemm(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride, img, s);
    return escha::launch_int8_gemv(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride, sms, s);
}

bool int8_uses_gemm(int Kin, int M) { return M >= escha::kInt8GemmMinM && Kin % 128 == 0; }

struct MoeWs {
    size_t err, logits, ids, w, ygu, shgu, shgate, sh, d, grp, img, shimg, fz, total;
};

MoeWs moe_ws_layout(const escha_moe_layer* L, int T, bool force_grouped = false) {
    MoeWs m{};
    size_t off = 0;
    const size_t slots = (size_t)T * L->topk;
    m.err = off;
    off += 256;
    m.logits = off;
    off += align_up((size_t)T * L->n_experts * 2);
    m.ids = off;
    off += align_up(slots * 4);
    m.w = off;
    off += align_up(slots * 4);
    m.ygu = off;
    off += align_up(slots * 2 * (size_t)L->inter * 4);
    m.shgu = off;
    off += align_up((size_t)T * 2 * (size_t)L->sh_inter * 4);
    m.shgate = off;
    off += align_up((size_t)T * 4);
    m.sh = off;
    off += align_up(L->sh_inter > 0 ? (size_t)T * L->hidden * 4 : 0);
    const bool grouped = force_grouped || T > escha::kSlotModeMaxT;
    m.d = off;
    off += align_up(grouped ? slots * (size_t)L->hidden * 4 : 0);
    const escha::GroupPlan g = escha::group_plan(T, L->topk, L->n_experts, L->hidden, L->inter, L->sh_inter);
    m.grp = off;
    off += align_up(grouped ? g.int_bytes : 0);
    m.img = off;
    off += align_up(grouped ? g.img_bytes : 0);
    m.shimg = off;  // the shared expert runs beside the routed path, with its own scratch
    off += align_up(grouped ? g.shared_img_bytes : 0);
    m.fz = off;  // one token: counters, split partials and finished experts of the fused kernel
    if (T == 1 && !grouped) {
        const escha::FusedPlan p = escha::fused_plan(L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter);
        off += align_up(p.ctr_bytes) + align_up(p.gu_part_bytes) + align_up(p.dn_part_bytes) + align_up(p.dres_bytes);
    }
    m.total = off;
    return m;
}

int check_layer(const escha_moe_layer* L) {
    if (!L) return fail(ESCHA_E_ARG, "moe_block: layer is null");
    if (L->hidden <= 0 || L->hidden % 256) return fail(ESCHA_E_SHAPE, "moe_block: hidden=%d must be a multiple of 256", L->hidden);
    if (L->hidden > 8192) return fail(ESCHA_E_SHAPE, "moe_block: hidden=%d above 8192", L->hidden);
    if (L->inter <= 0 || L->inter % 128 || L->inter > 8192)
        return fail(ESCHA_E_SHAPE, "moe_block: inter=%d must be a multiple of 128 (<= 8192)", L->inter);
    if (L->n_experts < 1 || L->n_experts > 256) return fail(ESCHA_E_SHAPE, "moe_block: n_experts=%d not in 1..256", L->n_experts);
    if (L->topk < 1 || L->topk > 8 || L->topk > L->n_experts)
        return fail(ESCHA_E_SHAPE, "moe_block: topk=%d not in 1..min(8, n_experts)", L->topk);
    if (!L->router_w || !L->gu_rin || !L->gu_rout || !L->dn_rin || !L->dn_rout)
        return fail(ESCHA_E_ARG, "moe_block: null router / rin / rout pointer");
    const void* ptrs[] = {L->router_w, L->gu_rin, L->gu_rout, L->dn_rin, L->dn_rout};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(ESCHA_E_ALIGN, "moe_block: a router / rin / rout pointer is not 16-byte aligned");
    int r = check_trellis(L->gu_codes, L->hidden, 2 * L->inter, L->gu_K, 128, "moe_block gate_up");
    if (r) return r;
    r = check_trellis(L->dn_codes, L->inter, L->hidden, L->dn_K, 128, "moe_block down");
    if (r) return r;
    if (L->sh_inter < 0 || L->sh_inter % 16) return fail(ESCHA_E_SHAPE, "moe_block: sh_inter=%d must be a multiple of 16", L->sh_inter);
    if (L->sh_inter > 0) {
        if (!L->sh_gu_w8 || !L->sh_gu_scale || !L->sh_dn_w8 || !L->sh_dn_scale || !L->sh_gate)
            return fail(ESCHA_E_ARG, "moe_block: null shared-expert pointer");
        const void* sp[] = {L->sh_gu_w8, L->sh_gu_scale, L->sh_dn_w8, L->sh_dn_scale, L->sh_gate};
        for (const void* p : sp)
            if (!aligned16(p)) return fail(ESCHA_E_ALIGN, "moe_block: a shared-expert pointer is not 16-byte aligned");
        if (L->sh_inter > 8192) return fail(ESCHA_E_SHAPE, "moe_block: sh_inter=%d above 8192", L->sh_inter);
    }
    return ESCHA_OK;
}

}  // namespace

extern "C" {

const char* escha_last_error(void) { return g_last_error.c_str(); }

int escha_version(void) { return 100; }

int escha_trellis_decode(const uint16_t* codes, int in, int out, int K, uint16_t* W, void* stream) {
    int r = check_trellis(codes, in, out, K, 16, "trellis_decode");
    if (r) return r;
    if (!W) return fail(ESCHA_E_ARG, "trellis_decode: W is null");
    if (!aligned16(W)) return fail(ESCHA_E_ALIGN, "trellis_decode: W not 16-byte aligned");
    int sms;
    if ((r = device_check(&sms))) return r;
    return cuda_status(escha::launch_trellis_decode(codes, in, out, K, W, static_cast<cudaStream_t>(stream)),
                       "trellis_decode launch");
}

size_t escha_trellis_gemv_workspace(int in, int out, int K, int batch) {
    (void)in;
    (void)out;
    (void)K;
    (void)batch;
    return 0;
}

int escha_trellis_gemv(const uint16_t* codes, int in, int out, int K, const void* x, int x_dtype, int batch,
                       const uint16_t* rin, const uint16_t* rout, float* y, void* ws, size_t ws_bytes, void* stream) {
    (void)ws;
    int r = check_trellis(codes, in, out, K, 128, "trellis_gemv");
    if (r) return r;
    if (in > 65536) return fail(ESCHA_E_SHAPE, "trellis_gemv: in=%d above 65536", in);
    if (!x || !rin || !rout || !y) return fail(ESCHA_E_ARG, "trellis_gemv: null x / rin / rout / y");
    if (x_dtype != ESCHA_F16 && x_dtype != ESCHA_F32)
        return fail(ESCHA_E_ARG, "trellis_gemv: x_dtype=%d must be ESCHA_F16 or ESCHA_F32", x_dtype);
    if (batch < 1) return fail(ESCHA_E_ARG, "trellis_gemv: batch=%d must be >= 1", batch);
    if (!aligned16(x) || !aligned16(rin) || !aligned16(rout) || !aligned16(y))
        return fail(ESCHA_E_ALIGN, "trellis_gemv: x / rin / rout / y not 16-byte aligned");
    if (ws_bytes < escha_trellis_gemv_workspace(in, out, K, batch))
        return fail(ESCHA_E_WORKSPACE, "trellis_gemv: workspace too small");
    int sms;
    if ((r = device_check(&sms))) return r;
    escha::GemvArgs a{};
    a.codes = codes;
    a.in = in;
    a.out = out;
    a.x_mode = x_dtype == ESCHA_F16 ? escha::kXmF16 : escha::kXmF32;
    a.x = x;
    a.x_stride = in;
    a.rin = rin;
    a.rout = rout;
    a.y = y;
    a.y_stride = out;
    a.batch = batch;
    const int nb = batch == 1 ? 1 : batch == 2 ? 2 : 4;
    const int items = (batch + nb - 1) / nb;
    return cuda_status(escha::launch_trellis_gemv(a, K, nb, items, sms, static_cast<cudaStream_t>(stream)),
                       "trellis_gemv launch");
}

int escha_codes_to_nt_major(const uint16_t* codes, int in, int out, int K, uint16_t* dst, void* stream) {
    int r = check_trellis(codes, in, out, K, 16, "codes_to_nt_major");
    if (r) return r;
    if (!dst) return fail(ESCHA_E_ARG, "codes_to_nt_major: dst is null");
    if (!aligned16(dst)) return fail(ESCHA_E_ALIGN, "codes_to_nt_major: dst not 16-byte aligned");
    const size_t bytes = (size_t)in * out * K * 2 / 16;  // 16 K words per 256 weights
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(codes), b0 = reinterpret_cast<uintptr_t>(dst);
    if (a0 < b0 + bytes && b0 < a0 + bytes) return fail(ESCHA_E_ARG, "codes_to_nt_major: dst overlaps codes");
    int sms;
    if ((r = device_check(&sms))) return r;
    return cuda_status(escha::launch_codes_to_nt_major(codes, in, out, K, dst, static_cast<cudaStream_t>(stream)),
                       "codes_to_nt_major launch");
}

size_t escha_dense_linear_workspace(int in, int out, int K, int M) {
    (void)K;
    if (in <= 0 || out <= 0 || M <= 0) return 0;
    const DenseWs w = dense_ws_layout(in, out, M);
    return w.total;
}

int escha_dense_linear(const uint16_t* codes, int in, int out, int K, int nt_major, const void* x, int x_dtype, int M,
                       const uint16_t* rin, const uint16_t* rout, const float* bias, float* y, void* ws,
                       size_t ws_bytes, void* stream) {
    int r = check_trellis(codes, in, out, K, 128, "dense_linear");
    if (r) return r;
    if (in > 65536) return fail(ESCHA_E_SHAPE, "dense_linear: in=%d above 65536", in);
    if (nt_major != 0 && nt_major != 1) return fail(ESCHA_E_ARG, "dense_linear: nt_major=%d must be 0 or 1", nt_major);
    if (!x || !rin || !rout || !y || !ws) return fail(ESCHA_E_ARG, "dense_linear: null x / rin / rout / y / ws");
    if (x_dtype != ESCHA_F16 && x_dtype != ESCHA_F32)
        return fail(ESCHA_E_ARG, "dense_linear: x_dtype=%d must be ESCHA_F16 or ESCHA_F32", x_dtype);
    if (M < 1 || M > kDenseMaxM) return fail(ESCHA_E_ARG, "dense_linear: M=%d outside [1, %d]", M, kDenseMaxM);
    if (!aligned16(x) || !aligned16(rin) || !aligned16(rout) || !aligned16(y) || !aligned16(ws) ||
        (bias && !aligned16(bias)))
        return fail(ESCHA_E_ALIGN, "dense_linear: x / rin / rout / bias / y / ws not 16-byte aligned");
    const DenseWs w = dense_ws_layout(in, out, M);
    if (ws_bytes < w.total) return fail(ESCHA_E_WORKSPACE, "dense_linear: workspace too small");
    int sms;
    if ((r = device_check(&sms))) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    int* err = reinterpret_cast<int*>(base + w.err);
    if ((r = cuda_status(cudaMemsetAsync(err, 0, sizeof(int), s), "dense_linear status reset"))) return r;
    if (dense_uses_gemv(in, out, M)) {
        escha::GemvArgs a{};
        a.codes = codes;
        a.in = in;
        a.out = out;
        a.x_mode = x_dtype == ESCHA_F16 ? escha::kXmF16 : escha::kXmF32;
        a.x = x;
        a.x_stride = in;
        a.rin = rin;
        a.rout = rout;
        a.y = y;
        a.y_stride = out;
        a.batch = M;
        a.nt_major = nt_major;
        a.bias = bias;
        const int nb = M == 1 ? 1 : M == 2 ? 2 : 4;
        return cuda_status(escha::launch_trellis_gemv(a, K, nb, (M + nb - 1) / nb, sms, s), "dense_linear gemv launch");
    }
    escha::DenseArgs d{};
    d.codes = codes;
    d.in = in;
    d.out = out;
    d.K = K;
    d.nt_major = nt_major;
    d.x = x;
    d.x_f32 = x_dtype == ESCHA_F32;
    d.M = M;
    d.cap = dense_cap(M);
    d.rin = rin;
    d.rout = rout;
    d.bias = bias;
    d.y = y;
    d.img = reinterpret_cast<uint8_t*>(base + w.img);
    d.img_rows = w.img_rows;
    d.splits = w.splits;
    d.part = reinterpret_cast<float*>(base + w.part);
    d.err = err;
    return cuda_status(escha::launch_dense_grouped(d, s), "dense_linear grouped launch");
}

size_t escha_moe_block_workspace(const escha_moe_layer* L, int T) {
    if (!L || T < 1 || L->topk < 1) return 0;
    return moe_ws_layout(L, T).total;
}

}  // extern "C"

namespace {

int record(cudaEvent_t* ev, int i, cudaStream_t s) {
    if (!ev || !ev[i]) return ESCHA_OK;
    return cuda_status(cudaEventRecord(ev[i], s), "cudaEventRecord");
}

// Kernel arguments of a MoE-block call over the workspace layout m (the
// grouping fields are filled for every T; only the grouped path uses them).
escha::MoeArgs moe_args(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out, float* w_out,
                        char* base, const MoeWs& m) {
    escha::MoeArgs a{};
    a.T = T;
    a.hidden = L->hidden;
    a.inter = L->inter;
    a.E = L->n_experts;
    a.topk = L->topk;
    a.sh_inter = L->sh_inter;
    a.x = x;
    a.router_w = L->router_w;
    a.gu_codes = L->gu_codes;
    a.gu_K = L->gu_K;
    a.gu_rin = L->gu_rin;
    a.gu_rout = L->gu_rout;
    a.dn_codes = L->dn_codes;
    a.dn_K = L->dn_K;
    a.dn_rin = L->dn_rin;
    a.dn_rout = L->dn_rout;
    a.sh_gu_w8 = L->sh_gu_w8;
    a.sh_gu_scale = L->sh_gu_scale;
    a.sh_dn_w8 = L->sh_dn_w8;
    a.sh_dn_scale = L->sh_dn_scale;
    a.sh_gate = L->sh_gate;
    a.out = out;
    a.ids = ids_out ? ids_out : reinterpret_cast<int32_t*>(base + m.ids);
    a.w = w_out ? w_out : reinterpret_cast<float*>(base + m.w);
    a.logits = reinterpret_cast<uint16_t*>(base + m.logits);
    a.ygu = reinterpret_cast<float*>(base + m.ygu);
    a.shgu = reinterpret_cast<float*>(base + m.shgu);
    a.shgate = reinterpret_cast<float*>(base + m.shgate);
    a.sh = reinterpret_cast<float*>(base + m.sh);
    a.err = reinterpret_cast<int*>(base + m.err);
    {
        const escha::GroupPlan gp = escha::group_plan(T, L->topk, L->n_experts, L->hidden, L->inter, L->sh_inter);
        const int E = L->n_experts, S = T * L->topk;
        a.grp_cap = gp.cap;
        a.grp_max_items = gp.max_items;
        a.grp_items = reinterpret_cast<int4*>(base + m.grp);  // 256-byte aligned region
        int* g = reinterpret_cast<int*>(a.grp_items + gp.max_items);
        a.grp_counts = g;
        a.grp_offsets = a.grp_counts + E;
        a.grp_poff = a.grp_offsets + E + 1;
        a.grp_nitems = a.grp_poff + E;
        a.grp_perm = a.grp_nitems + 1;
        a.grp_ppos = a.grp_perm + S;
        a.grp_img = reinterpret_cast<uint8_t*>(base + m.img);
        a.grp_img_rows = 2 * gp.pos_cap;
    }
    if (T == 1) {
        const escha::FusedPlan p = escha::fused_plan(L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter);
        size_t off = m.fz;
        a.fz_ctr = reinterpret_cast<unsigned*>(base + off);
        off += align_up(p.ctr_bytes);
        a.fz_gu_part = reinterpret_cast<float*>(base + off);
        off += align_up(p.gu_part_bytes);
        a.fz_dn_part = reinterpret_cast<float*>(base + off);
        off += align_up(p.dn_part_bytes);
        a.fz_dres = reinterpret_cast<float*>(base + off);
    }
    a.fz_wait_ns = g_fz_wait_ns.load();
    a.fz_skip_publish = g_fz_skip_publish.load();
    a.mbar_limit_log2 = g_mbar_limit_log2.load();
    a.skip_cluster_arrive = g_skip_cluster_arrive.load();
    return a;
}

// Route of a one-token block: the fused single-kernel path when the shape
// and the device allow it (and no diagnostic override forbids it).
struct FusedRoute {
    bool use;
    escha::FusedPlan plan;
};

std::mutex g_fz_mu;
struct FzFitKey {
    int dev, gu_K, dn_K, grid, smem;
};
std::vector<std::pair<FzFitKey, bool>> g_fz_fits;

int fused_route(const escha_moe_layer* L, int T, int sms, FusedRoute* out) {
    out->use = false;
    const int mode = g_moe_route_mode.load();
    if (T != 1 || mode != 2) return ESCHA_OK;
    const bool shape = escha::fused_shape_ok(L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter);
    if (!shape) {
        if (mode == 2) return fail(ESCHA_E_SHAPE, "moe_block: the one-token fused kernel does not cover this layer");
        return ESCHA_OK;
    }
    out->plan = escha::fused_plan(L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    bool fits = false, known = false;
    {
        std::lock_guard<std::mutex> lk(g_fz_mu);
        for (const auto& kv : g_fz_fits) {
            const FzFitKey& k = kv.first;
            if (k.dev == dev && k.gu_K == L->gu_K && k.dn_K == L->dn_K && k.grid == out->plan.grid &&
                k.smem == out->plan.smem) {
                fits = kv.second;
                known = true;
                break;
            }
        }
    }
    if (!known) {
        e = escha::fused_fits(out->plan, L->gu_K, L->dn_K, sms, &fits);
        if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "fused kernel occupancy: %s", cudaGetErrorString(e));
        std::lock_guard<std::mutex> lk(g_fz_mu);
        g_fz_fits.push_back({FzFitKey{dev, L->gu_K, L->dn_K, out->plan.grid, out->plan.smem}, fits});
    }
    if (!fits && mode == 2)
        return fail(ESCHA_E_SHAPE, "moe_block: the one-token fused grid (%d CTAs) cannot be resident at once",
                    out->plan.grid);
    out->use = fits;
    return ESCHA_OK;
}

// Second stream and fork / join events of this host thread on a device, on
// which the grouped path runs the shared expert beside the routed chain.
// Created on first use outside a stream capture (creation is not a stream
// operation, but it is kept out of captures); until then, or if creation
// fails, the shared expert runs in line on the caller's stream.
struct ForkCtx {
    bool tried = false;
    cudaStream_t s2 = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local ForkCtx g_fork[64];

ForkCtx* fork_ctx(cudaStream_t s) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    ForkCtx& f = g_fork[dev];
    if (!f.tried) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
        f.tried = true;
        if (cudaStreamCreateWithFlags(&f.s2, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();  // leave no sticky error behind; run in line from now on
            f.s2 = nullptr;
        }
    }
    return f.s2 ? &f : nullptr;
}

// Residual input of escha_moe_block_resid: h += add, x = RMSNorm(h).
struct ResidIn {
    float* h;
    const float* add;
    float eps;
    uint16_t* x;
};

int moe_block_impl(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out, float* w_out,
                   void* ws, size_t ws_bytes, void* stream, cudaEvent_t* ev, const ResidIn* rs = nullptr) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 1) return fail(ESCHA_E_ARG, "moe_block: T=%d must be >= 1", T);
    if (T > 8192) return fail(ESCHA_E_SHAPE, "moe_block: T=%d above 8192 tokens per call", T);
    if (!x || !out) return fail(ESCHA_E_ARG, "moe_block: null x / out");
    if (!aligned16(x) || !aligned16(out) || (ids_out && !aligned16(ids_out)) || (w_out && !aligned16(w_out)))
        return fail(ESCHA_E_ALIGN, "moe_block: x / out / ids_out / w_out not 16-byte aligned");
    const MoeWs m = moe_ws_layout(L, T);
    if (!ws || ws_bytes < m.total)
        return fail(ESCHA_E_WORKSPACE, "moe_block: workspace %zu bytes, need %zu", ws_bytes, m.total);
    if (!aligned16(ws)) return fail(ESCHA_E_ALIGN, "moe_block: workspace not 16-byte aligned");
    int sms;
    if ((r = device_check(&sms))) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    escha::MoeArgs a = moe_args(L, x, T, out, ids_out, w_out, base, m);
    FusedRoute fr{};
    if ((r = fused_route(L, T, sms, &fr))) return r;
    if (fr.use) {
        if (rs) {  // the router and shared CTAs normalise; one CTA stores h += add
            a.rs_h = rs->h;
            a.rs_add = rs->add;
            a.rs_eps = rs->eps;
            a.x_norm = rs->x;
        }
        if ((r = record(ev, 0, s))) return r;
        if ((r = cuda_status(escha::launch_moe_router(a, true, s), "router launch"))) return r;
        if ((r = record(ev, 1, s))) return r;
        if ((r = cuda_status(escha::launch_moe_fused(a, fr.plan, s), "fused experts launch"))) return r;
        for (int i = 2; i < 4; ++i)
            if ((r = record(ev, i, s))) return r;
        return ESCHA_OK;
    }
    a.fz_ctr = nullptr;  // the per-slot kernels use no counters
    if (rs) {
        if (T <= escha::kFusedNormMaxT && L->hidden <= 2048) {
            // the router grid normalises; the gate_up grid stores h += add
            a.rs_h = rs->h;
            a.rs_add = rs->add;
            a.rs_eps = rs->eps;
            a.x_norm = rs->x;
        } else if ((r = cuda_status(escha::launch_residual_rmsnorm(rs->h, rs->add, T, L->hidden, rs->eps, rs->x, s),
                                    "residual_rmsnorm launch"))) {
            return r;
        }
    }
    if (T > escha::kSlotModeMaxT) {
        float* d = reinterpret_cast<float*>(base + m.d);
        uint8_t* shimg = reinterpret_cast<uint8_t*>(base + m.shimg);
        // the shared expert needs only x: its int8 GEMMs run on a second
        // stream beside router -> grouping -> grouped GEMMs (except in the
        // timed variant, whose events bracket the phases on one stream)
        auto shared = [&](cudaStream_t st) -> int {
            int rr;
            if ((rr = cuda_status(int8_matmul(L->sh_gu_w8, L->sh_gu_scale, 2 * L->sh_inter, L->hidden, x, ESCHA_F16,
                                              L->hidden, 0, T, a.shgu, 2 * L->sh_inter, shimg, sms, st),
                                  "shared gate_up launch")))
                return rr;
            return cuda_status(int8_matmul(L->sh_dn_w8, L->sh_dn_scale, L->hidden, L->sh_inter, a.shgu, ESCHA_F32,
                                           2 * L->sh_inter, 1, T, a.sh, L->hidden, shimg, sms, st),
                               "shared down launch");
        };
        ForkCtx* fk = (L->sh_inter > 0 && !ev) ? fork_ctx(s) : nullptr;
        if (fk) {
            if ((r = cuda_status(cudaEventRecord(fk->fork, s), "fork record"))) return r;
            if ((r = cuda_status(cudaStreamWaitEvent(fk->s2, fk->fork, 0), "fork wait"))) return r;
            if ((r = shared(fk->s2))) return r;
            if ((r = cuda_status(cudaEventRecord(fk->join, fk->s2), "join record"))) return r;
        }
        if ((r = record(ev, 0, s))) return r;
        if ((r = cuda_status(escha::launch_moe_router(a, false, s), "router launch"))) return r;
        if ((r = record(ev, 1, s))) return r;
        if ((r = cuda_status(escha::launch_moe_grouped(a, d, sms, s), "grouped expert launch"))) return r;
        if ((r = record(ev, 2, s))) return r;
        if (L->sh_inter > 0 && !fk && (r = shared(s))) return r;
        if (fk && (r = cuda_status(cudaStreamWaitEvent(s, fk->join, 0), "join wait"))) return r;
        if ((r = cuda_status(escha::launch_moe_combine(a, d, s), "combine launch"))) return r;
        return record(ev, 3, s);
    }

    if ((r = record(ev, 0, s))) return r;
    if ((r = cuda_status(escha::launch_moe_router(a, true, s), "router launch"))) return r;
    if ((r = record(ev, 1, s))) return r;
    if ((r = cuda_status(escha::launch_moe_gate_up(a, sms, s), "gate_up launch"))) return r;
    if ((r = record(ev, 2, s))) return r;
    if ((r = cuda_status(escha::launch_moe_down(a, sms, s), "down/combine launch"))) return r;
    return record(ev, 3, s);
}

}  // namespace

// ---------------------------------------------------------------------------
// A sequence of one-token blocks in one cooperative launch (moe_multi.cu).
// ---------------------------------------------------------------------------
namespace {

struct SeqWs {
    size_t err, ctr, logits, xdg, shgu, shgate, sh, gu_part, dn_part, ids, w, total;
};

SeqWs seq_ws_layout(const escha::MbPlan& p) {
    SeqWs w{};
    size_t off = 0;
    w.err = off;
    off += 256;
    w.ctr = off;
    off += align_up(p.ctr_bytes);
    w.logits = off;
    off += align_up(p.logits_bytes);
    w.xdg = off;
    off += align_up(p.xdg_bytes);
    w.shgu = off;
    off += align_up(p.shgu_bytes);
    w.shgate = off;
    off += align_up(p.shgate_bytes);
    w.sh = off;
    off += align_up(p.sh_bytes);
    w.gu_part = off;
    off += align_up(p.gu_part_bytes);
    w.dn_part = off;
    off += align_up(p.dn_part_bytes);
    w.ids = off;
    off += align_up(p.ids_bytes);
    w.w = off;
    off += align_up(p.ids_bytes);
    w.total = off;
    return w;
}

// The layers of a sequence: each valid, all of one shape (K may differ per
// layer and projection), a shape the sequence kernel covers.
int seq_check(const escha_moe_layer* const* layers, int n, const char* name, escha::MbPlan* plan) {
    if (!layers) return fail(ESCHA_E_ARG, "%s: layers is null", name);
    if (n < 1 || n > escha::kMbMaxBlocks)
        return fail(ESCHA_E_ARG, "%s: n_blocks=%d not in 1..%d", name, n, escha::kMbMaxBlocks);
    for (int i = 0; i < n; ++i) {
        int r = check_layer(layers[i]);
        if (r) return r;
        const escha_moe_layer* a = layers[0];
        const escha_moe_layer* b = layers[i];
        if (b->hidden != a->hidden || b->inter != a->inter || b->n_experts != a->n_experts || b->topk != a->topk ||
            b->sh_inter != a->sh_inter)
            return fail(ESCHA_E_SHAPE, "%s: layer %d differs in shape from layer 0", name, i);
    }
    const escha_moe_layer* L = layers[0];
    if (!escha::multi_shape_ok(L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter))
        return fail(ESCHA_E_SHAPE,
                    "%s: the sequence kernel covers hidden <= 2048 (a multiple of 256), 2*inter/128 <= 32 and a "
                    "shared expert inter <= 512",
                    name);
    *plan = escha::multi_plan(n, L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter);
    return ESCHA_OK;
}

std::mutex g_seq_mu;
int g_seq_grid[64][2];  // per device: smem the grid was sized for, CTAs (every SM slot)

int seq_grid(int sms, int smem, int* grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(ESCHA_E_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_seq_mu);
    if (g_seq_grid[dev][1] == 0 || g_seq_grid[dev][0] != smem) {
        int g = 0;
        e = escha::multi_grid(sms, smem, &g);
        if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "sequence kernel occupancy: %s", cudaGetErrorString(e));
        if (g < 1) return fail(ESCHA_E_DEVICE, "the sequence kernel cannot be resident on this device");
        g_seq_grid[dev][0] = smem;
        g_seq_grid[dev][1] = g;
    }
    *grid = g_seq_grid[dev][1];
    return ESCHA_OK;
}

// The work queue of a sequence (escha::MbSeg): block after block for a
// stack; a three-stage software pipeline for independent blocks.
// at most 6 + 5 n + 1 segments (independent blocks) or n (stack)
static_assert(escha::kMbMaxSegs >= 5 * escha::kMbMaxBlocks + 7, "segment table");
void seq_segments(escha::MbArgs& m, int n, const escha::MbPlan& p, bool stack) {
    int ns = 0, pos = 0;
    auto add = [&](int b, int first, int count) {
        if (b < 0 || b >= n || count <= 0) return;
        escha::MbSeg& s = m.seg[ns++];
        s.block = static_cast<short>(b);
        s.first = static_cast<short>(first);
        s.count = static_cast<short>(count);
        s.pos = pos;
        pos += count;
    };
    // a block's units in order: R S, G X, F, D, C
    const int rs = p.nR + p.nS, g0 = rs, f0 = g0 + p.nG + p.nX, d0 = f0 + p.nF, c0 = d0 + p.nD;
    if (stack) {
        for (int b = 0; b < n; ++b) add(b, 0, p.U);
    } else {
        // stage s of the pipeline: R S of block s + kDepth + 1, G X of block
        // s + kDepth, F of block s + 1, D of block s, C of block s - 1 (the
        // first stages fill it, a last C empties it)
        constexpr int kDepth = 2;  // measured on GB300, 8 blocks per launch: depth 1 16.8 us per block, 2 16.3, 3 16.4
        for (int b = 0; b <= kDepth; ++b) add(b, 0, rs);
        for (int b = 0; b < kDepth; ++b) add(b, g0, p.nG + p.nX);
        add(0, f0, p.nF);
        for (int b = 0; b < n; ++b) {
            add(b + kDepth + 1, 0, rs);
            add(b + kDepth, g0, p.nG + p.nX);
            add(b + 1, f0, p.nF);
            add(b, d0, p.nD);
            add(b - 1, c0, p.nC);
        }
        add(n - 1, c0, p.nC);
    }
    m.n_segs = ns;
}

escha::MbArgs seq_args(const escha_moe_layer* const* layers, int n, const escha::MbPlan& p, char* base,
                       const SeqWs& w) {
    escha::MbArgs m{};
    escha::MbHead& h = m.h;
    const escha_moe_layer* L = layers[0];
    h.n_blocks = n;
    h.hidden = L->hidden;
    h.inter = L->inter;
    h.E = L->n_experts;
    h.topk = L->topk;
    h.sh_inter = L->sh_inter;
    h.ctr = reinterpret_cast<unsigned*>(base + w.ctr);
    h.logits = reinterpret_cast<uint16_t*>(base + w.logits);
    h.xdg = reinterpret_cast<float*>(base + w.xdg);
    h.shgu = reinterpret_cast<float*>(base + w.shgu);
    h.shgate = reinterpret_cast<float*>(base + w.shgate);
    h.sh = reinterpret_cast<float*>(base + w.sh);
    h.gu_part = reinterpret_cast<float*>(base + w.gu_part);
    h.dn_part = reinterpret_cast<float*>(base + w.dn_part);
    h.err = reinterpret_cast<int*>(base + w.err);
    h.wait_ns = g_fz_wait_ns.load();
    h.skip_publish = g_fz_skip_publish.load();
    h.gu_csize = p.gu_csize;
    h.gu_kt = p.gu_kt;
    h.dn_ks = p.dn_ks;
    h.nR = p.nR;
    h.nS = p.nS;
    h.nG = p.nG;
    h.nX = p.nX;
    h.nD = p.nD;
    h.nF = p.nF;
    h.nC = p.nC;
    h.U = p.U;
    h.xt_floats = p.xt_floats;
    h.smem = p.smem;
    for (int i = 0; i < n; ++i) {
        const escha_moe_layer* li = layers[i];
        escha::MbBlock& B = m.blk[i];
        B.router_w = li->router_w;
        B.gu_codes = li->gu_codes;
        B.gu_rin = li->gu_rin;
        B.gu_rout = li->gu_rout;
        B.dn_codes = li->dn_codes;
        B.dn_rin = li->dn_rin;
        B.dn_rout = li->dn_rout;
        B.sh_gu_w8 = li->sh_gu_w8;
        B.sh_gu_scale = li->sh_gu_scale;
        B.sh_dn_w8 = li->sh_dn_w8;
        B.sh_dn_scale = li->sh_dn_scale;
        B.sh_gate = li->sh_gate;
        B.gu_K = li->gu_K;
        B.dn_K = li->dn_K;
        B.ids = reinterpret_cast<int32_t*>(base + w.ids) + (size_t)i * L->topk;
        B.w = reinterpret_cast<float*>(base + w.w) + (size_t)i * L->topk;
    }
    return m;
}

}  // namespace

extern "C" {

// Independent one-token blocks on the per-slot kernels (one launch of each
// over all blocks' slots, token t running layer t): up to kMlMaxT blocks of
// one shape and one K pair, hidden <= 2048. Workspace: the per-slot path's
// for T = n, then the layer table.
bool ml_covers(const escha_moe_layer* const* layers, int n) {
    if (n < 1 || n > escha::kMlMaxT || layers[0]->hidden > 2048) return false;
    for (int i = 1; i < n; ++i)
        if (layers[i]->gu_K != layers[0]->gu_K || layers[i]->dn_K != layers[0]->dn_K) return false;
    return true;
}
size_t ml_table_offset(const escha_moe_layer* L, int n) { return align_up(moe_ws_layout(L, n).total); }
size_t ml_ws_bytes(const escha_moe_layer* L, int n) {
    return ml_table_offset(L, n) + align_up((size_t)n * sizeof(escha::MoeLayerPtrs));
}

int ml_blocks(const escha_moe_layer* const* layers, int n, const uint16_t* const* x, float* const* out,
              int32_t* const* ids_out, float* const* w_out, void* ws, int sms, cudaStream_t s, cudaEvent_t* ev) {
    const escha_moe_layer* L = layers[0];
    char* base = static_cast<char*>(ws);
    const MoeWs m = moe_ws_layout(L, n);
    escha::MoeArgs a = moe_args(L, x[0], n, out[0], nullptr, nullptr, base, m);
    a.fz_ctr = nullptr;
    a.lay = reinterpret_cast<escha::MoeLayerPtrs*>(base + ml_table_offset(L, n));
    a.lay_n = n;
    escha::MlTable tab{};
    for (int i = 0; i < n; ++i) {
        const escha_moe_layer* Li = layers[i];
        escha::MoeLayerPtrs& t = tab.l[i];
        t.router_w = Li->router_w;
        t.gu_codes = Li->gu_codes;
        t.gu_rin = Li->gu_rin;
        t.gu_rout = Li->gu_rout;
        t.dn_codes = Li->dn_codes;
        t.dn_rin = Li->dn_rin;
        t.dn_rout = Li->dn_rout;
        t.sh_gu_w8 = Li->sh_gu_w8;
        t.sh_gu_scale = Li->sh_gu_scale;
        t.sh_dn_w8 = Li->sh_dn_w8;
        t.sh_dn_scale = Li->sh_dn_scale;
        t.sh_gate = Li->sh_gate;
        t.x = x[i];
        t.out = out[i];
        t.ids = ids_out ? ids_out[i] : nullptr;
        t.w = w_out ? w_out[i] : nullptr;
    }
    int r;
    if ((r = record(ev, 0, s))) return r;
    if ((r = cuda_status(escha::launch_moe_router_ml(a, tab, s), "router launch"))) return r;
    if ((r = record(ev, 1, s))) return r;
    if ((r = cuda_status(escha::launch_moe_gate_up(a, sms, s), "gate_up launch"))) return r;
    if ((r = record(ev, 2, s))) return r;
    if ((r = cuda_status(escha::launch_moe_down(a, sms, s), "down/combine launch"))) return r;
    return record(ev, 3, s);
}

size_t escha_moe_seq_workspace(const escha_moe_layer* const* layers, int n_blocks) {
    if (!layers || n_blocks < 1 || n_blocks > escha::kMbMaxBlocks || !layers[0]) return 0;
    const escha_moe_layer* L = layers[0];
    if (L->topk < 1 || L->n_experts < 1) return 0;
    size_t need = seq_ws_layout(escha::multi_plan(n_blocks, L->hidden, L->inter, L->n_experts, L->topk, L->sh_inter)).total;
    if (n_blocks <= escha::kMlMaxT) need = std::max(need, ml_ws_bytes(L, n_blocks));
    return need;
}

namespace {
int moe_blocks_impl(const escha_moe_layer* const* layers, int n_blocks, const uint16_t* const* x, float* const* out,
                    int32_t* const* ids_out, float* const* w_out, void* ws, size_t ws_bytes, void* stream,
                    cudaEvent_t* ev) {
    escha::MbPlan p{};
    int r = seq_check(layers, n_blocks, "moe_blocks", &p);
    if (r) return r;
    if (!x || !out) return fail(ESCHA_E_ARG, "moe_blocks: null x / out array");
    for (int i = 0; i < n_blocks; ++i) {
        if (!x[i] || !out[i]) return fail(ESCHA_E_ARG, "moe_blocks: null x / out of block %d", i);
        if (!aligned16(x[i]) || !aligned16(out[i]) || (ids_out && ids_out[i] && (reinterpret_cast<uintptr_t>(ids_out[i]) & 3)) ||
            (w_out && w_out[i] && (reinterpret_cast<uintptr_t>(w_out[i]) & 3)))
            return fail(ESCHA_E_ALIGN, "moe_blocks: block %d: x / out not 16-byte or ids / w not 4-byte aligned", i);
    }
    const SeqWs w = seq_ws_layout(p);
    const size_t need = escha_moe_seq_workspace(layers, n_blocks);
    if (!ws || ws_bytes < need) return fail(ESCHA_E_WORKSPACE, "moe_blocks: workspace %zu bytes, need %zu", ws_bytes, need);
    if (!aligned16(ws)) return fail(ESCHA_E_ALIGN, "moe_blocks: workspace not 16-byte aligned");
    int sms, grid;
    if ((r = device_check(&sms))) return r;
    const int route = g_blocks_route.load();
    const bool ml = ml_covers(layers, n_blocks);
    if (route == 1 && !ml)
        return fail(ESCHA_E_SHAPE, "moe_blocks: the per-slot route takes up to %d blocks with one K pair", escha::kMlMaxT);
    if (ml && route != 2)
        return ml_blocks(layers, n_blocks, x, out, ids_out, w_out, ws, sms, static_cast<cudaStream_t>(stream), ev);
    if ((r = seq_grid(sms, p.smem, &grid))) return r;
    escha::MbArgs m = seq_args(layers, n_blocks, p, static_cast<char*>(ws), w);
    seq_segments(m, n_blocks, p, false);
    for (int i = 0; i < n_blocks; ++i) {
        m.blk[i].x = x[i];
        m.blk[i].out = out[i];
        if (ids_out && ids_out[i]) m.blk[i].ids = ids_out[i];
        if (w_out && w_out[i]) m.blk[i].w = w_out[i];
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((r = record(ev, 0, st))) return r;
    if ((r = cuda_status(escha::launch_moe_multi(m, grid, st), "moe_blocks launch"))) return r;
    for (int i = 1; i < 4; ++i)
        if ((r = record(ev, i, st))) return r;
    return ESCHA_OK;
}
}  // namespace

int escha_moe_blocks(const escha_moe_layer* const* layers, int n_blocks, const uint16_t* const* x, float* const* out,
                     int32_t* const* ids_out, float* const* w_out, void* ws, size_t ws_bytes, void* stream) {
    return moe_blocks_impl(layers, n_blocks, x, out, ids_out, w_out, ws, ws_bytes, stream, nullptr);
}

int escha_moe_blocks_timed(const escha_moe_layer* const* layers, int n_blocks, const uint16_t* const* x,
                           float* const* out, int32_t* const* ids_out, float* const* w_out, void* ws, size_t ws_bytes,
                           void* stream, void* const* events) {
    cudaEvent_t ev[4];
    for (int i = 0; i < 4; ++i) ev[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
    return moe_blocks_impl(layers, n_blocks, x, out, ids_out, w_out, ws, ws_bytes, stream, ev);
}

int escha_moe_stack(const escha_moe_layer* const* layers, int n_blocks, float* h, float eps, uint16_t* x_buf,
                    float* out_buf, int32_t* ids_out, float* w_out, void* ws, size_t ws_bytes, void* stream) {
    escha::MbPlan p{};
    int r = seq_check(layers, n_blocks, "moe_stack", &p);
    if (r) return r;
    if (!h || !x_buf || !out_buf) return fail(ESCHA_E_ARG, "moe_stack: null h / x_buf / out_buf");
    if (!(eps >= 0.f)) return fail(ESCHA_E_ARG, "moe_stack: eps must be >= 0");
    if (!aligned16(h) || !aligned16(x_buf) || !aligned16(out_buf) || (reinterpret_cast<uintptr_t>(ids_out) & 3) ||
        (reinterpret_cast<uintptr_t>(w_out) & 3))
        return fail(ESCHA_E_ALIGN, "moe_stack: h / x_buf / out_buf not 16-byte or ids / w not 4-byte aligned");
    const size_t H = layers[0]->hidden;
    auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
        return a0 < b0 + nb && b0 < a0 + na;
    };
    if (overlap(h, 4 * H, x_buf, 2 * H) || overlap(h, 4 * H, out_buf, 4 * H) || overlap(x_buf, 2 * H, out_buf, 4 * H))
        return fail(ESCHA_E_ARG, "moe_stack: h, x_buf and out_buf must not overlap");
    const SeqWs w = seq_ws_layout(p);
    if (!ws || ws_bytes < w.total) return fail(ESCHA_E_WORKSPACE, "moe_stack: workspace %zu bytes, need %zu", ws_bytes, w.total);
    if (!aligned16(ws)) return fail(ESCHA_E_ALIGN, "moe_stack: workspace not 16-byte aligned");
    int sms, grid;
    if ((r = device_check(&sms))) return r;
    if ((r = seq_grid(sms, p.smem, &grid))) return r;
    escha::MbArgs m = seq_args(layers, n_blocks, p, static_cast<char*>(ws), w);
    seq_segments(m, n_blocks, p, true);
    m.h.stack = 1;
    m.h.res = h;
    m.h.eps = eps;
    m.h.xbuf = x_buf;
    m.h.outbuf = out_buf;
    const int k = layers[0]->topk;
    for (int i = 0; i < n_blocks; ++i) {
        if (ids_out) m.blk[i].ids = ids_out + (size_t)i * k;
        if (w_out) m.blk[i].w = w_out + (size_t)i * k;
    }
    return cuda_status(escha::launch_moe_multi(m, grid, static_cast<cudaStream_t>(stream)), "moe_stack launch");
}

int escha_moe_block(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out, float* w_out,
                    void* ws, size_t ws_bytes, void* stream) {
    return moe_block_impl(L, x, T, out, ids_out, w_out, ws, ws_bytes, stream, nullptr);
}

int escha_moe_block_resid(const escha_moe_layer* L, float* h, const float* add, float eps, uint16_t* x, int T,
                          float* out, int32_t* ids_out, float* w_out, void* ws, size_t ws_bytes, void* stream) {
    int r = check_layer(L);
    if (r) return r;
    if (!h || !x) return fail(ESCHA_E_ARG, "moe_block_resid: null h / x");
    if (!(eps >= 0.f)) return fail(ESCHA_E_ARG, "moe_block_resid: eps must be >= 0");
    if (!aligned16(h) || (add && !aligned16(add)))
        return fail(ESCHA_E_ALIGN, "moe_block_resid: h / add not 16-byte aligned");
    if (T >= 1 && T <= 8192) {
        // x is written while h and add are read and before out is written:
        // it must not share memory with any of them
        const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), x1 = x0 + (size_t)T * L->hidden * 2;
        auto overlaps = [&](const void* p) {
            const uintptr_t p0 = reinterpret_cast<uintptr_t>(p), p1 = p0 + (size_t)T * L->hidden * 4;
            return p && p0 < x1 && x0 < p1;
        };
        if (overlaps(h) || overlaps(add) || overlaps(out))
            return fail(ESCHA_E_ARG, "moe_block_resid: x overlaps h, add or out");
    }
    const ResidIn rs{h, add, eps, x};
    return moe_block_impl(L, x, T, out, ids_out, w_out, ws, ws_bytes, stream, nullptr, &rs);
}

int escha_moe_block_path(const escha_moe_layer* L, int T) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 1 || T > 8192) return fail(ESCHA_E_SHAPE, "moe_block_path: T=%d not in 1..8192", T);
    if (T > escha::kSlotModeMaxT) return ESCHA_PATH_GROUPED;
    int sms;
    if ((r = device_check(&sms))) return r;
    FusedRoute fr{};
    if ((r = fused_route(L, T, sms, &fr))) return r;
    return fr.use ? ESCHA_PATH_FUSED : ESCHA_PATH_SLOT;
}

int escha_debug_set_blocks_route(int mode) {
    if (mode < 0 || mode > 2) return fail(ESCHA_E_ARG, "escha_debug_set_blocks_route: mode %d not in 0..2", mode);
    g_blocks_route.store(mode);
    return ESCHA_OK;
}

int escha_moe_blocks_path(const escha_moe_layer* const* layers, int n_blocks) {
    escha::MbPlan p{};
    int r = seq_check(layers, n_blocks, "moe_blocks_path", &p);
    if (r) return r;
    const int route = g_blocks_route.load();
    const bool ml = ml_covers(layers, n_blocks);
    if (route == 1 && !ml) return fail(ESCHA_E_SHAPE, "moe_blocks_path: the per-slot route does not cover these blocks");
    return ml && route != 2 ? ESCHA_PATH_SLOT : ESCHA_PATH_SEQUENCE;
}

int escha_debug_set_moe_route(int mode) {
    if (mode < 0 || mode > 2) return fail(ESCHA_E_ARG, "debug_set_moe_route: mode=%d not in 0..2", mode);
    g_moe_route_mode.store(mode);
    return ESCHA_OK;
}

int escha_debug_set_cluster_wait(int poll_limit_log2, int skip_arrive) {
    if (poll_limit_log2 < 8 || poll_limit_log2 > 30)
        return fail(ESCHA_E_ARG, "debug_set_cluster_wait: poll_limit_log2=%d not in [8, 30]", poll_limit_log2);
    if (skip_arrive != 0 && skip_arrive != 1)
        return fail(ESCHA_E_ARG, "debug_set_cluster_wait: skip_arrive=%d must be 0 or 1", skip_arrive);
    g_mbar_limit_log2.store(poll_limit_log2);
    g_skip_cluster_arrive.store(skip_arrive);
    return ESCHA_OK;
}

int escha_debug_set_fused_wait(long long wait_ns, int skip_publish) {
    if (wait_ns < 1000 || wait_ns > 60000000000ll)
        return fail(ESCHA_E_ARG, "debug_set_fused_wait: wait_ns=%lld not in [1e3, 6e10]", wait_ns);
    if (skip_publish != 0 && skip_publish != 1)
        return fail(ESCHA_E_ARG, "debug_set_fused_wait: skip_publish=%d must be 0 or 1", skip_publish);
    g_fz_wait_ns.store(wait_ns);
    g_fz_skip_publish.store(skip_publish);
    return ESCHA_OK;
}

int escha_moe_block_timed(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out,
                          float* w_out, void* ws, size_t ws_bytes, void* stream, void* const* events) {
    cudaEvent_t ev[4];
    for (int i = 0; i < 4; ++i) ev[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
    return moe_block_impl(L, x, T, out, ids_out, w_out, ws, ws_bytes, stream, ev);
}

size_t escha_moe_route_workspace(const escha_moe_layer* L, int T) {
    if (!L || T < 1 || L->topk < 1) return 0;
    return moe_ws_layout(L, T, true).total;
}

int escha_moe_route(const escha_moe_layer* L, const uint16_t* x, int T, uint16_t* logits_out, int32_t* ids_out,
                    float* w_out, int32_t* counts_out, int32_t* offsets_out, int32_t* perm_out, void* ws,
                    size_t ws_bytes, void* stream) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 1 || T > 8192) return fail(ESCHA_E_SHAPE, "moe_route: T=%d not in 1..8192", T);
    if (!x || !ids_out || !w_out) return fail(ESCHA_E_ARG, "moe_route: null x / ids_out / w_out");
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(ids_out) & 3) || (reinterpret_cast<uintptr_t>(w_out) & 3))
        return fail(ESCHA_E_ALIGN, "moe_route: x not 16-byte aligned or ids_out / w_out not 4-byte aligned");
    const MoeWs m = moe_ws_layout(L, T, true);
    if (!ws || ws_bytes < m.total)
        return fail(ESCHA_E_WORKSPACE, "moe_route: workspace %zu bytes, need %zu", ws_bytes, m.total);
    if (!aligned16(ws)) return fail(ESCHA_E_ALIGN, "moe_route: workspace not 16-byte aligned");
    int sms;
    if ((r = device_check(&sms))) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    const escha::MoeArgs a = moe_args(L, x, T, nullptr, ids_out, w_out, base, m);
    if ((r = cuda_status(escha::launch_moe_router(a, false, s), "router launch"))) return r;
    if ((r = cuda_status(escha::launch_moe_topk_group(a, s), "top-k / grouping launch"))) return r;
    const int E = L->n_experts;
    const size_t S = (size_t)T * L->topk;
    struct {
        void* dst;
        const void* src;
        size_t bytes;
    } copies[] = {{logits_out, a.logits, (size_t)T * E * 2},
                  {counts_out, a.grp_counts, (size_t)E * 4},
                  {offsets_out, a.grp_offsets, (size_t)(E + 1) * 4},
                  {perm_out, a.grp_perm, S * 4}};
    for (const auto& c : copies) {
        if (!c.dst) continue;
        if ((r = cuda_status(cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToDevice, s), "route copy")))
            return r;
    }
    return ESCHA_OK;
}

int escha_residual_rmsnorm(float* h, const float* add, int T, int hidden, float eps, uint16_t* x_out, void* stream) {
    if (!h) return fail(ESCHA_E_ARG, "residual_rmsnorm: null h");
    if (T < 1 || hidden < 1 || hidden > 8192) return fail(ESCHA_E_SHAPE, "residual_rmsnorm: T=%d hidden=%d", T, hidden);
    if (!(eps >= 0.f)) return fail(ESCHA_E_ARG, "residual_rmsnorm: eps must be >= 0");
    if (!aligned16(h) || (add && !aligned16(add)) || (x_out && !aligned16(x_out)))
        return fail(ESCHA_E_ALIGN, "residual_rmsnorm: pointer not 16-byte aligned");
    int r, sms;
    if ((r = device_check(&sms))) return r;
    return cuda_status(escha::launch_residual_rmsnorm(h, add, T, hidden, eps, x_out, static_cast<cudaStream_t>(stream)),
                       "residual_rmsnorm launch");
}

size_t int8_w8a16_workspace(int N, int Kin, int M) {
    (void)N;
    if (M < 1 || Kin < 16) return 0;
    return int8_uses_gemm(Kin, M) ? escha::int8_gemm_ws_bytes(N, Kin, M) : 0;
}

int int8_w8a16_matvec(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype, int M,
                      float* y, void* ws, size_t ws_bytes, void* stream) {
    if (!W || !scales || !x || !y) return fail(ESCHA_E_ARG, "int8_w8a16_matvec: null pointer");
    if (N < 1 || M < 1) return fail(ESCHA_E_ARG, "int8_w8a16_matvec: N=%d M=%d must be >= 1", N, M);
    if (Kin < 16 || Kin % 16 || Kin > 51200)
        return fail(ESCHA_E_SHAPE, "int8_w8a16_matvec: Kin=%d must be a multiple of 16 in 16..51200", Kin);
    if (x_dtype != ESCHA_F16 && x_dtype != ESCHA_BF16 && x_dtype != ESCHA_F32)
        return fail(ESCHA_E_ARG, "int8_w8a16_matvec: x_dtype=%d", x_dtype);
    if (!aligned16(W) || !aligned16(scales) || !aligned16(x) || !aligned16(y))
        return fail(ESCHA_E_ALIGN, "int8_w8a16_matvec: pointer not 16-byte aligned");
    const bool gemm = int8_uses_gemm(Kin, M);
    if (!gemm && M > 1 && Kin > 51168)
        return fail(ESCHA_E_SHAPE, "int8_w8a16_matvec: Kin=%d above 51168 for 2..15 tokens or Kin %% 128 != 0", Kin);
    if (gemm) {
        const size_t need = escha::int8_gemm_ws_bytes(N, Kin, M);
        if (!ws || ws_bytes < need)
            return fail(ESCHA_E_WORKSPACE, "int8_w8a16_matvec: workspace of %zu bytes, %zu needed", ws_bytes, need);
        if (!aligned16(ws)) return fail(ESCHA_E_ALIGN, "int8_w8a16_matvec: workspace not 16-byte aligned");
    }
    int r, sms;
    if ((r = device_check(&sms))) return r;
    return cuda_status(int8_matmul(W, scales, N, Kin, x, x_dtype, Kin, 0, M, y, N, gemm ? ws : nullptr, sms,
                                   static_cast<cudaStream_t>(stream)),
                       "int8 matmul launch");
}

int int8_w8a16_dequant(const int8_t* W, const float* scales, int N, int Kin, float* out, void* stream) {
    if (!W || !scales || !out) return fail(ESCHA_E_ARG, "int8_w8a16_dequant: null pointer");
    if (N < 1 || Kin < 1) return fail(ESCHA_E_SHAPE, "int8_w8a16_dequant: N=%d Kin=%d", N, Kin);
    int r, sms;
    if ((r = device_check(&sms))) return r;
    return cuda_status(escha::launch_int8_dequant(W, scales, N, Kin, out, static_cast<cudaStream_t>(stream)),
                       "int8 dequant launch");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// MoE block without any allocation by the caller.
//
// Some callers cannot allocate device memory when they run the block: an
// operator plugin inside a framework that owns every device allocation, code
// issuing work while a stream is being captured into a CUDA graph in a mode
// that forbids cudaMalloc, or a process whose memory must be fixed at
// start-up. For them the scratch lives in the buffer below, compiled into the
// library: every GPU that loads the library holds these bytes until the
// process exits. Host code cannot use the buffer's name as a device address,
// so its address is looked up once per device and kept.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ESCHA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];
unsigned long long g_noalloc_ctx[64];  // the context the address was looked up in

// Unique id of the current context (0 if it cannot be read): the driver's
// cuCtxGetCurrent / cuCtxGetId, reached through the runtime, so the library
// needs no link against the driver library.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrent)(CUcontext*);
    typedef CUresult (*GetId)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call for that device and again whenever the device's context has
// changed since (after cudaDeviceReset the module is loaded anew and the
// buffer can move).
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ESCHA_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(ESCHA_E_DEVICE, "device ordinal %d out of range", dev);
    const unsigned long long ctx = current_context_id();  // 0 before the runtime has made a context current
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(ESCHA_E_CUDA, "cudaGetSymbolAddress(built-in scratch): %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = current_context_id();  // the lookup has made the device's context current
    }
    *out = g_noalloc_ptr[dev];
    return ESCHA_OK;
}

}  // namespace

extern "C" {

int escha_moe_block_noalloc(const escha_moe_layer* L, const uint16_t* x, int T, float* out, int32_t* ids_out,
                            float* w_out, void* stream) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 1) return fail(ESCHA_E_ARG, "moe_block_noalloc: T=%d must be >= 1", T);
    const size_t need = moe_ws_layout(L, T).total;
    if (need > (size_t)ESCHA_NOALLOC_SCRATCH_BYTES)
        return fail(ESCHA_E_WORKSPACE,
                    "moe_block_noalloc: this layer at T=%d needs %zu bytes of scratch, more than the %zu-byte "
                    "built-in buffer; call escha_moe_block with a workspace instead",
                    T, need, (size_t)ESCHA_NOALLOC_SCRATCH_BYTES);
    void* ws = nullptr;
    if ((r = noalloc_scratch(&ws))) return r;
    // Nothing in the scratch has to start at zero: the status word is reset
    // by the router kernel and every other region is written before it is read.
    return moe_block_impl(L, x, T, out, ids_out, w_out, ws, (size_t)ESCHA_NOALLOC_SCRATCH_BYTES, stream, nullptr);
}

}  // extern "C"
