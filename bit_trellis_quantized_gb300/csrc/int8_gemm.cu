// int8 w8a16 GEMM on the 5th-generation tensor cores, for many tokens:
// y[m][o] = scale[o] * sum_i W[o][i] * x[m][i] (MTPLX PR #242, table
// "Improvements": int8 non-experts used as stored, no dequant at load; MLX
// model card, table "Exactness of every tensor": dequant = f32 scale * w8).
//
// Operands. An int8 weight is an integer in [-128, 127], exact in fp16 and in
// bf16, so A (128 weight rows per CTA) is the int8 block converted exactly to
// the activation's 16-bit type: fp16 x and bf16 x are then used as they are
// (exact products, f32 accumulation). f32 activations (and SwiGLU of an f32
// gate/up pair, act == 1) are split into bf16 hi + lo (16 significant bits,
// relative error <= 2^-17, full f32 range) and both rows enter the MMA; the
// epilogue adds the two columns. The row scale multiplies the finished sum.
//
// Kernels: a prep kernel writes the activations as the MMA's B image (K-major,
// 128-byte swizzled, every 64-value chunk holding all rows), then one CTA per
// (256 outputs, 256 image rows) runs the warp-specialised tensor-core loop:
// 8 warps convert int8 chunks into 3 shared-memory stages, a ninth issues the
// B bulk copies two chunks ahead and two M = 128 MMAs per K step that share
// the B chunk (so B, the re-read operand, comes from L2 once per 256 outputs).
#include <cuda_bf16.h>

#include "kernels.h"
#include "tc_mainloop.cuh"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kDtBf16 = 2, kDtF32 = 3;  // activation dtypes (ESCHA_BF16, ESCHA_F32); ESCHA_F16 is 1
constexpr int kRowsPerCta = 256;  // image rows (B rows) per CTA = MMA N at most
constexpr int kOutPerCta = 256;   // output rows per CTA: two M = 128 tiles sharing each B chunk
constexpr int kStages = 3;

__host__ __device__ __forceinline__ int img_rows_for(int parts, int M) { return (parts * M + 7) & ~7; }

// One warp per (token m, 128-value block).
__global__ void __launch_bounds__(256) int8_prep_kernel(const void* __restrict__ x, int x_dtype, long long x_stride,
                                                        int act, int M, int Kin, uint8_t* __restrict__ img,
                                                        int img_rows) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int nblk = Kin >> 7;
    const long long task = (long long)blockIdx.x * 8 + warp;
    if (task >= (long long)M * nblk) return;
    const int m = static_cast<int>(task / nblk), b = static_cast<int>(task % nblk);
    const int k = b * 128 + 4 * lane;
    uint8_t* base = img + (long long)(2 * b + (lane >> 4)) * img_rows * 128;
    const uint32_t k_in = static_cast<uint32_t>((4 * lane) & 63);
    if (act == 0 && x_dtype != kDtF32) {  // 16-bit x: copied as is
        const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + m * x_stride + k);
        *reinterpret_cast<uint2*>(base + tc::kmajor_off(static_cast<uint32_t>(m), k_in)) = v;
        return;
    }
    float v[4];
    const float* xr = static_cast<const float*>(x) + m * x_stride;
    if (act == 1) {
        const float4 g = *reinterpret_cast<const float4*>(xr + k);
        const float4 u = *reinterpret_cast<const float4*>(xr + Kin + k);
        v[0] = silu_f(g.x) * u.x;
        v[1] = silu_f(g.y) * u.y;
        v[2] = silu_f(g.z) * u.z;
        v[3] = silu_f(g.w) * u.w;
    } else {
        const float4 g = *reinterpret_cast<const float4*>(xr + k);
        v[0] = g.x;
        v[1] = g.y;
        v[2] = g.z;
        v[3] = g.w;
    }
    uint32_t hv[2], lv[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * q]), h1 = __float2bfloat16_rn(v[2 * q + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * q] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * q + 1] - __bfloat162float(h1));
        hv[q] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lv[q] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
    }
    *reinterpret_cast<uint2*>(base + tc::kmajor_off(2u * m, k_in)) = make_uint2(hv[0], hv[1]);
    *reinterpret_cast<uint2*>(base + tc::kmajor_off(2u * m + 1u, k_in)) = make_uint2(lv[0], lv[1]);
}

// Four int8 values (one 32-bit word) as two packed 16-bit pairs, exactly.
template <bool BF16>
__device__ __forceinline__ uint2 i8x4_to_16(uint32_t w) {
    if constexpr (BF16) {
        float f[4];
        i8x4_to_f32(w, f);
        const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
        return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
        // byte b biased to u = b + 128 under the fp16 exponent of 1024 (ulp 1):
        // 1024 + u, minus 1152, is b exactly
        const uint32_t u = w ^ 0x80808080u;
        const uint32_t p01 = __byte_perm(u, 0x64646464u, 0x4140);
        const uint32_t p23 = __byte_perm(u, 0x64646464u, 0x4342);
        const __half2 off = __half2half2(__ushort_as_half(0x6480));  // 1152
        const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&p01), off);
        const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&p23), off);
        return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
}

template <bool BF16, int PARTS>
__global__ void __launch_bounds__(tc::kMlThreads + 32, 1)
    int8_gemm_kernel(const int8_t* __restrict__ W, const float* __restrict__ scales, int N, int Kin,
                     const uint8_t* __restrict__ img, int img_rows, int M, float* __restrict__ y, long long y_stride,
                     int bps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr uint32_t kBStage = kRowsPerCta * 128;
    constexpr int kAStage = 2 * tc::kWsAStageBytes;
    uint8_t* Abuf = smem;                         // [3][2 tiles][16 KB]: 128 rows x 64 values, K-major
    uint8_t* Bbuf = smem + kStages * kAStage;     // [3][256 rows x 128 B]
    __shared__ tc::WsBars bars;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kOutPerCta;
    const int R0 = blockIdx.y * kRowsPerCta;

    pdl_wait();  // the B image is complete
    pdl_trigger();
    const int nrows = min(kRowsPerCta, img_rows - R0);  // a multiple of 8
    const int npad = (nrows + 15) & ~15;
    if (tid == 0) tc::ws_bars_init(bars);
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 512);  // two accumulators of 256 columns
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = tc::idesc_f16(128, npad, false, false, BF16);

    // K split z (blockIdx.z) covers blocks [z * bps, z * bps + nblk) of 128
    // values = chunks of 64 from 2 * z * bps; with more than one split, y
    // points at split z's partial sums ([M][N] each)
    const int b_first = blockIdx.z * bps;
    const int nblk = min(Kin / 128 - b_first, bps);
    if (gridDim.z > 1) {
        y += (long long)blockIdx.z * M * N;
        y_stride = N;
    }
    // producer warp w converts output rows 32w .. 32w + 31 of the CTA (M tile
    // w / 4): in part j (0..3) lane l takes row 32w + 8j + l/4, values
    // 16(l%4) .. +15 of the chunk, so four lanes read one row's 64 bytes and
    // each load instruction reads eight whole 64-byte row segments (one
    // row per lane left every sector half used for L1 to keep, and L1 is
    // small beside these shared-memory stages). Three register sets rotate:
    // chunk c + 2 loads into one while chunk c is converted from another, so
    // a load has two chunks of MMA time to arrive, and no set is ever copied
    // (a copy would wait for the load).
    const int r0 = (tid & 255) & ~31;  // the warp's first row
    const int8_t* wrow = W + (long long)min(n0 + r0 + (lane >> 2), N - 1) * Kin + b_first * 128 + 16 * (lane & 3);
    long long jstep[4];  // row j of the lane's four, clamped to the last weight row
#pragma unroll
    for (int j = 0; j < 4; ++j)
        jstep[j] = (long long)(min(n0 + r0 + 8 * j + (lane >> 2), N - 1) - min(n0 + r0 + (lane >> 2), N - 1)) * Kin;
    const int nch = 2 * nblk;
    uint4 w0[4], w1[4], w2[4];
    auto load = [&](uint4 (&w)[4], int c) {
        if (c < nch) {
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = __ldg(reinterpret_cast<const uint4*>(wrow + jstep[j] + c * 64));
        }
    };
    if (tid < tc::kMlThreads) {
        load(w0, 0);
        load(w1, 1);
    }
    auto convert = [&](const uint4 (&w)[4], uint8_t* A) {
        uint8_t* dst = A + (r0 >> 7) * tc::kWsAStageBytes;
        const uint32_t k0 = 16u * static_cast<uint32_t>(lane & 3);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t rr = static_cast<uint32_t>((r0 & 127) + 8 * j + (lane >> 2));
            const uint2 x0 = i8x4_to_16<BF16>(w[j].x), x1 = i8x4_to_16<BF16>(w[j].y);
            const uint2 x2 = i8x4_to_16<BF16>(w[j].z), x3 = i8x4_to_16<BF16>(w[j].w);
            *reinterpret_cast<uint4*>(dst + tc::kmajor_off(rr, k0)) = make_uint4(x0.x, x0.y, x1.x, x1.y);
            *reinterpret_cast<uint4*>(dst + tc::kmajor_off(rr, k0 + 8u)) = make_uint4(x2.x, x2.y, x3.x, x3.y);
        }
    };

    int rot = 0;  // c % 3
    const bool ok = tc::mma_mainloop_ws<kStages, false, 2>(
        Abuf, Bbuf, kBStage, img + (long long)R0 * 128 + 2ll * b_first * img_rows * 128, (long long)img_rows * 128,
        static_cast<uint32_t>(nrows) * 128u, nch, tmem, idesc, bars,
        [&](int c, uint8_t* A) {
            if (rot == 0) {
                load(w2, c + 2);
                convert(w0, A);
            } else if (rot == 1) {
                load(w0, c + 2);
                convert(w1, A);
            } else {
                load(w1, c + 2);
                convert(w2, A);
            }
            rot = rot == 2 ? 0 : rot + 1;
        },
        256u);

    // epilogue: TMEM lane = output row of an M tile, column = image row;
    // warps w (tile 0, columns 0..255) and w + 4 (tile 1, columns 256..511)
    // share lane quarter w % 4. A bounded wait that gave up leaves NaN in the
    // CTA's outputs.
    if (warp < 8) {
        const int q = warp & 3, mt = warp >> 2;
        const int n = n0 + 128 * mt + 32 * q + lane;
        const float sc = !ok ? __int_as_float(0x7fc00000) : (n < N ? scales[n] : 0.f);
        for (int c0 = 0; c0 < npad; c0 += 16) {
            float v[16];
            tc::tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + 256u * mt + c0, v);
            tc::tmem_ld_wait();
            if (n >= N) continue;
            if constexpr (PARTS == 1) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = R0 + c0 + i;
                    if (m < M) y[m * y_stride + n] = sc * v[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int m = (R0 + c0) / 2 + i;
                    if (m < M) y[m * y_stride + n] = sc * (v[2 * i] + v[2 * i + 1]);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// y[m][n] = sum over the splits z (in order) of part[z][m][n]; four
// consecutive n per thread when N % 4 == 0 (y_stride too), else one.
__global__ void __launch_bounds__(256) int8_split_reduce_kernel(const float* __restrict__ part, int ks, int M, int N,
                                                                float* __restrict__ y, long long y_stride) {
    pdl_wait();
    pdl_trigger();
    const long long MN = (long long)M * N;
    if ((N & 3) == 0 && (y_stride & 3) == 0) {
        const long long i = 4 * ((long long)blockIdx.x * 256 + threadIdx.x);
        if (i >= MN) return;
        float4 acc = *reinterpret_cast<const float4*>(part + i);
        for (int z = 1; z < ks; ++z) {
            const float4 v = *reinterpret_cast<const float4*>(part + z * MN + i);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        *reinterpret_cast<float4*>(y + (i / N) * y_stride + i % N) = acc;
        return;
    }
    const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
    if (i >= MN) return;
    float acc = part[i];
    for (int z = 1; z < ks; ++z) acc += part[z * MN + i];
    y[(i / N) * y_stride + i % N] = acc;
}

template <bool BF16, int PARTS>
cudaError_t launch_gemm(const int8_t* W, const float* scales, int N, int Kin, const uint8_t* img, int img_rows, int M,
                        float* y, long long y_stride, float* part, cudaStream_t s) {
    const int smem = kStages * (2 * tc::kWsAStageBytes + kRowsPerCta * 128) + 1024;
    const void* f = reinterpret_cast<const void*>(int8_gemm_kernel<BF16, PARTS>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nblk = Kin / 128;
    int bps = (nblk + int8_gemm_ksplit(N, Kin, M, PARTS) - 1) / int8_gemm_ksplit(N, Kin, M, PARTS);
    const int ks = (nblk + bps - 1) / bps;  // every split starts inside K
    float* out = ks > 1 ? part : y;
    void* args[] = {&W, &scales, &N, &Kin, &img, &img_rows, &M, &out, &y_stride, &bps};
    e = launch_kernel(f, dim3((N + kOutPerCta - 1) / kOutPerCta, (img_rows + kRowsPerCta - 1) / kRowsPerCta, ks),
                      dim3(tc::kMlThreads + 32), smem, true, s, args);
    if (e != cudaSuccess || ks == 1) return e;
    int ks_ = ks;
    void* rargs[] = {&part, &ks_, &M, &N, &y, &y_stride};
    const long long per_thread = ((N & 3) == 0 && (y_stride & 3) == 0) ? 4 : 1;
    const long long threads = ((long long)M * N + per_thread - 1) / per_thread;
    return launch_kernel(reinterpret_cast<const void*>(int8_split_reduce_kernel),
                         dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, true, s, rargs);
}

}  // namespace

// K splits of the GEMM: enough CTAs for about one wave of 152 SMs, at least
// two 128-value blocks per split, at most 8 splits. From 48 tiles on, a
// split of two is taken only while the doubled grid still fits one wave.
// A fixed function of the shape, so results do not depend on the device.
int int8_gemm_ksplit(int N, int Kin, int M, int parts) {
    const long long tiles =
        (long long)((N + kOutPerCta - 1) / kOutPerCta) * ((img_rows_for(parts, M) + kRowsPerCta - 1) / kRowsPerCta);
    const int nblk = Kin / 128;
    if (tiles >= 48) return (2 * tiles <= 152 && nblk >= 4) ? 2 : 1;
    int ks = static_cast<int>((152 + tiles - 1) / tiles);
    ks = min(ks, max(1, nblk / 2));
    return min(ks, 8);
}

size_t int8_gemm_image_bytes(int Kin, int M) { return (size_t)Kin * img_rows_for(2, M) * 2; }

size_t int8_gemm_ws_bytes(int N, int Kin, int M) {
    const int ks = max(int8_gemm_ksplit(N, Kin, M, 1), int8_gemm_ksplit(N, Kin, M, 2));
    const size_t img = (int8_gemm_image_bytes(Kin, M) + 255) & ~size_t(255);
    return img + (ks > 1 ? (size_t)ks * M * N * 4 : 0);
}

cudaError_t launch_int8_gemm(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                             long long x_stride, int act, int M, float* y, long long y_stride, void* img_v,
                             cudaStream_t s) {
    const int parts = (act == 1 || x_dtype == kDtF32) ? 2 : 1;
    int img_rows = img_rows_for(parts, M);
    uint8_t* img = static_cast<uint8_t*>(img_v);
    float* part = reinterpret_cast<float*>(img + ((int8_gemm_image_bytes(Kin, M) + 255) & ~size_t(255)));
    const long long tasks = (long long)M * (Kin / 128);
    void* pargs[] = {&x, &x_dtype, &x_stride, &act, &M, &Kin, &img, &img_rows};
    cudaError_t e = launch_kernel(reinterpret_cast<const void*>(int8_prep_kernel),
                                  dim3(static_cast<unsigned>((tasks + 7) / 8)), dim3(256), 0, true, s, pargs);
    if (e != cudaSuccess) return e;
    if (parts == 2) return launch_gemm<true, 2>(W, scales, N, Kin, img, img_rows, M, y, y_stride, part, s);
    if (x_dtype == kDtBf16) return launch_gemm<true, 1>(W, scales, N, Kin, img, img_rows, M, y, y_stride, part, s);
    return launch_gemm<false, 1>(W, scales, N, Kin, img, img_rows, M, y, y_stride, part, s);
}

}  // namespace escha
