// int8 w8a16: y[m][o] = sum_i (scale[o] * W[o][i]) * x[m][i], the int8
// weights used as stored (MTPLX PR #242 "serve Qwen3.6-35B-A3B-Escha-W2
// natively", table "Improvements": fused int8 matvec, no dequant at load; MLX
// model card, table "Exactness of every tensor": dequant = f32 scale * w8).
//
// GEMV design (small M). Memory-bound at M = 1: each warp streams 4 rows with
// 16-byte loads (16 weights per lane per row per step) and keeps the
// activations of up to 8 tokens in shared memory as f32. Bytes become floats
// without an integer-to-float conversion instruction: byte b (biased to
// b + 128) is placed in the mantissa of 2^23 and 2^23 + 128 is subtracted,
// which is exact. The row scale multiplies the finished dot product.
#include "kernels.h"
#include "trellis_core.cuh"

namespace escha {

namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kMaxTok = 8;

// Four signed bytes of v as exact floats.
__device__ __forceinline__ void bytes_to_f32(uint32_t v, float (&f)[4]) {
    const uint32_t u = v ^ 0x80808080u;  // b + 128 in each byte
    const float bias = 8388736.0f;       // 2^23 + 128
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
}

template <int MT>
__global__ void __launch_bounds__(256) int8_gemv_kernel(const int8_t* __restrict__ W, const float* __restrict__ scales,
                                                        int N, int Kin, const void* __restrict__ x, int x_dtype,
                                                        long long x_stride, int act, int M, float* __restrict__ y,
                                                        long long y_stride) {
    extern __shared__ __align__(16) float xs[];  // [MT][Kin]
    const int m0 = blockIdx.y * MT;
    const int mt = min(MT, M - m0);
    // 8 consecutive activations per thread and step, 16-byte loads, several
    // steps' loads in flight
#pragma unroll 4
    for (int c = threadIdx.x; c < MT * Kin / 8; c += blockDim.x) {
        const int idx = c * 8;
        const int t = idx / Kin, i = idx - t * Kin;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
        if (t < mt) {
            const long long row = (long long)(m0 + t) * x_stride;
            if (act == 1) {
                const float* yr = static_cast<const float*>(x) + row;
                const float4 g0 = *reinterpret_cast<const float4*>(yr + i);
                const float4 g1 = *reinterpret_cast<const float4*>(yr + i + 4);
                const float4 u0 = *reinterpret_cast<const float4*>(yr + Kin + i);
                const float4 u1 = *reinterpret_cast<const float4*>(yr + Kin + i + 4);
                v[0] = silu_f(g0.x) * u0.x;
                v[1] = silu_f(g0.y) * u0.y;
                v[2] = silu_f(g0.z) * u0.z;
                v[3] = silu_f(g0.w) * u0.w;
                v[4] = silu_f(g1.x) * u1.x;
                v[5] = silu_f(g1.y) * u1.y;
                v[6] = silu_f(g1.z) * u1.z;
                v[7] = silu_f(g1.w) * u1.w;
            } else if (x_dtype == 3) {
                const float* xr = static_cast<const float*>(x) + row + i;
                const float4 a0 = *reinterpret_cast<const float4*>(xr);
                const float4 a1 = *reinterpret_cast<const float4*>(xr + 4);
                v[0] = a0.x;
                v[1] = a0.y;
                v[2] = a0.z;
                v[3] = a0.w;
                v[4] = a1.x;
                v[5] = a1.y;
                v[6] = a1.z;
                v[7] = a1.w;
            } else {
                const uint4 hv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + row + i);
                const uint32_t w[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint16_t lo = static_cast<uint16_t>(w[q] & 0xFFFFu), hi = static_cast<uint16_t>(w[q] >> 16);
                    v[2 * q] = x_dtype == 1 ? h2f_bits(lo) : bf2f_bits(lo);
                    v[2 * q + 1] = x_dtype == 1 ? h2f_bits(hi) : bf2f_bits(hi);
                }
            }
        }
        *reinterpret_cast<float4*>(xs + xs_swz(idx)) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(xs + xs_swz(idx + 4)) = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * 8;
    for (int r0 = (blockIdx.x * 8 + warp) * kRowsPerWarp; r0 < N; r0 += warps_total * kRowsPerWarp) {
        float acc[kRowsPerWarp][MT];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[r][t] = 0.f;
        for (int i0 = lane * 16; i0 < Kin; i0 += 512) {
            uint4 wv[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int row = min(r0 + r, N - 1);
                wv[r] = ldg_stream_v4(W + (long long)row * Kin + i0);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float xq[MT][4];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const float4 xv = *reinterpret_cast<const float4*>(xs + xs_swz(t * Kin + i0 + 4 * q));
                    xq[t][0] = xv.x;
                    xq[t][1] = xv.y;
                    xq[t][2] = xv.z;
                    xq[t][3] = xv.w;
                }
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    const uint32_t word = q == 0 ? wv[r].x : q == 1 ? wv[r].y : q == 2 ? wv[r].z : wv[r].w;
                    float f[4];
                    bytes_to_f32(word, f);
#pragma unroll
                    for (int t = 0; t < MT; ++t)
#pragma unroll
                        for (int b = 0; b < 4; ++b) acc[r][t] = fmaf(f[b], xq[t][b], acc[r][t]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[r][t];
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                acc[r][t] = v;
            }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                if (r0 + r >= N) break;
                const float sc = scales[r0 + r];
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    if (t < mt) y[(long long)(m0 + t) * y_stride + r0 + r] = sc * acc[r][t];
            }
        }
    }
}

__global__ void int8_dequant_kernel(const int8_t* __restrict__ W, const float* __restrict__ scales, int N, int Kin,
                                    float* __restrict__ out) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)N * Kin) return;
    const int o = static_cast<int>(idx / Kin);
    out[idx] = __fmul_rn(scales[o], static_cast<float>(W[idx]));
}

// M = 1, enough loads in flight to stream the matrix at HBM rate. A tile is
// G row groups of 4 rows x all nch 512-column chunks of those rows. Warp w of
// a CTA always takes row group w / (8/G) and CPW chunks (w % (8/G) + j*(8/G)),
// so its activations (16 per lane and chunk) are loaded once; per iteration a
// CTA takes 4/CPW consecutive tiles and each warp issues all of its 4 x 4
// row loads (16 bytes per lane) before any arithmetic. CTAs walk the tiles
// grid-stride. Warp sums go to shared memory and are added per row in chunk
// order.
template <int CPW>
__global__ void __launch_bounds__(256) int8_gemv_m1_kernel(const int8_t* __restrict__ W,
                                                           const float* __restrict__ scales, int N, int Kin,
                                                           const void* __restrict__ x, int x_dtype,
                                                           float* __restrict__ y, int G, int nch) {
    constexpr int TPI = 4 / CPW;     // tiles per iteration
    extern __shared__ float part[];  // [TPI][G][4][nch]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpg = 8 / G;           // warps per row group
    const int g = warp / wpg, cw = warp % wpg;
    const int rows_per_tile = G * kRowsPerWarp;
    const int ntiles = (N + rows_per_tile - 1) / rows_per_tile;
    // The first tiles' weight loads go out before the wait for the preceding
    // kernel (weights are never its output); x and y only after it.
    uint4 wv[TPI][CPW][kRowsPerWarp];
    auto load_tiles = [&](int t0) {
#pragma unroll
        for (int tt = 0; tt < TPI; ++tt) {
            const int r0 = ((t0 + tt) * G + g) * kRowsPerWarp;
#pragma unroll
            for (int q = 0; q < CPW; ++q) {
                const int i0 = (cw + q * wpg) * 512 + lane * 16;
                if (cw + q * wpg >= nch || i0 >= Kin || t0 + tt >= ntiles) continue;
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    wv[tt][q][r] = ldg_stream_v4(W + (long long)min(r0 + r, N - 1) * Kin + i0);
            }
        }
    };
    const int first = blockIdx.x * TPI;
    if (first < ntiles) load_tiles(first);
    pdl_wait();
    pdl_trigger();
    float xv[CPW][16];
#pragma unroll
    for (int q = 0; q < CPW; ++q) {
        const int c = cw + q * wpg;
        const int i0 = c * 512 + lane * 16;
#pragma unroll
        for (int k = 0; k < 16; ++k) xv[q][k] = 0.f;
        if (c >= nch || i0 >= Kin) continue;
        if (x_dtype == 3) {
            const float4* xp = reinterpret_cast<const float4*>(static_cast<const float*>(x) + i0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 v = __ldg(xp + u);
                xv[q][4 * u] = v.x;
                xv[q][4 * u + 1] = v.y;
                xv[q][4 * u + 2] = v.z;
                xv[q][4 * u + 3] = v.w;
            }
        } else {
            const uint4* xp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + i0);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint4 v = __ldg(xp + u);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint16_t lo = static_cast<uint16_t>(w[k] & 0xFFFFu), hi = static_cast<uint16_t>(w[k] >> 16);
                    xv[q][8 * u + 2 * k] = x_dtype == 1 ? h2f_bits(lo) : bf2f_bits(lo);
                    xv[q][8 * u + 2 * k + 1] = x_dtype == 1 ? h2f_bits(hi) : bf2f_bits(hi);
                }
            }
        }
    }
    for (int t0 = first; t0 < ntiles; t0 += gridDim.x * TPI) {
        if (t0 != first) load_tiles(t0);
#pragma unroll
        for (int tt = 0; tt < TPI; ++tt) {
#pragma unroll
            for (int q = 0; q < CPW; ++q) {
                const int c = cw + q * wpg;
                if (c >= nch) break;
                float acc[kRowsPerWarp] = {0.f, 0.f, 0.f, 0.f};
                // Kin % 16 == 0: a lane's 16 columns are all in or all out
                if (c * 512 + lane * 16 < Kin && t0 + tt < ntiles) {
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r) {
                        const uint32_t words[4] = {wv[tt][q][r].x, wv[tt][q][r].y, wv[tt][q][r].z, wv[tt][q][r].w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            float f[4];
                            bytes_to_f32(words[u], f);
#pragma unroll
                            for (int b = 0; b < 4; ++b) acc[r] = fmaf(f[b], xv[q][4 * u + b], acc[r]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    float v = acc[r];
#pragma unroll
                    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                    if (lane == 0) part[((tt * G + g) * kRowsPerWarp + r) * nch + c] = v;
                }
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < TPI * rows_per_tile; i += blockDim.x) {
            const int row = t0 * rows_per_tile + i;
            if (row < N) {
                float s = 0.f;
                for (int c = 0; c < nch; ++c) s += part[i * nch + c];
                y[row] = scales[row] * s;
            }
        }
        __syncthreads();
    }
}

template <int CPW>
cudaError_t launch_m1(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype, float* y,
                      int G, int nch, int num_sms, cudaStream_t s) {
    const int rows_per_it = (4 / CPW) * G * kRowsPerWarp;
    const int smem = rows_per_it * nch * (int)sizeof(float);
    const long long its = (N + rows_per_it - 1) / rows_per_it;
    const int grid = static_cast<int>(its < 4LL * num_sms ? its : 4LL * num_sms);
    void* args[] = {const_cast<int8_t**>(&W), const_cast<float**>(&scales), &N, &Kin, const_cast<void**>(&x),
                    &x_dtype, &y, &G, &nch};
    return launch_kernel(reinterpret_cast<const void*>(int8_gemv_m1_kernel<CPW>), dim3(grid), dim3(256), smem, true,
                         s, args);
}

template <int MT>
cudaError_t launch_mt(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                      long long x_stride, int act, int M, float* y, long long y_stride, int num_sms, cudaStream_t s) {
    const int smem = ((MT * Kin + 31) / 32 * 32) * (int)sizeof(float);  // swizzle groups of 32 floats
    auto kern = int8_gemv_kernel<MT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long row_groups = (N + 8 * kRowsPerWarp - 1) / (8 * kRowsPerWarp);
    const int gx = static_cast<int>(row_groups < 8LL * num_sms ? row_groups : 8LL * num_sms);
    dim3 grid(gx, (M + MT - 1) / MT);
    kern<<<grid, 256, smem, s>>>(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_int8_gemv(const int8_t* W, const float* scales, int N, int Kin, const void* x, int x_dtype,
                             long long x_stride, int act, int M, float* y, long long y_stride, int num_sms,
                             cudaStream_t s) {
    const int nch = (Kin + 511) / 512;
    // Batch 1 with few rows: rows x chunks spread over the CTAs. With many
    // rows (four or more row groups of 32 per SM) the whole-row kernel below
    // already has enough loads in flight and needs no shared-memory reduction.
    // route by shape alone (sized for GB300's 152 SMs), so that which kernel,
    // and which summation order, serves a shape does not depend on the device
    if (M == 1 && act == 0 && nch <= 32 && N < 32 * 4 * 152) {
        // warps per row group = chunks rounded up to a power of two (at most 8)
        const int wpg = nch > 4 ? 8 : nch > 2 ? 4 : nch;
        const int G = 8 / wpg;
        const int cpw = (nch + wpg - 1) / wpg;  // chunks per warp: 1, 2 or 4 (up to 3 rounds up to 4)
        if (cpw == 1) return launch_m1<1>(W, scales, N, Kin, x, x_dtype, y, G, nch, num_sms, s);
        if (cpw == 2) return launch_m1<2>(W, scales, N, Kin, x, x_dtype, y, G, nch, num_sms, s);
        return launch_m1<4>(W, scales, N, Kin, x, x_dtype, y, G, nch, num_sms, s);
    }
    // tokens per pass whose f32 activations fit in shared memory
    const int cap = (200 * 1024 - 128) / (4 * Kin);
    if (cap < 1) return cudaErrorInvalidValue;
    if (M == 1 || cap < 2) return launch_mt<1>(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride, num_sms, s);
    if (M == 2 || cap < 4) return launch_mt<2>(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride, num_sms, s);
    if (M <= 4 || cap < 8) return launch_mt<4>(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride, num_sms, s);
    return launch_mt<kMaxTok>(W, scales, N, Kin, x, x_dtype, x_stride, act, M, y, y_stride, num_sms, s);
}

cudaError_t launch_int8_dequant(const int8_t* W, const float* scales, int N, int Kin, float* out, cudaStream_t s) {
    const long long total = (long long)N * Kin;
    int8_dequant_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, s>>>(W, scales, N, Kin, out);
    return cudaGetLastError();
}

}  // namespace escha
