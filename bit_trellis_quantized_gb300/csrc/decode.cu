// Dense decode of a trellis code tensor to fp16 weights W[in][out]: the
// diagnostic counterpart of the fused GEMV, used to check the decode bit for
// bit (hipfire PR #694, commit "Task 7 (G2): one-shot decode of Escha-W2
// packed trellis tiles into bare fp16 weights"). Not on the hot path.
//
// One thread per half-row (8 weights) of a 16x16 tile. Tile words form a
// cyclic bit stream, most significant bit of each word first; weight
// t = 16*r + q takes the 16 bits starting at bit t*K.
#include "common.cuh"
#include "kernels.h"

namespace escha {

namespace {

__global__ void trellis_decode_kernel(const uint16_t* __restrict__ codes, int KT, int NT, int K,
                                      uint16_t* __restrict__ W) {
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)KT * NT * 32;
    if (gid >= total) return;
    const int hr = static_cast<int>(gid & 31);  // half-row in the tile: row hr/2, columns 8*(hr%2)..+7
    const long long tile = gid >> 5;
    const int nt = static_cast<int>(tile % NT);
    const int kt = static_cast<int>(tile / NT);
    const int nwords = 16 * K;
    const uint16_t* tw = codes + tile * nwords;
    uint16_t outv[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int b = K * (8 * hr + m);
        const int a = b >> 4;
        const int o = b & 15;
        const uint32_t win = (static_cast<uint32_t>(tw[a]) << 16) | tw[(a + 1) % nwords];
        const uint32_t s = (win >> (16 - o)) & 0xFFFFu;
        outv[m] = __half_as_ushort(cb_decode_h(s));
    }
    const int r = hr >> 1;
    const long long row = (long long)(kt * 16 + r);
    uint16_t* dst = W + row * (NT * 16) + nt * 16 + 8 * (hr & 1);
    uint4 v;
    v.x = outv[0] | (static_cast<uint32_t>(outv[1]) << 16);
    v.y = outv[2] | (static_cast<uint32_t>(outv[3]) << 16);
    v.z = outv[4] | (static_cast<uint32_t>(outv[5]) << 16);
    v.w = outv[6] | (static_cast<uint32_t>(outv[7]) << 16);
    *reinterpret_cast<uint4*>(dst) = v;
}

}  // namespace

cudaError_t launch_trellis_decode(const uint16_t* codes, int in, int out, int K, uint16_t* W, cudaStream_t s) {
    const int KT = in / 16, NT = out / 16;
    const long long total = (long long)KT * NT * 32;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    trellis_decode_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(codes, KT, NT, K, W);
    return cudaGetLastError();
}

}  // namespace escha
