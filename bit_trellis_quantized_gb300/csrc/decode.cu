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

// Load-time move of whole tiles from the kt-major grid [in/16][out/16] to the
// nt-major grid [out/16][in/16], so that the tiles one output tile column
// walks through are adjacent (hipfire PR #694, commit on the nt-major tile
// grid). Tile contents are untouched. One thread per 16-byte piece of a
// destination tile (2K pieces of 16 bytes per tile), in destination order.
__global__ void codes_to_nt_major_kernel(const uint4* __restrict__ src, int KT, int NT, int pieces, uint4* __restrict__ dst) {
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)KT * NT * pieces;
    if (gid >= total) return;
    const long long tile_d = gid / pieces;
    const int c = static_cast<int>(gid % pieces);
    const long long nt = tile_d / KT, kt = tile_d % KT;
    dst[gid] = src[(kt * NT + nt) * pieces + c];
}

}  // namespace

cudaError_t launch_codes_to_nt_major(const uint16_t* src, int in, int out, int K, uint16_t* dst, cudaStream_t s) {
    const int KT = in / 16, NT = out / 16, pieces = 2 * K;
    const long long total = (long long)KT * NT * pieces;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    codes_to_nt_major_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, s>>>(
        reinterpret_cast<const uint4*>(src), KT, NT, pieces, reinterpret_cast<uint4*>(dst));
    return cudaGetLastError();
}

cudaError_t launch_trellis_decode(const uint16_t* codes, int in, int out, int K, uint16_t* W, cudaStream_t s) {
    const int KT = in / 16, NT = out / 16;
    const long long total = (long long)KT * NT * 32;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    trellis_decode_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(codes, KT, NT, K, W);
    return cudaGetLastError();
}

}  // namespace escha
