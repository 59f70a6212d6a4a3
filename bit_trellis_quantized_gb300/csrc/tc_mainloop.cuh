// Main loop shared by the tensor-core GEMMs whose A operand is made by the
// CTA's own threads (trellis decode, int8 -> 16-bit conversion) and whose B
// operand is a prepared image in global memory.
//
//   D[128][N] (TMEM, f32) = sum over K blocks of 128:  A_blk[128][128] * B_blk[N][128]^T
//
// Per K block, 256 threads produce A into one of two 32 KB shared buffers
// while the MMAs of the previous block run; one thread issues the eight
// K = 16 MMAs of the block and the bulk copy of the next block's B (two
// 64-value chunks of N rows x 128 B each, K-major 128-byte swizzled, copied
// as they lie in the image) into one of two B buffers.
//
// The B image holds, for every 64-value K chunk, all rows one after the
// other (row r at r * 128 B, 16-byte pieces swizzled by r % 8), so a CTA's
// rows are one contiguous range per chunk; a range starting at a multiple of
// 8 rows lands in shared memory with the swizzle phase the MMA expects.
#pragma once

#include "tcgen05.cuh"

namespace escha {
namespace tc {

constexpr int kMlThreads = 256;
constexpr int kABlockBytes = 32768;  // 128 x 128 16-bit values

struct MmaBars {
    unsigned long long full[2];  // B block landed
    unsigned long long done[2];  // MMAs of the block finished reading A and B
};

__device__ __forceinline__ void mma_bars_init(MmaBars& bars) {
    mbar_init_cta(smem_addr(&bars.full[0]), 1);
    mbar_init_cta(smem_addr(&bars.full[1]), 1);
    mbar_init_cta(smem_addr(&bars.done[0]), 1);
    mbar_init_cta(smem_addr(&bars.done[1]), 1);
    fence_proxy_async_smem();
}

// A_MN: A is MN-major (eight 4 KB slices, one per K = 16 step, atoms of 64 m
// 2048 B apart and of 8 k 1024 B apart) or K-major (two 16 KB chunks of 128
// rows x 64 values). `produce(b, A)` writes block b's A into A and is called
// by every thread. `img` points at the CTA's first row in chunk 0;
// consecutive chunks are `img_chunk_bytes` apart. Returns false in every
// thread when a bounded wait gave up.
//
// KSTEPS = 8: blocks of 128 values (A 32 KB, B two 64-value chunks);
// KSTEPS = 4: blocks of 64 values (A 16 KB, B one chunk); A_MN slices are
// 4 KB per K = 16 step either way.
template <bool A_MN, int KSTEPS = 8, class ProduceA>
__device__ __forceinline__ bool mma_mainloop(uint8_t* Abuf, uint8_t* Bbuf, uint32_t b_chunk_bytes, const uint8_t* img,
                                             long long img_chunk_bytes, uint32_t copy_bytes, int nblk, uint32_t tmem,
                                             uint32_t idesc, MmaBars& bars, ProduceA&& produce) {
    static_assert(KSTEPS == 4 || KSTEPS == 8, "blocks of 64 or 128 values");
    constexpr int kChunks = KSTEPS / 4;
    constexpr int kABytes = KSTEPS * 4096;
    const int tid = threadIdx.x;
    bool ok = true;
    auto issue_b = [&](int b) {
        const int buf = b & 1;
        const uint32_t bar = smem_addr(&bars.full[buf]);
        mbar_arrive_expect_tx(bar, kChunks * copy_bytes);
        uint8_t* dst = Bbuf + buf * kChunks * b_chunk_bytes;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
            bulk_g2s(smem_addr(dst + c * b_chunk_bytes), img + ((long long)kChunks * b + c) * img_chunk_bytes,
                     copy_bytes, bar);
    };
    if (tid == 0) issue_b(0);
    for (int b = 0; b < nblk; ++b) {
        const int buf = b & 1;
        // the MMAs of block b-2 have finished with this A buffer
        if (b >= 2 && !mbar_wait_parity_bounded(smem_addr(&bars.done[buf]), ((b >> 1) - 1) & 1)) ok = false;
        uint8_t* A = Abuf + buf * kABytes;
        produce(b, A);
        fence_proxy_async_smem();
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            fence_after_sync();
            if (!mbar_wait_parity_bounded(smem_addr(&bars.full[buf]), (b >> 1) & 1)) ok = false;
            const uint8_t* B = Bbuf + buf * kChunks * b_chunk_bytes;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const uint64_t ad =
                    A_MN ? smem_desc(smem_addr(A + kk * 4096), 2048u, 1024u, kSwizzle128B)
                         : smem_desc(smem_addr(A + (kk >> 2) * 16384) + (kk & 3) * 32u, 16u, 1024u, kSwizzle128B);
                const uint64_t bd =
                    smem_desc(smem_addr(B + (kk >> 2) * b_chunk_bytes) + (kk & 3) * 32u, 16u, 1024u, kSwizzle128B);
                mma_f16(tmem, ad, bd, idesc, b > 0 || kk > 0);
            }
            commit(smem_addr(&bars.done[buf]));
            if (b + 1 < nblk) {
                // the next B block goes into the buffer the MMAs of block b-1 read
                if (b >= 1 && !mbar_wait_parity_bounded(smem_addr(&bars.done[(b + 1) & 1]), ((b - 1) >> 1) & 1))
                    ok = false;
                issue_b(b + 1);
            }
        }
    }
    // the last commit covers every MMA issued before it; wait for the other
    // buffer's final phase too so that no arrival is pending at exit
    const int last = nblk - 1;
    if (!mbar_wait_parity_bounded(smem_addr(&bars.done[last & 1]), (last >> 1) & 1)) ok = false;
    if (nblk >= 2 && !mbar_wait_parity_bounded(smem_addr(&bars.done[(last - 1) & 1]), ((last - 1) >> 1) & 1))
        ok = false;
    fence_after_sync();
    return !__syncthreads_or(!ok);
}

}  // namespace tc
}  // namespace escha

namespace escha {
namespace tc {

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Two producer groups of 256 threads (warps 0-7 and 8-15) take alternate K
// blocks (group g: blocks g, g+2, ...). Each group has its own A buffer, B
// buffer, barrier pair and TMEM accumulator (columns g*acc_cols ..), so one
// group decodes while the other's MMAs run; the caller adds the two
// accumulators (group 1 holds nothing when nblk == 1). `produce(b, b_next, A)`
// writes block b's A and may prefetch block b_next (>= nblk: none); it is
// called by the group's 256 threads.
template <bool A_MN, class ProduceA>
__device__ __forceinline__ bool mma_mainloop_2grp(uint8_t* Abuf, uint8_t* Bbuf, uint32_t b_chunk_bytes,
                                                  const uint8_t* img, long long img_chunk_bytes, uint32_t copy_bytes,
                                                  int nblk, uint32_t tmem, uint32_t acc_cols, uint32_t idesc,
                                                  MmaBars& bars, ProduceA&& produce) {
    const int g = threadIdx.x >> 8;
    const bool leader = (threadIdx.x & 255) == 0;
    uint8_t* A = Abuf + g * kABlockBytes;
    uint8_t* B = Bbuf + g * 2 * b_chunk_bytes;
    const uint32_t full = smem_addr(&bars.full[g]), done = smem_addr(&bars.done[g]);
    const uint32_t acc = tmem + static_cast<uint32_t>(g) * acc_cols;
    bool ok = true;
    int k = 0;
    for (int b = g; b < nblk; b += 2, ++k) {
        // the group's previous MMAs have finished with its A and B buffers
        if (k >= 1 && !mbar_wait_parity_bounded(done, (k - 1) & 1)) ok = false;
        if (leader) {
            mbar_arrive_expect_tx(full, 2u * copy_bytes);
            bulk_g2s(smem_addr(B), img + (2ll * b) * img_chunk_bytes, copy_bytes, full);
            bulk_g2s(smem_addr(B + b_chunk_bytes), img + (2ll * b + 1) * img_chunk_bytes, copy_bytes, full);
        }
        produce(b, b + 2, A);
        fence_proxy_async_smem();
        fence_before_sync();
        named_barrier_sync(1 + g, 256);
        if (leader) {
            fence_after_sync();
            if (!mbar_wait_parity_bounded(full, k & 1)) ok = false;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad =
                    A_MN ? smem_desc(smem_addr(A + kk * 4096), 2048u, 1024u, kSwizzle128B)
                         : smem_desc(smem_addr(A + (kk >> 2) * 16384) + (kk & 3) * 32u, 16u, 1024u, kSwizzle128B);
                const uint64_t bd =
                    smem_desc(smem_addr(B + (kk >> 2) * b_chunk_bytes) + (kk & 3) * 32u, 16u, 1024u, kSwizzle128B);
                mma_f16(acc, ad, bd, idesc, k > 0 || kk > 0);
            }
            commit(done);
        }
    }
    if (k >= 1 && !mbar_wait_parity_bounded(done, (k - 1) & 1)) ok = false;
    fence_after_sync();
    return !__syncthreads_or(!ok);
}

}  // namespace tc
}  // namespace escha

namespace escha {
namespace tc {

// Warp-specialised main loop over 64-value K chunks in STAGES stages (A:
// 16 KB per chunk, K-major 128 rows x 64 values or MN-major four 4 KB slices;
// B: up to 256 rows x 128 B), for kernels of 256 producer threads (warps
// 0-7) + one issuer warp (warp 8):
//  * producers: for chunk c, wait until the MMAs of chunk c - STAGES released
//    stage c % STAGES, write A (`produce(c, A_stage)`), fence, arrive on
//    a_full;
//  * issuer (one thread): B copies run STAGES - 1 chunks ahead; per chunk wait
//    a_full and b_full, issue four K = 16 MMAs, commit to done; then wait for
//    the MMAs of chunk c - 1 and copy chunk c + STAGES - 1's B into the stage
//    they released.
// No CTA-wide barrier inside the loop. Returns false in every thread when a
// bounded wait gave up.
constexpr int kWsStages = 4;
constexpr int kWsAStageBytes = 16384;

struct WsBars {
    unsigned long long a_full[kWsStages];
    unsigned long long b_full[kWsStages];
    unsigned long long done[kWsStages];
};

__device__ __forceinline__ void ws_bars_init(WsBars& bars) {
    for (int s = 0; s < kWsStages; ++s) {
        mbar_init_cta(smem_addr(&bars.a_full[s]), kMlThreads);
        mbar_init_cta(smem_addr(&bars.b_full[s]), 1);
        mbar_init_cta(smem_addr(&bars.done[s]), 1);
    }
    fence_proxy_async_smem();
}

//
// MT = 2: two 128-row M tiles share each B chunk (A stage 2 x 16 KB, tile t at
// +16 KB), accumulating into TMEM columns [t * acc_cols, ...): the B operand is
// read from L2 once per 256 rows of A instead of once per 128.
template <int STAGES, bool A_MN, int MT = 1, class ProduceChunk>
__device__ __forceinline__ bool mma_mainloop_ws(uint8_t* Abuf, uint8_t* Bbuf, uint32_t b_stage_bytes,
                                                const uint8_t* img, long long img_chunk_bytes, uint32_t copy_bytes,
                                                int nch, uint32_t tmem, uint32_t idesc, WsBars& bars,
                                                ProduceChunk&& produce, uint32_t acc_cols = 0) {
    static_assert(STAGES >= 2 && STAGES <= kWsStages, "2 to 4 stages");
    static_assert(MT == 1 || MT == 2, "one or two M tiles");
    constexpr int kAStage = MT * kWsAStageBytes;
    const int tid = threadIdx.x;
    bool ok = true;
    if (tid < kMlThreads) {
        for (int c = 0; c < nch; ++c) {
            const int s = c % STAGES;
            if (c >= STAGES && !mbar_wait_parity_bounded(smem_addr(&bars.done[s]), ((c / STAGES) - 1) & 1))
                ok = false;
            produce(c, Abuf + s * kAStage);
            fence_proxy_async_smem();
            mbar_arrive_cta(smem_addr(&bars.a_full[s]));
        }
    } else if (tid == kMlThreads) {
        auto issue_b = [&](int c) {
            const uint32_t bar = smem_addr(&bars.b_full[c % STAGES]);
            mbar_arrive_expect_tx(bar, copy_bytes);
            bulk_g2s(smem_addr(Bbuf + (c % STAGES) * b_stage_bytes), img + (long long)c * img_chunk_bytes, copy_bytes,
                     bar);
        };
        for (int c = 0; c < nch && c < STAGES - 1; ++c) issue_b(c);
        for (int c = 0; c < nch; ++c) {
            const int s = c % STAGES;
            const uint32_t ph = (c / STAGES) & 1;
            if (!mbar_wait_parity_bounded(smem_addr(&bars.a_full[s]), ph)) ok = false;
            if (!mbar_wait_parity_bounded(smem_addr(&bars.b_full[s]), ph)) ok = false;
            fence_after_sync();
            const uint32_t a0 = smem_addr(Abuf + s * kAStage), b0 = smem_addr(Bbuf + s * b_stage_bytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = smem_desc(b0 + kk * 32u, 16u, 1024u, kSwizzle128B);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint32_t at = a0 + mt * kWsAStageBytes;
                    const uint64_t ad = A_MN ? smem_desc(at + kk * 4096u, 2048u, 1024u, kSwizzle128B)
                                             : smem_desc(at + kk * 32u, 16u, 1024u, kSwizzle128B);
                    mma_f16(tmem + mt * acc_cols, ad, bd, idesc, c > 0 || kk > 0);
                }
            }
            commit(smem_addr(&bars.done[s]));
            if (c + STAGES - 1 < nch) {
                // stage (c + STAGES - 1) % STAGES was last read by the MMAs of chunk c - 1
                if (c >= 1 && !mbar_wait_parity_bounded(smem_addr(&bars.done[(c - 1) % STAGES]),
                                                        ((c - 1) / STAGES) & 1))
                    ok = false;
                issue_b(c + STAGES - 1);
            }
        }
        // the final phase of every stage used: all MMAs complete, no arrival pending
        for (int s = 0; s < STAGES && s < nch; ++s) {
            const int last = s + ((nch - 1 - s) / STAGES) * STAGES;
            if (!mbar_wait_parity_bounded(smem_addr(&bars.done[s]), (last / STAGES) & 1)) ok = false;
        }
    }
    fence_before_sync();
    const bool bad = __syncthreads_or(!ok);
    fence_after_sync();
    return !bad;
}

}  // namespace tc
}  // namespace escha
