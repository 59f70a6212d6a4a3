// Blackwell 5th-generation tensor core primitives (tcgen05, sm_100a/sm_103a)
// as inline PTX, plus the shared-memory layouts the MMAs read.
//
// Operand layouts used here (both 128-byte swizzled, 1024-byte aligned atoms):
//
//  * K-major (element (row, k) of a tile whose rows hold 64 16-bit values
//    along K): rows are 128 B apart, 8-row groups ("atoms", 1 KB) follow each
//    other; inside a row the 16-byte chunk c is stored at chunk c ^ (row % 8).
//    Descriptor: start = tile + 32 B per 16-element K step, SBO = 1024 B.
//
//  * MN-major (element (m, k), m contiguous): an atom holds 64 m values
//    (128 B) for 8 consecutive k; inside the atom, the row of k is 128 B
//    long and chunk c of that row is stored at chunk c ^ (k % 8). Atoms for
//    the next 64 m are LBO bytes apart, atoms for the next 8 k SBO bytes
//    apart; a 16-element K step advances the start address by 2 * SBO.
//
// These encodings were checked on GB300 against a CPU matrix product (M=128,
// N = 16/64/256, K = 64, f16 operands, both A layouts); exchanging LBO and SBO
// in the MN-major descriptor gives wrong results, as it must.
#pragma once

#include <stdint.h>

namespace escha {
namespace tc {

// 64-bit shared-memory matrix descriptor: start address, leading- and
// stride-dimension byte offsets (all >> 4), version 1 (bits 46-47), swizzle
// mode in bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
    return d;
}

constexpr uint32_t kSwizzle128B = 2;

// 32-bit instruction descriptor of tcgen05.mma .kind::f16: D f32 (bits 4-5 =
// 1), A/B element type (bits 7-9 / 10-12: 0 = f16, 1 = bf16), A/B major-ness
// (bit 15 / 16: 0 = K-major, 1 = MN-major), N >> 3 (bits 17-22), M >> 4
// (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
           ((static_cast<uint32_t>(M) >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (row, k) in a K-major 128-byte-swizzled tile
// (64 16-bit values per row).
__host__ __device__ __forceinline__ uint32_t kmajor_off(uint32_t row, uint32_t k) {
    const uint32_t chunk = (k >> 3) ^ (row & 7u);
    return (row >> 3) * 1024u + (row & 7u) * 128u + chunk * 16u + (k & 7u) * 2u;
}

// Byte offset of element (m, k) in an MN-major 128-byte-swizzled tile with
// atoms of 64 m x 8 k; atoms along m are `lbo` bytes apart, along k `sbo`.
__host__ __device__ __forceinline__ uint32_t mnmajor_off(uint32_t m, uint32_t k, uint32_t lbo, uint32_t sbo) {
    const uint32_t chunk = ((m & 63u) >> 3) ^ (k & 7u);
    return (m >> 6) * lbo + (k >> 3) * sbo + (k & 7u) * 128u + chunk * 16u + (m & 7u) * 2u;
}

// ---- TMEM allocation (one warp) ------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- MMA (one thread) ------------------------------------------------------
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Arrive (once) on an mbarrier when all previously issued tcgen05 async
// operations of this thread have completed.
__device__ __forceinline__ void commit(uint32_t mbar_saddr) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_saddr)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Generic-proxy shared-memory writes made visible to the tensor core (async
// proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMEM -> registers (one warp, its 32 lanes; 16 consecutive columns) ---
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- mbarrier (CTA-local) -------------------------------------------------
__device__ __forceinline__ void mbar_init_cta(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test_parity(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for `parity`; returns false (and leaves the barrier) when the
// iteration limit is hit.
__device__ __forceinline__ bool mbar_wait_parity_bounded(uint32_t bar, uint32_t parity, long long limit = 1ll << 24) {
    for (long long it = 0; it < limit; ++it)
        if (mbar_test_parity(bar, parity)) return true;
    return false;
}
// One arrival that also announces `bytes` of bulk-copy data to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// ---- bulk copy global -> shared (the TMA's untiled form) -----------------
// Both addresses 16-byte aligned, bytes a multiple of 16; completion is
// signalled to the mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_saddr, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_saddr),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

}  // namespace tc
}  // namespace escha
