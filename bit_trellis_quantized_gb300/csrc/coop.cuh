// Hand-over between the CTAs of one cooperative grid (sm_103a): arrival
// counters in global memory and bounded waits on them. A wait that runs out
// sets a status word and returns false, so a kernel built on these always
// ends; the caller skips the work that needed the data.
#pragma once

#include <stdint.h>

namespace escha {

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Arrival counts: the CTA's writes before the barrier that precedes the add
// are released with it (acq_rel also acquires the other arrivals' writes,
// for the CTA that turns out to be last); red: release only.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A 64-bit word published whole: the writer's earlier writes are released
// with it, and a reader that sees it acquires them.
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One thread: true once *p >= target; after wait_ns without it, records
// `code` in *err unless an earlier wait already did (so the status word names
// the first wait that ran out, not the waits that then starve behind it) and
// returns false. Between polls the thread sleeps a little, so that waiting
// CTAs take few issue slots from the warps working beside them on the SM and
// few L2 accesses from everyone.
__device__ __forceinline__ bool wait_geq(const unsigned* p, unsigned target, long long wait_ns, int* err, int code) {
    if (ld_acquire(p) >= target) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        __nanosleep(200);
        if (ld_acquire(p) >= target) return true;
        if (static_cast<long long>(global_ns() - t0) > wait_ns) {
            atomicCAS(err, 0, code);
            return false;
        }
    }
}

// The whole CTA: thread 0 waits, the others learn the outcome at the barrier.
__device__ __forceinline__ bool cta_wait_geq(const unsigned* p, unsigned target, long long wait_ns, int* err, int code) {
    int ok = 1;
    if (threadIdx.x == 0) ok = wait_geq(p, target, wait_ns, err, code);
    return __syncthreads_and(ok) != 0;
}

}  // namespace escha
