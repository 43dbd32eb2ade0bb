// Inline-PTX wrappers shared by the library's TMA / mbarrier kernels (sm_103a): shared-memory
// addresses, mbarrier set-up, arrivals and bounded waits, 2-D tensor loads and proxy fences.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace slmoe {

// Every mbarrier wait gives up after this long (%globaltimer, ns) unless a launch sets its own
// limit: the kernel then sets its abort flag, every role leaves its loop and the launch
// reports status[2].
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;

// Bounded-wait state of one thread block, in shared memory: the abort flag every role polls
// and the time limit of each wait.
struct WaitCtl {
    int abort;
    int pad;
    unsigned long long limit_ns;
};

__device__ __forceinline__ uint32_t su32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of the given parity.  False = gave up (the limit ran out, or
// another role set the abort flag meanwhile).
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, volatile WaitCtl *wc) {
    const uint32_t a = su32(b);
    if (mbar_try(a, parity)) return true;
    const uint64_t t0 = gtimer();
    const uint64_t limit = wc->limit_ns;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(a, parity)) return true;
        if ((it & 255u) == 0) {
            if (wc->abort) return false;
            if (gtimer() - t0 > limit) {
                wc->abort = 1;
                return false;
            }
        }
    }
}
// Set-up of a block's wait state by one thread (limit_ns = 0 takes the default).
__device__ __forceinline__ void wait_ctl_init(volatile WaitCtl *wc, unsigned long long limit_ns) {
    wc->abort = 0;
    wc->limit_ns = limit_ns ? limit_ns : WAIT_LIMIT_NS;
}
// The same wait with its own time limit and no abort flag: used to drain copies still in
// flight after an abort, so that nothing lands in shared memory after the block exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *b, uint32_t parity) {
    const uint32_t a = su32(b);
    const uint64_t t0 = gtimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try(a, parity)) return true;
        if ((it & 255u) == 0 && gtimer() - t0 > WAIT_LIMIT_NS) return false;
    }
}
// After an abort: wait (bounded) for the last fill of every stage of a TMA ring whose producer
// stopped at ring position (stage, phase), so that no copy lands in shared memory after the
// block has exited.  Stages below `stage` were last filled in the current lap (parity phase),
// the others in the lap before (parity phase ^ 1), if the ring has wrapped at least once.
__device__ __forceinline__ void drain_ring(uint64_t *full, int stages, int stage, uint32_t phase, bool wrapped) {
    for (int i = 0; i < stages; ++i) {
        if (i < stage) mbar_wait_drain(&full[i], phase);
        else if (wrapped) mbar_wait_drain(&full[i], phase ^ 1);
    }
}
// 2-D tiled TMA load of one box at (c0 = innermost, c1) into shared memory; completion is
// counted in bytes on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(map), "r"(su32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
// TMA store of a box from shared memory, a 1-D bulk store, and the waits of their bulk groups
// (this thread's groups only)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
                 "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
// The same box added element-wise into global memory (the reduction done by the memory
// system; the element type is the tensor map's).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one group still reading shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// no group still reading shared memory
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every group complete (its writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Named barrier of the four warps of one half of the epilogue (ids 1 and 2), and the same
// barrier returning whether the predicate held in every thread.
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool group_all(int id, bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

}  // namespace slmoe
