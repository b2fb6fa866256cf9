// Bulk-copy (TMA) and mbarrier helpers for the streaming kernels (sm_90+,
// used here on sm_103a).  One producer thread moves global data into
// shared-memory stages with cp.async.bulk (contiguous ranges) or
// cp.async.bulk.tensor (boxes of a tensor map); each stage has a "full"
// mbarrier (the copy engine completes its transaction count) and an "empty"
// mbarrier (every consumer warp arrives once it no longer reads the stage).
//
// Every wait is bounded in time.  A wait that runs out returns false; the
// caller records SPLITZIP_ERR_TIMEOUT and carries on, so no thread ever spins
// forever and every barrier is still reached.
#pragma once

#include <cstdint>

namespace splitzip {

// About one second at 2 GHz: far above any real wait (microseconds).
constexpr long long kWaitLimitCycles = 2000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false once more than
// `limit` SM clock cycles have passed without it.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// The wait every streaming kernel uses (limit kWaitLimitCycles).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, kWaitLimitCycles);
}

// Global -> shared bulk copy; completes `bytes` of the barrier's transaction
// count.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Tiled tensor-map copy of one box of a 2-D tensor into shared memory;
// completes the box's bytes on the barrier (elements outside the tensor are
// written as zeros and still counted).  `map` is the address of a
// __grid_constant__ CUtensorMap kernel parameter; x (innermost, in elements)
// times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tensor_load_2d(void* dst, const void* map, int32_t x, int32_t y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier for a subset of the CTA's warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads:
// every participant gets the same answer, so a decision taken on it keeps all
// of them on the same path through later barriers.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// Named barrier that also counts the participating threads whose predicate
// is true (the same count in every participant).
__device__ __forceinline__ uint32_t named_barrier_popc(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.popc.u32 %0, %2, %3, p;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred)), "r"(id), "r"(threads)
        : "memory");
    return r;
}

// Before a producer thread leaves: wait (bounded) until the last bulk copy of
// every stage has landed, so no copy is still writing into shared memory when
// the CTA exits.  `issued` = number of stage uses so far.
__device__ __forceinline__ bool drain_stages(uint64_t* full_bar, uint32_t stages, uint32_t issued) {
    bool ok = true;
    for (uint32_t s = 0; s < stages && s < issued; ++s) {
        // the last use of stage (issued - 1 - s) % stages
        const uint32_t it = issued - 1 - s;
        ok &= mbar_wait(&full_bar[it % stages], (it / stages) & 1u);
    }
    return ok;
}

// A 16-byte-aligned window that covers [p, p + bytes): the bulk copy moves the
// window, the reader skips `offset` bytes.
struct Window {
    const uint8_t* src;
    uint32_t bytes;
    uint32_t offset;
};

__device__ __forceinline__ Window window_of(const uint8_t* p, uint64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15);
    const uintptr_t hi = (reinterpret_cast<uintptr_t>(p) + bytes + 15) & ~uintptr_t(15);
    Window w;
    w.src = reinterpret_cast<const uint8_t*>(lo);
    w.bytes = uint32_t(hi - lo);
    w.offset = uint32_t(reinterpret_cast<uintptr_t>(p) - lo);
    return w;
}

}  // namespace splitzip
