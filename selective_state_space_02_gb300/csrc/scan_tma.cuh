// TMA (cp.async.bulk.tensor) and mbarrier helpers, inline PTX for sm_103a,
// plus the host-side tensor-map encoder (driver entry point, no libcuda link).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace ssm {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the barrier's phase with this parity has completed.  The wait is
// bounded by `limit` SM cycles: past the bound bit 0 of *status is set and the
// wait returns false instead of spinning forever.
__device__ __forceinline__ bool wait_parity(uint64_t *bar, uint32_t parity, unsigned int *status,
                                            long long limit = (1ll << 31)) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long start = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - start > limit) {
            atomicOr(status, 1u);
            return false;
        }
    }
    return true;
}

// 2-D tiled TMA load of box [rows][cols] at (col0, row0) into shared memory,
// completing `bar`'s transaction count.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int col0, int row0,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col0), "r"(row0), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completing `bar`'s transaction count.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy from shared to global memory in the issuing thread's current
// bulk group (same size and alignment rules).
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the shared-memory sources of all but the newest N committed bulk
// groups of this thread have been read (the memory may then be reused).
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Host: encode a row-major [rows][cols] tensor of `elem` bytes per element,
// box [box_rows][box_cols], zero fill out of bounds; `swizzle` 128 or 64
// selects that shared-memory swizzle (box rows of exactly that many bytes,
// destinations on 1024-byte boundaries), 0 none.  Returns false if the
// driver entry point is unavailable or rejects the map.
bool encode_tile_map(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_cols, int swizzle = 0);

// Host: the same for a float32 tensor whose rows hold `cols` values.
bool encode_f32_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols);

}  // namespace ssm
