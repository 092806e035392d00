// tma.cuh -- thin inline-PTX wrappers for the sm_90+/sm_100 asynchronous copy
// machinery used by the staged scan kernels: shared-memory mbarriers, tiled
// TMA tensor loads and stores (cp.async.bulk.tensor), bulk-group completion
// and the generic->async proxy fence.  Every wait here is bounded in wall
// time: a wait that gives up records kDeviceErrTimeout in the library's device error
// word (and, if given, in a caller status word) and returns false, so that a
// kernel always runs to its end instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// Device-side error bits (OR-ed together).
constexpr unsigned kDeviceErrTimeout = 1u;  // a bounded wait gave up
constexpr unsigned kDeviceErrRange = 2u;    // an access fell outside its tensor and was skipped

// Library-wide device error word, defined once in ssm_scan.cu (the library is
// built with relocatable device code, so every kernel translation unit shares
// it); read and cleared by ssm_device_status.
extern __device__ unsigned int g_ssm_device_error;

// Wall-clock budget of one wait (ns, read from %globaltimer).  A healthy wait
// here lasts microseconds; after two seconds the wait gives up.
constexpr unsigned long long kWaitBudgetNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive on the barrier and add `bytes` to the transaction count of its
// current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Plain arrive (count 1) on the barrier's current phase; release semantics
// for this thread's prior memory accesses.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete; bounded by
// budget_ns of wall time (kWaitBudgetNs unless the caller gives another).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* status,
                                          unsigned long long budget_ns = kWaitBudgetNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long start = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - start > budget_ns) {
            atomicOr(&g_ssm_device_error, kDeviceErrTimeout);
            if (status) atomicOr(status, kDeviceErrTimeout);
            return false;
        }
    }
    return true;
}

// 2-D / 3-D tiled tensor loads global -> shared, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// 2-D tiled tensor store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_addr(src))
                 : "memory");
}

// 3-D tiled tensor store shared -> global (bulk-group completion).  Elements of
// the box that fall outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z, const void* src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until at most N committed bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream still runs;
// grid_dep_wait() blocks until that kernel has completed and its writes are
// visible (a no-op without the launch attribute), and grid_dep_launch() lets
// the next such kernel start launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Byte offset of 16-byte chunk c (0..3) of row r inside a tile whose rows are
// 64 bytes and which TMA wrote with CU_TENSOR_MAP_SWIZZLE_64B: address bits
// [4:5] are XOR-ed with bits [7:8], i.e. with (r >> 1) & 3.  The tile base must
// be 512-byte aligned.
__device__ __forceinline__ uint32_t swz64(int r, int c) {
    return static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// The same for 32-byte rows written with CU_TENSOR_MAP_SWIZZLE_32B: address bit
// 4 is XOR-ed with bit 7, i.e. with (r >> 2) & 1.  The tile base must be
// 256-byte aligned.
__device__ __forceinline__ uint32_t swz32(int r, int c) {
    return static_cast<uint32_t>(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
}

// The same for 128-byte rows written with CU_TENSOR_MAP_SWIZZLE_128B: address
// bits [4:6] are XOR-ed with bits [7:9], i.e. with r & 7.  The tile base must
// be 1024-byte aligned.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Byte offset of 16-byte chunk c of row r in a tile of RB-byte rows written
// by TMA with the swizzle of that row width (32, 64 or 128 bytes).
template <int RB>
__device__ __forceinline__ uint32_t swz_rows(int r, int c) {
    static_assert(RB == 32 || RB == 64 || RB == 128, "tile rows are 32, 64 or 128 bytes");
    if constexpr (RB == 32) return swz32(r, c);
    else if constexpr (RB == 64) return swz64(r, c);
    else return swz128(r, c);
}

}  // namespace ssm
