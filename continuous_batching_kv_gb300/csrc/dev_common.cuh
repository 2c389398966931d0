// Device helpers shared by the kvattn kernels: the visibility rule, mbarrier
// and TMA wrappers (inline PTX for sm_103a), bounded waits, error reporting.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace kvd {

// Device error codes written to the cache's error word.
enum : int32_t {
    DERR_NONE = 0,
    DERR_TMA_TIMEOUT = 1,     // an mbarrier wait for a TMA load gave up
    DERR_MMA_TIMEOUT = 2,     // an mbarrier wait for a tensor-core commit gave up
    DERR_BOUNDS = 3,          // an index check failed
    DERR_TMEM = 4,            // TMEM allocation returned an unusable address
    DERR_SELFTEST = 5,        // the wait self-test's wait gave up (as it must)
};

// A bounded wait gives up after this many SM clock cycles (~1 s at 2 GHz).
constexpr long long WAIT_LIMIT_CYCLES = 2000000000ll;

__device__ __forceinline__ void report(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  pdl_wait: the calling thread waits until the
// grids this one depends on have completed and their writes are visible (it
// returns at once in a grid launched without the programmatic attribute).
// pdl_trigger: this CTA lets the next grid of the stream, if that grid was
// launched with the attribute, start now; the next grid still waits for this
// one in its own pdl_wait before it reads what this one writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Everything a kernel needs to decide whether row i sees cell j.
// "llama.cpp and the ubatch", "The mask is doing the work": the cell must be
// occupied, hold the row's first sequence id, not come from a later ubatch of
// the same batch (a larger epoch, "Batch、Ubatch 与解码主循环", Part D), and --
// the position part, tested here -- not be later than the row under causal
// attention nor n_swa or more positions behind it under a sliding window
// (n_swa 0: none).  Positions are >= 0, so row_pos - cell_pos cannot overflow.
__device__ __forceinline__ bool pos_visible(int32_t causal, int32_t n_swa, int32_t row_pos, int32_t cell_pos) {
    return (!causal || cell_pos <= row_pos) && (n_swa <= 0 || row_pos - cell_pos < n_swa);
}

// The same test for hot loops: the positions a row sees form one interval
// lo .. lim (lim = row_pos under causal attention, else INT32_MAX; lo = row_pos -
// n_swa + 1 under a window, else INT32_MIN).  Positions are >= 0, so lo does not
// overflow and lo <= lim; a cell position p is inside iff p - lo <= lim - lo in
// unsigned arithmetic: one subtract and one compare per cell.
struct PosRange {
    int32_t lo;
    uint32_t span;
};
__device__ __forceinline__ PosRange pos_range(int32_t causal, int32_t n_swa, int32_t row_pos) {
    const int32_t lim = causal ? row_pos : INT32_MAX;
    const int32_t lo = n_swa > 0 ? row_pos - n_swa + 1 : INT32_MIN;
    return PosRange{lo, (uint32_t)lim - (uint32_t)lo};
}
__device__ __forceinline__ bool pos_in(const PosRange &r, int32_t cell_pos) {
    return (uint32_t)cell_pos - (uint32_t)r.lo <= r.span;
}

// ---- shared-memory addresses ---------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
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
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking probe: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false if the wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > WAIT_LIMIT_CYCLES) return false;
    }
    return true;
}

// True in one lane of the converged warp (elect.sync over all 32 lanes).
__device__ __forceinline__ bool elect_one() {
    uint32_t p;
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
    return p != 0;
}

// ---- thread-block clusters -------------------------------------------------------
// All threads of all CTAs of the cluster meet (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of this CTA's shared address `a` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t map_cluster(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
    return v;
}

// ---- TMA ------------------------------------------------------------------------
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Warm L2 with box (x, y) of a tensor map (no data returned, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *m, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y) : "memory");
}

// Warm L2 with the 128-byte line holding p.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 2-D tiled load of box (x, y) into shared memory, completing on `bar`.
// x (the innermost coordinate) must be a multiple of 8 for 16-bit data.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, int32_t x, int32_t y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y),
          "r"(smem_u32(bar))
        : "memory");
}

// Bulk copy of `bytes` contiguous bytes (a multiple of 16, both addresses
// 16-byte aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bulk copy of `bytes` contiguous bytes (a multiple of 16, both addresses
// 16-byte aligned) from shared to global memory, in this thread's current bulk
// group; bulk_commit closes the group, bulk_wait_read<N> waits until at most N
// of this thread's groups still read their shared source, bulk_wait_all until
// every group of this thread has completed its writes.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 2-D tiled store of box (x, y) from shared memory, in this thread's current bulk
// group.  x (innermost) must be a multiple of 4 for 32-bit data; x, y >= 0.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, int32_t x, int32_t y, const void *src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}

// Order this thread's async-proxy global accesses with its generic ones.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// 3-D tiled load of box (x, y, z) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, int32_t x, int32_t y, int32_t z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile
// written by TMA with 128-byte swizzling (rows of 128 bytes, 1024-byte atoms).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace kvd
