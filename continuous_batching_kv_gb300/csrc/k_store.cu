// K1: the K/V scatter (set_rows) and the cell-mirror delta apply.
//
// "What does llama.cpp's KV cache actually look like in memory?", sections
// "One row, one token's keys" and "The tensor's three dimensions": a layer's
// K tensor is rows of n_head_kv * head_dim fp16 values, one row per cell,
// streams stacked as slabs of kv_size rows; V has the same layout.  Each
// ubatch row's K (V) values go to the row of its reserved cell.

#include "dev_common.cuh"
#include "kernels.h"

namespace {

// One 16-byte chunk per thread; consecutive threads cover consecutive chunks
// of one row, so loads and stores are fully coalesced 16-byte vectors.
__global__ void __launch_bounds__(256) k_store(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                               const uint4 *__restrict__ kin,
                                               const uint4 *__restrict__ vin,
                                               const kvi::DevRow *__restrict__ rows, int32_t n_tokens,
                                               int32_t chunks_per_row, int64_t n_cells,
                                               int32_t *err) {
    // Launched as a programmatic dependent of the kernel before it: wait for it
    // before reading the rows (the caller may have just produced them) or
    // writing the cache; then let the attention kernel that follows set up.
    // Until then, warm L2 with this thread's first 128-byte lines of K and V (a
    // prefetch returns nothing, so racing the previous kernel's writes is harmless).
    const int64_t total = (int64_t)n_tokens * chunks_per_row;
    {
        const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        if (t0 < total && (t0 & 7) == 0) {
            kvd::prefetch_l2(kin + t0);
            kvd::prefetch_l2(vin + t0);
        }
    }
    kvd::pdl_wait();
    kvd::pdl_trigger();
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int32_t r = (int32_t)(t / chunks_per_row);
        const int32_t c = (int32_t)(t - (int64_t)r * chunks_per_row);
        const int64_t cell = rows[r].cell;
        if (cell < 0 || cell >= n_cells) {
            kvd::report(err, kvd::DERR_BOUNDS);
            continue;
        }
        const int64_t dst = cell * chunks_per_row + c;
        const uint4 kv = __ldg(kin + t);
        const uint4 vv = __ldg(vin + t);
        kc[dst] = kv;
        vc[dst] = vv;
    }
}

// Host -> device upload through mapped pinned memory: the kernel reads the host
// buffer directly, so the upload does not queue on a copy engine behind the
// caller's own transfers.  16-byte chunks, then the remaining bytes.
__global__ void __launch_bounds__(256) k_upload(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                int64_t n16, int32_t tail) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
    if (blockIdx.x == 0 && threadIdx.x < (unsigned)tail)
        reinterpret_cast<uint8_t *>(dst + n16)[threadIdx.x] = reinterpret_cast<const uint8_t *>(src + n16)[threadIdx.x];
}

__global__ void k_apply_deltas(const kvi::Delta *__restrict__ d, int32_t n, int32_t n_words,
                               int32_t *pos, uint32_t *epoch, uint64_t *bits) {
    int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const kvi::Delta r = d[i];
    pos[r.cell] = r.pos;
    epoch[r.cell] = r.epoch;
    for (int32_t w = 0; w < n_words; ++w) bits[(int64_t)r.cell * n_words + w] = r.bits[w];
}

// The bounded-wait path, exercised: one thread waits on an mbarrier that nothing
// arrives at, with the limit every wait of the attention kernels uses; when the
// wait gives up (after ~1 s), the error word is set, as a kernel whose copy or
// commit never came would set it, and the kernel returns normally.
__global__ void k_wait_selftest(int32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    kvd::mbar_init(&bar, 1);
    kvd::fence_mbar_init();
    if (!kvd::mbar_wait_bounded(&bar, 0)) kvd::report(err, kvd::DERR_SELFTEST);
}

}  // namespace

namespace kvk {

cudaError_t launch_wait_selftest(int32_t *err, cudaStream_t st) {
    k_wait_selftest<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

cudaError_t launch_store(void *k_cache, void *v_cache, const void *k_cur, const void *v_cur,
                         const kvi::DevRow *rows, int32_t n_tokens, int32_t row_bytes,
                         int64_t n_cells, int32_t *err, int32_t n_sm, cudaStream_t st) {
    const int32_t cpr = row_bytes / 16;
    const int64_t total = (int64_t)n_tokens * cpr;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)n_sm * 16) blocks = (int64_t)n_sm * 16;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_store, (uint4 *)k_cache, (uint4 *)v_cache, (const uint4 *)k_cur,
                                       (const uint4 *)v_cur, rows, n_tokens, cpr, n_cells, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_upload(const void *src, void *dst, size_t bytes, int32_t n_sm, cudaStream_t st) {
    const int64_t n16 = (int64_t)(bytes / 16);
    int64_t blocks = (n16 + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > (int64_t)n_sm * 4) blocks = (int64_t)n_sm * 4;
    k_upload<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16,
                                                (int32_t)(bytes % 16));
    return cudaGetLastError();
}

cudaError_t load_store_kernels() {
    cudaFuncAttributes fa;
    cudaError_t e;
    if ((e = cudaFuncGetAttributes(&fa, k_store)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, k_upload)) != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, k_apply_deltas);
}

cudaError_t launch_apply_deltas(const kvi::Delta *d, int32_t n, int32_t n_words, int32_t *pos,
                                uint32_t *epoch, uint64_t *bits, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    k_apply_deltas<<<(n + 255) / 256, 256, 0, st>>>(d, n, n_words, pos, epoch, bits);
    return cudaGetLastError();
}

}  // namespace kvk
