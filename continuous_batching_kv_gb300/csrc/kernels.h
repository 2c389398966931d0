// Launch interfaces of the kvattn kernels (host side of each .cu file).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace kvk {

// One unit of attention work: tile-list entries [t0, t1) of one block, run
// by CTA column `cta`.  A block's items are consecutive; an item's index
// (within its path) names its split-K partial slot.
// Most CTA columns a prefill grid may have (the planner stages one entry per column).
constexpr int32_t PLAN_MAX_COLS = 1024;

struct WorkItem {
    int32_t block;
    int32_t t0;
    int32_t t1;
    int32_t cta;
};

// Read-only view of one ubatch's planning inputs and the cell mirror.
struct UbView {
    const int32_t *cell_pos;      // mirror
    const uint32_t *cell_epoch;
    const uint64_t *cell_bits;
    int32_t n_words;
    uint32_t ub_epoch;
    int32_t causal;
    int32_t kv_size;
    int32_t n_kv;
    int32_t n_tokens;
    int32_t n_blocks;
    int32_t n_dec_blocks;
    const kvi::DevRow *rows;      // [n_tokens]
    const int32_t *perm;          // [n_tokens]
    const kvi::DevBlock *blocks;  // [n_blocks]
    const int32_t *seq_blk_off;   // [n_seq_max + 1]
    const int32_t *seq_blk;       // [n_blocks]
    int32_t n_swa;                // sliding window in positions (0: none)
};

// Attention plan buffers (library-owned device memory).
constexpr int32_t DEC_FIRST = 16;   // ints per decode start record (see Plan::dec_first)

struct Plan {
    uint32_t *flags;        // [max_blocks][tile_stride]: bits 0..15 visible (row, cell)
                            // pairs in the 64-cell tile, bits 16..23 which 8-cell groups
                            // hold a visible pair
    int32_t *tiles;         // [max_blocks][tile_stride] compacted tile lists
    int32_t *cum;           // [max_blocks][tile_stride] decode cost of the listed tiles before each:
                            // a fully visible tile 8, another 2 + its number of visible 8-cell groups
    int32_t *wcount;        // [max_blocks] total decode cost of each block's list
    int32_t *counts;        // [max_blocks]
    WorkItem *work;         // decode items [0, cap_dec), prefill items [cap_dec, +cap_pf)
    int32_t *n_work;        // [2] decode / prefill item counts
    int32_t *blk_item0;     // [max_blocks] first item of each block
    int32_t *blk_nitems;    // [max_blocks]
    int32_t *counters;      // [max_blocks * n_head_kv] split-K completion counters (zero between launches)
    int32_t *cta_item0;     // decode [gx_dec + 1], then prefill [gx_pf + 1]: each CTA column's items
    int32_t *pf_rows;       // [gx_pf][PF_M]: the ubatch row behind each query vector of each prefill
                            // CTA column's first item (-1: none), so that Q loads without the
                            // chain item -> block -> row permutation
    int32_t *pf_first;      // [gx_pf][4]: each prefill CTA column's first pair: TMA rows of its two
                            // tiles (-TILE: no second tile), 1 if fully visible; [0] < 0: none
    int32_t *dec_first;     // [gx_dec][DEC_FIRST]: each decode CTA column's start record, so that
                            // its first window needs no dependent load: the first item's first
                            // four list entries (tile, -1 past the item) and their flags, its
                            // block, t0, t1, the block's first cache row (stream * kv_size), row
                            // count and first sequence id; block -1: no item
    int32_t *err;
    int32_t tile_stride;
    int32_t cap_dec, cap_pf;
    int32_t pf_cluster;     // prefill CTAs per thread-block cluster along the columns (1: none);
                            // > 1: a split block's pieces are the last items of one cluster's
                            // columns and are merged through distributed shared memory
    int32_t gqa;            // query heads per KV head
};

// k_store.cu
cudaError_t launch_store(void *k_cache, void *v_cache, const void *k_cur, const void *v_cur,
                         const kvi::DevRow *rows, int32_t n_tokens, int32_t row_bytes,
                         int64_t n_cells, int32_t *err, int32_t n_sm, cudaStream_t st);
// src: mapped pinned host memory (device-visible address); dst: device memory
cudaError_t launch_upload(const void *src, void *dst, size_t bytes, int32_t n_sm, cudaStream_t st);
cudaError_t launch_apply_deltas(const kvi::Delta *d, int32_t n, int32_t n_words, int32_t *pos,
                                uint32_t *epoch, uint64_t *bits, cudaStream_t st);
// one wait that runs out (~1 s), reported to err as DERR_SELFTEST
cudaError_t launch_wait_selftest(int32_t *err, cudaStream_t st);

// Per device, at cache creation (the device current): load every kernel's
// module and set the attributes launches rely on, so that later calls obtain
// no device memory for code or static data (modules load lazily otherwise).
cudaError_t load_store_kernels();
cudaError_t load_plan_kernels();
cudaError_t load_decode_kernels();
cudaError_t load_prefill_kernels();
int prefill_max_active_clusters(int cluster);

// k_plan.cu
cudaError_t launch_plan(const UbView &u, const Plan &p, int32_t n_stream, int32_t gx_dec, int32_t gx_pf,
                        cudaStream_t st);
cudaError_t launch_mask(const UbView &u, uint16_t *mask, cudaStream_t st);

// k_decode.cu
struct DecodeArgs {
    UbView u;
    Plan p;
    const __half *q;        // [n_tokens][n_head][128]
    float *o;               // [n_tokens][n_head][128]
    float *part;            // split-K partials [cap_dec][n_head_kv][DEC_QMAX][2 + 128]
    int32_t n_head, n_head_kv, gqa;
    float scale_log2;       // log2(e) / sqrt(head_dim)
    int32_t *err;
    int32_t nq_max;         // most query vectors in one decode block of this ubatch (1..DEC_QMAX)
    int32_t early_ok;       // as in PrefillArgs
};
// tm: the layer's K and V maps with 64-row boxes, then with 8-row boxes
cudaError_t launch_decode(const CUtensorMap *tm, const DecodeArgs &a, int32_t grid_x, cudaStream_t st);
int32_t decode_ctas_per_sm();

// k_prefill.cu
struct PrefillArgs {
    UbView u;
    Plan p;
    const __half *q;
    float *o;
    float *part;            // O rows of the partials: [cap_pf][n_head_kv][PF_M][128]
    float *part_ml;         // their (m, l): [cap_pf][n_head_kv][PF_M][2]
    int32_t n_head, n_head_kv, gqa;
    int32_t gx_dec;         // decode grid columns (offset of the prefill cta_item0 table)
    int32_t q_tma;          // 1: Q of blocks with consecutive rows loads by TMA through tm_q
    float scale_log2;
    int32_t *err;
    int32_t cluster;        // Plan::pf_cluster of the launch (its cluster dimension along x)
    int32_t early_ok;       // 1: the plan, tables and cell mirror were complete before the
                            // previous kernel of the stream began, so they may be read before
                            // waiting for it (the kernel is launched as a programmatic dependent)
};
// tm_part: the partials' O rows as a 2-D fp32 matrix (32 x 32 boxes, 128-byte swizzle);
// tm_q: q as a 3-D fp16 tensor (d, head, token) with (64, gqa, 128 / gqa) boxes, used when
// a.q_tma is set
cudaError_t launch_prefill(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const CUtensorMap *tm_part,
                           const CUtensorMap *tm_q, const PrefillArgs &a, int32_t grid_x, cudaStream_t st);

}  // namespace kvk
