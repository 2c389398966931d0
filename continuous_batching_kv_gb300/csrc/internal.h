// Internal structures shared by the host (host.cpp) and device (device.cu)
// halves of libkvattn.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cstddef>
#include <new>
#include <string>
#include <vector>

#include "../../include/kvattn.h"

namespace kvi {

// Attention paths a block of rows can take.
enum : int32_t { PATH_DECODE = 0, PATH_PREFILL = 1 };

// Rows of one group (same stream, same first sequence id) are cut into
// blocks.  A decode block holds at most DEC_QMAX query vectors (rows x GQA
// group size); a prefill block fills two 128-lane MMA tiles.
constexpr int DEC_QMAX = 16;
constexpr int PF_M = 256;
// A group takes the prefill path when it has at least this many query vectors.
constexpr int PF_MIN_QV = 64;
constexpr int PF_CLUSTER = 4;             // prefill CTAs per thread-block cluster (see device.cu)
// Cells per plan tile, and cells per TMA sub-box inside it.
constexpr int TILE = 64;
constexpr int SUB = 8;

// One row of a ubatch as the device sees it (ubatch row order).
struct DevRow {
    int32_t cell;    // global cell index: stream * kv_size + local cell
    int32_t pos;
    int32_t seq0;
    int32_t stream;
};

// A block of rows sharing (stream, seq0) that attends together.
struct DevBlock {
    int32_t row0;    // first entry in the block-sorted row permutation
    int32_t n_rows;
    int32_t seq0;
    int32_t stream;
    int32_t path;    // PATH_DECODE / PATH_PREFILL
    int32_t pos_min;
    int32_t pos_max;
    int32_t tok0;    // first ubatch row when the block's rows are consecutive ubatch rows in
                     // order (perm[row0 + i] == tok0 + i), else -1
    int32_t contig;  // 1: the rows' positions are pos_min .. pos_max, each once (in any order)
};

// Host-side per-ubatch tables (filled at split / prepare time).
struct UbatchHost {
    int32_t n_tokens = 0, n_seq_tokens = 0, n_seqs = 0;
    int32_t n_kv = 0;
    uint32_t epoch = 0;            // serial of this ubatch: cells it filled carry it
    std::vector<int32_t> rows, pos, seq0, streams, cells, seq_unq;
    std::vector<int32_t> ids_off, ids;   // CSR: every sequence id of each row
    // attention planning (built at prepare)
    std::vector<int32_t> perm;     // block-sorted ubatch row indices
    std::vector<DevBlock> blocks;
    int32_t n_dec_blocks = 0, n_pf_blocks = 0;
    std::vector<int32_t> seq_blk_off;   // [n_seq_max + 1] CSR: blocks per sequence
    std::vector<int32_t> seq_blk;       // block ids
};

}  // namespace kvi

struct kv_split {
    uint64_t id = 0;
    kv_cache *owner = nullptr;
    bool prepared = false;
    uint64_t rm_gen = 0;           // cache removal generation at prepare time
    int32_t n_tokens = 0;
    std::vector<kvi::UbatchHost> ub;
    std::vector<std::vector<uint8_t>> stored;   // [layer][ub] K/V stored
    // device upload layout (byte offsets inside the per-split table image)
    std::vector<uint8_t> image;    // DevRow / perm / DevBlock / CSR arrays of all ubatches
    std::vector<size_t> off_rows, off_perm, off_blocks, off_seq_off, off_seq_blk;
};

namespace kvi {

struct DeviceState;   // defined in device.cu

struct CellState {
    int32_t n_stream = 1, kv_size = 0, n_words = 1;
    std::vector<int32_t> pos;      // [n_cells], -1 = empty
    std::vector<int32_t> nseq;     // [n_cells], 0 = empty
    std::vector<uint64_t> bits;    // [n_cells * n_words]
    std::vector<uint32_t> epoch;   // [n_cells]
    std::vector<int32_t> first_free;   // per stream: every cell below is occupied
    std::vector<int32_t> used_max_p1;  // per stream
};

// A change of one cell for the device mirror.
struct Delta {
    int32_t cell;
    int32_t pos;
    uint32_t epoch;
    int32_t nseq;
    uint64_t bits[4];
};

}  // namespace kvi

struct kv_cache {
    kv_params prm{};               // normalised copy (pointers below)
    int32_t n_batch = 0, n_ubatch = 0, kv_size = 0, n_words = 1, gqa = 1;
    int32_t pf_min_qv = 0;         // groups with this many query vectors take the prefill path (0: never)
    std::vector<int32_t> seq_to_stream;
    std::vector<void *> k_layers, v_layers;
    bool has_device = false;

    kvi::CellState cells;
    uint64_t next_split_id = 1;
    uint32_t next_epoch = 1;
    uint64_t rm_gen = 0;

    // device mirror bookkeeping
    std::vector<kvi::Delta> pending;     // at most one record per cell (the latest)
    std::vector<int32_t> pending_idx;    // [n_cells] index into pending, or -1
    bool pending_reset = false;
    uint64_t dev_tables_split = 0;      // split whose tables are on the device
    kvi::DeviceState *dev = nullptr;
    uint64_t launches = 0;          // kernels launched (all entry points)

    std::string err;
    int set_err(int code, const std::string &msg) { err = msg; return code; }
};


// An entry point's body, run so that no C++ exception crosses the C boundary: a
// failed host allocation (or any other exception) becomes KV_E_NOMEM.
template <class F>
int guarded(kv_cache *c, F &&body) noexcept {
    try {
        return body();
    } catch (...) {
        if (c) {
            try {
                c->err = "host allocation failed";
            } catch (...) {
            }
        }
        return KV_E_NOMEM;
    }
}

// device.cu
namespace kvi {
int device_init(kv_cache *c);
void device_free(kv_cache *c);
}  // namespace kvi
