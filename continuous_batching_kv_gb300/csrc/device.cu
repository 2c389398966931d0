// Device half of libkvattn: workspace, TMA descriptors, the cell-mirror
// upload, and the two device entry points kv_store and ubatch_attention.
//
// "Batch、Ubatch 与解码主循环", Part F: after the batch is split and cells are
// reserved, each ubatch runs in order; inside it every layer stores its K/V
// rows and attends.  The host owns the cell metadata; the device keeps a
// mirror (position, sequence bitset, reserving-ubatch serial per cell) that
// is brought up to date, from a list of changed cells, at the first device
// call after each reservation or removal.

#include <algorithm>
#include <cstdio>
#include <cstring>

#include <cudaTypedefs.h>

#include "dev_common.cuh"
#include "kernels.h"

namespace kvi {

struct DeviceState {
    int device = 0;
    int n_sm = 148;
    // cell mirror
    int32_t *d_pos = nullptr;
    uint32_t *d_epoch = nullptr;
    uint64_t *d_bits = nullptr;
    // uploads
    int32_t delta_cap = 0;                      // deltas the staging buffers hold without growing
    uint8_t *d_tables = nullptr;
    size_t tables_cap = 0;
    // two pinned staging buffers used in turn, so preparing a split never waits
    // for the upload of the one before it
    uint8_t *h_stage[2] = {nullptr, nullptr};   // mapped pinned memory: the host writes, kernels read
    uint8_t *d_stage[2] = {nullptr, nullptr};   // their device-visible addresses
    size_t stage_cap[2] = {0, 0};
    cudaEvent_t stage_ev[2] = {nullptr, nullptr};
    bool stage_pending[2] = {false, false};
    int stage_slot = 0;
    // attention plan and split-K scratch
    kvk::Plan plan{};
    int32_t max_blocks = 0;
    int32_t gx_dec = 1, gx_pf = 1;          // CTA columns of the decode / prefill grids
    float *d_part_dec = nullptr;
    float *d_part_pf = nullptr;      // prefill partials: O rows [rows][128], then (m, l) [rows][2]
    int64_t pf_part_rows = 0;        // cap_pf * n_head_kv * PF_M
    CUtensorMap tm_part{};           // the O rows as a 2-D fp32 matrix, 32 x 32 boxes, 128-byte swizzle
    int32_t *d_err = nullptr;
    // device address of the library's fixed static-scratch array on this device
    // (looked up at kv_init, which also makes the runtime load and back it)
    unsigned char *static_scratch = nullptr;
    // one TMA descriptor per K / V tensor
    std::vector<CUtensorMap> tm_k, tm_v;
    std::vector<CUtensorMap> tm_dec;   // per layer: K, V with 64-row boxes, K, V with 8-row boxes
    // Two sets of plan arrays (plan, plan2).  While a split's ubatch runs its layers, the
    // plan of its next ubatch is built into the other set on a side stream, ordered
    // after everything the caller's stream had been given; the ubatch's first call then
    // has its stream wait for that build instead of running the plan kernels itself.
    kvk::Plan plan2{};
    uint64_t pb_split[2] = {0, 0};      // (split, ubatch) each set holds; split 0: none
    int32_t pb_ub[2] = {-1, -1};
    bool pb_pending[2] = {false, false};   // built on the side stream, not yet waited for
    cudaEvent_t pb_ready[2] = {nullptr, nullptr};
    cudaEvent_t call_ev = nullptr;      // the caller's stream, when a look-ahead build starts
    cudaStream_t side = nullptr;
    int32_t pb_cur = 0;                 // the set the last attention call used
    size_t bytes = 0;
    std::vector<void *> allocs;
};

}  // namespace kvi

using namespace kvi;

namespace {

// Split-K scratch of ubatch_attention_static_scratch: one fixed array in this
// file's device image.  Every process that loads the library holds it on each
// device where a cache is created (kv_init looks up its address, which loads
// this module there) until the process exits.  In host code the name is a
// host-side stand-in; only the address from cudaGetSymbolAddress may be given
// to a kernel.
constexpr size_t STATIC_SCRATCH_BYTES = KV_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

constexpr int32_t DEC_PART_FLOATS = DEC_QMAX * 132;
constexpr int32_t PF_PART_FLOATS = PF_M * 132;

int cuda_fail(kv_cache *c, cudaError_t e, const char *what) {
    char buf[256];
    std::snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
    return c->set_err(KV_E_CUDA, buf);
}

template <class T>
cudaError_t dev_alloc(DeviceState *d, T **p, size_t n) {
    void *v = nullptr;
    size_t bytes = std::max<size_t>(n * sizeof(T), 16);
    cudaError_t e = cudaMalloc(&v, bytes);
    if (e != cudaSuccess) return e;
    d->allocs.push_back(v);
    d->bytes += bytes;
    *p = static_cast<T *>(v);
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A K or V tensor as a 2-D fp16 matrix: n_stream*kv_size rows of
// n_head_kv*128 values; boxes of box_rows (64 or 8) rows x 64 values, 128-byte
// swizzle (an 8-row box lands in shared memory exactly as rows 8g .. 8g + 7 of
// a 64-row box at the same 1 KiB-aligned offset).
bool make_kv_map(CUtensorMap *m, void *base, int32_t n_head_kv, int64_t n_rows, uint32_t box_rows = TILE) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)n_head_kv * 128, (cuuint64_t)n_rows};
    cuuint64_t strides[1] = {(cuuint64_t)n_head_kv * 128 * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t tables_bound(const kv_cache *c) {
    const size_t n = (size_t)c->n_batch;
    const size_t per_ub = 4 * ((size_t)c->prm.n_seq_max + 1) + 6 * 16;
    return 56 * n + n * per_ub + 4096;
}

kvk::UbView make_view(const kv_cache *c, const kv_split *sp, int32_t ub) {
    const DeviceState *d = c->dev;
    const UbatchHost &u = sp->ub[ub];
    kvk::UbView v{};
    v.cell_pos = d->d_pos;
    v.cell_epoch = d->d_epoch;
    v.cell_bits = d->d_bits;
    v.n_words = c->n_words;
    v.ub_epoch = u.epoch;
    v.causal = c->prm.causal;
    v.n_swa = c->prm.n_swa;
    v.kv_size = c->kv_size;
    v.n_kv = u.n_kv;
    v.n_tokens = u.n_tokens;
    v.n_blocks = (int32_t)u.blocks.size();
    v.n_dec_blocks = u.n_dec_blocks;
    v.rows = reinterpret_cast<const DevRow *>(d->d_tables + sp->off_rows[ub]);
    v.perm = reinterpret_cast<const int32_t *>(d->d_tables + sp->off_perm[ub]);
    v.blocks = reinterpret_cast<const DevBlock *>(d->d_tables + sp->off_blocks[ub]);
    v.seq_blk_off = reinterpret_cast<const int32_t *>(d->d_tables + sp->off_seq_off[ub]);
    v.seq_blk = reinterpret_cast<const int32_t *>(d->d_tables + sp->off_seq_blk[ub]);
    return v;
}

// Order st after the look-ahead plan build into set i: a stream wait, or, while st is
// being captured into a graph (which cannot wait for work outside it), a host wait.
cudaError_t wait_build(DeviceState *d, int i, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone) return cudaEventSynchronize(d->pb_ready[i]);
    return cudaStreamWaitEvent(st, d->pb_ready[i], 0);
}

// Bring the device mirror and this split's tables up to date (stream-ordered).
int sync_device(kv_cache *c, const kv_split *sp, cudaStream_t st) {
    DeviceState *d = c->dev;
    const bool need_tables = c->dev_tables_split != sp->id;
    if (!c->pending_reset && c->pending.empty() && !need_tables) return KV_OK;
    cudaError_t e;
    // a look-ahead plan build reads the mirror and the tables: the uploads wait for it
    for (int i = 0; i < 2; ++i) {
        if (!d->pb_pending[i]) continue;
        if ((e = wait_build(d, i, st)) != cudaSuccess) return cuda_fail(c, e, "plan wait");
        d->pb_pending[i] = false;
    }
    const int sl = d->stage_slot;
    if (d->stage_pending[sl]) {   // this staging buffer is reused: wait for its last copy
        e = cudaEventSynchronize(d->stage_ev[sl]);
        if (e != cudaSuccess) return cuda_fail(c, e, "stage event");
        d->stage_pending[sl] = false;
    }
    if (c->pending_reset) {
        const size_t n = (size_t)c->prm.n_ctx;
        if ((e = cudaMemsetAsync(d->d_pos, 0xff, n * sizeof(int32_t), st)) != cudaSuccess ||
            (e = cudaMemsetAsync(d->d_epoch, 0, n * sizeof(uint32_t), st)) != cudaSuccess ||
            (e = cudaMemsetAsync(d->d_bits, 0, n * c->n_words * sizeof(uint64_t), st)) != cudaSuccess)
            return cuda_fail(c, e, "mirror reset");
        c->pending_reset = false;
    }
    const size_t nd = c->pending.size();
    const size_t dbytes = nd * sizeof(Delta);
    const size_t tbytes = need_tables ? sp->image.size() : 0;
    if (tbytes > d->tables_cap) return c->set_err(KV_E_INVAL, "split tables exceed bound");
    if (dbytes + tbytes > d->stage_cap[sl]) {   // rare (large removals): grow
        if (d->h_stage[sl]) cudaFreeHost(d->h_stage[sl]);
        d->h_stage[sl] = nullptr;
        d->d_stage[sl] = nullptr;
        size_t cap = dbytes + tbytes;
        if ((e = cudaHostAlloc((void **)&d->h_stage[sl], cap, cudaHostAllocMapped)) != cudaSuccess ||
            (e = cudaHostGetDevicePointer((void **)&d->d_stage[sl], d->h_stage[sl], 0)) != cudaSuccess)
            return cuda_fail(c, e, "stage grow");
        d->stage_cap[sl] = cap;
    }
    uint8_t *stage = d->h_stage[sl];
    if (nd) std::memcpy(stage, c->pending.data(), dbytes);
    if (tbytes) std::memcpy(stage + dbytes, sp->image.data(), tbytes);
    // both uploads are kernels reading the mapped staging buffer (no copy engine)
    if (nd) {
        if ((e = kvk::launch_apply_deltas(reinterpret_cast<const Delta *>(d->d_stage[sl]), (int32_t)nd, c->n_words,
                                          d->d_pos, d->d_epoch, d->d_bits, st)) != cudaSuccess)
            return cuda_fail(c, e, "apply deltas");
        c->launches += 1;
    }
    if (tbytes) {
        if ((e = kvk::launch_upload(d->d_stage[sl] + dbytes, d->d_tables, tbytes, d->n_sm, st)) != cudaSuccess)
            return cuda_fail(c, e, "table upload");
        c->launches += 1;
        c->dev_tables_split = sp->id;
        for (int i = 0; i < 2; ++i) {
            d->pb_split[i] = 0;
            d->pb_ub[i] = -1;
        }
    }
    if ((e = cudaEventRecord(d->stage_ev[sl], st)) != cudaSuccess) return cuda_fail(c, e, "stage record");
    d->stage_pending[sl] = true;
    d->stage_slot = sl ^ 1;
    for (const Delta &r : c->pending) c->pending_idx[r.cell] = -1;
    c->pending.clear();
    return KV_OK;
}

kvk::Plan &plan_set(DeviceState *d, int i) { return i == 0 ? d->plan : d->plan2; }

// The plan set holding (split, ubatch) for a call on stream st: one built ahead on the
// side stream (st then waits for that build), one built before, or else one built now
// on st into the set the last call used (the other may hold a look-ahead build).
// fresh: the plan was not complete before this call's first kernel was issued.
// Returns the set, or -1 with rc set.
int plan_for(kv_cache *c, const kv_split *sp, int32_t ub, cudaStream_t st, bool &fresh, int &rc) {
    DeviceState *d = c->dev;
    fresh = false;
    rc = KV_OK;
    cudaError_t e;
    for (int i = 0; i < 2; ++i) {
        if (d->pb_split[i] != sp->id || d->pb_ub[i] != ub) continue;
        if (d->pb_pending[i]) {
            if ((e = wait_build(d, i, st)) != cudaSuccess) {
                rc = cuda_fail(c, e, "plan wait");
                return -1;
            }
            d->pb_pending[i] = false;
            fresh = true;
        }
        d->pb_cur = i;
        return i;
    }
    int i = d->pb_cur;
    if (d->pb_pending[i]) i ^= 1;   // the set a look-ahead build is writing is left alone
    if ((e = kvk::launch_plan(make_view(c, sp, ub), plan_set(d, i), c->prm.n_stream, d->gx_dec, d->gx_pf, st)) !=
        cudaSuccess) {
        d->pb_split[i] = 0;
        d->pb_ub[i] = -1;
        rc = cuda_fail(c, e, "plan launch");
        return -1;
    }
    c->launches += 3;
    d->pb_split[i] = sp->id;
    d->pb_ub[i] = ub;
    d->pb_pending[i] = false;
    d->pb_cur = i;
    fresh = true;
    return i;
}

// Build the plan of (split, ubatch) ahead on the side stream, into the set the current
// call does not use, after everything already issued on st (which may still read that
// set).  Not while st is being captured into a graph: the side stream's work would be
// left outside the capture's joins.
int plan_ahead(kv_cache *c, const kv_split *sp, int32_t ub, cudaStream_t st) {
    DeviceState *d = c->dev;
    const int i = d->pb_cur ^ 1;
    if (d->pb_split[i] == sp->id && d->pb_ub[i] == ub) return KV_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(c, e, "capture query");
    if (cs != cudaStreamCaptureStatusNone) return KV_OK;
    d->pb_split[i] = 0;   // holds nothing usable until the build is issued
    d->pb_ub[i] = -1;
    if ((e = cudaEventRecord(d->call_ev, st)) != cudaSuccess || (e = cudaStreamWaitEvent(d->side, d->call_ev, 0)) != cudaSuccess ||
        (e = kvk::launch_plan(make_view(c, sp, ub), plan_set(d, i), c->prm.n_stream, d->gx_dec, d->gx_pf, d->side)) !=
            cudaSuccess ||
        (e = cudaEventRecord(d->pb_ready[i], d->side)) != cudaSuccess)
        return cuda_fail(c, e, "look-ahead plan");
    c->launches += 3;
    d->pb_split[i] = sp->id;
    d->pb_ub[i] = ub;
    d->pb_pending[i] = true;
    return KV_OK;
}

// The most query vectors in one decode block of the ubatch (rows x GQA group).
int32_t decode_nq_max(const kv_cache *c, const UbatchHost &u) {
    int32_t r = 1;
    for (int32_t b = 0; b < u.n_dec_blocks; ++b) r = std::max(r, u.blocks[b].n_rows * c->gqa);
    return r;
}

int check_call(kv_cache *c, const kv_split *sp, int32_t ub, int32_t layer) {
    if (!c || !sp || sp->owner != c) return KV_E_INVAL;
    if (!c->has_device) return c->set_err(KV_E_NO_DEVICE, "host-only cache");
    if (!sp->prepared) return c->set_err(KV_E_ORDER, "split not prepared");
    if (sp->rm_gen != c->rm_gen) return c->set_err(KV_E_STALE, "split prepared before a removal");
    if (ub < 0 || ub >= (int32_t)sp->ub.size()) return c->set_err(KV_E_INVAL, "ubatch index");
    if (layer < 0 || layer >= c->prm.n_layer) return c->set_err(KV_E_INVAL, "layer index");
    return KV_OK;
}

}  // namespace

namespace kvi {

int device_init(kv_cache *c) {
    DeviceState *d = new (std::nothrow) DeviceState();
    if (!d) return c->set_err(KV_E_NOMEM, "device state");
    c->dev = d;
    cudaError_t e;
    if ((e = cudaGetDevice(&d->device)) != cudaSuccess) return cuda_fail(c, e, "cudaGetDevice");
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d->device) == cudaSuccess && sms > 0)
        d->n_sm = sms;
    const int64_t n_cells = c->prm.n_ctx;
    if ((e = dev_alloc(d, &d->d_pos, n_cells)) != cudaSuccess ||
        (e = dev_alloc(d, &d->d_epoch, n_cells)) != cudaSuccess ||
        (e = dev_alloc(d, &d->d_bits, n_cells * c->n_words)) != cudaSuccess)
        return cuda_fail(c, e, "mirror alloc");
    if ((e = cudaMemset(d->d_pos, 0xff, n_cells * sizeof(int32_t))) != cudaSuccess ||
        (e = cudaMemset(d->d_epoch, 0, n_cells * sizeof(uint32_t))) != cudaSuccess ||
        (e = cudaMemset(d->d_bits, 0, n_cells * c->n_words * sizeof(uint64_t))) != cudaSuccess)
        return cuda_fail(c, e, "mirror clear");
    d->delta_cap = std::max<int32_t>(c->n_batch, 4096);
    d->tables_cap = tables_bound(c);
    if ((e = dev_alloc(d, &d->d_tables, d->tables_cap)) != cudaSuccess) return cuda_fail(c, e, "table alloc");
    for (int sl = 0; sl < 2; ++sl) {
        d->stage_cap[sl] = d->tables_cap + (size_t)d->delta_cap * sizeof(Delta);
        if ((e = cudaHostAlloc((void **)&d->h_stage[sl], d->stage_cap[sl], cudaHostAllocMapped)) != cudaSuccess ||
            (e = cudaHostGetDevicePointer((void **)&d->d_stage[sl], d->h_stage[sl], 0)) != cudaSuccess)
            return cuda_fail(c, e, "stage alloc");
        if ((e = cudaEventCreateWithFlags(&d->stage_ev[sl], cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(c, e, "event");
    }

    // plan and split-K scratch
    const int32_t hkv = c->prm.n_head_kv;
    d->max_blocks = c->n_ubatch;
    const int32_t max_pf_blocks = std::max<int32_t>(1, (c->n_ubatch * c->gqa + PF_MIN_QV - 1) / PF_MIN_QV);
    d->gx_dec = std::max<int32_t>(1, d->n_sm * kvk::decode_ctas_per_sm() / hkv);
    d->gx_pf = std::min<int32_t>(kvk::PLAN_MAX_COLS, std::max<int32_t>(1, d->n_sm / hkv));
    // Prefill CTAs in clusters of PF_CLUSTER columns (a split block's pieces merge over
    // distributed shared memory) when the grid has room for at least two clusters a row
    d->plan.pf_cluster = 1;
    if (d->gx_pf >= 2 * PF_CLUSTER) {
        d->gx_pf -= d->gx_pf % PF_CLUSTER;
        d->plan.pf_cluster = PF_CLUSTER;
    }
    kvk::Plan &p = d->plan;
    p.tile_stride = (c->kv_size + TILE - 1) / TILE;
    p.cap_dec = d->gx_dec + d->max_blocks;
    p.cap_pf = d->gx_pf + max_pf_blocks;
    const size_t fl = (size_t)d->max_blocks * p.tile_stride;
    if ((e = dev_alloc(d, &p.flags, fl)) != cudaSuccess || (e = dev_alloc(d, &p.tiles, fl)) != cudaSuccess ||
        (e = dev_alloc(d, &p.cum, fl)) != cudaSuccess || (e = dev_alloc(d, &p.wcount, d->max_blocks)) != cudaSuccess ||
        (e = dev_alloc(d, &p.counts, d->max_blocks)) != cudaSuccess ||
        (e = dev_alloc(d, &p.work, (size_t)p.cap_dec + p.cap_pf)) != cudaSuccess ||
        (e = dev_alloc(d, &p.n_work, 2)) != cudaSuccess ||
        (e = dev_alloc(d, &p.blk_item0, d->max_blocks)) != cudaSuccess ||
        (e = dev_alloc(d, &p.blk_nitems, d->max_blocks)) != cudaSuccess ||
        (e = dev_alloc(d, &p.counters, (size_t)d->max_blocks * hkv)) != cudaSuccess ||
        (e = dev_alloc(d, &p.cta_item0, (size_t)d->gx_dec + d->gx_pf + 2)) != cudaSuccess ||
        (e = dev_alloc(d, &p.pf_rows, (size_t)d->gx_pf * PF_M)) != cudaSuccess ||
        (e = dev_alloc(d, &p.pf_first, (size_t)d->gx_pf * 4)) != cudaSuccess ||
        (e = dev_alloc(d, &p.dec_first, (size_t)d->gx_dec * kvk::DEC_FIRST)) != cudaSuccess ||
        (e = dev_alloc(d, &d->d_part_dec, (size_t)p.cap_dec * hkv * DEC_PART_FLOATS)) != cudaSuccess ||
        (e = dev_alloc(d, &d->d_part_pf, (size_t)p.cap_pf * hkv * PF_PART_FLOATS)) != cudaSuccess ||
        (e = dev_alloc(d, &d->d_err, 1)) != cudaSuccess)
        return cuda_fail(c, e, "plan alloc");
    p.err = d->d_err;
    p.gqa = c->gqa;
    {
        kvk::Plan &q = d->plan2;
        q = p;   // shared: the split-K counters, the error word and the sizes
        if ((e = dev_alloc(d, &q.flags, fl)) != cudaSuccess || (e = dev_alloc(d, &q.tiles, fl)) != cudaSuccess ||
            (e = dev_alloc(d, &q.cum, fl)) != cudaSuccess || (e = dev_alloc(d, &q.wcount, d->max_blocks)) != cudaSuccess ||
            (e = dev_alloc(d, &q.counts, d->max_blocks)) != cudaSuccess ||
            (e = dev_alloc(d, &q.work, (size_t)q.cap_dec + q.cap_pf)) != cudaSuccess ||
            (e = dev_alloc(d, &q.n_work, 2)) != cudaSuccess ||
            (e = dev_alloc(d, &q.blk_item0, d->max_blocks)) != cudaSuccess ||
            (e = dev_alloc(d, &q.blk_nitems, d->max_blocks)) != cudaSuccess ||
            (e = dev_alloc(d, &q.cta_item0, (size_t)d->gx_dec + d->gx_pf + 2)) != cudaSuccess ||
            (e = dev_alloc(d, &q.pf_rows, (size_t)d->gx_pf * PF_M)) != cudaSuccess ||
            (e = dev_alloc(d, &q.pf_first, (size_t)d->gx_pf * 4)) != cudaSuccess ||
            (e = dev_alloc(d, &q.dec_first, (size_t)d->gx_dec * kvk::DEC_FIRST)) != cudaSuccess)
            return cuda_fail(c, e, "plan alloc");
        if ((e = cudaStreamCreateWithFlags(&d->side, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&d->call_ev, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&d->pb_ready[0], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&d->pb_ready[1], cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(c, e, "plan stream");
    }
    d->pf_part_rows = (int64_t)p.cap_pf * hkv * PF_M;
    {
        auto enc = get_encode();
        cuuint64_t dims[2] = {128, (cuuint64_t)d->pf_part_rows};
        cuuint64_t strides[1] = {128 * sizeof(float)};
        cuuint32_t box[2] = {32, 32};
        cuuint32_t estr[2] = {1, 1};
        if (!enc || enc(&d->tm_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d->d_part_pf, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return c->set_err(KV_E_CUDA, "cuTensorMapEncodeTiled failed (partials)");
    }
    if ((e = cudaMemset(p.counters, 0, (size_t)d->max_blocks * hkv * sizeof(int32_t))) != cudaSuccess ||
        (e = cudaMemset(d->d_err, 0, sizeof(int32_t))) != cudaSuccess)
        return cuda_fail(c, e, "plan clear");

    d->tm_k.resize(c->prm.n_layer);
    d->tm_v.resize(c->prm.n_layer);
    const int64_t rows = (int64_t)c->prm.n_stream * c->kv_size;
    d->tm_dec.resize(4 * (size_t)c->prm.n_layer);
    for (int32_t l = 0; l < c->prm.n_layer; ++l) {
        CUtensorMap *td = &d->tm_dec[4 * (size_t)l];
        if (!make_kv_map(&d->tm_k[l], c->k_layers[l], hkv, rows) ||
            !make_kv_map(&d->tm_v[l], c->v_layers[l], hkv, rows) ||
            !make_kv_map(&td[2], c->k_layers[l], hkv, rows, 8) ||
            !make_kv_map(&td[3], c->v_layers[l], hkv, rows, 8))
            return c->set_err(KV_E_CUDA, "cuTensorMapEncodeTiled failed");
        td[0] = d->tm_k[l];
        td[1] = d->tm_v[l];
    }
    if ((e = kvk::load_store_kernels()) != cudaSuccess || (e = kvk::load_plan_kernels()) != cudaSuccess ||
        (e = kvk::load_decode_kernels()) != cudaSuccess || (e = kvk::load_prefill_kernels()) != cudaSuccess)
        return cuda_fail(c, e, "kernel load");
    // no cluster launch where no cluster of attention CTAs can be resident
    if (d->plan.pf_cluster > 1 && kvk::prefill_max_active_clusters(d->plan.pf_cluster) < 1) d->plan.pf_cluster = 1;
    d->plan2.pf_cluster = d->plan.pf_cluster;
    // The static-scratch array's address on this device (the current one).  With
    // lazy module loading this lookup is what loads the module and backs the array,
    // so it happens here, where memory is obtained anyway, and not during a call
    // that promises to obtain none.
    {
        void *ps = nullptr;
        if ((e = cudaGetSymbolAddress(&ps, g_static_scratch)) != cudaSuccess)
            return cuda_fail(c, e, "static scratch address");
        d->static_scratch = static_cast<unsigned char *>(ps);
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(c, e, "init sync");
    return KV_OK;
}

void device_free(kv_cache *c) {
    DeviceState *d = c->dev;
    if (!d) return;
    for (int sl = 0; sl < 2; ++sl)
        if (d->stage_pending[sl] && d->stage_ev[sl]) cudaEventSynchronize(d->stage_ev[sl]);
    if (d->side) cudaStreamSynchronize(d->side);
    for (void *p : d->allocs) cudaFree(p);
    for (int i = 0; i < 2; ++i)
        if (d->pb_ready[i]) cudaEventDestroy(d->pb_ready[i]);
    if (d->call_ev) cudaEventDestroy(d->call_ev);
    if (d->side) cudaStreamDestroy(d->side);
    for (int sl = 0; sl < 2; ++sl) {
        if (d->h_stage[sl]) cudaFreeHost(d->h_stage[sl]);
        if (d->stage_ev[sl]) cudaEventDestroy(d->stage_ev[sl]);
    }
    delete d;
    c->dev = nullptr;
}

}  // namespace kvi

extern "C" {

int kv_store(kv_cache *c, const kv_split *sp, int32_t ub, int32_t layer, const void *k_cur,
             const void *v_cur, void *stream) {
    return guarded(c, [&]() -> int {
        int rc = check_call(c, sp, ub, layer);
        if (rc != KV_OK) return rc;
        if (!k_cur || !v_cur || ((uintptr_t)k_cur & 15) || ((uintptr_t)v_cur & 15))
            return c->set_err(KV_E_INVAL, "k_cur / v_cur must be 16-byte aligned device pointers");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        if ((rc = sync_device(c, sp, st)) != KV_OK) return rc;
        const UbatchHost &u = sp->ub[ub];
        DeviceState *d = c->dev;
        const DevRow *rows = reinterpret_cast<const DevRow *>(d->d_tables + sp->off_rows[ub]);
        cudaError_t e = kvk::launch_store(c->k_layers[layer], c->v_layers[layer], k_cur, v_cur, rows, u.n_tokens,
                                          c->prm.n_head_kv * c->prm.head_dim * 2, (int64_t)c->prm.n_ctx, d->d_err,
                                          d->n_sm, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "store launch");
        c->launches += 1;
        const_cast<kv_split *>(sp)->stored[layer][ub] = 1;
        return KV_OK;
    });
}

int ubatch_attention(kv_cache *c, const kv_split *sp, int32_t ub, int32_t layer, const void *q, float *o,
                     void *mask_out, void *stream) {
    return guarded(c, [&]() -> int {
        int rc = check_call(c, sp, ub, layer);
        if (rc != KV_OK) return rc;
        if (!q || !o || ((uintptr_t)q & 15) || ((uintptr_t)o & 15))
            return c->set_err(KV_E_INVAL, "q / o must be 16-byte aligned device pointers");
        for (int32_t k = 0; k <= ub; ++k)
            if (!sp->stored[layer][k]) return c->set_err(KV_E_ORDER, "attention before its K/V were stored");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        // Nothing of this call precedes the attention kernels when the device is in
        // sync, the plan is cached and no mask is asked for: then the plan, tables
        // and mirror were complete before the previous kernel began.
        bool early_ok = !c->pending_reset && c->pending.empty() && c->dev_tables_split == sp->id && !mask_out;
        if ((rc = sync_device(c, sp, st)) != KV_OK) return rc;
        DeviceState *d = c->dev;
        const UbatchHost &u = sp->ub[ub];
        kvk::UbView v = make_view(c, sp, ub);
        cudaError_t e;
        bool fresh = false;
        const int pi = plan_for(c, sp, ub, st, fresh, rc);
        if (pi < 0) return rc;
        if (fresh) early_ok = false;
        const kvk::Plan &plan = plan_set(d, pi);
        if (mask_out) {
            if ((e = kvk::launch_mask(v, static_cast<uint16_t *>(mask_out), st)) != cudaSuccess)
                return cuda_fail(c, e, "mask launch");
            c->launches += 1;
        }
        const float scale_log2 = 1.4426950408889634f / sqrtf((float)c->prm.head_dim);
        if (u.n_dec_blocks > 0) {
            kvk::DecodeArgs a{};
            a.u = v;
            a.p = plan;
            a.q = static_cast<const __half *>(q);
            a.o = o;
            a.part = d->d_part_dec;
            a.n_head = c->prm.n_head;
            a.n_head_kv = c->prm.n_head_kv;
            a.gqa = c->gqa;
            a.scale_log2 = scale_log2;
            a.err = d->d_err;
            a.nq_max = decode_nq_max(c, u);
            a.early_ok = early_ok ? 1 : 0;
            if ((e = kvk::launch_decode(&d->tm_dec[4 * (size_t)layer], a, d->gx_dec, st)) != cudaSuccess)
                return cuda_fail(c, e, "decode launch");
            c->launches += 1;
        }
        if (u.n_pf_blocks > 0) {
            kvk::PrefillArgs a{};
            a.u = v;
            a.p = plan;
            a.q = static_cast<const __half *>(q);
            a.o = o;
            a.part = d->d_part_pf;
            a.part_ml = d->d_part_pf + d->pf_part_rows * 128;
            a.gx_dec = d->gx_dec;
            a.n_head = c->prm.n_head;
            a.n_head_kv = c->prm.n_head_kv;
            a.gqa = c->gqa;
            a.scale_log2 = scale_log2;
            a.err = d->d_err;
            a.early_ok = early_ok ? 1 : 0;
            a.cluster = plan.pf_cluster;
            // Q as a (d, head, token) tensor: a GQA group's query vectors of 128 / gqa
            // consecutive rows are one (64, gqa, 128 / gqa) box per 64-value d half; used
            // when every prefill block of the ubatch has consecutive rows
            CUtensorMap tm_q{};
            bool all_consecutive = true;
            for (int32_t b = u.n_dec_blocks; b < (int32_t)u.blocks.size() && all_consecutive; ++b)
                all_consecutive = u.blocks[b].tok0 >= 0;
            if (128 % c->gqa == 0 && all_consecutive) {
                auto enc = get_encode();
                cuuint64_t dims[3] = {128, (cuuint64_t)c->prm.n_head, (cuuint64_t)u.n_tokens};
                cuuint64_t strides[2] = {128 * 2, (cuuint64_t)c->prm.n_head * 128 * 2};
                cuuint32_t box[3] = {64, (cuuint32_t)c->gqa, (cuuint32_t)(128 / c->gqa)};
                cuuint32_t estr[3] = {1, 1, 1};
                a.q_tma = enc && enc(&tm_q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
                                  ? 1
                                  : 0;
            }
            if ((e = kvk::launch_prefill(&d->tm_k[layer], &d->tm_v[layer], &d->tm_part, &tm_q, a, d->gx_pf, st)) !=
                cudaSuccess)
                return cuda_fail(c, e, "prefill launch");
            c->launches += 1;
        }
        // the next ubatch of the split gets its plan while this one runs its layers
        if (layer == 0 && ub + 1 < (int32_t)sp->ub.size()) return plan_ahead(c, sp, ub + 1, st);
        return KV_OK;
    });
}

int kv_device_error(kv_cache *c) {
    if (!c || !c->has_device) return KV_E_INVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(c, e, "sync");
    int32_t v = 0;
    if ((e = cudaMemcpy(&v, c->dev->d_err, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(c, e, "error word read");
    if (v) {
        // a kernel gave up part-way: clear the word, and the split-K completion
        // counters it may have left counted, so that the next launch starts clean
        cudaMemset(c->dev->d_err, 0, sizeof(int32_t));
        cudaMemset(c->dev->plan.counters, 0, (size_t)c->dev->max_blocks * c->prm.n_head_kv * sizeof(int32_t));
        cudaDeviceSynchronize();
    }
    return v;
}

int kv_selftest_wait(kv_cache *c, void *stream) {
    if (!c || !c->has_device) return KV_E_INVAL;
    return guarded(c, [&]() -> int {
        cudaError_t e = kvk::launch_wait_selftest(c->dev->d_err, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(c, e, "wait self-test launch");
        c->launches += 1;
        return KV_OK;
    });
}

size_t kv_device_bytes(const kv_cache *c) { return (c && c->dev) ? c->dev->bytes : 0; }

uint64_t kv_launch_count(const kv_cache *c) { return c ? c->launches : 0; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Attention without allocation: the decode path with its split-K scratch in a
// fixed array of the library's device image instead of memory obtained at
// kv_init.  The array is shared by every call on a device; each call clears
// the completion counters (which must start at zero) on its own stream.
// ---------------------------------------------------------------------------

namespace {

// True when sync_device would have to grow its delta or staging buffer.
bool sync_would_allocate(const kv_cache *c, const kv_split *sp) {
    const DeviceState *d = c->dev;
    const size_t nd = c->pending.size();
    const size_t tbytes = c->dev_tables_split != sp->id ? sp->image.size() : 0;
    return nd * sizeof(Delta) + tbytes > d->stage_cap[d->stage_slot] ||
           tbytes > d->tables_cap;
}

}  // namespace

extern "C" int ubatch_attention_static_scratch(kv_cache *c, const kv_split *sp, int32_t ub, int32_t layer,
                                               const void *q, float *o, void *mask_out, void *stream) {
    return guarded(c, [&]() -> int {
        int rc = check_call(c, sp, ub, layer);
        if (rc != KV_OK) return rc;
        if (!q || !o || ((uintptr_t)q & 15) || ((uintptr_t)o & 15))
            return c->set_err(KV_E_INVAL, "q / o must be 16-byte aligned device pointers");
        for (int32_t k = 0; k <= ub; ++k)
            if (!sp->stored[layer][k]) return c->set_err(KV_E_ORDER, "attention before its K/V were stored");
        DeviceState *d = c->dev;
        const UbatchHost &u = sp->ub[ub];
        if (u.n_pf_blocks > 0)
            return c->set_err(KV_E_INVAL, "static-scratch attention runs the decode path only; this ubatch has "
                                          "prefill blocks (use ubatch_attention)");
        const int32_t hkv = c->prm.n_head_kv;
        const size_t cnt_bytes = ((size_t)u.n_dec_blocks * hkv * sizeof(int32_t) + 255) & ~(size_t)255;
        const size_t part_bytes = ((size_t)d->gx_dec + u.n_dec_blocks) * hkv * DEC_PART_FLOATS * sizeof(float);
        if (cnt_bytes + part_bytes > STATIC_SCRATCH_BYTES) {
            char buf[200];
            std::snprintf(buf, sizeof buf, "static-scratch attention needs %zu bytes of scratch for %d decode blocks, "
                          "more than the %zu available", cnt_bytes + part_bytes, u.n_dec_blocks, STATIC_SCRATCH_BYTES);
            return c->set_err(KV_E_INVAL, buf);
        }
        int cur = -1;
        cudaError_t e = cudaGetDevice(&cur);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetDevice");
        if (cur != d->device)
            return c->set_err(KV_E_INVAL, "static-scratch attention: make the cache's device current");
        if (sync_would_allocate(c, sp))
            return c->set_err(KV_E_INVAL, "static-scratch attention: device tables need a larger upload buffer "
                                          "(call kv_store for this split first)");
        unsigned char *scratch = d->static_scratch;   // looked up at kv_init
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        if ((rc = sync_device(c, sp, st)) != KV_OK) return rc;
        kvk::UbView v = make_view(c, sp, ub);
        bool fresh = false;
        const int pi = plan_for(c, sp, ub, st, fresh, rc);
        if (pi < 0) return rc;
        if (mask_out) {
            if ((e = kvk::launch_mask(v, static_cast<uint16_t *>(mask_out), st)) != cudaSuccess)
                return cuda_fail(c, e, "mask launch");
            c->launches += 1;
        }
        if (u.n_dec_blocks == 0) return KV_OK;
        int32_t *counters = reinterpret_cast<int32_t *>(scratch);
        if ((e = cudaMemsetAsync(counters, 0, cnt_bytes, st)) != cudaSuccess) return cuda_fail(c, e, "counter clear");
        kvk::DecodeArgs a{};
        a.u = v;
        a.p = plan_set(d, pi);
        a.p.counters = counters;
        a.q = static_cast<const __half *>(q);
        a.o = o;
        a.part = reinterpret_cast<float *>(scratch + cnt_bytes);
        a.n_head = c->prm.n_head;
        a.n_head_kv = hkv;
        a.gqa = c->gqa;
        a.scale_log2 = 1.4426950408889634f / sqrtf((float)c->prm.head_dim);
        a.err = d->d_err;
        a.nq_max = decode_nq_max(c, u);
        // the counters were just cleared by a copy engine, not a kernel: wait for it
        a.early_ok = 0;
        if ((e = kvk::launch_decode(&d->tm_dec[4 * (size_t)layer], a, d->gx_dec, st)) != cudaSuccess)
            return cuda_fail(c, e, "decode launch");
        c->launches += 1;
        return KV_OK;
    });
}
