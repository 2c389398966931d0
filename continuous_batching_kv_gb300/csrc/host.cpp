// Host half of libkvattn: parameters, batch validation, the three ubatch
// splitters, the first-fit cell-slot finder, n_kv and sequence removal.
//
// Pages restated here (by title and section):
//   "llama.cpp and the ubatch" -- "Three things called batch" (n_batch /
//     n_ubatch clamps, the n_batch refusal), "Prefill and decode are not the
//     same shape" (n_kv padding), "Part 1" (split_simple, split_equal).
//   "Batch、Ubatch 与解码主循环" -- Part A (batch fields, auto-fill), Part B
//     (ubatch fields), Part C (the three splitters and the strategy choice),
//     Part F (validate, split, reserve; return 1 when the cache is full).
//   "What does llama.cpp's KV cache actually look like in memory?" --
//     "Unified versus non-unified" (streams), "The tensor's three dimensions".
//   "Iteration-Level Batching: Reforming the Batch at Every Token" -- "The
//     loop that replaces the batch" (retired sequences release their cache).

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <new>
#include <set>

#include "internal.h"

using namespace kvi;

namespace {

constexpr int32_t N_PAD_MODEL = 1;
constexpr int32_t N_PAD_FLOOR = 256;

bool log_on() {
    static int on = -1;
    if (on < 0) {
        const char *e = std::getenv("KV_LOG");
        on = (e && e[0] == '1') ? 1 : 0;
    }
    return on == 1;
}

int32_t pad_up(int32_t x, int32_t n) { return ((x + n - 1) / n) * n; }

inline bool bit_has(const uint64_t *w, int32_t q) { return (w[q >> 6] >> (q & 63)) & 1ull; }

// ---- cell state ---------------------------------------------------------------

void cells_init(CellState &cs, int32_t n_stream, int32_t kv_size, int32_t n_words) {
    cs.n_stream = n_stream;
    cs.kv_size = kv_size;
    cs.n_words = n_words;
    size_t n = (size_t)n_stream * kv_size;
    cs.pos.assign(n, -1);
    cs.nseq.assign(n, 0);
    cs.bits.assign(n * n_words, 0ull);
    cs.epoch.assign(n, 0u);
    cs.first_free.assign(n_stream, 0);
    cs.used_max_p1.assign(n_stream, 0);
}

// Next empty cell of stream s at or after `from`, or -1.
int32_t next_empty(const CellState &cs, int32_t s, int32_t from) {
    const int32_t *ns = cs.nseq.data() + (size_t)s * cs.kv_size;
    for (int32_t j = from; j < cs.kv_size; ++j)
        if (ns[j] == 0) return j;
    return -1;
}

void refresh_used_max(CellState &cs, int32_t s) {
    const int32_t *ns = cs.nseq.data() + (size_t)s * cs.kv_size;
    int32_t u = cs.used_max_p1[s];
    while (u > 0 && ns[u - 1] == 0) --u;
    cs.used_max_p1[s] = u;
}

// UBATCH, "Prefill and decode are not the same shape": the highest occupied
// cell + 1, padded to max(model pad, 256), at least one quantum, at most the
// stream's size.
int32_t n_kv_of(const CellState &cs, int32_t s) {
    int32_t q = std::max(N_PAD_MODEL, N_PAD_FLOOR);
    int32_t padded = std::max(q, pad_up(cs.used_max_p1[s], q));
    return std::min(cs.kv_size, padded);
}

int32_t seq_pos_max(const kv_cache *c, int32_t q) {
    const CellState &cs = c->cells;
    int32_t s = c->seq_to_stream[q];
    int32_t best = -1;
    size_t base = (size_t)s * cs.kv_size;
    for (int32_t j = 0; j < cs.used_max_p1[s]; ++j) {
        size_t g = base + j;
        if (cs.nseq[g] && bit_has(&cs.bits[g * cs.n_words], q)) best = std::max(best, cs.pos[g]);
    }
    return best;
}

// ---- splitting ----------------------------------------------------------------

struct RowSet {  // a row's sequence set, as a sorted id list
    std::vector<int32_t> ids;
    bool operator==(const RowSet &o) const { return ids == o.ids; }
    bool operator<(const RowSet &o) const { return ids < o.ids; }
};

bool overlaps(const RowSet &a, const RowSet &b) {
    size_t i = 0, j = 0;
    while (i < a.ids.size() && j < b.ids.size()) {
        if (a.ids[i] == b.ids[j]) return true;
        if (a.ids[i] < b.ids[j]) ++i; else ++j;
    }
    return false;
}

struct SplitIn {
    int32_t n;
    std::vector<int32_t> pos;
    std::vector<int32_t> ids;       // every row's ids, first id first, as given, row after row
    std::vector<int32_t> ids_off;   // [n + 1]: row r's ids are ids[ids_off[r] .. ids_off[r + 1])
    std::vector<RowSet> set;        // sorted, built only for the splits that compare sets
    const int32_t *ids_of(int32_t r) const { return ids.data() + ids_off[r]; }
    int32_t n_ids(int32_t r) const { return ids_off[r + 1] - ids_off[r]; }
    void build_sets() {
        set.resize(n);
        for (int32_t r = 0; r < n; ++r) {
            set[r].ids.assign(ids_of(r), ids_of(r) + n_ids(r));
            std::sort(set[r].ids.begin(), set[r].ids.end());
        }
    }
};

void add_ubatch(kv_split *sp, const SplitIn &in, const std::vector<int32_t> &rows,
                int32_t n_seq_tokens, int32_t n_seqs, const kv_cache *c) {
    UbatchHost u;
    u.n_tokens = (int32_t)rows.size();
    u.n_seq_tokens = n_seq_tokens;
    u.n_seqs = n_seqs;
    u.rows = rows;
    u.ids_off.reserve(rows.size() + 1);
    u.pos.reserve(rows.size());
    u.seq0.reserve(rows.size());
    u.streams.reserve(rows.size());
    u.ids_off.push_back(0);
    for (int32_t r : rows) {
        const int32_t *ids = in.ids_of(r);
        u.ids.insert(u.ids.end(), ids, ids + in.n_ids(r));
        u.ids_off.push_back((int32_t)u.ids.size());
        u.pos.push_back(in.pos[r]);
        u.seq0.push_back(ids[0]);
        u.streams.push_back(c->seq_to_stream[ids[0]]);
    }
    // the distinct ids, ascending
    u.seq_unq = u.ids;
    std::sort(u.seq_unq.begin(), u.seq_unq.end());
    u.seq_unq.erase(std::unique(u.seq_unq.begin(), u.seq_unq.end()), u.seq_unq.end());
    sp->ub.push_back(std::move(u));
}

// BATCH-ZH, Part C (1); UBATCH, "Part 1": submission order, at most n_ubatch,
// sequence ids ignored.  Each row counts as its own set.
void split_simple(kv_split *sp, const SplitIn &in, int32_t n_ub, const kv_cache *c) {
    for (int32_t a = 0; a < in.n; a += n_ub) {
        std::vector<int32_t> rows;
        for (int32_t r = a; r < std::min(in.n, a + n_ub); ++r) rows.push_back(r);
        add_ubatch(sp, in, rows, 1, (int32_t)rows.size(), c);
    }
}

// BATCH-ZH, Part C (2): choose non-overlapping sequence sets (first
// appearance among unused rows, at most n_ubatch of them), order them by
// smallest id, take the same number of rows from each: the fewest unused rows
// any chosen set has, capped at n_ubatch / n_sets; rows set-major.
void split_equal(kv_split *sp, const SplitIn &in, int32_t n_ub, const kv_cache *c) {
    std::vector<uint8_t> used(in.n, 0);
    // rows of each distinct set, in submission order
    std::map<RowSet, std::vector<int32_t>> rows_of;
    for (int32_t r = 0; r < in.n; ++r) rows_of[in.set[r]].push_back(r);
    std::map<RowSet, size_t> cursor;
    int32_t left = in.n;
    int32_t first_unused = 0;
    while (left > 0) {
        while (used[first_unused]) ++first_unused;
        std::vector<const RowSet *> chosen;
        for (int32_t r = first_unused; r < in.n; ++r) {
            if (used[r]) continue;
            const RowSet &s = in.set[r];
            bool skip = false;
            for (const RowSet *x : chosen) {
                if (*x == s || overlaps(*x, s)) { skip = true; break; }
            }
            if (skip) continue;
            if ((int32_t)chosen.size() == n_ub) break;
            chosen.push_back(&rows_of.find(s)->first);
        }
        std::stable_sort(chosen.begin(), chosen.end(),
                         [](const RowSet *a, const RowSet *b) { return a->ids[0] < b->ids[0]; });
        int32_t n_sets = (int32_t)chosen.size();
        int32_t take = n_ub / n_sets;
        for (const RowSet *x : chosen) {
            int32_t rem = (int32_t)(rows_of[*x].size() - cursor[*x]);
            take = std::min(take, rem);
        }
        std::vector<int32_t> rows;
        for (const RowSet *x : chosen) {
            size_t &cur = cursor[*x];
            const std::vector<int32_t> &lst = rows_of[*x];
            for (int32_t t = 0; t < take; ++t) {
                int32_t r = lst[cur++];
                rows.push_back(r);
                used[r] = 1;
            }
        }
        left -= (int32_t)rows.size();
        add_ubatch(sp, in, rows, take, n_sets, c);
    }
}

// BATCH-ZH, Part C (3): one sequence set per ubatch -- the set of the first
// unused row, then up to n_ubatch unused rows with exactly that set.
void split_seq(kv_split *sp, const SplitIn &in, int32_t n_ub, const kv_cache *c) {
    std::map<RowSet, std::vector<int32_t>> rows_of;
    for (int32_t r = 0; r < in.n; ++r) rows_of[in.set[r]].push_back(r);
    std::map<RowSet, size_t> cursor;
    std::vector<uint8_t> used(in.n, 0);
    int32_t first_unused = 0;
    int32_t left = in.n;
    while (left > 0) {
        while (used[first_unused]) ++first_unused;
        const RowSet &s = in.set[first_unused];
        size_t &cur = cursor[s];
        const std::vector<int32_t> &lst = rows_of[s];
        std::vector<int32_t> rows;
        while (cur < lst.size() && (int32_t)rows.size() < n_ub) {
            rows.push_back(lst[cur]);
            used[lst[cur]] = 1;
            ++cur;
        }
        left -= (int32_t)rows.size();
        add_ubatch(sp, in, rows, (int32_t)rows.size(), 1, c);
    }
}

// ---- attention planning tables ---------------------------------------------

// Group a ubatch's rows by first sequence id (which fixes the stream), keep
// ubatch order inside a group, and cut each group into blocks: groups with at
// least PF_MIN_QV query vectors take the tensor-core prefill path in blocks
// of PF_M query vectors, the rest the decode path in blocks of at most
// DEC_QMAX query vectors.
void build_blocks(UbatchHost &u, const kv_cache *c) {
    const int32_t G = c->gqa;
    std::map<int32_t, std::vector<int32_t>> groups;   // seq0 -> ubatch rows
    std::vector<int32_t> order;
    for (int32_t i = 0; i < u.n_tokens; ++i) {
        auto it = groups.find(u.seq0[i]);
        if (it == groups.end()) {
            order.push_back(u.seq0[i]);
            groups[u.seq0[i]].push_back(i);
        } else {
            it->second.push_back(i);
        }
    }
    u.perm.clear();
    u.blocks.clear();
    std::vector<DevBlock> dec, pf;
    std::vector<std::vector<int32_t>> dec_rows, pf_rows;
    for (int32_t q : order) {
        const std::vector<int32_t> &g = groups[q];
        int32_t nq = (int32_t)g.size() * G;
        bool prefill = c->pf_min_qv > 0 && nq >= c->pf_min_qv;
        int32_t per = prefill ? std::max(1, PF_M / G) : std::max(1, DEC_QMAX / G);
        for (size_t a = 0; a < g.size(); a += per) {
            std::vector<int32_t> rows(g.begin() + a, g.begin() + std::min(g.size(), a + per));
            DevBlock b{};
            b.tok0 = -1;
            b.n_rows = (int32_t)rows.size();
            b.seq0 = q;
            b.stream = c->seq_to_stream[q];
            b.path = prefill ? PATH_PREFILL : PATH_DECODE;
            b.pos_min = INT32_MAX;
            b.pos_max = INT32_MIN;
            for (int32_t i : rows) {
                b.pos_min = std::min(b.pos_min, u.pos[i]);
                b.pos_max = std::max(b.pos_max, u.pos[i]);
            }
            // positions pos_min .. pos_max, each once: the rows that see a cell are then
            // counted from the interval of positions that see it, with no pass over them
            b.contig = 0;
            if ((int64_t)b.pos_max - b.pos_min + 1 == (int64_t)rows.size()) {
                std::vector<char> seen(rows.size(), 0);
                bool ok = true;
                for (int32_t i : rows) {
                    char &f = seen[(size_t)(u.pos[i] - b.pos_min)];
                    ok = ok && !f;
                    f = 1;
                }
                b.contig = ok ? 1 : 0;
            }
            (prefill ? pf : dec).push_back(b);
            (prefill ? pf_rows : dec_rows).push_back(rows);
        }
    }
    // decode blocks first, then prefill blocks
    u.n_dec_blocks = (int32_t)dec.size();
    u.n_pf_blocks = (int32_t)pf.size();
    for (size_t k = 0; k < dec.size(); ++k) {
        dec[k].row0 = (int32_t)u.perm.size();
        u.perm.insert(u.perm.end(), dec_rows[k].begin(), dec_rows[k].end());
        u.blocks.push_back(dec[k]);
    }
    for (size_t k = 0; k < pf.size(); ++k) {
        pf[k].row0 = (int32_t)u.perm.size();
        u.perm.insert(u.perm.end(), pf_rows[k].begin(), pf_rows[k].end());
        bool consecutive = true;
        for (size_t i = 1; i < pf_rows[k].size() && consecutive; ++i)
            consecutive = pf_rows[k][i] == pf_rows[k][0] + (int32_t)i;
        pf[k].tok0 = consecutive ? pf_rows[k][0] : -1;
        u.blocks.push_back(pf[k]);
    }
    // CSR: blocks of each sequence
    int32_t nsm = c->prm.n_seq_max;
    u.seq_blk_off.assign(nsm + 1, 0);
    for (const DevBlock &b : u.blocks) u.seq_blk_off[b.seq0 + 1]++;
    for (int32_t q = 0; q < nsm; ++q) u.seq_blk_off[q + 1] += u.seq_blk_off[q];
    u.seq_blk.assign(u.blocks.size(), 0);
    std::vector<int32_t> fill(u.seq_blk_off.begin(), u.seq_blk_off.end() - 1);
    for (size_t k = 0; k < u.blocks.size(); ++k) u.seq_blk[fill[u.blocks[k].seq0]++] = (int32_t)k;
}

template <class T>
size_t append(std::vector<uint8_t> &img, const T *p, size_t n) {
    size_t off = (img.size() + 15) & ~size_t(15);
    img.resize(off + n * sizeof(T));
    if (n) std::memcpy(img.data() + off, p, n * sizeof(T));
    return off;
}

// One flat image of every ubatch's device tables, uploaded on first device use.
void build_image(kv_split *sp, const kv_cache *c) {
    sp->image.clear();
    size_t n = sp->ub.size();
    sp->off_rows.resize(n); sp->off_perm.resize(n); sp->off_blocks.resize(n);
    sp->off_seq_off.resize(n); sp->off_seq_blk.resize(n);
    for (size_t k = 0; k < n; ++k) {
        const UbatchHost &u = sp->ub[k];
        std::vector<DevRow> rows(u.n_tokens);
        for (int32_t i = 0; i < u.n_tokens; ++i) {
            rows[i].cell = u.streams[i] * c->kv_size + u.cells[i];
            rows[i].pos = u.pos[i];
            rows[i].seq0 = u.seq0[i];
            rows[i].stream = u.streams[i];
        }
        sp->off_rows[k] = append(sp->image, rows.data(), rows.size());
        sp->off_perm[k] = append(sp->image, u.perm.data(), u.perm.size());
        sp->off_blocks[k] = append(sp->image, u.blocks.data(), u.blocks.size());
        sp->off_seq_off[k] = append(sp->image, u.seq_blk_off.data(), u.seq_blk_off.size());
        sp->off_seq_blk[k] = append(sp->image, u.seq_blk.data(), u.seq_blk.size());
    }
    sp->image.resize((sp->image.size() + 15) & ~size_t(15));
}

void push_delta(kv_cache *c, size_t g) {
    const CellState &cs = c->cells;
    Delta d{};
    d.cell = (int32_t)g;
    d.pos = cs.pos[g];
    d.epoch = cs.epoch[g];
    d.nseq = cs.nseq[g];
    for (int32_t w = 0; w < cs.n_words; ++w) d.bits[w] = cs.bits[g * cs.n_words + w];
    // The device applies all records of one upload in parallel, so a cell
    // changed twice (freed, then reserved again) keeps only its latest record.
    int32_t &slot = c->pending_idx[g];
    if (slot >= 0) {
        c->pending[slot] = d;
    } else {
        slot = (int32_t)c->pending.size();
        c->pending.push_back(d);
    }
}

}  // namespace

// ============================================================================
// C interface
// ============================================================================

extern "C" {

int kv_init(const kv_params *p, kv_cache **out) {
    return guarded(nullptr, [&]() -> int {
        if (!out) return KV_E_INVAL;
        *out = nullptr;
        if (!p) return KV_E_INVAL;
        if (p->n_ctx < 1 || p->n_batch < 1 || p->n_ubatch < 0 || p->n_seq_max < 1 ||
            p->n_seq_max > KV_MAX_SEQ || p->n_stream < 1 || p->n_stream > p->n_seq_max ||
            p->n_ctx % p->n_stream != 0 || p->n_layer < 1 || p->n_head < 1 || p->n_head_kv < 1 ||
            p->n_head % p->n_head_kv != 0 || p->n_head / p->n_head_kv > 8 ||
            p->head_dim != KV_HEAD_DIM || (p->causal != 0 && p->causal != 1) || p->n_swa < 0)
            return KV_E_INVAL;
        if ((p->k_layers == nullptr) != (p->v_layers == nullptr)) return KV_E_INVAL;
        kv_cache *c = new (std::nothrow) kv_cache();
        if (!c) return KV_E_NOMEM;
        c->prm = *p;
        // UBATCH, "Three things called batch": the two clamps.
        c->n_batch = p->causal ? std::min(p->n_ctx, p->n_batch) : p->n_batch;
        int32_t req_ub = p->n_ubatch == 0 ? p->n_batch : p->n_ubatch;
        c->n_ubatch = std::min(c->n_batch, req_ub);
        c->kv_size = p->n_ctx / p->n_stream;
        c->n_words = (p->n_seq_max + 63) / 64;
        c->gqa = p->n_head / p->n_head_kv;
        c->pf_min_qv = PF_MIN_QV;
        c->seq_to_stream.resize(p->n_seq_max);
        for (int32_t q = 0; q < p->n_seq_max; ++q) {
            int32_t s = p->seq_to_stream ? p->seq_to_stream[q] : q % p->n_stream;
            if (s < 0 || s >= p->n_stream) { delete c; return KV_E_INVAL; }
            c->seq_to_stream[q] = s;
        }
        c->prm.seq_to_stream = nullptr;
        c->prm.k_layers = c->prm.v_layers = nullptr;
        cells_init(c->cells, p->n_stream, c->kv_size, c->n_words);
        if (p->k_layers) {
            c->pending_idx.assign((size_t)p->n_ctx, -1);
            c->k_layers.assign(p->k_layers, p->k_layers + p->n_layer);
            c->v_layers.assign(p->v_layers, p->v_layers + p->n_layer);
            for (int32_t l = 0; l < p->n_layer; ++l) {
                if (!c->k_layers[l] || !c->v_layers[l] ||
                    ((uintptr_t)c->k_layers[l] & 15) || ((uintptr_t)c->v_layers[l] & 15)) {
                    delete c;
                    return KV_E_INVAL;
                }
            }
            c->has_device = true;
            int rc = device_init(c);
            if (rc != KV_OK) {
                if (log_on()) std::fprintf(stderr, "kvattn: device init failed: %s\n", c->err.c_str());
                device_free(c);
                delete c;
                return rc;
            }
        }
        if (log_on())
            std::fprintf(stderr, "kvattn: n_ctx %d n_stream %d kv_size %d n_batch %d n_ubatch %d "
                         "layers %d heads %d/%d; K+V %.1f MiB\n", p->n_ctx, p->n_stream, c->kv_size,
                         c->n_batch, c->n_ubatch, p->n_layer, p->n_head, p->n_head_kv,
                         (double)p->n_ctx * p->n_head_kv * p->head_dim * 2 * 2 * p->n_layer / 1048576.0);
        *out = c;
        return KV_OK;
    });
}

void kv_free(kv_cache *c) {
    if (!c) return;
    if (c->has_device) device_free(c);
    delete c;
}

int32_t kv_n_batch(const kv_cache *c) { return c ? c->n_batch : KV_E_INVAL; }
int32_t kv_n_ubatch(const kv_cache *c) { return c ? c->n_ubatch : KV_E_INVAL; }
int32_t kv_kv_size(const kv_cache *c) { return c ? c->kv_size : KV_E_INVAL; }
const char *kv_last_error(const kv_cache *c) { return c ? c->err.c_str() : "null cache"; }

int kv_split_ubatches(kv_cache *c, const kv_batch *b, int32_t mode, kv_split **out) {
    return guarded(c, [&]() -> int {
        if (!c || !b || !out) return KV_E_INVAL;
        *out = nullptr;
        if (mode < KV_SPLIT_AUTO || mode > KV_SPLIT_SEQ) return c->set_err(KV_E_INVAL, "bad split mode");
        const int32_t n = b->n_tokens;
        if (n < 1) return c->set_err(KV_E_INVAL, "empty batch");
        if (n > c->n_batch) return c->set_err(KV_E_BATCH_TOO_LARGE, "n_tokens > n_batch");
        const int32_t nsm = c->prm.n_seq_max;
        SplitIn in;
        in.n = n;
        in.ids_off.resize((size_t)n + 1);
        in.ids_off[0] = 0;
        in.ids.reserve(n);
        std::vector<int32_t> sorted;   // a row's ids, for the repeat check (rows of two or more)
        for (int32_t i = 0; i < n; ++i) {
            const size_t at = in.ids.size();
            if (!b->seq_id) {
                in.ids.push_back(0);
            } else if (!b->n_seq_id) {
                if (!b->seq_id[i]) return c->set_err(KV_E_INVAL, "null seq_id row");
                in.ids.push_back(b->seq_id[i][0]);
            } else {
                int32_t k = b->n_seq_id[i];
                if (k < 1 || k > nsm) return c->set_err(KV_E_INVAL, "bad n_seq_id");
                if (!b->seq_id[i]) return c->set_err(KV_E_INVAL, "null seq_id row");
                in.ids.insert(in.ids.end(), b->seq_id[i], b->seq_id[i] + k);
            }
            const int32_t *ids = in.ids.data() + at;
            const int32_t k = (int32_t)(in.ids.size() - at);
            for (int32_t t = 0; t < k; ++t)
                if (ids[t] < 0 || ids[t] >= nsm) return c->set_err(KV_E_SEQ_RANGE, "sequence id out of range");
            if (k > 1) {
                sorted.assign(ids, ids + k);
                std::sort(sorted.begin(), sorted.end());
                if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
                    return c->set_err(KV_E_INVAL, "repeated sequence id in one slot");
            }
            const int32_t st = c->seq_to_stream[ids[0]];
            for (int32_t t = 1; t < k; ++t)
                if (c->seq_to_stream[ids[t]] != st)
                    return c->set_err(KV_E_CROSS_STREAM, "slot spans streams");
            if (b->pos && b->pos[i] < 0) return c->set_err(KV_E_INVAL, "negative position");
            in.ids_off[i + 1] = (int32_t)in.ids.size();
        }
        in.pos.resize(n);
        if (b->pos) {
            for (int32_t i = 0; i < n; ++i) in.pos[i] = b->pos[i];
        } else {
            // BATCH-ZH, Part A: a NULL pos is filled by counting up per sequence.
            std::map<int32_t, int32_t> last;   // sequence -> largest pos so far
            for (int32_t i = 0; i < n; ++i) {
                int32_t q = in.ids_of(i)[0];
                auto it = last.find(q);
                int32_t best = it != last.end() ? it->second : seq_pos_max(c, q);
                in.pos[i] = best + 1;
                for (int32_t t = 0; t < in.n_ids(i); ++t) {
                    const int32_t x = in.ids_of(i)[t];
                    auto jt = last.find(x);
                    int32_t prev = jt != last.end() ? jt->second : seq_pos_max(c, x);
                    last[x] = std::max(prev, in.pos[i]);
                }
            }
        }
        kv_split *sp = new (std::nothrow) kv_split();
        if (!sp) return c->set_err(KV_E_NOMEM, "split alloc");
        sp->id = c->next_split_id++;
        sp->owner = c;
        sp->n_tokens = n;
        if (mode == KV_SPLIT_AUTO) mode = c->prm.n_stream == 1 ? KV_SPLIT_SIMPLE : KV_SPLIT_EQUAL;
        if (mode == KV_SPLIT_SIMPLE) {
            split_simple(sp, in, c->n_ubatch, c);
        } else {
            in.build_sets();
            if (mode == KV_SPLIT_EQUAL) split_equal(sp, in, c->n_ubatch, c);
            else split_seq(sp, in, c->n_ubatch, c);
        }
        *out = sp;
        return KV_OK;
    });
}

int32_t kv_split_count(const kv_split *s) { return s ? (int32_t)s->ub.size() : KV_E_INVAL; }

int kv_split_ubatch(const kv_split *s, int32_t k, kv_ubatch_info *out) {
    if (!s || !out || k < 0 || k >= (int32_t)s->ub.size()) return KV_E_INVAL;
    const UbatchHost &u = s->ub[k];
    out->n_tokens = u.n_tokens;
    out->n_seq_tokens = u.n_seq_tokens;
    out->n_seqs = u.n_seqs;
    out->n_seqs_unq = (int32_t)u.seq_unq.size();
    out->n_kv = s->prepared ? u.n_kv : 0;
    out->rows = u.rows.data();
    out->pos = u.pos.data();
    out->seq0 = u.seq0.data();
    out->seq_id_unq = u.seq_unq.data();
    out->streams = u.streams.data();
    out->cells = s->prepared ? u.cells.data() : nullptr;
    return KV_OK;
}

void kv_split_free(kv_split *s) { delete s; }

int kv_prepare_cells(kv_cache *c, kv_split *sp) {
    return guarded(c, [&]() -> int {
        if (!c || !sp || sp->owner != c) return KV_E_INVAL;
        if (sp->prepared) return c->set_err(KV_E_ORDER, "split already prepared");
        CellState &cs = c->cells;
        const int32_t W = cs.n_words;
        // undo log: cells filled so far (all were empty before)
        std::vector<size_t> filled;
        std::vector<int32_t> saved_first_free = cs.first_free, saved_used = cs.used_max_p1;
        uint32_t epoch = c->next_epoch;
        bool ok = true;
        for (UbatchHost &u : sp->ub) {
            u.cells.assign(u.n_tokens, -1);
            u.epoch = epoch++;
            for (int32_t i = 0; i < u.n_tokens && ok; ++i) {
                int32_t s = u.streams[i];
                int32_t j = next_empty(cs, s, cs.first_free[s]);
                if (j < 0) { ok = false; break; }
                cs.first_free[s] = j + 1;
                size_t g = (size_t)s * cs.kv_size + j;
                cs.pos[g] = u.pos[i];
                uint64_t *w = &cs.bits[g * W];
                for (int32_t x = 0; x < W; ++x) w[x] = 0;
                for (int32_t t = u.ids_off[i]; t < u.ids_off[i + 1]; ++t)
                    w[u.ids[t] >> 6] |= 1ull << (u.ids[t] & 63);
                cs.nseq[g] = u.ids_off[i + 1] - u.ids_off[i];
                cs.epoch[g] = u.epoch;
                filled.push_back(g);
                u.cells[i] = j;
                cs.used_max_p1[s] = std::max(cs.used_max_p1[s], j + 1);
            }
            if (!ok) break;
            int32_t nkv = 0;
            std::set<int32_t> touched(u.streams.begin(), u.streams.end());
            for (int32_t s : touched) nkv = std::max(nkv, n_kv_of(cs, s));
            u.n_kv = nkv;
        }
        if (!ok) {
            for (size_t g : filled) {
                cs.pos[g] = -1;
                cs.nseq[g] = 0;
                cs.epoch[g] = 0;
                for (int32_t x = 0; x < W; ++x) cs.bits[g * W + x] = 0;
            }
            cs.first_free = saved_first_free;
            cs.used_max_p1 = saved_used;
            for (UbatchHost &u : sp->ub) { u.cells.clear(); u.n_kv = 0; }
            return c->set_err(KV_NO_SLOT, "no free cell");
        }
        c->next_epoch = epoch;
        sp->prepared = true;
        sp->rm_gen = c->rm_gen;
        if (c->has_device) {
            for (size_t g : filled) push_delta(c, g);
            for (UbatchHost &u : sp->ub) build_blocks(u, c);
            build_image(sp, c);
            sp->stored.assign(c->prm.n_layer, std::vector<uint8_t>(sp->ub.size(), 0));
        }
        return KV_OK;
    });
}

int kv_seq_rm(kv_cache *c, int32_t seq, int32_t p0, int32_t p1) {
    return guarded(c, [&]() -> int {
        if (!c) return KV_E_INVAL;
        if (seq >= c->prm.n_seq_max) return c->set_err(KV_E_SEQ_RANGE, "sequence id out of range");
        CellState &cs = c->cells;
        const int32_t W = cs.n_words;
        const int64_t hi = p1 < 0 ? INT64_MAX : (int64_t)p1;
        const bool all = seq < 0 && p0 <= 0 && p1 < 0;
        bool changed = false;
        for (int32_t s = 0; s < cs.n_stream; ++s) {
            if (seq >= 0 && c->seq_to_stream[seq] != s) continue;
            size_t base = (size_t)s * cs.kv_size;
            for (int32_t j = 0; j < cs.used_max_p1[s]; ++j) {
                size_t g = base + j;
                if (!cs.nseq[g]) continue;
                if (cs.pos[g] < p0 || cs.pos[g] >= hi) continue;
                uint64_t *w = &cs.bits[g * W];
                if (seq < 0) {
                    for (int32_t x = 0; x < W; ++x) w[x] = 0;
                    cs.nseq[g] = 0;
                } else if (bit_has(w, seq)) {
                    w[seq >> 6] &= ~(1ull << (seq & 63));
                    cs.nseq[g] -= 1;
                } else {
                    continue;
                }
                if (cs.nseq[g] == 0) {
                    cs.pos[g] = -1;
                    cs.epoch[g] = 0;
                    cs.first_free[s] = std::min(cs.first_free[s], j);
                }
                changed = true;
                if (c->has_device && !all) push_delta(c, g);
            }
            refresh_used_max(cs, s);
        }
        if (changed || all) {
            c->rm_gen++;
            if (c->has_device && all) {
                // the whole mirror is cleared on the device instead of cell by cell
                for (const Delta &d : c->pending) c->pending_idx[d.cell] = -1;
                c->pending.clear();
                c->pending_reset = true;
            }
        }
        return KV_OK;
    });
}

int kv_seq_cp(kv_cache *c, int32_t src, int32_t dst, int32_t p0, int32_t p1) {
    return guarded(c, [&]() -> int {
        if (!c) return KV_E_INVAL;
        if (src < 0 || src >= c->prm.n_seq_max || dst < 0 || dst >= c->prm.n_seq_max)
            return c->set_err(KV_E_SEQ_RANGE, "sequence id out of range");
        const int32_t s = c->seq_to_stream[src];
        if (c->seq_to_stream[dst] != s) return c->set_err(KV_E_CROSS_STREAM, "copy between streams");
        if (src == dst) return KV_OK;
        CellState &cs = c->cells;
        const int32_t W = cs.n_words;
        const int64_t hi = p1 < 0 ? INT64_MAX : (int64_t)p1;
        const size_t base = (size_t)s * cs.kv_size;
        bool changed = false;
        for (int32_t j = 0; j < cs.used_max_p1[s]; ++j) {
            const size_t g = base + j;
            if (!cs.nseq[g] || cs.pos[g] < p0 || cs.pos[g] >= hi) continue;
            uint64_t *w = &cs.bits[g * W];
            if (!bit_has(w, src) || bit_has(w, dst)) continue;
            w[dst >> 6] |= 1ull << (dst & 63);
            cs.nseq[g] += 1;
            changed = true;
            if (c->has_device) push_delta(c, g);
        }
        if (changed) c->rm_gen++;   // splits prepared before see another cell state
        return KV_OK;
    });
}

int32_t kv_seq_pos_max(const kv_cache *c, int32_t seq) {
    if (!c || seq < 0 || seq >= c->prm.n_seq_max) return KV_E_SEQ_RANGE;
    return seq_pos_max(c, seq);
}

int kv_cells_read(const kv_cache *c, int32_t stream, int32_t *pos_out, uint64_t *bits_out) {
    if (!c || stream < 0 || stream >= c->prm.n_stream || !pos_out) return KV_E_INVAL;
    const CellState &cs = c->cells;
    size_t base = (size_t)stream * cs.kv_size;
    std::memcpy(pos_out, cs.pos.data() + base, sizeof(int32_t) * cs.kv_size);
    if (bits_out)
        std::memcpy(bits_out, cs.bits.data() + base * cs.n_words,
                    sizeof(uint64_t) * cs.kv_size * cs.n_words);
    return KV_OK;
}

int32_t kv_stream_n_kv(const kv_cache *c, int32_t stream) {
    if (!c || stream < 0 || stream >= c->prm.n_stream) return KV_E_INVAL;
    return n_kv_of(c->cells, stream);
}

}  // extern "C"
