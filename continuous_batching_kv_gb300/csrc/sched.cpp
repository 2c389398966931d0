// Iteration-level (continuous) batching: the host-side scheduler loop.
//
// "Iteration-Level Batching: Reforming the Batch at Every Token", "The loop that
// replaces the batch": before every pass, retire the finished sequences and
// release their cache, admit waiting requests while the token budget and the
// cache budget both allow, assemble the batch (a new sequence's whole prompt, one
// token per running sequence).  "The budget that actually binds": positions per
// pass, and cache cells (reserved here for prompt + max_new at admission, the
// page's conservative policy).  No allocation on the per-pass path once the
// arrays have grown to the largest batch (the page: schedulers avoid allocating
// memory on the critical path).

#include <algorithm>
#include <deque>
#include <vector>

#include "internal.h"

namespace {

struct Req {
    int32_t L = 0, N = 0;        // prompt tokens, new tokens
    int32_t seq = -1;
    int32_t generated = 0;
};

}  // namespace

struct kv_sched {
    kv_cache *c = nullptr;
    kv_sched_params p{};
    int32_t free_cells = 0;
    int32_t next_rid = 0;
    std::deque<Req> waiting;
    std::vector<Req> running;            // admission order
    bool batch_open = false;             // a batch was assembled and not advanced yet
    int64_t passes = 0, useful = 0;
    // the last batch (owned here)
    std::vector<int32_t> pos, seq, n_seq_id, retired;
    std::vector<const int32_t *> seq_ptr;
    std::vector<uint8_t> used;           // [n_seq_max] sequence id in use
};

extern "C" {

int kv_sched_init(kv_cache *c, const kv_sched_params *p, kv_sched **out) {
    return guarded(c, [&]() -> int {
        if (!c || !p || !out) return KV_E_INVAL;
        if (c->prm.n_stream != 1) return c->set_err(KV_E_INVAL, "the scheduler drives a unified cache");
        if (p->max_seqs < 1 || p->max_seqs > c->prm.n_seq_max || p->token_budget < p->max_seqs)
            return c->set_err(KV_E_INVAL, "scheduler: 1 <= max_seqs <= n_seq_max, token_budget >= max_seqs");
        if (p->token_budget > c->n_batch)   // a pass's batch is one kv_split_ubatches call
            return c->set_err(KV_E_INVAL, "scheduler: token_budget > n_batch");
        kv_sched *s = new kv_sched;
        s->c = c;
        s->p = *p;
        s->free_cells = c->kv_size;
        s->used.assign((size_t)c->prm.n_seq_max, 0);
        *out = s;
        return KV_OK;
    });
}

void kv_sched_free(kv_sched *s) { delete s; }

int kv_sched_submit(kv_sched *s, int32_t prompt_len, int32_t max_new) {
    return guarded(s ? s->c : nullptr, [&]() -> int {
        if (!s) return KV_E_INVAL;
        if (prompt_len < 1 || max_new < 1 || prompt_len > s->p.token_budget ||
            (int64_t)prompt_len + max_new > s->c->kv_size)
            return s->c->set_err(KV_E_INVAL, "request can never run");
        Req r;
        r.L = prompt_len;
        r.N = max_new;
        s->waiting.push_back(r);
        return s->next_rid++;
    });
}

int kv_sched_next(kv_sched *s, kv_sched_batch *out) {
    return guarded(s ? s->c : nullptr, [&]() -> int {
        if (!s || !out) return KV_E_INVAL;
        if (s->batch_open) return s->c->set_err(KV_E_ORDER, "the previous batch was not advanced");
        // 1. retire the finished sequences, releasing their reservations and cells
        s->retired.clear();
        size_t keep = 0;
        for (size_t i = 0; i < s->running.size(); ++i) {
            Req &r = s->running[i];
            if (r.generated == r.N) {
                s->retired.push_back(r.seq);
                s->free_cells += r.L + r.N;
                s->used[(size_t)r.seq] = 0;
                int rc = kv_seq_rm(s->c, r.seq, 0, -1);
                if (rc != KV_OK) return rc;
            } else {
                s->running[keep++] = r;
            }
        }
        s->running.resize(keep);
        // 2. admit, first come first served, while both budgets allow
        int64_t tokens = (int64_t)s->running.size();   // one position per running sequence
        const size_t n_old = s->running.size();
        if (!s->p.fixed || s->running.empty()) {
            while (!s->waiting.empty()) {
                Req r = s->waiting.front();
                if ((int32_t)s->running.size() >= s->p.max_seqs || r.L + r.N > s->free_cells ||
                    tokens + r.L > s->p.token_budget)
                    break;
                s->waiting.pop_front();
                int32_t q = 0;
                while (s->used[(size_t)q]) ++q;        // running < max_seqs <= n_seq_max: one is free
                s->used[(size_t)q] = 1;
                r.seq = q;
                s->free_cells -= r.L + r.N;
                tokens += r.L;
                s->running.push_back(r);
            }
        }
        // 3. assemble: running sequences one token each, then the new prompts
        s->pos.clear();
        s->seq.clear();
        for (size_t i = 0; i < s->running.size(); ++i) {
            const Req &r = s->running[i];
            if (i < n_old) {
                s->pos.push_back(r.L + r.generated - 1);
                s->seq.push_back(r.seq);
            } else {
                for (int32_t t = 0; t < r.L; ++t) {
                    s->pos.push_back(t);
                    s->seq.push_back(r.seq);
                }
            }
        }
        const size_t n = s->pos.size();
        s->n_seq_id.assign(n, 1);
        s->seq_ptr.resize(n);
        for (size_t i = 0; i < n; ++i) s->seq_ptr[i] = &s->seq[i];
        out->batch.n_tokens = (int32_t)n;
        out->batch.pos = s->pos.data();
        out->batch.n_seq_id = s->n_seq_id.data();
        out->batch.seq_id = s->seq_ptr.data();
        out->n_retired = (int32_t)s->retired.size();
        out->retired = s->retired.data();
        s->batch_open = n > 0;
        return KV_OK;
    });
}

int kv_sched_advance(kv_sched *s) {
    if (!s) return KV_E_INVAL;
    if (!s->batch_open) return KV_OK;
    for (Req &r : s->running) r.generated += 1;
    s->passes += 1;
    s->useful += (int64_t)s->running.size();
    s->batch_open = false;
    return KV_OK;
}

int kv_sched_stats(const kv_sched *s, kv_sched_info *out) {
    if (!s || !out) return KV_E_INVAL;
    out->passes = s->passes;
    out->useful = s->useful;
    out->running = (int32_t)s->running.size();
    out->waiting = (int32_t)s->waiting.size();
    out->free_cells = s->free_cells;
    return KV_OK;
}

}  // extern "C"
