/*
 * The C interface from C (no GPU): a host-only cache (no K/V tensors), a split,
 * cell reservation, a sequence copy, and the iteration-level batching loop with
 * its batches handed to kv_split_ubatches as they are.  Prints one line of
 * figures on success; exits non-zero on the first unexpected result.
 */
#include <stdio.h>
#include <stdlib.h>

#include "kvattn.h"

#define CHECK(x)                                                              \
    do {                                                                      \
        if (!(x)) {                                                           \
            fprintf(stderr, "failed: %s (line %d)\n", #x, __LINE__);          \
            return 1;                                                         \
        }                                                                     \
    } while (0)

int main(void) {
    kv_params p = {0};
    p.n_ctx = 4096;
    p.n_batch = 512;
    p.n_ubatch = 128;
    p.n_seq_max = 8;
    p.n_stream = 1;
    p.n_layer = 1;
    p.n_head = 16;
    p.n_head_kv = 8;
    p.head_dim = 128;
    p.causal = 1;
    kv_cache *c = NULL;
    CHECK(kv_init(&p, &c) == KV_OK && c != NULL);
    CHECK(kv_n_ubatch(c) == 128);

    /* a 300-token prompt of sequence 0: ubatches of 128, 128, 44 */
    int32_t pos[300], one[300], zero = 0;
    const int32_t *ids[300];
    for (int i = 0; i < 300; ++i) {
        pos[i] = i;
        one[i] = 1;
        ids[i] = &zero;
    }
    kv_batch b = {300, pos, one, ids};
    kv_split *s = NULL;
    CHECK(kv_split_ubatches(c, &b, KV_SPLIT_AUTO, &s) == KV_OK);
    CHECK(kv_split_count(s) == 3);
    kv_ubatch_info u;
    CHECK(kv_split_ubatch(s, 2, &u) == KV_OK && u.n_tokens == 44);
    CHECK(kv_prepare_cells(c, s) == KV_OK);
    kv_split_free(s);
    CHECK(kv_seq_pos_max(c, 0) == 299);

    /* sequence 1 shares positions 0 .. 99 (BATCH-ZH, Part E) */
    CHECK(kv_seq_cp(c, 0, 1, 0, 100) == KV_OK);
    CHECK(kv_seq_pos_max(c, 1) == 99);
    CHECK(kv_seq_cp(c, 0, 9, 0, -1) == KV_E_SEQ_RANGE);
    CHECK(kv_seq_rm(c, -1, 0, -1) == KV_OK);       /* clear */
    CHECK(kv_seq_pos_max(c, 0) == -1);

    /* the batching loop: ITER's eight output lengths, fixed and continuous */
    static const int32_t lengths[8] = {64, 128, 256, 512, 512, 1024, 1024, 2048};
    int64_t passes[2] = {0, 0};
    for (int fixed = 1; fixed >= 0; --fixed) {
        kv_params q = p;
        q.n_ctx = 1 << 16;
        q.n_batch = 2048;
        q.n_ubatch = 512;
        kv_cache *cc = NULL;
        CHECK(kv_init(&q, &cc) == KV_OK);
        kv_sched_params sp = {8, 2048, fixed};
        kv_sched *sch = NULL;
        CHECK(kv_sched_init(cc, &sp, &sch) == KV_OK);
        for (int r = 0; r < 16; ++r) CHECK(kv_sched_submit(sch, 32, lengths[r % 8]) == r);
        for (;;) {
            kv_sched_batch nb;
            CHECK(kv_sched_next(sch, &nb) == KV_OK);
            if (nb.batch.n_tokens == 0) break;
            kv_split *ss = NULL;
            CHECK(kv_split_ubatches(cc, &nb.batch, KV_SPLIT_AUTO, &ss) == KV_OK);
            CHECK(kv_prepare_cells(cc, ss) == KV_OK);    /* reservations make room */
            kv_split_free(ss);
            CHECK(kv_sched_advance(sch) == KV_OK);
        }
        kv_sched_info st;
        CHECK(kv_sched_stats(sch, &st) == KV_OK);
        CHECK(st.useful == 2 * 5568 && st.running == 0 && st.waiting == 0);
        CHECK(st.free_cells == kv_kv_size(cc));
        passes[fixed] = st.passes;
        kv_sched_free(sch);
        kv_free(cc);
    }
    /* ITER: a fixed batch of the eight lengths takes 2048 passes per group */
    CHECK(passes[1] == 2 * 2048);
    CHECK(passes[0] < passes[1]);
    kv_free(c);
    printf("ok fixed_passes=%lld continuous_passes=%lld\n", (long long)passes[1], (long long)passes[0]);
    return 0;
}
