/*
 * kvattn.h -- ubatch attention over a cell-indexed KV cache, C interface.
 *
 * One ubatch of token slots (each slot: a position and a set of sequence ids)
 * attends to a KV cache whose rows ("cells") are shared by all layers.  The
 * host side splits a batch into ubatches and reserves cells; the device side
 * scatters K/V rows into the cache, builds the KQ mask from the cells'
 * positions and sequence sets, and runs GQA flash attention.
 *
 * Pages this interface restates (cited by title and section):
 *   "llama.cpp and the ubatch"                                  (UBATCH)
 *   "Batch、Ubatch 与解码主循环"                                  (BATCH-ZH)
 *   "What does llama.cpp's KV cache actually look like in memory?" (KV-MEM)
 *   "Iteration-Level Batching: Reforming the Batch at Every Token" (ITER)
 *
 * Conventions
 *   - Every function returning int returns KV_OK (0), KV_NO_SLOT (1) or a
 *     negative KV_E_* code.  No function aborts or prints unless KV_LOG=1.
 *   - Device pointers are plain CUDA device addresses on the current device;
 *     `stream` arguments are cudaStream_t values passed as void* (NULL = the
 *     legacy default stream).  All device work is asynchronous on `stream`.
 *     A cache's device calls are ordered on one stream (the library keeps one
 *     attention plan and its scratch per cache); besides, the library's own
 *     side stream builds the next ubatch's plan ahead, ordered after the
 *     caller's stream (see ubatch_attention).
 *   - The caller owns every buffer it passes in (K/V caches, q, k_cur, v_cur,
 *     o, mask_out).  The library owns kv_cache and kv_split handles and the
 *     device memory it allocates in kv_init (cell-metadata mirror, per-ubatch
 *     row tables, attention plan and split-K scratch).
 *   - A kv_cache is not thread-safe; use one host thread per cache (a kv_sched
 *     belongs to its cache's thread too).
 *   - A call that allocates host memory returns KV_E_NOMEM when that fails; no
 *     C++ exception leaves the library.
 */
#ifndef KVATTN_H
#define KVATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define KV_OK                  0
#define KV_NO_SLOT             1   /* no free cell for some row; cache unchanged (BATCH-ZH, Part F: the decode call returns 1) */
#define KV_E_INVAL            (-1) /* bad argument: empty batch, bad n_seq_id, repeated id, negative pos, bad params, bad index */
#define KV_E_BATCH_TOO_LARGE  (-2) /* n_tokens > effective n_batch (UBATCH, "Three things called batch": the engine refuses it) */
#define KV_E_SEQ_RANGE        (-3) /* a sequence id outside [0, n_seq_max) */
#define KV_E_CROSS_STREAM     (-4) /* one slot's sequence ids map to different streams */
#define KV_E_ORDER            (-5) /* device call out of order (attention before this layer stored ubatches 0..ub, or a split not prepared) */
#define KV_E_STALE            (-6) /* the split was prepared before a later kv_seq_rm / kv_seq_cp that changed a cell */
#define KV_E_CUDA             (-7) /* a CUDA call failed; kv_last_error() has the text */
#define KV_E_NOMEM            (-8) /* host or device allocation failed */
#define KV_E_NO_DEVICE        (-9) /* device call on a host-only cache (k_layers == NULL in kv_init) */

/* ---- split strategies (BATCH-ZH, Part C) -------------------------------- */
#define KV_SPLIT_AUTO    0  /* split_simple when n_stream == 1, else split_equal(sequential) */
#define KV_SPLIT_SIMPLE  1
#define KV_SPLIT_EQUAL   2
#define KV_SPLIT_SEQ     3

#define KV_MAX_SEQ       256   /* largest n_seq_max */
#define KV_HEAD_DIM      128   /* the only head_dim the kernels are built for */

typedef struct kv_cache kv_cache;
typedef struct kv_split kv_split;

/*
 * kv_params -- context parameters.
 *
 * UBATCH, "Three things called batch": n_batch is the logical limit on one
 * call, n_ubatch the physical ubatch size; at creation n_ubatch is clamped to
 * n_batch, and under causal attention n_batch is clamped to n_ctx.  A
 * requested n_ubatch of 0 means n_batch.  KV-MEM, "Unified versus
 * non-unified": n_ctx cells are split evenly over n_stream streams
 * (kv_size = n_ctx / n_stream cells per stream; 1 stream = unified cache).
 *
 *   n_ctx         total cells over all streams; n_ctx % n_stream == 0
 *   n_batch       requested logical batch limit, >= 1
 *   n_ubatch      requested ubatch size, 0 = n_batch
 *   n_seq_max     number of sequence ids, 1..KV_MAX_SEQ
 *   n_stream      1..n_seq_max
 *   n_layer       layers (each has its own K and V tensor)
 *   n_head        query heads; n_head % n_head_kv == 0, n_head / n_head_kv <= 8
 *   n_head_kv     KV heads
 *   head_dim      must be KV_HEAD_DIM
 *   causal        1 = causal attention (mask later positions), 0 = not
 *   n_swa         sliding window in positions, 0 = none: a cell n_swa or more
 *                 positions behind the row is masked (UBATCH, "The mask is
 *                 doing the work": "outside the sliding window"); >= 0
 *   seq_to_stream NULL (sequence q lives in stream q % n_stream) or an array
 *                 of n_seq_max stream indices, copied by kv_init
 *   k_layers, v_layers
 *                 NULL (a host-only cache: splitting and cell reservation
 *                 work, device calls return KV_E_NO_DEVICE), or arrays of
 *                 n_layer device pointers, each to a caller-owned fp16 tensor
 *                 of n_stream * kv_size rows of n_head_kv * head_dim values
 *                 (ggml shape [n_embd_k_gqa, kv_size, n_stream], KV-MEM, "The
 *                 tensor's three dimensions"), 16-byte aligned.  Copied.
 */
typedef struct kv_params {
    int32_t n_ctx;
    int32_t n_batch;
    int32_t n_ubatch;
    int32_t n_seq_max;
    int32_t n_stream;
    int32_t n_layer;
    int32_t n_head;
    int32_t n_head_kv;
    int32_t head_dim;
    int32_t causal;
    int32_t n_swa;
    const int32_t *seq_to_stream;
    void *const *k_layers;
    void *const *v_layers;
} kv_params;

/*
 * kv_batch -- one list of token slots (UBATCH, "Three things called batch";
 * BATCH-ZH, Part A), host memory, read only during kv_split_ubatches.
 *
 *   n_tokens  number of slots, 1..n_batch
 *   pos       [n_tokens] positions, or NULL: slot i then gets 1 + the largest
 *             position its first sequence already holds in the cache or in
 *             earlier slots of this batch, or 0 if none
 *   n_seq_id  [n_tokens] ids per slot (1..n_seq_max), or NULL: 1 each
 *   seq_id    [n_tokens] pointers to each slot's ids, or NULL: every slot in
 *             sequence 0.  The first id, seq_id[i][0], is the one the slot's
 *             query masks with (UBATCH, "The mask is doing the work"); all
 *             ids own the cell the slot is stored in (prefix sharing).
 */
typedef struct kv_batch {
    int32_t n_tokens;
    const int32_t *pos;
    const int32_t *n_seq_id;
    const int32_t *const *seq_id;
} kv_batch;

/*
 * kv_ubatch_info -- read-only view of one ubatch of a split (BATCH-ZH,
 * Part B).  Arrays are owned by the split and live until kv_split_free.
 *
 *   n_tokens     rows; == n_seq_tokens * n_seqs
 *   n_seq_tokens rows taken from each sequence set (1 for split_simple)
 *   n_seqs       number of sequence sets
 *   n_seqs_unq   distinct sequence ids
 *   n_kv         attention width after this ubatch's cells are reserved
 *                (UBATCH, "Prefill and decode are not the same shape"),
 *                0 before kv_prepare_cells
 *   rows         [n_tokens] batch index of each ubatch row
 *   pos          [n_tokens] position of each row
 *   seq0         [n_tokens] first sequence id of each row
 *   seq_id_unq   [n_seqs_unq] distinct ids, ascending
 *   streams      [n_tokens] stream of each row
 *   cells        [n_tokens] stream-local cell of each row, NULL before
 *                kv_prepare_cells
 */
typedef struct kv_ubatch_info {
    int32_t n_tokens;
    int32_t n_seq_tokens;
    int32_t n_seqs;
    int32_t n_seqs_unq;
    int32_t n_kv;
    const int32_t *rows;
    const int32_t *pos;
    const int32_t *seq0;
    const int32_t *seq_id_unq;
    const int32_t *streams;
    const int32_t *cells;
} kv_ubatch_info;

/* ---- lifetime ----------------------------------------------------------- */

/*
 * kv_init -- normalise the parameters and create an empty cache.
 * UBATCH, "Three things called batch" (the two clamps); KV-MEM, "28 layers,
 * 56 tensors" (one K and one V tensor per layer) and "Unified versus
 * non-unified" (n_stream partitions).  With device tensors it also allocates
 * the device cell-metadata mirror and attention workspace on the current
 * device (about 40 B per cell plus O(n_ubatch) tables and split-K scratch)
 * and builds one TMA descriptor per K/V tensor.
 * Errors: KV_E_INVAL (bad params), KV_E_NOMEM, KV_E_CUDA.  *out is NULL on error.
 */
int kv_init(const kv_params *p, kv_cache **out);

/* kv_free -- release the cache and its device memory (not the caller's K/V). */
void kv_free(kv_cache *c);

/* Effective sizes after the clamps, and the derived per-stream cell count. */
int32_t kv_n_batch(const kv_cache *c);
int32_t kv_n_ubatch(const kv_cache *c);
int32_t kv_kv_size(const kv_cache *c);

/* Text of the last error on this cache (never NULL; "" if none). */
const char *kv_last_error(const kv_cache *c);

/* ---- host side: split and reserve ------------------------------------- */

/*
 * kv_split_ubatches -- validate/auto-fill a batch and split it into ubatches.
 * BATCH-ZH, Part F step 1 (validate and fill) and Part C (split_simple,
 * split_equal, split_seq; KV_SPLIT_AUTO is the cache's own choice: one
 * stream -> split_simple, several -> split_equal(n_ubatch, sequential)).
 *   mode  one of KV_SPLIT_*
 *   out   receives a new split handle (free with kv_split_free)
 * Errors: KV_E_INVAL, KV_E_BATCH_TOO_LARGE, KV_E_SEQ_RANGE,
 * KV_E_CROSS_STREAM, KV_E_NOMEM.  The cache is not modified.
 */
int kv_split_ubatches(kv_cache *c, const kv_batch *b, int32_t mode, kv_split **out);

/* Number of ubatches in a split (>= 1), or a negative code. */
int32_t kv_split_count(const kv_split *s);

/* Fill *out with ubatch k's view.  KV_E_INVAL if k is out of range. */
int kv_split_ubatch(const kv_split *s, int32_t k, kv_ubatch_info *out);

/* Free a split handle (NULL is ignored). */
void kv_split_free(kv_split *s);

/*
 * kv_prepare_cells -- reserve one cell per row of every ubatch of the split.
 * BATCH-ZH, Part C ("策略选择": slots are reserved for all ubatches before
 * any runs) and Part F (a full cache returns 1).  First fit: ubatches in
 * order, rows in order, each row takes the lowest-index empty cell of its
 * stream; the cell records the row's position and all of its ids.
 * All or nothing: on KV_NO_SLOT the cache is exactly as before.
 * A split can be prepared once (KV_E_ORDER on a second call).
 */
int kv_prepare_cells(kv_cache *c, kv_split *s);

/*
 * kv_seq_rm -- remove sequence `seq` (every sequence if seq < 0) from cells
 * with p0 <= pos < p1 (p1 < 0: no upper bound); a cell left with no sequence
 * becomes free.  ITER, "The loop that replaces the batch": finished
 * sequences are retired and their cache released.  Splits prepared before
 * this call become stale (their device calls return KV_E_STALE).
 * Errors: KV_E_SEQ_RANGE.
 */
int kv_seq_rm(kv_cache *c, int32_t seq, int32_t p0, int32_t p1);

/*
 * kv_seq_cp -- let sequence `dst` share the cells of sequence `src` with
 * p0 <= pos < p1 (p1 < 0: no upper bound): `dst` joins each such cell's
 * sequence set, so both sequences' rows see the same K/V rows, no data moves.
 * BATCH-ZH, Part E: a prompt shared by several sequences is one set of cells
 * whose sequence set holds them all; this gives that state to a prefix stored
 * for one sequence (the same cells as storing it with both ids).  Cells that
 * already hold `dst` are left alone; src == dst does nothing.  Splits prepared
 * before a call that changed a cell become stale (KV_E_STALE).
 * Errors: KV_E_SEQ_RANGE (either id outside 0 .. n_seq_max - 1),
 * KV_E_CROSS_STREAM (the two sequences live in different streams: sharing
 * would need the K/V rows copied into the other stream's cache).
 */
int kv_seq_cp(kv_cache *c, int32_t src, int32_t dst, int32_t p0, int32_t p1);

/* Largest position sequence `seq` holds in the cache, or -1. */
int32_t kv_seq_pos_max(const kv_cache *c, int32_t seq);

/*
 * kv_cells_read -- copy the host cell state of one stream (for checks):
 * pos_out[kv_size] (-1 = empty) and, if bits_out is not NULL,
 * bits_out[kv_size * ((n_seq_max + 63) / 64)] sequence bitsets (sequence q is
 * bit q % 64 of word q / 64).  KV_E_INVAL on a bad stream.
 */
int kv_cells_read(const kv_cache *c, int32_t stream, int32_t *pos_out, uint64_t *bits_out);

/* n_kv of one stream for the current cell state (UBATCH, n_kv section). */
int32_t kv_stream_n_kv(const kv_cache *c, int32_t stream);

/* ---- device side ---------------------------------------------------------- */

/*
 * kv_store -- scatter ubatch `ub`'s K and V rows into layer `layer`'s cache.
 * KV-MEM, "One row, one token's keys" and "The tensor's three dimensions":
 * row i goes to byte offset (stream*kv_size + cell) * n_head_kv*head_dim*2 of
 * the layer's K (V) tensor.
 *   k_cur, v_cur  device fp16 [n_tokens][n_head_kv*head_dim], ubatch row
 *                 order, 16-byte aligned rows
 *   stream        cudaStream_t
 * Errors: KV_E_INVAL (bad ub/layer/pointer), KV_E_ORDER (split not
 * prepared), KV_E_STALE, KV_E_NO_DEVICE, KV_E_CUDA (launch failure).
 */
int kv_store(kv_cache *c, const kv_split *s, int32_t ub, int32_t layer,
             const void *k_cur, const void *v_cur, void *stream);

/*
 * ubatch_attention -- attention of ubatch `ub` at layer `layer`.
 * UBATCH, "The mask is doing the work" (a cell is visible to row i iff it
 * is occupied, holds seq_id[i][0], and under causal attention its position is
 * <= pos_i; masked cells contribute nothing) and "Chunked prefill is the same
 * mechanism" ([U, C+U] scores).  The cell state seen is the one right after
 * this ubatch's cells were reserved: later ubatches of the same split are
 * not visible yet (BATCH-ZH, Part D).
 *   o[i][h][:] = sum_j softmax_j(q[i][h] . K[j][hk] / sqrt(head_dim) + M[i][j]) V[j][hk]
 *   with hk = h * n_head_kv / n_head; rows that see no cell get zeros.
 *   q         device fp16 [n_tokens][n_head][head_dim], ubatch row order
 *   o         device fp32 [n_tokens][n_head][head_dim]
 *   mask_out  NULL, or device fp16 bits [n_tokens][n_kv]: 0x0000 visible,
 *             0xFC00 (-inf) masked, column j = cell j of the row's stream
 * Requires kv_store(ub', layer) for every ub' <= ub of this split first
 * (KV_E_ORDER otherwise).  Errors: as kv_store.
 * The call runs the plan kernels (the tile lists and the work split of the
 * ubatch) unless the plan of (split, ub) is already on the device.  A layer-0
 * call of ubatch ub also starts the plan of ubatch ub + 1 of the same split on
 * a side stream of the cache, after everything issued on `stream` so far; the
 * first call of ub + 1 then makes `stream` wait for it.  Not while `stream` is
 * being captured into a CUDA graph.
 */
int ubatch_attention(kv_cache *c, const kv_split *s, int32_t ub, int32_t layer,
                     const void *q, float *o, void *mask_out, void *stream);

/*
 * ubatch_attention_static_scratch -- the same result as ubatch_attention for
 * a ubatch whose query blocks all take the decode path (the rows that share
 * a first sequence id number fewer than 64 * n_head_kv / n_head, as in a
 * decode iteration), computed without obtaining any device or host memory
 * during the call.  The pages have no counterpart of this call: it exists
 * for callers that cannot allocate while a step runs -- a server that has
 * handed all free device memory to its own pool at start-up, or a decode
 * loop that must not stall on the device-wide synchronisation cudaMalloc /
 * cudaFree may imply, or fail half-way on an out-of-memory.
 *
 * The split-K partial results and the per-block completion counters live in
 * one fixed array of KV_STATIC_SCRATCH_BYTES in the library's device image.
 * Needed: 256-byte-rounded (decode blocks x n_head_kv x 4) bytes of counters
 * plus (decode CTA columns + decode blocks) x n_head_kv x 8448 bytes of
 * partials, where decode CTA columns = 2 x SMs / n_head_kv; with 8 KV heads
 * on 152 SMs that is about 300 single-row sequences.
 *   Arguments, layout and ownership: as ubatch_attention.
 *   Errors: as ubatch_attention, and KV_E_INVAL (no work done) when a block
 *   of the ubatch takes the tensor-core prefill path, when the scratch would
 *   exceed KV_STATIC_SCRATCH_BYTES, when the current device is not the
 *   cache's, or when bringing the device tables up to date would need a
 *   larger upload buffer (call kv_store for this split first).
 * Every call on a device, for any cache, shares the one array: calls whose
 * device work overlaps in time (other streams, other threads) race on it and
 * give wrong results; order them on one stream.  Each call clears the
 * counters on its stream before its kernel; the array otherwise keeps the
 * last call's contents.  The array's device memory is taken when kv_init
 * creates a device cache (kv_init looks up its address on the current
 * device, which loads the library's device image there), so this call itself
 * obtains none; the 24 MiB stay held on that device until the process exits
 * and are not counted by kv_device_bytes.
 */
#define KV_STATIC_SCRATCH_BYTES (24u << 20)
int ubatch_attention_static_scratch(kv_cache *c, const kv_split *s, int32_t ub, int32_t layer,
                                    const void *q, float *o, void *mask_out, void *stream);

/* Device error codes (the first one a kernel reported since the word was last read). */
#define KV_DERR_TMA_TIMEOUT 1 /* a bounded wait for a TMA copy gave up */
#define KV_DERR_MMA_TIMEOUT 2 /* a bounded wait for a tensor-core commit gave up */
#define KV_DERR_BOUNDS      3 /* an index or layout check failed */
#define KV_DERR_TMEM        4 /* tensor memory allocation returned an unusable address */
#define KV_DERR_SELFTEST    5 /* kv_selftest_wait's wait gave up, as it must */

/*
 * kv_device_error -- synchronise the cache's device work and return the
 * device error word: 0 if no kernel reported a fault, else one of the
 * KV_DERR_* codes (a bounded wait gave up or an index check failed); clears it.
 */
int kv_device_error(kv_cache *c);

/*
 * kv_selftest_wait -- the failure path of the kernels' bounded waits, run on
 * purpose: launches one thread on the cache's device (on `stream`, a
 * cudaStream_t, NULL = the legacy default stream) that waits on a shared-memory
 * barrier nothing completes, with the same limit as every wait of the attention
 * kernels (2e9 SM cycles, about 1 s); when the wait gives up, the thread writes
 * KV_DERR_SELFTEST to the device error word and returns.  No memory is touched
 * but that word; the device stays usable.  Returns KV_OK once launched (the
 * word reads nonzero from kv_device_error after the kernel ends), KV_E_INVAL
 * for a host-only cache.  A fault-free stand-in for a copy or a commit that
 * never arrives.
 */
int kv_selftest_wait(kv_cache *c, void *stream);

/* Bytes of device memory the library allocated for this cache (cell mirror,
 * tables, plan, split-K scratch).  Not counted: the fixed
 * KV_STATIC_SCRATCH_BYTES array of ubatch_attention_static_scratch, held once
 * per device by the process from the first kv_init on that device. */
size_t kv_device_bytes(const kv_cache *c);

/* Number of CUDA kernels this cache has launched so far (all entry points). */
uint64_t kv_launch_count(const kv_cache *c);

/* ------------------------------------------------------------------------
 * Iteration-level (continuous) batching over one cache.  ITER, "The loop that
 * replaces the batch": before every pass the scheduler retires the finished
 * sequences (kv_seq_rm of all their cells), admits waiting requests first come,
 * first served while both budgets allow, and assembles the batch -- a newly
 * admitted sequence contributes its whole prompt (positions 0 .. L - 1), a
 * running one a single token (position L + generated - 1).  "The budget that
 * actually binds": the token budget counts positions per pass; the cache budget
 * is the page's conservative one, prompt + max_new cells reserved at admission
 * and released at retirement.  A request of N new tokens takes N passes.  A new
 * sequence takes the smallest sequence id not running.  Host only: the caller
 * runs each batch through kv_split_ubatches / kv_prepare_cells / kv_store /
 * ubatch_attention, then calls kv_sched_advance.  The cache must be unified
 * (n_stream 1) and used by this scheduler alone.
 * ------------------------------------------------------------------------ */
typedef struct kv_sched kv_sched;

typedef struct kv_sched_params {
    int32_t max_seqs;      /* sequences running at once: 1 .. n_seq_max */
    int32_t token_budget;  /* positions per pass: max_seqs .. n_batch (a pass is one batch) */
    int32_t fixed;         /* 1: admit only into an empty batch (a classical fixed batch) */
} kv_sched_params;

typedef struct kv_sched_batch {
    kv_batch batch;        /* this pass's tokens, one sequence id each: pass it to kv_split_ubatches */
    int32_t n_retired;     /* sequences retired before this pass, and their ids */
    const int32_t *retired;
} kv_sched_batch;          /* arrays owned by the scheduler, valid until its next kv_sched_next */

typedef struct kv_sched_info {
    int64_t passes;        /* passes advanced */
    int64_t useful;        /* tokens produced: the sequences of each advanced pass, summed */
    int32_t running;       /* sequences admitted and not retired */
    int32_t waiting;       /* requests not admitted yet */
    int32_t free_cells;    /* cells no running sequence has reserved */
} kv_sched_info;           /* duty cycle (ITER, "Two resources idled by a fixed batch"):
                              useful / (passes * max_seqs) */

/* Errors: KV_E_INVAL (bad parameters, n_stream != 1, max_seqs > n_seq_max,
 * token_budget > n_batch). */
int kv_sched_init(kv_cache *c, const kv_sched_params *p, kv_sched **out);
void kv_sched_free(kv_sched *s);

/* Queue a request of prompt_len prompt tokens and max_new new tokens; returns
 * its id (0, 1, ...), or KV_E_INVAL when it could never run (a prompt longer
 * than the token budget, prompt + max_new over the cache, a length < 1). */
int kv_sched_submit(kv_sched *s, int32_t prompt_len, int32_t max_new);

/* Retire, admit, assemble (see above).  out->batch.n_tokens == 0: nothing is
 * left to run.  Errors: KV_E_ORDER (the previous batch was not advanced). */
int kv_sched_next(kv_sched *s, kv_sched_batch *out);

/* The pass of the last batch ran: each of its sequences has one more token. */
int kv_sched_advance(kv_sched *s);

int kv_sched_stats(const kv_sched *s, kv_sched_info *out);

#ifdef __cplusplus
}
#endif

#endif /* KVATTN_H */
