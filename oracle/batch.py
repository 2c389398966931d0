"""Batch validation, auto-fill and the three ubatch splitters.

A batch is a list of token slots (UBATCH, "Three things called batch";
BATCH-ZH, Part A): each slot has a position and a list of sequence ids.  The
oracle represents it as two Python lists ``pos`` (or None) and ``seq_ids``
(list of lists, or None).

A ubatch (BATCH-ZH, Part B) is represented as a dict with

* ``rows``          indices into the batch, in ubatch row order,
* ``n_tokens``      len(rows) == n_seq_tokens * n_seqs,
* ``n_seq_tokens``  tokens taken from each sequence set,
* ``n_seqs``        number of sequence sets,
* ``seq_id_unq``    sorted distinct sequence ids of the ubatch.

Error codes mirror the C interface: 0 ok, negative = error.

Pins: the page's worked splits (5000 tokens at n_batch 2048 give calls of
2048/2048/904 and 10 ubatches; 1000 tokens give 512 + 488, 1500 give
512/512/476), the clamps, and brute-forced invariants on every small batch
(each row once, per-sequence order kept, rectangular ubatches, disjoint
sequence sets).  split_equal's choice among overlapping sequence sets and its
"sequential" order, and split_seq's exact rows, follow a written reading of
the pages that nothing on them fixes further: parity unpinned for those
tie-breaks (the library must match this reading bit for bit, but no page
value confirms the reading itself).
"""

E_INVAL = -1
E_BATCH_TOO_LARGE = -2
E_SEQ_RANGE = -3
E_CROSS_STREAM = -4


def caller_chunks(n_tokens, n_batch):
    """Sizes of the decode calls a caller makes for a long input.

    UBATCH, "Three things called batch": a call may hold at most n_batch slots
    (the engine asserts it), so a 5000-token prompt at n_batch 2048 is handed
    over as calls of 2048, 2048 and 904.
    """
    out = []
    left = n_tokens
    while left > 0:
        take = min(n_batch, left)
        out.append(take)
        left -= take
    return out


def validate_and_fill(n_tokens, pos, n_seq_id, seq_id, n_batch, n_seq_max,
                      seq_to_stream, cell_state):
    """Validate a batch and fill the fields the caller left out.

    BATCH-ZH, Part A (field table) and Part F (step 1 of the decode loop): the
    allocator validates the batch and fills missing pos / seq_id.  UBATCH,
    "Three things called batch": more than n_batch slots is refused.

    Readings where the pages are silent:
    * seq_id None -> every row belongs to sequence 0; n_seq_id None with
      seq_id given -> each row has the single sequence seq_id[i][0];
    * pos None -> row i gets 1 + the largest position already held by its
      sequence seq_id[i][0], over the cache and the earlier rows of this batch
      that belong to that sequence, or 0 when there is none;
    * a row's ids must be distinct, in [0, n_seq_max), and map to one cache
      stream (KV-MEM, "Unified versus non-unified": a stream is one partition,
      so a shared cell cannot span two).

    Checks run row by row in this order: n_tokens, then for each row the
    n_seq_id count, the id range, duplicates, the stream, the position.

    Returns (err, pos_list, seq_sets) where seq_sets[i] is the row's ids with
    the first id kept first (masking uses seq_id[i][0]).
    """
    if n_tokens < 1:
        return E_INVAL, None, None
    if n_tokens > n_batch:
        return E_BATCH_TOO_LARGE, None, None

    seq_lists = []
    for i in range(n_tokens):
        if seq_id is None:
            ids = [0]
        elif n_seq_id is None:
            ids = [int(seq_id[i][0])]
        else:
            k = int(n_seq_id[i])
            if k < 1 or k > n_seq_max:
                return E_INVAL, None, None
            ids = [int(x) for x in seq_id[i][:k]]
        for s in ids:
            if s < 0 or s >= n_seq_max:
                return E_SEQ_RANGE, None, None
        if len(set(ids)) != len(ids):
            return E_INVAL, None, None
        streams = {seq_to_stream[s] for s in ids}
        if len(streams) != 1:
            return E_CROSS_STREAM, None, None
        if pos is not None and int(pos[i]) < 0:
            return E_INVAL, None, None
        seq_lists.append(ids)

    if pos is not None:
        pos_list = [int(p) for p in pos[:n_tokens]]
    else:
        pos_list = []
        for i in range(n_tokens):
            s = seq_lists[i][0]
            best = cell_state.seq_pos_max(s)
            for k in range(i):
                if s in seq_lists[k] and pos_list[k] > best:
                    best = pos_list[k]
            pos_list.append(best + 1)
    return 0, pos_list, seq_lists


def _ubatch(rows, n_seq_tokens, n_seqs, seq_lists):
    unq = sorted({s for r in rows for s in seq_lists[r]})
    return {
        "rows": list(rows),
        "n_tokens": len(rows),
        "n_seq_tokens": n_seq_tokens,
        "n_seqs": n_seqs,
        "seq_id_unq": unq,
    }


def split_simple(used, n_ubatch, seq_lists):
    """Next ubatch of split_simple, or None when every row is used.

    UBATCH, "Part 1": slots are taken in submission order up to n_ubatch, with
    no regard to sequence ids.  BATCH-ZH, Part C (1): 1000 tokens at 512 give
    512 + 488.  Reading: each row counts as its own sequence set, so
    n_seq_tokens = 1 and n_seqs = n_tokens (BATCH-ZH, Part B:
    n_tokens = n_seq_tokens * n_seqs).
    """
    rows = []
    for r in range(len(used)):
        if len(rows) == n_ubatch:
            break
        if not used[r]:
            rows.append(r)
    if not rows:
        return None
    for r in rows:
        used[r] = True
    return _ubatch(rows, 1, len(rows), seq_lists)


def split_equal(used, n_ubatch, seq_lists):
    """Next ubatch of split_equal(n_ubatch, sequential=true), or None.

    BATCH-ZH, Part C (2): choose non-overlapping sequence sets, then take the
    same number of tokens from each set until the total nears n_ubatch or a set
    runs out.  UBATCH, "Part 1": equal-length chunks with ordered sequence ids.

    Reading, step by step:
    1. a row's set is the (unordered) set of its ids; walk the unused rows in
       submission order and collect each new set unless it shares an id with a
       set already collected (identical sets are one set); stop at n_ubatch sets;
    2. order the collected sets by their smallest id ("ordered sequence ids");
    3. n_seq_tokens = min(fewest unused rows over the sets, n_ubatch // n_sets);
    4. the ubatch is set-major: for each set in that order, its first
       n_seq_tokens unused rows in submission order.
    The exact tie-breaks are this reading's, not the pages' (parity pinned by
    the written rule and by invariants only).
    """
    chosen = []
    for r in range(len(used)):
        if used[r]:
            continue
        s = frozenset(seq_lists[r])
        if s in chosen:
            continue
        if any(s & c for c in chosen):
            continue
        if len(chosen) == n_ubatch:
            break
        chosen.append(s)
    if not chosen:
        return None
    chosen.sort(key=min)
    rows_of = []
    for c in chosen:
        rows_of.append([r for r in range(len(used))
                        if not used[r] and frozenset(seq_lists[r]) == c])
    n_seqs = len(chosen)
    n_seq_tokens = min(min(len(x) for x in rows_of), n_ubatch // n_seqs)
    rows = []
    for x in rows_of:
        rows.extend(x[:n_seq_tokens])
    for r in rows:
        used[r] = True
    return _ubatch(rows, n_seq_tokens, n_seqs, seq_lists)


def split_seq(used, n_ubatch, seq_lists):
    """Next ubatch of split_seq, or None.

    BATCH-ZH, Part C (3): every ubatch holds the tokens of a single sequence
    set.  Reading: the set of the first unused row, then up to n_ubatch unused
    rows with exactly that set, in submission order; n_seqs = 1.
    """
    first = None
    for r in range(len(used)):
        if not used[r]:
            first = r
            break
    if first is None:
        return None
    s = frozenset(seq_lists[first])
    rows = [r for r in range(len(used))
            if not used[r] and frozenset(seq_lists[r]) == s][:n_ubatch]
    for r in rows:
        used[r] = True
    return _ubatch(rows, len(rows), 1, seq_lists)


SPLIT_AUTO, SPLIT_SIMPLE, SPLIT_EQUAL, SPLIT_SEQ = 0, 1, 2, 3


def init_batch(n_tokens, seq_lists, n_ubatch, n_stream, mode=SPLIT_AUTO):
    """All ubatches of one batch, in order.

    BATCH-ZH, Part C, "策略选择": the cache resets the splitter, then loops
    split_simple when there is one stream and split_equal(n_ubatch, true)
    otherwise, until a split returns no tokens.  ``mode`` forces one splitter
    (split_seq is reachable only this way; the pages use it on other paths).
    """
    if mode == SPLIT_AUTO:
        mode = SPLIT_SIMPLE if n_stream == 1 else SPLIT_EQUAL
    fn = {SPLIT_SIMPLE: split_simple, SPLIT_EQUAL: split_equal,
          SPLIT_SEQ: split_seq}[mode]
    used = [False] * n_tokens
    out = []
    while True:
        ub = fn(used, n_ubatch, seq_lists)
        if ub is None:
            break
        out.append(ub)
    return out
