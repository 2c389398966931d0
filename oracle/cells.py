"""Per-stream cell state, the first-fit slot finder and n_kv.

KV-MEM, "The tensor's three dimensions" and "Unified versus non-unified": the
cache has n_stream streams of kv_size cells; a cell is one row index shared by
every layer's K and V tensors.  A cell is empty or holds one position and a
set of sequences (UBATCH, "Three things called batch": one token can belong to
several sequences, which is how a shared prefix lives in the cache once).

State per stream s and cell j:
* ``pos[s, j]``   the cell's position (-1 when empty);
* ``nseq[s, j]``  how many sequences the cell belongs to (0 = empty);
* ``bits[s, j, w]`` a plain bitset of those sequences: sequence q is bit
  q % 64 of word q // 64.

Pins: the n_kv examples (700 cells used -> 768; the kv_size clamp), first-fit
on an empty cache giving cells 0..n-1, the all-or-nothing failure (state
unchanged, return 1) and the prefix-sharing example of BATCH-ZH, Part E.  The
slot-finder policy beyond that (first fit from cell 0, cells not necessarily
contiguous, rows in ubatch order) is not stated by the pages: parity
unpinned for that policy.
"""

import numpy as np

NO_SLOT = 1  # the decode call's "no KV slot" return (BATCH-ZH, Part F)

# UBATCH, n_kv section: the quantum is max(model pad, 256) and the model pad is
# 1 on the paths the page looked at, so 256 always wins.
MODEL_N_PAD = 1
N_PAD_FLOOR = 256


def pad_up(x, n):
    """Round x up to a multiple of n (the GGML_PAD of UBATCH, n_kv section)."""
    return ((x + n - 1) // n) * n


class CellState:
    def __init__(self, n_stream, kv_size, n_seq_max, seq_to_stream=None):
        self.n_stream = n_stream
        self.kv_size = kv_size
        self.n_seq_max = n_seq_max
        self.n_words = (n_seq_max + 63) // 64
        if seq_to_stream is None:
            # Reading: with more sequences than streams, sequence q lives in
            # stream q mod n_stream unless the caller gives a map.
            seq_to_stream = [q % n_stream for q in range(n_seq_max)]
        self.seq_to_stream = [int(x) for x in seq_to_stream]
        self.pos = np.full((n_stream, kv_size), -1, dtype=np.int64)
        self.nseq = np.zeros((n_stream, kv_size), dtype=np.int32)
        self.bits = np.zeros((n_stream, kv_size, self.n_words), dtype=np.uint64)

    def copy(self):
        c = CellState.__new__(CellState)
        c.n_stream, c.kv_size, c.n_seq_max = self.n_stream, self.kv_size, self.n_seq_max
        c.n_words = self.n_words
        c.seq_to_stream = list(self.seq_to_stream)
        c.pos = self.pos.copy()
        c.nseq = self.nseq.copy()
        c.bits = self.bits.copy()
        return c

    def same_as(self, other):
        return (np.array_equal(self.pos, other.pos)
                and np.array_equal(self.nseq, other.nseq)
                and np.array_equal(self.bits, other.bits))

    # -- the queries named in UBATCH, "The mask is doing the work" ------------
    def is_empty(self, s, j):
        return self.nseq[s, j] == 0

    def seq_has(self, s, j, q):
        return bool((int(self.bits[s, j, q // 64]) >> (q % 64)) & 1)

    def pos_get(self, s, j):
        return int(self.pos[s, j])

    def seqs_of(self, s, j):
        return [q for q in range(self.n_seq_max) if self.seq_has(s, j, q)]

    # -- vectorised forms of the same queries ----------------------------------------
    def empty_mask(self, s):
        return self.nseq[s] == 0

    def has_seq_mask(self, s, q):
        word = self.bits[s, :, q // 64]
        return ((word >> np.uint64(q % 64)) & np.uint64(1)).astype(bool)

    def used_max_p1(self, s):
        """1 + index of the highest non-empty cell of stream s, or 0."""
        occupied = np.flatnonzero(self.nseq[s] != 0)
        return 0 if occupied.size == 0 else int(occupied[-1]) + 1

    def seq_pos_max(self, q):
        """Largest position held by sequence q in the cache, or -1."""
        s = self.seq_to_stream[q]
        held = self.has_seq_mask(s, q)
        return int(self.pos[s][held].max()) if held.any() else -1

    def n_used(self, s):
        return int((self.nseq[s] != 0).sum())

    # -- writes ------------------------------------------------------------------
    def fill(self, s, j, p, seqs):
        self.pos[s, j] = p
        self.bits[s, j, :] = 0
        for q in seqs:
            self.bits[s, j, q // 64] |= np.uint64(1) << np.uint64(q % 64)
        self.nseq[s, j] = len(seqs)

    # -- n_kv ------------------------------------------------------------------
    def n_kv_stream(self, s):
        """Padded attention width of stream s.

        UBATCH, "Prefill and decode are not the same shape": n_kv is the
        highest occupied cell + 1 rounded up to the quantum, at least one
        quantum, and at most the stream's cell count.  With a quantum of 256,
        700 live cells are reported as 768.
        """
        quantum = max(MODEL_N_PAD, N_PAD_FLOOR)
        padded = max(quantum, pad_up(self.used_max_p1(s), quantum))
        return min(self.kv_size, padded)

    # -- removal (retire a sequence) ----------------------------------------------
    def seq_rm(self, q, p0, p1):
        """Drop sequence q (every sequence when q < 0) from cells with p0 <= pos < p1.

        ITER, "The loop that replaces the batch": finished sequences are retired
        and their cache released.  p1 < 0 means no upper bound.  A cell left
        with no sequence becomes empty.
        """
        hi = np.iinfo(np.int64).max if p1 < 0 else p1
        for s in range(self.n_stream):
            if q >= 0 and self.seq_to_stream[q] != s:
                continue
            for j in range(self.kv_size):
                if self.nseq[s, j] == 0:
                    continue
                if not (p0 <= self.pos[s, j] < hi):
                    continue
                if q < 0:
                    self.fill(s, j, -1, [])
                elif self.seq_has(s, j, q):
                    keep = [x for x in self.seqs_of(s, j) if x != q]
                    self.fill(s, j, self.pos[s, j] if keep else -1, keep)


    def seq_cp(self, src, dst, p0, p1):
        """Let sequence dst share src's cells with p0 <= pos < p1; returns 0, or
        "cross-stream" when the two sequences live in different streams.

        BATCH-ZH, Part E: a prompt shared by several sequences is one set of
        cells whose sequence set holds them all.  Reading (the pages give no copy
        call): copying src to dst adds dst to the set of each cell of src in the
        range, which is the state that storing those tokens with both ids gives.
        Nothing else changes; p1 < 0 means no upper bound.
        """
        s = self.seq_to_stream[src]
        if self.seq_to_stream[dst] != s:
            return "cross-stream"
        hi = np.iinfo(np.int64).max if p1 < 0 else p1
        for j in range(self.kv_size):
            if self.nseq[s, j] == 0 or not (p0 <= self.pos[s, j] < hi):
                continue
            if self.seq_has(s, j, src) and not self.seq_has(s, j, dst):
                self.fill(s, j, self.pos[s, j], self.seqs_of(s, j) + [dst])
        return 0

def prepare(state, ubatches, pos_list, seq_lists, keep_snapshots=True):
    """Reserve a cell for every row of every ubatch, all or nothing.

    BATCH-ZH, Part C ("策略选择": reserve slots for each ubatch) and Part F
    (a full cache makes the decode call return 1).  Reading of the slot
    policy, which the pages leave open: ubatches in order, rows in ubatch
    order; each row takes the lowest-index empty cell of the stream of its
    first sequence, and that cell gets the row's position and its whole
    sequence set.  If any row finds no empty cell the state is left exactly as
    it was and NO_SLOT is returned.

    Returns (code, cells, n_kv, snapshots): cells[k][i] is the stream-local
    cell of row i of ubatch k, n_kv[k] the attention width after ubatch k,
    and snapshots[k] the cell state right after ubatch k -- what the mask of
    ubatch k sees, since later ubatches of the same batch have not run yet
    (BATCH-ZH, Part D).  snapshots is None unless keep_snapshots.
    """
    work = state.copy()
    all_cells, all_nkv, snaps = [], [], []
    for ub in ubatches:
        rows = ub["rows"]
        streams = [work.seq_to_stream[seq_lists[r][0]] for r in rows]
        # First fit, row by row.  Within one ubatch cells only get filled, so
        # the k-th row that lands in a stream takes that stream's k-th lowest
        # empty cell.
        free = {s: np.flatnonzero(work.empty_mask(s)) for s in set(streams)}
        taken = {s: 0 for s in free}
        cells = []
        for r, s in zip(rows, streams):
            if taken[s] >= len(free[s]):
                return NO_SLOT, None, None, None
            j = int(free[s][taken[s]])
            taken[s] += 1
            work.fill(s, j, pos_list[r], seq_lists[r])
            cells.append(j)
        all_cells.append(cells)
        all_nkv.append(max(work.n_kv_stream(s) for s in set(streams)))
        if keep_snapshots:
            snaps.append(work.copy())
    state.pos, state.nseq, state.bits = work.pos, work.nseq, work.bits
    return 0, all_cells, all_nkv, (snaps if keep_snapshots else None)


def stream_of_rows(state, ub, seq_lists):
    return [state.seq_to_stream[seq_lists[r][0]] for r in ub["rows"]]
