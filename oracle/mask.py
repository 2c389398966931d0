"""The KQ mask of one ubatch.

UBATCH, "The mask is doing the work": a query sees a key only if the key's
cell is occupied, belongs to the query's sequence, and (under causal
attention) does not hold a later position; every other entry is negative
infinity before the softmax.  The query's sequence is its first id,
seq_id[i][0], while a cell holding several sequences is visible to each of
them.  The same passage lists a sliding-window term ("outside the sliding
window") without defining it; the reading taken: with a window of n_swa
positions, a cell is outside the window of a row at position p when
p - pos_j >= n_swa (the row sees its last n_swa positions, itself included;
later cells are not affected); n_swa = 0 means no window.

Encoding (a reading; the pages give only "negative infinity"): an additive
F16 mask, +0.0 (bit pattern 0x0000) where visible and -inf (0xFC00) where
masked, laid out [n_tokens, n_kv] row-major, column j being cell j of the
row's own stream.
"""

import numpy as np

F16_ZERO = 0x0000
F16_NEG_INF = 0xFC00


def visible(state, s, j, q, p, causal, n_swa=0):
    """The per-pair rule, written out once, in the order the page lists it."""
    if state.is_empty(s, j):
        return False
    if not state.seq_has(s, j, q):
        return False
    if causal and state.pos_get(s, j) > p:
        return False
    if n_swa > 0 and p - state.pos_get(s, j) >= n_swa:
        return False
    return True


def visible_row(state, s, q, p, n_kv, causal, n_swa=0):
    """Vector form of ``visible`` over cells 0..n_kv-1 of stream s."""
    ok = ~state.empty_mask(s)[:n_kv]
    ok &= state.has_seq_mask(s, q)[:n_kv]
    if causal:
        ok &= state.pos[s, :n_kv] <= p
    if n_swa > 0:
        ok &= p - state.pos[s, :n_kv].astype(np.int64) < n_swa
    return ok


def kq_mask(state, row_pos, row_seq0, row_stream, n_kv, causal, n_swa=0):
    """F16 bit patterns (uint16) of the mask, shape [n_tokens, n_kv]."""
    n = len(row_pos)
    out = np.full((n, n_kv), F16_NEG_INF, dtype=np.uint16)
    for i in range(n):
        ok = visible_row(state, row_stream[i], row_seq0[i], row_pos[i], n_kv, causal, n_swa)
        out[i, ok] = F16_ZERO
    return out


def kq_mask_bruteforce(state, row_pos, row_seq0, row_stream, n_kv, causal, n_swa=0):
    """Same mask, one pair at a time (for small cases)."""
    n = len(row_pos)
    out = np.full((n, n_kv), F16_NEG_INF, dtype=np.uint16)
    for i in range(n):
        for j in range(n_kv):
            if visible(state, row_stream[i], j, row_seq0[i], row_pos[i], causal, n_swa):
                out[i, j] = F16_ZERO
    return out
