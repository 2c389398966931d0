"""Float64 masked-softmax GQA attention over the cache, and the K/V scatter.

UBATCH, "The mask is doing the work" and "Chunked prefill is the same
mechanism": each query row is compared with the keys of every cell it may see,
the masked softmax weights the values, and masked cells contribute nothing.
ITER, "The budget that actually binds": with grouped-query attention several
query heads read one KV head.

Readings (not stated on the pages):
* softmax scale 1/sqrt(head_dim);
* query head h reads KV head floor(h * n_head_kv / n_head), i.e. contiguous
  groups of n_head / n_head_kv query heads per KV head;
* a row that sees no cell at all gets an output of zeros.

Layout of the oracle's cache (KV-MEM, "The tensor's three dimensions"): per
layer K and V arrays of shape [n_stream, kv_size, n_head_kv, head_dim], fp16,
which is the same byte order as the ggml tensor [n_embd_k_gqa, kv_size,
n_stream] (fastest dimension first).
"""

import numpy as np

from .mask import visible_row


def kv_store(k_cache, v_cache, streams, cells, k_cur, v_cur):
    """Write row i of k_cur / v_cur into cell cells[i] of stream streams[i].

    KV-MEM, "One row, one token's keys": one row of a layer's K tensor holds
    one token's keys for all KV heads side by side; V likewise.
    """
    for i, (s, j) in enumerate(zip(streams, cells)):
        k_cache[s, j] = k_cur[i]
        v_cache[s, j] = v_cur[i]


def attend_row(q_row, k_cache, v_cache, s, vis, n_head, n_head_kv):
    """Output [n_head, d] float64 for one query row given its visible cells."""
    d = q_row.shape[-1]
    scale = 1.0 / np.sqrt(d)
    group = n_head // n_head_kv
    out = np.zeros((n_head, d), dtype=np.float64)
    idx = np.flatnonzero(vis)
    if idx.size == 0:
        return out
    for h in range(n_head):
        hk = (h * n_head_kv) // n_head
        assert hk == h // group
        keys = k_cache[s, idx, hk, :].astype(np.float64)      # [m, d]
        vals = v_cache[s, idx, hk, :].astype(np.float64)      # [m, d]
        scores = (keys @ q_row[h].astype(np.float64)) * scale  # [m]
        w = np.exp(scores - scores.max())
        out[h] = (w @ vals) / w.sum()
    return out


def ubatch_attention(q, k_cache, v_cache, state, row_pos, row_seq0, row_stream,
                     n_kv, causal, n_head, n_head_kv, rows=None, n_swa=0):
    """o[i, h, :] for the ubatch rows (all rows, or the listed subset).

    ``state`` must be the cell state this ubatch sees (after its own cells were
    reserved and stored).  Returns float64 [len(rows), n_head, d].
    """
    if rows is None:
        rows = range(len(row_pos))
    rows = list(rows)
    d = q.shape[-1]
    out = np.zeros((len(rows), n_head, d), dtype=np.float64)
    for n, i in enumerate(rows):
        vis = visible_row(state, row_stream[i], row_seq0[i], row_pos[i], n_kv, causal, n_swa)
        out[n] = attend_row(q[i], k_cache, v_cache, row_stream[i], vis, n_head, n_head_kv)
    return out


def attend_row_loops(q_row, keys, vals, n_head, n_head_kv):
    """Pure-Python loops over one row's visible keys (tiny cases only).

    ``keys``/``vals``: lists of [n_head_kv][d] float lists for the visible
    cells.  Returns [n_head][d] floats.
    """
    import math
    d = len(q_row[0])
    scale = 1.0 / math.sqrt(d)
    out = []
    for h in range(n_head):
        hk = (h * n_head_kv) // n_head
        if not keys:
            out.append([0.0] * d)
            continue
        scores = []
        for k in keys:
            acc = 0.0
            for t in range(d):
                acc += float(q_row[h][t]) * float(k[hk][t])
            scores.append(acc * scale)
        m = max(scores)
        w = [math.exp(x - m) for x in scores]
        z = sum(w)
        row = []
        for t in range(d):
            acc = 0.0
            for wj, v in zip(w, vals):
                acc += wj * float(v[hk][t])
            row.append(acc / z)
        out.append(row)
    return out
