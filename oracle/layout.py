"""Cache sizes, strides, byte offsets and the fixed-batch duty cycle.

KV-MEM: a layer's K tensor is [values per token, cells per stream, streams]
in fastest-first order; with F16 each value takes 2 bytes.  ITER gives the
same per-token arithmetic for a 32-layer model and the duty cycle of a
fixed batch.
"""

F16_BYTES = 2


def row_values(n_head_kv, head_dim):
    """Values in one K (or V) row: KV-MEM, "One row, one token's keys"."""
    return n_head_kv * head_dim


def row_bytes(n_head_kv, head_dim, elt=F16_BYTES):
    return row_values(n_head_kv, head_dim) * elt


def bytes_per_token(n_layer, n_head_kv, head_dim, elt=F16_BYTES):
    """K and V bytes one token holds over all layers (KV-MEM, ITER)."""
    return row_bytes(n_head_kv, head_dim, elt) * n_layer * 2


def cache_bytes(n_cells, n_layer, n_head_kv, head_dim, elt=F16_BYTES):
    """Whole reserved cache: every cell, every layer, K and V (KV-MEM,
    "llama.cpp reserves space for the configured capacity")."""
    return n_cells * bytes_per_token(n_layer, n_head_kv, head_dim, elt)


def strides(n_head_kv, head_dim, kv_size, elt=F16_BYTES):
    """ggml byte strides nb[0..2] of a layer's K tensor (KV-MEM, "The
    tensor's three dimensions"): value, row (cell), stream slab."""
    nb0 = elt
    nb1 = nb0 * row_values(n_head_kv, head_dim)
    nb2 = nb1 * kv_size
    return nb0, nb1, nb2


def shape(n_head_kv, head_dim, n_ctx, n_stream):
    """ne[0..2] of a layer's K tensor: the total capacity n_ctx split evenly
    over the streams (KV-MEM, "Unified versus non-unified")."""
    return row_values(n_head_kv, head_dim), n_ctx // n_stream, n_stream


def byte_offset(stream, cell, head, elem, n_head_kv, head_dim, kv_size, elt=F16_BYTES):
    """Offset of one value from the start of its layer's K tensor (KV-MEM,
    "The tensor's three dimensions": cell row, then head, then element)."""
    nb0, nb1, nb2 = strides(n_head_kv, head_dim, kv_size, elt)
    return stream * nb2 + cell * nb1 + (head * head_dim + elem) * nb0


def duty_cycle(lengths):
    """Useful positions over executed positions of a fixed batch.

    ITER, "Two resources idled by a fixed batch": the batch runs for the
    longest member's length, every member occupying a row throughout, so the
    useful fraction is sum(lengths) / (count * max(lengths)).  Returned as the
    exact pair (useful, executed).
    """
    return sum(lengths), len(lengths) * max(lengths)
