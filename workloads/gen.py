"""Seeded fp16 rows.

Every value is N(0, 1) drawn with ``numpy.random.default_rng`` and cast to
fp16.  A row is addressed by (config id, layer, content sequence, kind, pos),
kind 0 = Q, 1 = K, 2 = V.  Rows are generated in blocks of BLOCK positions,
each block from its own seed tuple, so identical (content, pos) always gives
identical bytes (a sequence that duplicates another's tokens duplicates its
K/V exactly) and a long sequence never needs its earlier rows regenerated.
"""

import numpy as np

BLOCK = 256
KIND_Q, KIND_K, KIND_V = 0, 1, 2


def _block(cfg, layer, content, kind, blk, width):
    rng = np.random.default_rng([int(cfg), int(layer), int(content), int(kind), int(blk)])
    return rng.standard_normal((BLOCK, width), dtype=np.float32).astype(np.float16)


def rows(cfg, layer, content, kind, pos, width):
    """fp16 [len(pos), width]: row n is the value row of (content, pos[n])."""
    pos = np.asarray(pos, dtype=np.int64)
    content = np.broadcast_to(np.asarray(content, dtype=np.int64), pos.shape)
    out = np.empty((pos.size, width), dtype=np.float16)
    cache = {}
    for n in range(pos.size):
        key = (int(content[n]), int(pos[n]) // BLOCK)
        blk = cache.get(key)
        if blk is None:
            blk = _block(cfg, layer, key[0], kind, key[1], width)
            cache[key] = blk
        out[n] = blk[int(pos[n]) % BLOCK]
    return out


def rows_fast(cfg, layer, content, kind, p0, n, width):
    """Rows for positions p0 .. p0+n-1 of one content sequence (contiguous)."""
    out = np.empty((n, width), dtype=np.float16)
    p = p0
    while p < p0 + n:
        blk = p // BLOCK
        lo = p % BLOCK
        take = min(BLOCK - lo, p0 + n - p)
        out[p - p0:p - p0 + take] = _block(cfg, layer, content, kind, blk, width)[lo:lo + take]
        p += take
    return out


def batch_rows(cfg, layer, kind, pos, content, width):
    """Rows for a list of (pos, content) pairs, grouping contiguous runs."""
    pos = np.asarray(pos, dtype=np.int64)
    content = np.asarray(content, dtype=np.int64)
    out = np.empty((pos.size, width), dtype=np.float16)
    i = 0
    n = pos.size
    while i < n:
        j = i + 1
        while j < n and content[j] == content[i] and pos[j] == pos[j - 1] + 1:
            j += 1
        out[i:j] = rows_fast(cfg, layer, int(content[i]), kind, int(pos[i]), j - i, width)
        i = j
    return out


def uniform_f16(seed, shape, lo=-1.0, hi=1.0):
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=shape).astype(np.float16)
