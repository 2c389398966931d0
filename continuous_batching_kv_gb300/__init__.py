"""Python binding of libkvattn: ubatch attention over a cell-indexed KV cache.

Argument marshalling only.  Every step of the path runs in the native library
(host C++ for splitting and cell reservation, CUDA kernels for the K/V
scatter, the mask and attention); this module converts Python lists, numpy
arrays and torch tensors to the C interface declared in include/kvattn.h and
raises ``KvError`` for negative return codes.  There is no fallback: if the
library is missing, importing this package fails.

The functions keep the C names:

    kv_init, kv_free, kv_n_batch, kv_n_ubatch, kv_kv_size, kv_last_error,
    kv_split_ubatches, kv_split_count, kv_split_ubatch, kv_split_free,
    kv_prepare_cells, kv_seq_rm, kv_seq_cp, kv_seq_pos_max, kv_cells_read,
    kv_stream_n_kv, kv_store, ubatch_attention, ubatch_attention_static_scratch,
    kv_device_error, kv_selftest_wait, kv_device_bytes, kv_launch_count,
    kv_sched_init, kv_sched_free, kv_sched_submit, kv_sched_next, kv_sched_advance, kv_sched_stats
    (and kv_split_sched_batch: kv_split_ubatches of a scheduler batch)
"""

import ctypes as C
import itertools
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvattn.so")

KV_OK, KV_NO_SLOT = 0, 1
KV_E_INVAL, KV_E_BATCH_TOO_LARGE, KV_E_SEQ_RANGE, KV_E_CROSS_STREAM = -1, -2, -3, -4
KV_E_ORDER, KV_E_STALE, KV_E_CUDA, KV_E_NOMEM, KV_E_NO_DEVICE = -5, -6, -7, -8, -9
KV_SPLIT_AUTO, KV_SPLIT_SIMPLE, KV_SPLIT_EQUAL, KV_SPLIT_SEQ = 0, 1, 2, 3
KV_MAX_SEQ, KV_HEAD_DIM = 256, 128
KV_STATIC_SCRATCH_BYTES = 24 << 20
KV_DERR_TMA_TIMEOUT, KV_DERR_MMA_TIMEOUT, KV_DERR_BOUNDS, KV_DERR_TMEM, KV_DERR_SELFTEST = 1, 2, 3, 4, 5

EXPORTS = [
    "kv_init", "kv_free", "kv_n_batch", "kv_n_ubatch", "kv_kv_size", "kv_last_error",
    "kv_split_ubatches", "kv_split_count", "kv_split_ubatch", "kv_split_free",
    "kv_prepare_cells", "kv_seq_rm", "kv_seq_cp", "kv_seq_pos_max", "kv_cells_read", "kv_stream_n_kv",
    "kv_store", "ubatch_attention", "ubatch_attention_static_scratch", "kv_device_error",
    "kv_selftest_wait", "kv_device_bytes", "kv_launch_count",
    "kv_sched_init", "kv_sched_free", "kv_sched_submit", "kv_sched_next", "kv_sched_advance",
    "kv_sched_stats",
]


class KvError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("kvattn error %d: %s" % (code, msg))
        self.code = code


class kv_params(C.Structure):
    _fields_ = [("n_ctx", C.c_int32), ("n_batch", C.c_int32), ("n_ubatch", C.c_int32),
                ("n_seq_max", C.c_int32), ("n_stream", C.c_int32), ("n_layer", C.c_int32),
                ("n_head", C.c_int32), ("n_head_kv", C.c_int32), ("head_dim", C.c_int32),
                ("causal", C.c_int32), ("n_swa", C.c_int32), ("seq_to_stream", C.POINTER(C.c_int32)),
                ("k_layers", C.POINTER(C.c_void_p)), ("v_layers", C.POINTER(C.c_void_p))]


class kv_batch(C.Structure):
    _fields_ = [("n_tokens", C.c_int32), ("pos", C.POINTER(C.c_int32)),
                ("n_seq_id", C.POINTER(C.c_int32)),
                ("seq_id", C.POINTER(C.POINTER(C.c_int32)))]


class kv_ubatch_info(C.Structure):
    _fields_ = [("n_tokens", C.c_int32), ("n_seq_tokens", C.c_int32), ("n_seqs", C.c_int32),
                ("n_seqs_unq", C.c_int32), ("n_kv", C.c_int32),
                ("rows", C.POINTER(C.c_int32)), ("pos", C.POINTER(C.c_int32)),
                ("seq0", C.POINTER(C.c_int32)), ("seq_id_unq", C.POINTER(C.c_int32)),
                ("streams", C.POINTER(C.c_int32)), ("cells", C.POINTER(C.c_int32))]


class kv_sched_params(C.Structure):
    _fields_ = [("max_seqs", C.c_int32), ("token_budget", C.c_int32), ("fixed", C.c_int32)]


class kv_sched_batch(C.Structure):
    _fields_ = [("batch", kv_batch), ("n_retired", C.c_int32), ("retired", C.POINTER(C.c_int32))]


class kv_sched_info(C.Structure):
    _fields_ = [("passes", C.c_int64), ("useful", C.c_int64), ("running", C.c_int32),
                ("waiting", C.c_int32), ("free_cells", C.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libkvattn.so is not built; run "
                          "`python continuous_batching_kv_gb300/build.py` (needs nvcc)")
    lib = C.CDLL(LIB_PATH)
    P = C.c_void_p
    sig = {
        "kv_init": (C.c_int, [C.POINTER(kv_params), C.POINTER(P)]),
        "kv_free": (None, [P]),
        "kv_n_batch": (C.c_int32, [P]),
        "kv_n_ubatch": (C.c_int32, [P]),
        "kv_kv_size": (C.c_int32, [P]),
        "kv_last_error": (C.c_char_p, [P]),
        "kv_split_ubatches": (C.c_int, [P, C.POINTER(kv_batch), C.c_int32, C.POINTER(P)]),
        "kv_split_count": (C.c_int32, [P]),
        "kv_split_ubatch": (C.c_int, [P, C.c_int32, C.POINTER(kv_ubatch_info)]),
        "kv_split_free": (None, [P]),
        "kv_prepare_cells": (C.c_int, [P, P]),
        "kv_seq_rm": (C.c_int, [P, C.c_int32, C.c_int32, C.c_int32]),
        "kv_seq_cp": (C.c_int, [P, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
        "kv_seq_pos_max": (C.c_int32, [P, C.c_int32]),
        "kv_cells_read": (C.c_int, [P, C.c_int32, C.POINTER(C.c_int32), C.POINTER(C.c_uint64)]),
        "kv_stream_n_kv": (C.c_int32, [P, C.c_int32]),
        "kv_store": (C.c_int, [P, P, C.c_int32, C.c_int32, P, P, P]),
        "ubatch_attention": (C.c_int, [P, P, C.c_int32, C.c_int32, P, P, P, P]),
        "ubatch_attention_static_scratch": (C.c_int, [P, P, C.c_int32, C.c_int32, P, P, P, P]),
        "kv_device_error": (C.c_int, [P]),
        "kv_selftest_wait": (C.c_int, [P, P]),
        "kv_device_bytes": (C.c_size_t, [P]),
        "kv_launch_count": (C.c_uint64, [P]),
        "kv_sched_init": (C.c_int, [P, C.POINTER(kv_sched_params), C.POINTER(P)]),
        "kv_sched_free": (None, [P]),
        "kv_sched_submit": (C.c_int, [P, C.c_int32, C.c_int32]),
        "kv_sched_next": (C.c_int, [P, C.POINTER(kv_sched_batch)]),
        "kv_sched_advance": (C.c_int, [P]),
        "kv_sched_stats": (C.c_int, [P, C.POINTER(kv_sched_info)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def _ptr(x):
    """Device (or host) address of a torch tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(c, rc):
    if rc < 0:
        msg = lib.kv_last_error(c).decode() if c else ""
        raise KvError(rc, msg)
    return rc


class Cache:
    """Handle returned by kv_init (keeps the marshalled arrays alive)."""

    def __init__(self, ptr, keep):
        self.ptr = ptr
        self._keep = keep

    @property
    def _as_parameter_(self):
        return self.ptr


class Split:
    """Handle returned by kv_split_ubatches."""

    def __init__(self, ptr, cache):
        self.ptr = ptr
        self.cache = cache

    @property
    def _as_parameter_(self):
        return self.ptr


# ---- lifetime -----------------------------------------------------------------

def kv_init(n_ctx, n_batch=2048, n_ubatch=512, n_seq_max=1, n_stream=1, n_layer=1,
            n_head=16, n_head_kv=8, head_dim=128, causal=True, seq_to_stream=None,
            k_layers=None, v_layers=None, n_swa=0):
    """Create a cache.  k_layers / v_layers: lists of device tensors (or
    addresses), one per layer, each [n_stream * kv_size, n_head_kv * head_dim]
    fp16; None for a host-only cache.  causal=False: bidirectional attention;
    n_swa > 0: a sliding window of n_swa positions (see kv_params in kvattn.h)."""
    p = kv_params()
    p.n_ctx, p.n_batch, p.n_ubatch = n_ctx, n_batch, n_ubatch
    p.n_seq_max, p.n_stream, p.n_layer = n_seq_max, n_stream, n_layer
    p.n_head, p.n_head_kv, p.head_dim, p.causal = n_head, n_head_kv, head_dim, int(bool(causal))
    p.n_swa = n_swa
    keep = []
    if seq_to_stream is not None:
        arr = (C.c_int32 * len(seq_to_stream))(*seq_to_stream)
        keep.append(arr)
        p.seq_to_stream = C.cast(arr, C.POINTER(C.c_int32))
    if k_layers is not None:
        ka = (C.c_void_p * len(k_layers))(*[_ptr(t) for t in k_layers])
        va = (C.c_void_p * len(v_layers))(*[_ptr(t) for t in v_layers])
        keep += [ka, va, list(k_layers), list(v_layers)]
        p.k_layers = C.cast(ka, C.POINTER(C.c_void_p))
        p.v_layers = C.cast(va, C.POINTER(C.c_void_p))
    out = C.c_void_p()
    rc = lib.kv_init(C.byref(p), C.byref(out))
    if rc != 0:
        raise KvError(rc, "kv_init failed")
    return Cache(out.value, keep)


def kv_free(c):
    if c.ptr:
        lib.kv_free(c.ptr)
        c.ptr = None


def kv_n_batch(c):
    return lib.kv_n_batch(c)


def kv_n_ubatch(c):
    return lib.kv_n_ubatch(c)


def kv_kv_size(c):
    return lib.kv_kv_size(c)


def kv_last_error(c):
    return lib.kv_last_error(c).decode()


# ---- host side -------------------------------------------------------------------

def _seq_arrays(seq_id):
    """The per-slot id lists as (flat int32 ids, per-slot counts, per-slot
    offsets).  seq_id: a list of id lists, a 2-D integer array (every slot has
    the same number of ids), or a (flat ids, counts) pair."""
    if isinstance(seq_id, tuple):
        flat = np.ascontiguousarray(seq_id[0], dtype=np.int32)
        counts = np.ascontiguousarray(seq_id[1], dtype=np.int32)
    elif isinstance(seq_id, np.ndarray) and seq_id.ndim == 2:
        flat = np.ascontiguousarray(seq_id, dtype=np.int32).reshape(-1)
        counts = np.full(seq_id.shape[0], seq_id.shape[1], dtype=np.int32)
    else:
        counts = np.fromiter((len(ids) for ids in seq_id), dtype=np.int32, count=len(seq_id))
        flat = np.fromiter(itertools.chain.from_iterable(seq_id), dtype=np.int32, count=int(counts.sum()))
    offs = np.zeros(counts.shape[0], dtype=np.int64)
    if counts.shape[0] > 1:
        np.cumsum(counts[:-1], out=offs[1:])
    if flat.size == 0:
        flat = np.zeros(1, dtype=np.int32)
    return flat, counts, offs


def kv_split_ubatches(c, pos, seq_id=None, n_seq_id=None, mode=KV_SPLIT_AUTO, n_tokens=None):
    """Split a batch.  pos: list / array of positions or None (auto-fill);
    seq_id: list of id lists (first id first), a 2-D id array, a (flat ids,
    counts) pair, or None (all sequence 0); n_seq_id: counts, default the
    lists' lengths (pass False for the C NULL: one id per slot)."""
    if n_tokens is None:
        n_tokens = len(pos) if pos is not None else (len(seq_id[1]) if isinstance(seq_id, tuple) else len(seq_id))
    b = kv_batch()
    b.n_tokens = n_tokens
    keep = []
    if pos is not None:
        pa = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
        keep.append(pa)
        b.pos = pa.ctypes.data_as(C.POINTER(C.c_int32))
    if seq_id is not None:
        flat, counts, offs = _seq_arrays(seq_id)
        ptrs = (offs * 4 + flat.ctypes.data).astype(np.uint64)   # one pointer per slot into flat
        keep += [flat, ptrs]
        b.seq_id = C.cast(C.c_void_p(ptrs.ctypes.data), C.POINTER(C.POINTER(C.c_int32)))
        if n_seq_id is None:
            n_seq_id = counts
    if n_seq_id is not None and n_seq_id is not False:
        na = np.ascontiguousarray(np.asarray(n_seq_id, dtype=np.int32))
        keep.append(na)
        b.n_seq_id = na.ctypes.data_as(C.POINTER(C.c_int32))
    out = C.c_void_p()
    _check(c, lib.kv_split_ubatches(c, C.byref(b), mode, C.byref(out)))
    return Split(out.value, c)


def kv_split_sched_batch(c, b, mode=KV_SPLIT_AUTO):
    """kv_split_ubatches of a scheduler batch (a SchedBatch from kv_sched_next),
    passed through as the C struct it is."""
    out = C.c_void_p()
    _check(c, lib.kv_split_ubatches(c, C.byref(b.raw.batch), mode, C.byref(out)))
    return Split(out.value, c)


def kv_split_count(s):
    return lib.kv_split_count(s)


def kv_split_ubatch(s, k):
    """Ubatch k as a dict of Python ints and numpy arrays (copies)."""
    info = kv_ubatch_info()
    rc = lib.kv_split_ubatch(s, k, C.byref(info))
    if rc != 0:
        raise KvError(rc, "bad ubatch index")
    n = info.n_tokens

    def arr(p, m):
        return np.ctypeslib.as_array(p, shape=(m,)).copy() if p and m else np.zeros(0, np.int32)

    return {"n_tokens": n, "n_seq_tokens": info.n_seq_tokens, "n_seqs": info.n_seqs,
            "n_seqs_unq": info.n_seqs_unq, "n_kv": info.n_kv,
            "rows": arr(info.rows, n), "pos": arr(info.pos, n), "seq0": arr(info.seq0, n),
            "seq_id_unq": arr(info.seq_id_unq, info.n_seqs_unq),
            "streams": arr(info.streams, n),
            "cells": arr(info.cells, n) if info.cells else None}


def kv_split_free(s):
    if s.ptr:
        lib.kv_split_free(s.ptr)
        s.ptr = None


def kv_prepare_cells(c, s):
    """0 on success, KV_NO_SLOT (1) if the cache is full (cache unchanged)."""
    return _check(c, lib.kv_prepare_cells(c, s))


def kv_seq_rm(c, seq, p0=0, p1=-1):
    return _check(c, lib.kv_seq_rm(c, seq, p0, p1))


def kv_seq_cp(c, src, dst, p0=0, p1=-1):
    return _check(c, lib.kv_seq_cp(c, src, dst, p0, p1))


def kv_seq_pos_max(c, seq):
    return lib.kv_seq_pos_max(c, seq)


def kv_cells_read(c, stream, n_seq_max):
    kv_size = lib.kv_kv_size(c)
    nw = (n_seq_max + 63) // 64
    pos = np.zeros(kv_size, np.int32)
    bits = np.zeros(kv_size * nw, np.uint64)
    _check(c, lib.kv_cells_read(c, stream, pos.ctypes.data_as(C.POINTER(C.c_int32)),
                                bits.ctypes.data_as(C.POINTER(C.c_uint64))))
    return pos, bits.reshape(kv_size, nw)


def kv_stream_n_kv(c, stream):
    return _check(c, lib.kv_stream_n_kv(c, stream))


# ---- device side ---------------------------------------------------------------------

def kv_store(c, s, ub, layer, k_cur, v_cur, stream=None):
    return _check(c, lib.kv_store(c, s, ub, layer, _ptr(k_cur), _ptr(v_cur), _stream(stream)))


def ubatch_attention(c, s, ub, layer, q, o, mask_out=None, stream=None):
    return _check(c, lib.ubatch_attention(c, s, ub, layer, _ptr(q), _ptr(o), _ptr(mask_out),
                                          _stream(stream)))


def ubatch_attention_static_scratch(c, s, ub, layer, q, o, mask_out=None, stream=None):
    """ubatch_attention for an all-decode ubatch, obtaining no memory during the
    call: its split-K scratch is a fixed array in the library's device image,
    shared by every call on the device (order such calls on one stream)."""
    return _check(c, lib.ubatch_attention_static_scratch(c, s, ub, layer, _ptr(q), _ptr(o),
                                                         _ptr(mask_out), _stream(stream)))


def kv_device_error(c):
    return _check(c, lib.kv_device_error(c))


def kv_selftest_wait(c, stream=None):
    """Launch one wait that nothing completes; it gives up after the kernels'
    wait limit (~1 s) and sets the device error word to KV_DERR_SELFTEST."""
    return _check(c, lib.kv_selftest_wait(c, _stream(stream)))


def kv_device_bytes(c):
    return lib.kv_device_bytes(c)


def kv_launch_count(c):
    return lib.kv_launch_count(c)


# ---- iteration-level batching (host) -----------------------------------------------

class Sched:
    """Handle returned by kv_sched_init (keeps its cache alive)."""

    def __init__(self, ptr, cache):
        self.ptr = ptr
        self.cache = cache

    @property
    def _as_parameter_(self):
        return self.ptr


class SchedBatch:
    """One pass's batch from kv_sched_next: n_tokens, pos and seq (copies),
    retired ids; raw is the C struct (its arrays live until the next call)."""

    def __init__(self, raw):
        self.raw = raw
        n = raw.batch.n_tokens
        self.n_tokens = n
        self.pos = np.ctypeslib.as_array(raw.batch.pos, (n,)).copy() if n else np.zeros(0, np.int32)
        self.seq = np.array([raw.batch.seq_id[i][0] for i in range(n)], dtype=np.int32)
        self.retired = [raw.retired[i] for i in range(raw.n_retired)]


def kv_sched_init(c, max_seqs, token_budget, fixed=False):
    p = kv_sched_params(max_seqs, token_budget, 1 if fixed else 0)
    out = C.c_void_p()
    _check(c, lib.kv_sched_init(c, C.byref(p), C.byref(out)))
    return Sched(out.value, c)


def kv_sched_free(s):
    lib.kv_sched_free(s)
    s.ptr = None


def kv_sched_submit(s, prompt_len, max_new):
    return _check(s.cache, lib.kv_sched_submit(s, prompt_len, max_new))


def kv_sched_next(s):
    raw = kv_sched_batch()
    _check(s.cache, lib.kv_sched_next(s, C.byref(raw)))
    return SchedBatch(raw)


def kv_sched_advance(s):
    return _check(s.cache, lib.kv_sched_advance(s))


def kv_sched_stats(s):
    st = kv_sched_info()
    _check(s.cache, lib.kv_sched_stats(s, C.byref(st)))
    return {"passes": st.passes, "useful": st.useful, "running": st.running,
            "waiting": st.waiting, "free_cells": st.free_cells}
