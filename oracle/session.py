"""The whole path, end to end, on the CPU: one object per cache.

BATCH-ZH, Part F: a decode call validates and fills the batch, splits it into
ubatches and reserves cells for all of them (returning 1 if the cache is
full), then runs the ubatches one after another; inside each, every layer
stores the ubatch's K/V rows and attends with the KQ mask.  KV-MEM,
"28 layers, 56 tensors": every layer owns one K and one V tensor.
"""

import numpy as np

from . import params as P
from . import batch as B
from . import cells as C
from . import mask as M
from . import attention as A


class Split:
    """One decode call's ubatches after cell reservation."""

    def __init__(self, ubatches, pos, seq_lists, cells, n_kv, snapshots, streams):
        self.ubatches = ubatches
        self.pos = pos
        self.seq_lists = seq_lists
        self.cells = cells
        self.n_kv = n_kv
        self.snapshots = snapshots
        self.streams = streams  # streams[k][i]: stream of row i of ubatch k

    def row_pos(self, k):
        return [self.pos[r] for r in self.ubatches[k]["rows"]]

    def row_seq0(self, k):
        return [self.seq_lists[r][0] for r in self.ubatches[k]["rows"]]


class OracleKV:
    def __init__(self, n_ctx, n_batch=P.DEFAULT_N_BATCH, n_ubatch=P.DEFAULT_N_UBATCH,
                 n_seq_max=1, n_stream=1, n_layer=1, n_head=16, n_head_kv=8,
                 head_dim=128, causal=True, seq_to_stream=None, keep_kv=True, n_swa=0):
        assert n_ctx % n_stream == 0
        self.n_batch, self.n_ubatch = P.clamp(n_ctx, n_batch, n_ubatch, causal)
        self.n_ctx, self.n_stream = n_ctx, n_stream
        self.kv_size = n_ctx // n_stream
        self.n_seq_max = n_seq_max
        self.n_layer, self.n_head, self.n_head_kv, self.head_dim = n_layer, n_head, n_head_kv, head_dim
        self.causal = causal
        self.n_swa = n_swa      # sliding window in positions (0: none)
        self.state = C.CellState(n_stream, self.kv_size, n_seq_max, seq_to_stream)
        self.k = self.v = None
        if keep_kv:
            shp = (n_stream, self.kv_size, n_head_kv, head_dim)
            self.k = [np.zeros(shp, dtype=np.float16) for _ in range(n_layer)]
            self.v = [np.zeros(shp, dtype=np.float16) for _ in range(n_layer)]

    def split(self, pos, seq_id, n_seq_id=None, mode=B.SPLIT_AUTO, keep_snapshots=True,
              n_tokens=None):
        """Validate, split and reserve cells.  Returns (code, Split or None)."""
        if n_tokens is None:
            n_tokens = len(pos) if pos is not None else len(seq_id)
        if seq_id is not None and n_seq_id is None:
            # Python lists carry their own lengths; the C interface's "count
            # array omitted" case is validate_and_fill's n_seq_id=None.
            n_seq_id = [len(s) for s in seq_id]
        err, pos_l, seq_l = B.validate_and_fill(
            n_tokens, pos, n_seq_id, seq_id, self.n_batch, self.n_seq_max,
            self.state.seq_to_stream, self.state)
        if err != 0:
            return err, None
        ubs = B.init_batch(n_tokens, seq_l, self.n_ubatch, self.n_stream, mode)
        code, cells, n_kv, snaps = C.prepare(self.state, ubs, pos_l, seq_l, keep_snapshots)
        if code != 0:
            return code, None
        streams = [C.stream_of_rows(self.state, ub, seq_l) for ub in ubs]
        return 0, Split(ubs, pos_l, seq_l, cells, n_kv, snaps, streams)

    def store(self, sp, k, layer, k_cur, v_cur):
        """k_cur/v_cur: [n_tokens of ubatch k, n_head_kv * head_dim] fp16."""
        n = sp.ubatches[k]["n_tokens"]
        shp = (n, self.n_head_kv, self.head_dim)
        A.kv_store(self.k[layer], self.v[layer], sp.streams[k], sp.cells[k],
                   np.asarray(k_cur).reshape(shp), np.asarray(v_cur).reshape(shp))

    def mask(self, sp, k):
        return M.kq_mask(sp.snapshots[k], sp.row_pos(k), sp.row_seq0(k),
                         sp.streams[k], sp.n_kv[k], self.causal, self.n_swa)

    def attention(self, sp, k, layer, q, rows=None, state=None):
        """q: [n_tokens of ubatch k, n_head, head_dim] fp16 -> float64 output."""
        st = state if state is not None else sp.snapshots[k]
        return A.ubatch_attention(np.asarray(q), self.k[layer], self.v[layer], st,
                                  sp.row_pos(k), sp.row_seq0(k), sp.streams[k],
                                  sp.n_kv[k], self.causal, self.n_head, self.n_head_kv,
                                  rows=rows, n_swa=self.n_swa)

    def seq_rm(self, q, p0, p1):
        return self.state.seq_rm(q, p0, p1)

    def seq_cp(self, src, dst, p0, p1):
        return self.state.seq_cp(src, dst, p0, p1)
