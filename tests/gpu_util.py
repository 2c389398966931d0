"""Shared driver for the GPU parity tests: one workload through the library
(C interface, CUDA kernels) and through the CPU oracle, on the same seeded
inputs.  Test infrastructure only."""

import numpy as np

import os

ATOL = 2e-3      # max-abs error, fp16 in / fp32 accumulate
RTOL_L2 = 1e-2   # relative L2 error

# worst (max-abs, rel-L2, outputs compared) per test, printed at the end of the
# session (tests/conftest.py) so that the margin to the tolerance is on record
MARGINS = {}


def _record(amax, rel, n):
    name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
    a, r, m = MARGINS.get(name, (0.0, 0.0, 0))
    MARGINS[name] = (max(a, amax), max(r, rel), m + n)


def check_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape, what)
    assert np.isfinite(got).all(), "non-finite output " + what
    err = np.abs(got - ref)
    amax = float(err.max()) if err.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / nref if nref > 0 else float(np.linalg.norm(got))
    _record(amax, rel, int(got.size))
    assert amax <= ATOL, "max-abs %.3g > %.3g %s" % (amax, ATOL, what)
    assert rel <= RTOL_L2, "rel-L2 %.3g > %.3g %s" % (rel, RTOL_L2, what)
    return amax, rel


# ---- the oracle's attention over many rows, in worker processes ----------------
# Workers are started with "spawn" (a process forked after the first GPU call can
# hang) and receive the oracle's K/V arrays once; each task is one chunk of one
# ubatch's rows, computed by the oracle's own ubatch_attention.

_W = {}


def _worker_init(k_layers, v_layers):
    _W["k"], _W["v"] = k_layers, v_layers


def _worker_rows(task):
    from oracle import attention as A
    (layer, q, state, row_pos, row_seq0, row_stream, n_kv, causal, n_head, n_head_kv, rows, n_swa) = task
    return A.ubatch_attention(q, _W["k"][layer], _W["v"][layer], state, row_pos, row_seq0, row_stream,
                              n_kv, causal, n_head, n_head_kv, rows=rows, n_swa=n_swa)


def oracle_rows_parallel(o, jobs, chunk=32):
    """jobs: list of (sp, k, layer, q [n, H, d], rows).  Returns the oracle's
    float64 outputs per job, computed in a pool of spawned processes."""
    import multiprocessing as mp
    tasks, where = [], []
    for j, (sp, k, layer, q, rows) in enumerate(jobs):
        for a in range(0, len(rows), chunk):
            tasks.append((layer, q, sp.snapshots[k], sp.row_pos(k), sp.row_seq0(k), sp.streams[k],
                          sp.n_kv[k], o.causal, o.n_head, o.n_head_kv, rows[a:a + chunk], o.n_swa))
            where.append(j)
    n_proc = max(1, min(16, os.cpu_count() or 1))
    ctx = mp.get_context("spawn")
    # one BLAS thread per worker (the workers are the parallelism); the children
    # read these when they import NumPy
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update({v: "1" for v in saved})
    try:
        with ctx.Pool(n_proc, initializer=_worker_init, initargs=(o.k, o.v)) as pool:
            res = pool.map(_worker_rows, tasks, chunksize=1)
    finally:
        for v, x in saved.items():
            if x is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = x
    out = [[] for _ in jobs]
    for j, r in zip(where, res):
        out[j].append(r)
    return [np.concatenate(x, axis=0) for x in out]


class Pair:
    """A library cache on cuda:0 and an oracle cache fed identical inputs."""

    def __init__(self, cfg, poison=False, oracle=True):
        import torch
        import continuous_batching_kv_gb300 as kv
        from oracle.session import OracleKV
        self.torch, self.kv = torch, kv
        self.cfg = cfg
        sh, prm = cfg["shape"], cfg["params"]
        self.H, self.Hk, self.d, self.L = sh["n_head"], sh["n_head_kv"], sh["head_dim"], sh["n_layer"]
        width = self.Hk * self.d
        fill = float("nan") if poison else 0.0
        self.kt = [torch.full((prm["n_ctx"], width), fill, dtype=torch.float16, device="cuda")
                   for _ in range(self.L)]
        self.vt = [torch.full((prm["n_ctx"], width), fill, dtype=torch.float16, device="cuda")
                   for _ in range(self.L)]
        # the cache's initial bytes, and which rows a store has written (per layer)
        self.fill_bits = np.float16(fill).view(np.uint16)
        self.kv_size = prm["n_ctx"] // prm["n_stream"]
        self.written = [np.zeros(prm["n_ctx"], dtype=bool) for _ in range(self.L)]
        self.c = kv.kv_init(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                            n_seq_max=prm["n_seq_max"], n_stream=prm["n_stream"], n_layer=self.L,
                            n_head=self.H, n_head_kv=self.Hk, head_dim=self.d,
                            causal=prm.get("causal", True), seq_to_stream=prm.get("seq_to_stream"),
                            k_layers=self.kt, v_layers=self.vt, n_swa=prm.get("n_swa", 0))
        self.o = None
        if oracle:
            self.o = OracleKV(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                              n_seq_max=prm["n_seq_max"], n_stream=prm["n_stream"], n_layer=self.L,
                              n_head=self.H, n_head_kv=self.Hk, head_dim=self.d,
                              causal=prm.get("causal", True), seq_to_stream=prm.get("seq_to_stream"),
                              n_swa=prm.get("n_swa", 0))

    def close(self):
        self.kv.kv_free(self.c)

    def seq_cp(self, src, dst, p0=0, p1=-1):
        """Share src's cells with dst on both sides."""
        self.kv.kv_seq_cp(self.c, src, dst, p0, p1)
        if self.o is not None:
            assert self.o.seq_cp(src, dst, p0, p1) == 0

    def check_store(self):
        """K1 bytes: every layer's K and V tensors read back and compared bit for
        bit -- rows a store wrote against the oracle's scatter (same layout:
        [n_stream][kv_size][n_head_kv][head_dim] fp16), other rows against the
        cache's initial fill (nothing else may be written)."""
        assert self.o is not None
        for layer in range(self.L):
            w = self.written[layer]
            for dev, ref in ((self.kt[layer], self.o.k[layer]), (self.vt[layer], self.o.v[layer])):
                got = dev.cpu().numpy().view(np.uint16)
                exp = ref.reshape(got.shape).view(np.uint16)
                assert np.array_equal(got[w], exp[w]), "stored rows differ, layer %d" % layer
                rest = got[~w]
                if np.isnan(self.fill_bits.view(np.float16)):
                    assert np.isnan(rest.view(np.float16)).all(), "unwritten rows changed, layer %d" % layer
                else:
                    assert (rest == self.fill_bits).all(), "unwritten rows changed, layer %d" % layer

    def qkv(self, layer, pos, content):
        from workloads import gen
        cid = self.cfg["id"]
        q = gen.batch_rows(cid, layer, gen.KIND_Q, pos, content, self.H * self.d)
        k = gen.batch_rows(cid, layer, gen.KIND_K, pos, content, self.Hk * self.d)
        v = gen.batch_rows(cid, layer, gen.KIND_V, pos, content, self.Hk * self.d)
        return q, k, v

    def run_call(self, call, attend=True, rows_sample=None, check_mask=False, layers=None, split=None,
                 defer=False):
        """Split, reserve, store every layer, and (if attend) attend and compare.

        rows_sample(n) -> list of ubatch rows to compare (None: all rows).
        split: a split handle made by the caller from the same batch (e.g. from a
        scheduler batch), used instead of splitting `call` here.  defer: compare
        after the whole call, the oracle's rows computed in worker processes.
        Returns a list of (ubatch, layer, amax, rel) and the outputs by
        (seq tuple, pos)."""
        torch, kv = self.torch, self.kv
        s = split if split is not None else kv.kv_split_ubatches(self.c, call["pos"], call["seq"])
        assert kv.kv_prepare_cells(self.c, s) == 0
        deferred = []
        if self.o is not None:
            code, sp = self.o.split(call["pos"], call["seq"], keep_snapshots=attend)
            assert code == 0
        stats, outs = [], {}
        layers = range(self.L) if layers is None else layers
        for k in range(kv.kv_split_count(s)):
            u = kv.kv_split_ubatch(s, k)
            rows = list(u["rows"])
            pos = [call["pos"][r] for r in rows]
            con = [call["content"][r] for r in rows]
            n = len(rows)
            if self.o is not None:
                assert rows == sp.ubatches[k]["rows"]
                assert list(u["cells"]) == sp.cells[k] and u["n_kv"] == sp.n_kv[k]
            for layer in range(self.L):
                q, kk, vv = self.qkv(layer, pos, con)
                kv.kv_store(self.c, s, k, layer, torch.from_numpy(kk).cuda(), torch.from_numpy(vv).cuda())
                self.written[layer][np.asarray(u["streams"], dtype=np.int64) * self.kv_size +
                                    np.asarray(u["cells"], dtype=np.int64)] = True
                if self.o is not None:
                    self.o.store(sp, k, layer, kk, vv)
                if not attend or layer not in layers:
                    continue
                qd = torch.from_numpy(q).cuda()
                od = torch.empty((n, self.H, self.d), dtype=torch.float32, device="cuda")
                md = None
                if check_mask:
                    md = torch.empty((n, u["n_kv"]), dtype=torch.int16, device="cuda")
                kv.ubatch_attention(self.c, s, k, layer, qd, od, md)
                torch.cuda.synchronize()
                assert kv.kv_device_error(self.c) == 0, "device error ubatch %d layer %d" % (k, layer)
                got = od.cpu().numpy()
                for n_, r in enumerate(rows):
                    outs[(tuple(call["seq"][r]), call["pos"][r], layer)] = got[n_]
                if self.o is not None:
                    if check_mask:
                        ref_m = self.o.mask(sp, k)
                        got_m = md.cpu().numpy().view(np.uint16)
                        assert np.array_equal(got_m, ref_m), "mask mismatch ubatch %d" % k
                    sel = list(range(n)) if rows_sample is None else rows_sample(n)
                    if defer:
                        deferred.append(((sp, k, layer, q.reshape(n, self.H, self.d), sel), got[sel]))
                        continue
                    ref = self.o.attention(sp, k, layer, q.reshape(n, self.H, self.d), rows=sel)
                    amax, rel = check_close(got[sel], ref, "ubatch %d layer %d" % (k, layer))
                    stats.append((k, layer, amax, rel))
        assert kv.kv_device_error(self.c) == 0
        if deferred:
            refs = oracle_rows_parallel(self.o, [j for j, _ in deferred])
            for ((_, k, layer, _, _), got), ref in zip(deferred, refs):
                amax, rel = check_close(got, ref, "ubatch %d layer %d" % (k, layer))
                stats.append((k, layer, amax, rel))
        kv.kv_split_free(s)
        return stats, outs


def sample_rows(n, m=24, seed=0):
    """First, last, and a seeded spread of rows."""
    if n <= m:
        return list(range(n))
    rng = np.random.default_rng(seed + n)
    mid = rng.choice(np.arange(1, n - 1), size=m - 2, replace=False)
    return sorted({0, n - 1, *mid.tolist()})
