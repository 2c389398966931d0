"""Shared driver for the GPU parity tests: one workload through the library
(C interface, CUDA kernels) and through the CPU oracle, on the same seeded
inputs.  Test infrastructure only."""

import numpy as np

ATOL = 2e-3      # max-abs error, fp16 in / fp32 accumulate
RTOL_L2 = 1e-2   # relative L2 error


def check_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape, what)
    assert np.isfinite(got).all(), "non-finite output " + what
    err = np.abs(got - ref)
    amax = float(err.max()) if err.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / nref if nref > 0 else float(np.linalg.norm(got))
    assert amax <= ATOL, "max-abs %.3g > %.3g %s" % (amax, ATOL, what)
    assert rel <= RTOL_L2, "rel-L2 %.3g > %.3g %s" % (rel, RTOL_L2, what)
    return amax, rel


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

    def qkv(self, layer, pos, content):
        from workloads import gen
        cid = self.cfg["id"]
        q = gen.batch_rows(cid, layer, gen.KIND_Q, pos, content, self.H * self.d)
        k = gen.batch_rows(cid, layer, gen.KIND_K, pos, content, self.Hk * self.d)
        v = gen.batch_rows(cid, layer, gen.KIND_V, pos, content, self.Hk * self.d)
        return q, k, v

    def run_call(self, call, attend=True, rows_sample=None, check_mask=False, layers=None):
        """Split, reserve, store every layer, and (if attend) attend and compare.

        rows_sample(n) -> list of ubatch rows to compare (None: all rows).
        Returns a list of (ubatch, layer, amax, rel) and the outputs by
        (seq tuple, pos)."""
        torch, kv = self.torch, self.kv
        s = kv.kv_split_ubatches(self.c, call["pos"], call["seq"])
        assert kv.kv_prepare_cells(self.c, s) == 0
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
                    ref = self.o.attention(sp, k, layer, q.reshape(n, self.H, self.d), rows=sel)
                    amax, rel = check_close(got[sel], ref, "ubatch %d layer %d" % (k, layer))
                    stats.append((k, layer, amax, rel))
        assert kv.kv_device_error(self.c) == 0
        kv.kv_split_free(s)
        return stats, outs


def sample_rows(n, m=24, seed=0):
    """First, last, and a seeded spread of rows."""
    if n <= m:
        return list(range(n))
    rng = np.random.default_rng(seed + n)
    mid = rng.choice(np.arange(1, n - 1), size=m - 2, replace=False)
    return sorted({0, n - 1, *mid.tolist()})
