"""The multi-GPU mode is replicas only: every rank runs the whole path on its
own copy of the workload, and the only collective is the max over ranks of
the timed region.  Checked here with two gloo ranks on the CPU: the host
side of the path (split, cell reservation, n_kv) comes out identical on both
ranks, and the timing reduction returns the slowest rank's time."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _host_path_digest(cfg):
    """Split and reserve every call of a workload on a host-only cache; return
    the ubatch rows, cells and n_kv seen."""
    import continuous_batching_kv_gb300 as kv
    sh, prm = cfg["shape"], cfg["params"]
    c = kv.kv_init(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                   n_seq_max=prm["n_seq_max"], n_stream=prm["n_stream"], n_layer=sh["n_layer"],
                   n_head=sh["n_head"], n_head_kv=sh["n_head_kv"], head_dim=sh["head_dim"],
                   seq_to_stream=prm.get("seq_to_stream"))
    out = []
    try:
        for call in cfg["setup"] + cfg["measured"]:
            s = kv.kv_split_ubatches(c, call["pos"], call["seq"])
            assert kv.kv_prepare_cells(c, s) == 0
            for k in range(kv.kv_split_count(s)):
                u = kv.kv_split_ubatch(s, k)
                out.append((tuple(u["rows"]), tuple(u["cells"]), u["n_kv"]))
            kv.kv_split_free(s)
    finally:
        kv.kv_free(c)
    return out


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from workloads import configs
        digest = _host_path_digest(configs.config(4, n_layer=1))
        got = [None] * world
        dist.all_gather_object(got, digest)
        same = all(g == got[0] for g in got)
        ms = bench.max_over_ranks(10.0 + rank, "cpu")
        q.put((rank, same, ms, [len(r) for r, _, _ in digest[-7:]]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_and_time_is_max_over_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same, ms, sizes in res:
        assert same, "rank %d saw a different split / cell assignment" % rank
        assert ms == 10.0 + (world - 1)
        assert sizes == [34] + [512] * 5 + [438]   # the mixed iteration's split_equal ubatches
