"""GPU parity: the CUDA path (through the C interface) against the CPU oracle.

Splits, cells and masks bit-exact; attention within max-abs 2e-3 and
relative L2 1e-2 (fp16 inputs, fp32 accumulation and output).
"""

import numpy as np
import pytest

from workloads import configs
from tests.gpu_util import Pair, sample_rows, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import continuous_batching_kv_gb300  # noqa: F401  (fails loudly if the library is missing)


def _run(cfg, rows_sample=None, check_mask=False, poison=False, layers=None, check_store=False, defer=False):
    p = Pair(cfg, poison=poison)
    try:
        for call in cfg["setup"]:
            p.run_call(call, attend=False)
        stats = []
        outs = {}
        for call in cfg["measured"]:
            st, o = p.run_call(call, attend=True, rows_sample=rows_sample, check_mask=check_mask,
                               layers=layers, defer=defer)
            stats += st
            outs.update(o)
        if check_store:
            p.check_store()
        return stats, outs
    finally:
        p.close()


def test_config1_prompt_then_decode_all_rows_and_masks():
    stats, _ = _run(configs.config(1), check_mask=True, check_store=True)
    assert len(stats) == 5


def test_config1_nan_poisoned_cache():
    # unused cells hold NaN: masked cells must contribute nothing at all
    stats, outs = _run(configs.config(1), check_mask=True, poison=True, check_store=True)
    assert all(np.isfinite(v).all() for v in outs.values())


def test_config2_prefill_5000_all_rows():
    # every row of all 10 ubatches at layer 1 (the plan built at layer 0 is reused,
    # as in a model's later layers); the oracle's rows run in worker processes
    cfg = configs.config(2, n_layer=2)
    stats, _ = _run(cfg, check_mask=True, layers=[1], defer=True)
    assert len(stats) == 10


def test_config2_nan_poisoned_cache_prefill_path():
    # the tensor-core path multiplies whole tiles: unused cells (NaN) must
    # have their V rows cleared before the PV product
    cfg = configs.config(2, n_layer=1)
    cfg["measured"] = cfg["measured"][:1]
    stats, outs = _run(cfg, rows_sample=lambda n: sample_rows(n, 32), poison=True)
    assert len(stats) == 4
    assert all(np.isfinite(v).all() for v in outs.values())


def test_config3_decode_unified_all_rows():
    stats, _ = _run(configs.config(3, n_layer=2), check_mask=True)
    assert len(stats) == 2


def test_config4_mixed_prefix_streams_and_twins():
    cfg = configs.config(4, n_layer=1)
    stats, outs = _run(cfg, rows_sample=lambda n: sample_rows(n, 40), check_mask=True, check_store=True)
    assert len(stats) == 7
    # prefix cells shared by 16 sequences give the same output as duplicated copies
    for s in range(16):
        a = outs[((s,), 1280, 0)]
        b = outs[((s + 16,), 1280, 0)]
        check_close(a, b.astype(np.float64), "twin %d" % s)


def test_config5_full_size_one_layer_all_rows():
    cfg = configs.config(5, n_layer=1)
    stats, _ = _run(cfg)
    assert len(stats) == 1


def test_ragged_kv_size_and_streams():
    # kv_size not a multiple of the 64-cell tile, two streams, prefix sharing
    cfg = {"id": 7, "name": "ragged", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=2 * 100, n_batch=200, n_ubatch=37, n_seq_max=4, n_stream=2,
                          seq_to_stream=[0, 1, 0, 1]),
           "setup": [],
           "measured": [
               {"pos": list(range(30)), "seq": [[0, 2]] * 30, "content": [0] * 30},
               {"pos": list(range(30, 97)) + list(range(40)),
                "seq": [[0]] * 67 + [[1, 3]] * 40, "content": [0] * 67 + [1] * 40},
               {"pos": [97, 30, 40, 40], "seq": [[0], [2], [1], [3]], "content": [0, 2, 1, 3]},
           ]}
    stats, _ = _run(cfg, check_mask=True, check_store=True)
    assert len(stats) >= 5


def test_non_causal_prefill_decode_and_prefix():
    # causal = 0: a row sees every occupied cell of its sequence, later positions
    # included, but not the cells that later ubatches of the same split fill
    # (300 prompt tokens at n_ubatch 128: the first ubatch must not see the other
    # two's cells); then a prompt shared by sequences 1 and 2, and decode rows
    cfg = {"id": 14, "name": "non-causal", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=1024, n_batch=512, n_ubatch=128, n_seq_max=3, n_stream=1,
                          causal=False),
           "setup": [],
           "measured": [
               {"pos": list(range(300)), "seq": [[0]] * 300, "content": [0] * 300},
               {"pos": list(range(200)) + [300], "seq": [[1, 2]] * 200 + [[0]],
                "content": [1] * 200 + [0]},
               {"pos": [301, 200, 200], "seq": [[0], [1], [2]], "content": [0, 1, 2]},
           ]}
    stats, _ = _run(cfg, check_mask=True)
    assert len(stats) >= 6


def test_prefill_split_without_clusters_many_kv_heads():
    # 32 KV heads leave a few prefill CTA columns per head (too few for clusters of
    # four), so split blocks write partials to global memory and merge there
    shape = dict(configs.QWEN, n_layer=1, n_head=32, n_head_kv=32)
    cfg = {"id": 15, "name": "kv32", "shape": shape,
           "params": dict(n_ctx=2048, n_batch=2048, n_ubatch=512, n_seq_max=1, n_stream=1),
           "setup": [],
           "measured": [{"pos": list(range(1200)), "seq": [[0]] * 1200, "content": [0] * 1200}]}
    stats, _ = _run(cfg, rows_sample=lambda n: sample_rows(n, 48), check_mask=True)
    assert len(stats) == 3


@pytest.mark.parametrize("causal,n_swa", [(True, 100), (False, 100), (True, 1)])
def test_sliding_window(causal, n_swa):
    # a window of n_swa positions (a cell that far or further behind the row is
    # masked): 300 prompt tokens in ubatches of 128 (the window cuts tiles, so
    # both kernels take their per-cell paths), a mixed ubatch with a prompt
    # shared by sequences 1 and 2, then decode rows; masks bit-exact
    cfg = {"id": 16, "name": "swa", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=1024, n_batch=512, n_ubatch=128, n_seq_max=3, n_stream=1,
                          causal=causal, n_swa=n_swa),
           "setup": [],
           "measured": [
               {"pos": list(range(300)), "seq": [[0]] * 300, "content": [0] * 300},
               {"pos": list(range(150)) + [300], "seq": [[1, 2]] * 150 + [[0]],
                "content": [1] * 150 + [0]},
               {"pos": [301, 150, 150], "seq": [[0], [1], [2]], "content": [0, 1, 2]},
           ]}
    stats, _ = _run(cfg, check_mask=True)
    assert len(stats) >= 6


def test_random_small_batches():
    rng = np.random.default_rng(5)
    calls = []
    nxt = [0, 0, 0]
    for _ in range(6):
        n = int(rng.integers(1, 60))
        pos, seq, con = [], [], []
        for _ in range(n):
            q = int(rng.integers(0, 3))
            pos.append(nxt[q]); seq.append([q]); con.append(q)
            nxt[q] += 1
        calls.append({"pos": pos, "seq": seq, "content": con})
    cfg = {"id": 8, "name": "random", "shape": dict(configs.LLAMA, n_layer=1),
           "params": dict(n_ctx=512, n_batch=64, n_ubatch=24, n_seq_max=3, n_stream=1),
           "setup": [], "measured": calls}
    stats, _ = _run(cfg, check_mask=True)
    assert stats


def test_retire_and_reuse_cells():
    import torch
    import continuous_batching_kv_gb300 as kv
    cfg = {"id": 9, "name": "retire", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=256, n_batch=256, n_ubatch=64, n_seq_max=4, n_stream=1),
           "setup": [], "measured": []}
    p = Pair(cfg)
    try:
        p.run_call({"pos": list(range(40)), "seq": [[0]] * 40, "content": [0] * 40})
        p.run_call({"pos": list(range(30)), "seq": [[1]] * 30, "content": [1] * 30})
        # retire sequence 0 (ITER: finished sequences release their cache)
        kv.kv_seq_rm(p.c, 0, 0, -1)
        p.o.seq_rm(0, 0, -1)
        st, _ = p.run_call({"pos": list(range(50)), "seq": [[2]] * 50, "content": [2] * 50})
        assert st
        st, _ = p.run_call({"pos": [30, 50], "seq": [[1], [2]], "content": [1, 2]})
        assert st
    finally:
        p.close()


def test_seq_cp_shares_a_prefix():
    # a 100-token prompt of sequence 0, shared whole with sequence 2 and up to
    # position 60 with sequence 1 (no K/V moves: the cells gain the ids); then a
    # decode row each.  Sequence 2 continues sequence 0's content, so its row must
    # give sequence 0's output: prefix-shared cells equal duplicated ones.
    cfg = {"id": 15, "name": "seq-cp", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=512, n_batch=256, n_ubatch=64, n_seq_max=4, n_stream=1),
           "setup": [], "measured": []}
    p = Pair(cfg)
    try:
        p.run_call({"pos": list(range(100)), "seq": [[0]] * 100, "content": [0] * 100})
        p.seq_cp(0, 2)
        p.seq_cp(0, 1, 0, 60)
        st, outs = p.run_call({"pos": [100, 60, 100], "seq": [[0], [1], [2]], "content": [0, 1, 0]},
                              check_mask=True)
        assert len(st) == 1
        np.testing.assert_allclose(outs[((2,), 100, 0)], outs[((0,), 100, 0)], rtol=0, atol=1e-5)
    finally:
        p.close()


def test_large_removal_grows_upload_buffers():
    # 5000 cells of sequence 0, then its removal: more changed cells than the
    # staging buffers hold (4096 deltas), so they are re-allocated (mapped pinned
    # memory) before the next device call; a new prompt and a decode row follow
    import continuous_batching_kv_gb300 as kv
    cfg = {"id": 10, "name": "large-removal", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=8192, n_batch=2048, n_ubatch=512, n_seq_max=2, n_stream=1),
           "setup": [], "measured": []}
    p = Pair(cfg)
    try:
        for c0 in range(0, 5000, 2048):
            n = min(2048, 5000 - c0)
            p.run_call({"pos": list(range(c0, c0 + n)), "seq": [[0]] * n, "content": [0] * n}, attend=False)
        kv.kv_seq_rm(p.c, 0, 0, -1)
        p.o.seq_rm(0, 0, -1)
        st, _ = p.run_call({"pos": list(range(300)), "seq": [[1]] * 300, "content": [1] * 300}, rows_sample=sample_rows)
        assert st
        st, _ = p.run_call({"pos": [300], "seq": [[1]], "content": [1]})
        assert st
    finally:
        p.close()


def test_device_call_errors():
    import torch
    import continuous_batching_kv_gb300 as kv
    k = [torch.zeros((64, 1024), dtype=torch.float16, device="cuda")]
    v = [torch.zeros((64, 1024), dtype=torch.float16, device="cuda")]
    c = kv.kv_init(n_ctx=64, n_batch=64, n_ubatch=8, n_layer=1, k_layers=k, v_layers=v)
    q = torch.zeros((8, 16, 128), dtype=torch.float16, device="cuda")
    o = torch.zeros((8, 16, 128), dtype=torch.float32, device="cuda")
    kc = torch.zeros((8, 1024), dtype=torch.float16, device="cuda")
    s = kv.kv_split_ubatches(c, list(range(16)), [[0]] * 16)
    with pytest.raises(kv.KvError) as e:
        kv.kv_store(c, s, 0, 0, kc, kc)
    assert e.value.code == kv.KV_E_ORDER            # not prepared
    kv.kv_prepare_cells(c, s)
    with pytest.raises(kv.KvError) as e:
        kv.ubatch_attention(c, s, 1, 0, q, o)
    assert e.value.code == kv.KV_E_ORDER            # ubatches 0..1 not stored
    kv.kv_store(c, s, 0, 0, kc, kc)
    kv.kv_store(c, s, 1, 0, kc, kc)
    kv.ubatch_attention(c, s, 1, 0, q, o)
    with pytest.raises(kv.KvError) as e:
        kv.kv_store(c, s, 0, 1, kc, kc)
    assert e.value.code == kv.KV_E_INVAL            # layer out of range
    kv.kv_seq_rm(c, 0, 3, -1)
    with pytest.raises(kv.KvError) as e:
        kv.ubatch_attention(c, s, 1, 0, q, o)
    assert e.value.code == kv.KV_E_STALE
    assert kv.kv_device_error(c) == 0
    kv.kv_free(c)


def test_plans_built_ahead_unsynchronised_and_out_of_order():
    # every ubatch's plan after the first is built ahead on the library's side stream
    # while the previous ubatch runs; issue the calls back to back with no host
    # synchronisation, then again in an order that leaves some look-ahead builds unused
    # and misses others, and compare every output with the oracle
    import torch
    import continuous_batching_kv_gb300 as kv
    cfg = configs.config(2, n_layer=2)
    p = Pair(cfg)
    try:
        call = cfg["measured"][0]
        s = kv.kv_split_ubatches(p.c, call["pos"], call["seq"])
        assert kv.kv_prepare_cells(p.c, s) == 0
        code, sp = p.o.split(call["pos"], call["seq"], keep_snapshots=True)
        assert code == 0
        nub = kv.kv_split_count(s)
        assert nub >= 4
        qs = {}
        for k in range(nub):
            u = kv.kv_split_ubatch(s, k)
            rows = list(u["rows"])
            pos = [call["pos"][r] for r in rows]
            con = [call["content"][r] for r in rows]
            for layer in range(p.L):
                q, kk, vv = p.qkv(layer, pos, con)
                kv.kv_store(p.c, s, k, layer, torch.from_numpy(kk).cuda(), torch.from_numpy(vv).cuda())
                p.o.store(sp, k, layer, kk, vv)
                qs[(k, layer)] = q.reshape(len(rows), p.H, p.d)
        orders = [[(k, layer) for k in range(nub) for layer in range(p.L)],
                  [(k, 0) for k in (1, 0, 3, 2)] + [(k, 1) for k in (0, 2, 1, 3)] + [(k, 0) for k in range(4, nub)]
                  + [(k, 1) for k in range(4, nub)]]
        # inputs and outputs on the device before the calls, so that nothing between
        # them waits for the device
        qd = {key: torch.from_numpy(q).cuda() for key, q in qs.items()}
        for order in orders:
            outs = {key: torch.empty(q.shape, dtype=torch.float32, device="cuda") for key, q in qs.items()}
            torch.cuda.synchronize()
            for k, layer in order:
                kv.ubatch_attention(p.c, s, k, layer, qd[(k, layer)], outs[(k, layer)])
            torch.cuda.synchronize()
            assert kv.kv_device_error(p.c) == 0
            for (k, layer), od in outs.items():
                ref = p.o.attention(sp, k, layer, qs[(k, layer)])
                check_close(od.cpu().numpy(), ref, "ubatch %d layer %d" % (k, layer))
        kv.kv_split_free(s)
    finally:
        p.close()


def test_bounded_wait_gives_up_reports_and_the_next_calls_are_clean():
    # a wait that nothing completes runs to the kernels' limit, the error word says
    # so (and is cleared by reading it), and later attention calls on the same cache
    # still match the oracle
    import time
    import torch
    import continuous_batching_kv_gb300 as kv
    cfg = configs.config(1)
    p = Pair(cfg)
    try:
        for call in cfg["setup"]:
            p.run_call(call, attend=False)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        kv.kv_selftest_wait(p.c)
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
        assert kv.kv_device_error(p.c) == kv.KV_DERR_SELFTEST
        assert kv.kv_device_error(p.c) == 0
        assert waited > 0.2, "the wait gave up after %.3f s, before its limit" % waited
        stats = []
        for call in cfg["measured"]:
            st, _ = p.run_call(call, attend=True, check_mask=True)
            stats += st
        assert len(stats) == 5
    finally:
        p.close()


@pytest.mark.parametrize("fixed", [False, True])
def test_batching_loop_through_scheduler(fixed):
    # ITER, "The loop that replaces the batch": the native scheduler retires,
    # admits and assembles each pass; every pass's batch goes through
    # kv_split_ubatches -> kv_prepare_cells -> kv_store -> ubatch_attention on two
    # layers, and the oracle scheduler + oracle cache are driven the same way.
    # Prompts up to 70 tokens at n_ubatch 48 put both kernels on the path (a
    # sequence's 24+ rows in one ubatch take the tensor-core path), mixed with
    # decode rows; retirements free cells that later admissions take.
    import random
    import continuous_batching_kv_gb300 as kv
    from oracle import sched as S
    kv_size, budget, n_seq_max, max_seqs = 640, 96, 6, 4
    cfg = {"id": 17, "name": "loop", "shape": dict(configs.QWEN, n_layer=2),
           "params": dict(n_ctx=kv_size, n_batch=budget, n_ubatch=48, n_seq_max=n_seq_max, n_stream=1),
           "setup": [], "measured": []}
    p = Pair(cfg)
    rng = random.Random(31 + fixed)
    try:
        sch = kv.kv_sched_init(p.c, max_seqs=max_seqs, token_budget=budget, fixed=fixed)
        osch = S.Scheduler(kv_size=kv_size, n_seq_max=n_seq_max, max_seqs=max_seqs, token_budget=budget,
                           fixed=fixed)
        for _ in range(16):
            L, N = rng.randint(1, 70), rng.randint(1, 12)
            assert kv.kv_sched_submit(sch, L, N) == osch.submit(L, N)
        passes = 0
        while True:
            b = kv.kv_sched_next(sch)
            retired, pos, seq = osch.next_batch()
            assert b.retired == retired and list(b.pos) == pos and list(b.seq) == seq
            for q in retired:
                p.o.seq_rm(q, 0, -1)
            if not pos:
                break
            by_seq = {r.seq: r.rid for r in osch.running}
            call = {"pos": pos, "seq": [[q] for q in seq], "content": [100 + by_seq[q] for q in seq]}
            sp = kv.kv_split_sched_batch(p.c, b)
            st, _ = p.run_call(call, check_mask=True, split=sp)
            assert st
            kv.kv_sched_advance(sch)
            osch.advance()
            passes += 1
        info = kv.kv_sched_stats(sch)
        assert (info["passes"], info["useful"]) == (osch.passes, osch.useful) and passes == osch.passes
        assert passes >= 20
        p.check_store()
        kv.kv_sched_free(sch)
    finally:
        p.close()
