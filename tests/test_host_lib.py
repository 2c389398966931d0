"""The native host half (C++) against the CPU oracle, bit-exact, no GPU.

Splits, auto-filled positions, reserved cells, n_kv, the cell state after
every call, removal, and error codes must all match the oracle exactly.
"""

import os
import random
import re

import numpy as np
import pytest

import continuous_batching_kv_gb300 as kv
from oracle import batch as B, params as P
from oracle.cells import NO_SLOT
from oracle.session import OracleKV
from oracle import sched as S
from workloads import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    hdr = open(os.path.join(ROOT, "include", "kvattn.h")).read()
    decl = re.findall(r"^\s*(?:int|void|int32_t|uint64_t|size_t|const char \*)\s*\*?\s*(\w+)\s*\(", hdr, re.M)
    assert len(decl) >= 19
    for name in decl:
        assert hasattr(kv.lib, name), name
    assert sorted(decl) == sorted(kv.EXPORTS)


def _pair(n_ctx, n_batch, n_ubatch, n_seq_max, n_stream, s2s=None, causal=True):
    c = kv.kv_init(n_ctx=n_ctx, n_batch=n_batch, n_ubatch=n_ubatch, n_seq_max=n_seq_max,
                   n_stream=n_stream, n_layer=1, n_head=4, n_head_kv=2, causal=causal,
                   seq_to_stream=s2s)
    o = OracleKV(n_ctx=n_ctx, n_batch=n_batch, n_ubatch=n_ubatch, n_seq_max=n_seq_max,
                 n_stream=n_stream, n_layer=1, n_head=4, n_head_kv=2, head_dim=128,
                 causal=causal, seq_to_stream=s2s, keep_kv=False)
    return c, o


def _compare_state(c, o):
    for s in range(o.n_stream):
        pos, bits = kv.kv_cells_read(c, s, o.n_seq_max)
        np.testing.assert_array_equal(pos, o.state.pos[s])
        np.testing.assert_array_equal(bits, o.state.bits[s])
        assert kv.kv_stream_n_kv(c, s) == o.state.n_kv_stream(s)


def _call_both(c, o, pos, seqs, mode=kv.KV_SPLIT_AUTO, n_seq_id=None):
    """Split + prepare on both sides; compare everything; return the code."""
    err_o, sp_o = o.split(pos, seqs, mode=mode, n_seq_id=n_seq_id, keep_snapshots=False,
                          n_tokens=(len(pos) if pos is not None else len(seqs)))
    try:
        s = kv.kv_split_ubatches(c, pos, seqs, n_seq_id=n_seq_id, mode=mode)
    except kv.KvError as e:
        assert err_o == e.code, (err_o, e.code)
        return e.code
    if err_o == NO_SLOT:
        assert kv.kv_prepare_cells(c, s) == kv.KV_NO_SLOT
        kv.kv_split_free(s)
        _compare_state(c, o)
        return NO_SLOT
    assert err_o == 0, err_o
    assert kv.kv_split_count(s) == len(sp_o.ubatches)
    assert kv.kv_prepare_cells(c, s) == 0
    for k, ub in enumerate(sp_o.ubatches):
        u = kv.kv_split_ubatch(s, k)
        assert list(u["rows"]) == ub["rows"]
        assert u["n_tokens"] == ub["n_tokens"]
        assert u["n_seq_tokens"] == ub["n_seq_tokens"]
        assert u["n_seqs"] == ub["n_seqs"]
        assert list(u["seq_id_unq"]) == ub["seq_id_unq"]
        assert list(u["pos"]) == [sp_o.pos[r] for r in ub["rows"]]
        assert list(u["seq0"]) == [sp_o.seq_lists[r][0] for r in ub["rows"]]
        assert list(u["streams"]) == sp_o.streams[k]
        assert list(u["cells"]) == sp_o.cells[k]
        assert u["n_kv"] == sp_o.n_kv[k]
    kv.kv_split_free(s)
    _compare_state(c, o)
    return 0


def test_clamps_match_oracle():
    for (n_ctx, nb, nu, causal) in [(64, 2048, 512, True), (4096, 64, 512, True), (64, 2048, 512, False),
                                    (8192, 2048, 0, True), (32768, 4096, 512, True), (100, 7, 3, True)]:
        c = kv.kv_init(n_ctx=n_ctx, n_batch=nb, n_ubatch=nu, causal=causal)
        assert (kv.kv_n_batch(c), kv.kv_n_ubatch(c)) == P.clamp(n_ctx, nb, nu, causal)
        kv.kv_free(c)


def test_page_split_examples():
    c, o = _pair(8192, 2048, 512, 1, 1)
    sizes = []
    for n in B.caller_chunks(5000, 2048):
        p0 = sum(sizes)
        s = kv.kv_split_ubatches(c, list(range(p0, p0 + n)), [[0]] * n)
        sizes += [kv.kv_split_ubatch(s, k)["n_tokens"] for k in range(kv.kv_split_count(s))]
        assert kv.kv_prepare_cells(c, s) == 0
        kv.kv_split_free(s)
    assert sizes[:9] == [512] * 9 and sizes[9:] == [392] and sum(sizes) == 5000
    c2 = kv.kv_init(n_ctx=8192, n_batch=2048, n_ubatch=512)
    s = kv.kv_split_ubatches(c2, list(range(1000)), [[0]] * 1000)
    assert [kv.kv_split_ubatch(s, k)["n_tokens"] for k in range(kv.kv_split_count(s))] == [512, 488]


@pytest.mark.parametrize("mode", [kv.KV_SPLIT_AUTO, kv.KV_SPLIT_SIMPLE, kv.KV_SPLIT_EQUAL, kv.KV_SPLIT_SEQ])
@pytest.mark.parametrize("n_stream", [1, 3])
def test_random_calls_match_oracle(mode, n_stream):
    rng = random.Random(1000 * mode + n_stream)
    n_seq = 6
    s2s = [q % n_stream for q in range(n_seq)]
    c, o = _pair(n_ctx=48 * n_stream, n_batch=40, n_ubatch=7, n_seq_max=n_seq, n_stream=n_stream, s2s=s2s)
    for step in range(40):
        n = rng.randint(1, 40)
        seqs = []
        for _ in range(n):
            first = rng.randrange(n_seq)
            same = [q for q in range(n_seq) if s2s[q] == s2s[first] and q != first]
            extra = rng.sample(same, rng.randint(0, min(2, len(same)))) if rng.random() < 0.3 else []
            seqs.append([first] + extra)
        pos = None if rng.random() < 0.3 else [rng.randint(0, 60) for _ in range(n)]
        code = _call_both(c, o, pos, seqs, mode=mode)
        assert code in (0, NO_SLOT)
        if rng.random() < 0.3:
            q = rng.randrange(-1, n_seq)
            p0, p1 = rng.randint(0, 30), rng.choice([-1, rng.randint(0, 60)])
            assert kv.kv_seq_rm(c, q, p0, p1) == 0
            o.seq_rm(q, p0, p1)
            _compare_state(c, o)
        if rng.random() < 0.3:
            src, dst = rng.randrange(n_seq), rng.randrange(n_seq)
            p0, p1 = rng.randint(0, 30), rng.choice([-1, rng.randint(0, 60)])
            if o.seq_cp(src, dst, p0, p1) == "cross-stream":
                with pytest.raises(kv.KvError) as ei:
                    kv.kv_seq_cp(c, src, dst, p0, p1)
                assert ei.value.code == kv.KV_E_CROSS_STREAM
            else:
                assert kv.kv_seq_cp(c, src, dst, p0, p1) == 0
            _compare_state(c, o)
        for q in range(n_seq):
            assert kv.kv_seq_pos_max(c, q) == o.state.seq_pos_max(q)


def test_error_codes_match_oracle():
    c, o = _pair(64, 16, 8, 4, 2, s2s=[0, 0, 1, 1])
    cases = [
        (list(range(17)), None, None),             # too large
        ([0], [[4]], None),                        # seq out of range
        ([0], [[0, 0]], None),                     # repeated id
        ([0], [[0, 2]], None),                     # cross stream
        ([-1], [[0]], None),                       # negative pos
        ([0], [[0]], [0]),                         # n_seq_id 0
    ]
    for pos, seqs, nsi in cases:
        err_o, _ = o.split(pos, seqs, n_seq_id=nsi, keep_snapshots=False, n_tokens=len(pos))
        with pytest.raises(kv.KvError) as ei:
            kv.kv_split_ubatches(c, pos, seqs, n_seq_id=nsi)
        assert ei.value.code == err_o, (pos, seqs)
    with pytest.raises(kv.KvError) as ei:
        kv.kv_split_ubatches(c, [], [], n_tokens=0)
    assert ei.value.code == kv.KV_E_INVAL
    for src, dst, code in ((0, 4, kv.KV_E_SEQ_RANGE), (-1, 0, kv.KV_E_SEQ_RANGE), (0, 2, kv.KV_E_CROSS_STREAM)):
        with pytest.raises(kv.KvError) as ei:
            kv.kv_seq_cp(c, src, dst, 0, -1)
        assert ei.value.code == code


def test_auto_fill_and_null_seq():
    c, o = _pair(64, 16, 16, 4, 1)
    assert _call_both(c, o, None, None if False else [[0]] * 3) == 0
    assert _call_both(c, o, None, [[1], [0, 1], [1]]) == 0
    s = kv.kv_split_ubatches(c, None, None, n_tokens=2)     # seq_id NULL -> sequence 0
    u = kv.kv_split_ubatch(s, 0)
    assert list(u["seq0"]) == [0, 0] and list(u["pos"]) == [4, 5]


def test_all_or_nothing_restores_state():
    c, o = _pair(32, 32, 4, 2, 1)
    assert _call_both(c, o, list(range(30)), [[0]] * 30) == 0
    assert _call_both(c, o, [30, 31, 32], [[0]] * 3) == NO_SLOT
    assert _call_both(c, o, [30, 31], [[1]] * 2) == 0


def test_split_handle_rules():
    c = kv.kv_init(n_ctx=64, n_batch=16, n_ubatch=8)
    s = kv.kv_split_ubatches(c, [0, 1], [[0], [0]])
    assert kv.kv_prepare_cells(c, s) == 0
    with pytest.raises(kv.KvError) as ei:
        kv.kv_prepare_cells(c, s)
    assert ei.value.code == kv.KV_E_ORDER
    with pytest.raises(kv.KvError) as ei:          # host-only cache: no device calls
        kv.kv_store(c, s, 0, 0, 16, 16)
    assert ei.value.code == kv.KV_E_NO_DEVICE


@pytest.mark.parametrize("cid", [1, 2, 3, 4])
def test_workload_configs_match_oracle(cid):
    cfg = configs.config(cid)
    prm = cfg["params"]
    c, o = _pair(prm["n_ctx"], prm["n_batch"], prm["n_ubatch"], prm["n_seq_max"], prm["n_stream"],
                 s2s=prm.get("seq_to_stream"))
    for call in cfg["setup"] + cfg["measured"]:
        assert _call_both(c, o, call["pos"], call["seq"]) == 0


def test_workload_worked_numbers():
    # config 3: decode rows land on cells 5568..5575 with n_kv 5632
    cfg = configs.config(3)
    prm = cfg["params"]
    c = kv.kv_init(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                   n_seq_max=prm["n_seq_max"])
    for call in cfg["setup"]:
        s = kv.kv_split_ubatches(c, call["pos"], call["seq"])
        assert kv.kv_prepare_cells(c, s) == 0
    call = cfg["measured"][0]
    s = kv.kv_split_ubatches(c, call["pos"], call["seq"])
    assert kv.kv_prepare_cells(c, s) == 0
    u = kv.kv_split_ubatch(s, 0)
    assert list(u["cells"]) == list(range(5568, 5576)) and u["n_kv"] == 5632
    # config 4: the mixed iteration splits as [34, 512 x 5, 438]
    cfg = configs.config(4)
    prm = cfg["params"]
    c = kv.kv_init(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                   n_seq_max=prm["n_seq_max"], n_stream=prm["n_stream"],
                   seq_to_stream=prm["seq_to_stream"])
    for call in cfg["setup"]:
        s = kv.kv_split_ubatches(c, call["pos"], call["seq"])
        assert kv.kv_prepare_cells(c, s) == 0
    call = cfg["measured"][0]
    s = kv.kv_split_ubatches(c, call["pos"], call["seq"])
    assert [kv.kv_split_ubatch(s, k)["n_tokens"] for k in range(kv.kv_split_count(s))] == [34] + [512] * 5 + [438]
    assert kv.kv_prepare_cells(c, s) == 0
    fill = [int((kv.kv_cells_read(c, st, 64)[0] >= 0).sum()) for st in range(4)]
    assert fill == [5136, 7686, 7905, 7905]


@pytest.mark.parametrize("fixed", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_scheduler_matches_oracle(fixed, seed):
    # the native scheduler against the oracle's, pass by pass; every batch is
    # split and placed in both caches and the cell states compared (retirement
    # frees the cells the next admissions take)
    rng = random.Random(100 * seed + fixed)
    kv_size, budget = 300, 48
    c, o = _pair(n_ctx=kv_size, n_batch=budget, n_ubatch=16, n_seq_max=6, n_stream=1)
    sch = kv.kv_sched_init(c, max_seqs=4, token_budget=budget, fixed=fixed)
    osch = S.Scheduler(kv_size=kv_size, n_seq_max=6, max_seqs=4, token_budget=budget, fixed=fixed)
    for _ in range(40):
        L, N = rng.randint(1, 60), rng.randint(1, 40)
        rid = osch.submit(L, N)
        if rid is None:
            with pytest.raises(kv.KvError) as ei:
                kv.kv_sched_submit(sch, L, N)
            assert ei.value.code == kv.KV_E_INVAL
        else:
            assert kv.kv_sched_submit(sch, L, N) == rid
    passes = 0
    while True:
        b = kv.kv_sched_next(sch)
        retired, pos, seq = osch.next_batch()
        for q in retired:
            o.seq_rm(q, 0, -1)
        assert b.retired == retired and list(b.pos) == pos and list(b.seq) == seq
        if not pos:
            break
        s = kv.kv_split_sched_batch(c, b)
        assert kv.kv_prepare_cells(c, s) == 0
        code, _ = o.split(pos, [[q] for q in seq], keep_snapshots=False)
        assert code == 0
        _compare_state(c, o)
        kv.kv_split_free(s)
        kv.kv_sched_advance(sch)
        osch.advance()
        passes += 1
    st = kv.kv_sched_stats(sch)
    assert (st["passes"], st["useful"], st["running"], st["waiting"]) == (osch.passes, osch.useful, 0, 0)
    assert st["free_cells"] == kv_size and passes == osch.passes
    kv.kv_sched_free(sch)


def test_scheduler_errors():
    c = kv.kv_init(n_ctx=64, n_batch=16, n_ubatch=8, n_seq_max=4, n_stream=2)
    with pytest.raises(kv.KvError) as ei:
        kv.kv_sched_init(c, 2, 16)                  # needs a unified cache
    assert ei.value.code == kv.KV_E_INVAL
    c = kv.kv_init(n_ctx=64, n_batch=16, n_ubatch=8, n_seq_max=4)
    for ms, tb in ((5, 16), (0, 16), (4, 3), (2, 17)):   # 17 > n_batch 16
        with pytest.raises(kv.KvError):
            kv.kv_sched_init(c, ms, tb)
    sch = kv.kv_sched_init(c, 2, 16)
    assert kv.kv_sched_submit(sch, 4, 2) == 0
    b = kv.kv_sched_next(sch)
    assert b.n_tokens == 4
    with pytest.raises(kv.KvError) as ei:
        kv.kv_sched_next(sch)                       # the batch was not advanced
    assert ei.value.code == kv.KV_E_ORDER
    kv.kv_sched_free(sch)


def test_init_rejects_a_negative_window():
    with pytest.raises(kv.KvError) as ei:
        kv.kv_init(n_ctx=64, n_swa=-1)
    assert ei.value.code == kv.KV_E_INVAL
    c = kv.kv_init(n_ctx=64, n_swa=16)          # a window is a host-side parameter only
    s = kv.kv_split_ubatches(c, list(range(10)), [[0]] * 10)
    assert kv.kv_prepare_cells(c, s) == 0
