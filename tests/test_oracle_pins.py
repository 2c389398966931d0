"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a value a
page prints (fixtures under tests/golden/, each with its citation), a closed
form, an independent library routine (torch's scaled_dot_product_attention),
brute force on tiny inputs, or an invariant the pages state.
"""

import itertools
import math
import random

import numpy as np
import pytest

from oracle import params as P, batch as B, cells as C, mask as M, attention as A
from oracle import layout as L
from oracle import sched as S
from oracle.session import OracleKV
from workloads import gen
from tests.conftest import golden


# ----------------------------------------------------------------------------
# splits and clamps
# ----------------------------------------------------------------------------

def test_caller_chunks_pin():
    g = golden("splits.json")
    for case in g["caller_chunks"]:
        assert B.caller_chunks(case["n_tokens"], case["n_batch"]) == case["calls"]


def test_ubatches_per_call_pin():
    g = golden("splits.json")
    for case in g["ubatches_per_call"]:
        per_call = []
        for n in B.caller_chunks(case["n_tokens"], case["n_batch"]):
            seqs = [[0]] * n
            per_call.append(len(B.init_batch(n, seqs, case["n_ubatch"], 1)))
        assert per_call == case["per_call"]
        assert sum(per_call) == case["total"]


def test_split_simple_sizes_pin():
    g = golden("splits.json")
    for case in g["split_simple_sizes"]:
        ubs = B.init_batch(case["n_tokens"], [[0]] * case["n_tokens"], case["n_ubatch"], 1)
        assert [u["n_tokens"] for u in ubs] == case["sizes"]
    for case in g["split_simple_ranges"]:
        n_batch, n_ub = P.clamp(8192, case["n_batch"], case["n_ubatch"], True)
        ubs = B.init_batch(case["n_tokens"], [[0]] * case["n_tokens"], n_ub, 1)
        assert [[u["rows"][0], u["rows"][-1]] for u in ubs] == case["ranges"]
        for u in ubs:
            assert u["rows"] == list(range(u["rows"][0], u["rows"][-1] + 1))


def test_clamps_pin():
    g = golden("clamps.json")
    assert (P.DEFAULT_N_BATCH, P.DEFAULT_N_UBATCH) == (g["defaults"]["n_batch"], g["defaults"]["n_ubatch"])
    for c in g["cases"]:
        assert P.clamp(c["n_ctx"], c["n_batch"], c["n_ubatch"], c["causal"]) == (c["eff_batch"], c["eff_ubatch"])


def _all_batches(max_rows, n_seq):
    subsets = [list(s) for r in range(1, n_seq + 1) for s in itertools.combinations(range(n_seq), r)]
    for n in range(1, max_rows + 1):
        for rows in itertools.product(range(len(subsets)), repeat=n):
            yield [subsets[i] for i in rows]


def _check_split_invariants(seq_lists, ubs, n_ubatch, mode):
    n = len(seq_lists)
    seen = [r for u in ubs for r in u["rows"]]
    assert sorted(seen) == list(range(n)), "every row exactly once"
    for u in ubs:
        assert u["n_tokens"] == len(u["rows"]) >= 1
        assert u["n_tokens"] <= n_ubatch
        assert u["n_tokens"] == u["n_seq_tokens"] * u["n_seqs"]
        assert u["seq_id_unq"] == sorted({s for r in u["rows"] for s in seq_lists[r]})
    # rows that carry the same sequence set keep their submission order
    order = {r: k for k, r in enumerate(seen)}
    for a in range(n):
        for b in range(a + 1, n):
            if set(seq_lists[a]) == set(seq_lists[b]):
                assert order[a] < order[b]
    if mode == B.SPLIT_EQUAL:
        for u in ubs:
            groups = [u["rows"][k * u["n_seq_tokens"]:(k + 1) * u["n_seq_tokens"]]
                      for k in range(u["n_seqs"])]
            sets = []
            for g in groups:
                ss = {frozenset(seq_lists[r]) for r in g}
                assert len(ss) == 1, "one set per group"
                sets.append(ss.pop())
            for x, y in itertools.combinations(sets, 2):
                assert not (x & y), "sets in one ubatch are disjoint"
            mins = [min(s) for s in sets]
            assert mins == sorted(mins), "ordered sequence ids"
    if mode == B.SPLIT_SEQ:
        for u in ubs:
            assert len({frozenset(seq_lists[r]) for r in u["rows"]}) == 1
            assert u["n_seqs"] == 1
    if mode == B.SPLIT_SIMPLE:
        assert seen == list(range(n))
        assert all(u["n_tokens"] == n_ubatch for u in ubs[:-1])


@pytest.mark.parametrize("mode", [B.SPLIT_SIMPLE, B.SPLIT_EQUAL, B.SPLIT_SEQ])
def test_split_invariants_bruteforce(mode):
    for seq_lists in _all_batches(4, 3):
        for n_ub in (1, 2, 3, 8):
            ubs = B.init_batch(len(seq_lists), seq_lists, n_ub, 2, mode)
            _check_split_invariants(seq_lists, ubs, n_ub, mode)
    rng = random.Random(7)
    subsets = [list(s) for r in (1, 2, 3) for s in itertools.combinations(range(3), r)]
    for _ in range(1500):
        seq_lists = [rng.choice(subsets) for _ in range(6)]
        n_ub = rng.choice([1, 2, 3, 4, 6, 16])
        ubs = B.init_batch(6, seq_lists, n_ub, 2, mode)
        _check_split_invariants(seq_lists, ubs, n_ub, mode)


def test_split_equal_mixed_iteration_shape():
    # 32 one-token decode sequences plus two 1500-token prompts at n_ubatch 512
    # over several streams: the first ubatch takes one row from each of the 34
    # sets (512 // 34 = 15 > 1 remaining of the decode sets); then the two
    # prompts advance 256 rows each.
    seq_lists = [[s] for s in range(32)] + [[32]] * 1500 + [[33]] * 1500
    ubs = B.init_batch(len(seq_lists), seq_lists, 512, 4)
    assert [u["n_tokens"] for u in ubs] == [34] + [512] * 5 + [438]
    assert ubs[0]["rows"] == list(range(33)) + [32 + 1500]


def test_init_batch_strategy_choice():
    # BATCH-ZH Part C: one stream -> split_simple (ignores ids), several -> split_equal
    seq_lists = [[0], [1], [0], [1]]
    one = B.init_batch(4, seq_lists, 4, 1)
    assert [u["rows"] for u in one] == [[0, 1, 2, 3]]
    many = B.init_batch(4, seq_lists, 4, 2)
    assert [u["rows"] for u in many] == [[0, 2, 1, 3]]


# ----------------------------------------------------------------------------
# validation and auto-fill
# ----------------------------------------------------------------------------

def _fill(n, pos, n_seq_id, seq_id, n_batch=16, n_seq_max=4, s2s=(0, 0, 1, 1), state=None):
    st = state or C.CellState(2, 16, n_seq_max, list(s2s))
    return B.validate_and_fill(n, pos, n_seq_id, seq_id, n_batch, n_seq_max, list(s2s), st)


def test_validation_errors():
    assert _fill(0, [], None, None)[0] == B.E_INVAL
    assert _fill(17, list(range(17)), None, None)[0] == B.E_BATCH_TOO_LARGE
    assert _fill(1, [0], [1], [[4]])[0] == B.E_SEQ_RANGE
    assert _fill(1, [0], [1], [[-1]])[0] == B.E_SEQ_RANGE
    assert _fill(1, [0], [2], [[0, 0]])[0] == B.E_INVAL
    assert _fill(1, [0], [0], [[0]])[0] == B.E_INVAL
    assert _fill(1, [0], [2], [[0, 2]])[0] == B.E_CROSS_STREAM
    assert _fill(1, [-3], [1], [[0]])[0] == B.E_INVAL
    assert _fill(2, [0, 1], [2, 2], [[0, 1], [1, 0]])[0] == 0


def test_auto_fill():
    err, pos, seqs = _fill(3, None, None, None)
    assert err == 0 and pos == [0, 1, 2] and seqs == [[0], [0], [0]]
    st = C.CellState(2, 16, 4, [0, 0, 1, 1])
    st.fill(0, 5, 6, [0, 1])
    err, pos, seqs = _fill(4, None, [1, 1, 1, 2], [[0], [2], [0], [1, 0]], state=st)
    assert err == 0
    # seq 0 already holds pos 6 -> 7, 8; seq 2 is new -> 0; row 3's first id is 1,
    # which holds pos 6 in the cache (shared cell) -> 7
    assert pos == [7, 0, 8, 7]


# ----------------------------------------------------------------------------
# cells, n_kv, slot finder
# ----------------------------------------------------------------------------

def test_n_kv_pin():
    for case in golden("n_kv.json")["cases"]:
        st = C.CellState(1, case["kv_size"], 1)
        for j in range(case["used"]):
            st.fill(0, j, j, [0])
        assert st.n_kv_stream(0) == case["n_kv"]


def test_n_kv_closed_form():
    # quantum 256, at least one quantum, at most the stream size
    for kv_size, used, want in [(4096, 0, 256), (4096, 1, 256), (4096, 256, 256), (4096, 257, 512),
                                (4096, 769, 1024), (64, 7, 64), (300, 290, 300), (8192, 5000, 5120)]:
        st = C.CellState(1, kv_size, 1)
        for j in range(used):
            st.fill(0, j, j, [0])
        assert st.n_kv_stream(0) == want
    # n_kv counts the highest occupied cell, not the number of occupied cells
    st = C.CellState(1, 4096, 1)
    st.fill(0, 700, 0, [0])
    assert st.n_kv_stream(0) == 768


def test_first_fit_and_all_or_nothing():
    kv = OracleKV(n_ctx=32, n_batch=32, n_ubatch=4, n_seq_max=2, n_stream=2,
                  n_layer=1, n_head=2, n_head_kv=1, head_dim=4, keep_kv=False)
    code, sp = kv.split(list(range(10)), [[0]] * 10)
    assert code == 0
    assert [c for cs in sp.cells for c in cs] == list(range(10))
    code, sp = kv.split(list(range(3)), [[1]] * 3)
    assert code == 0 and sp.cells == [[0, 1, 2]]  # stream 1 is separate
    before = kv.state.copy()
    code, sp = kv.split(list(range(10, 17)), [[0]] * 7)   # stream 0 has 6 free
    assert code == C.NO_SLOT and sp is None
    assert kv.state.same_as(before)
    code, sp = kv.split(list(range(10, 16)), [[0]] * 6)
    assert code == 0 and [c for cs in sp.cells for c in cs] == list(range(10, 16))


def test_seq_rm_frees_cells_and_keeps_shared_prefix():
    kv = OracleKV(n_ctx=16, n_batch=16, n_ubatch=16, n_seq_max=3, n_stream=1,
                  n_layer=1, n_head=2, n_head_kv=1, head_dim=4, keep_kv=False)
    kv.split([0, 1], [[0, 1, 2], [0, 1, 2]])
    kv.split([2, 2, 2], [[0], [1], [2]])
    assert kv.state.n_used(0) == 5
    kv.seq_rm(1, 0, -1)
    assert kv.state.n_used(0) == 4            # seq 1's own cell freed, prefix kept
    assert kv.state.seqs_of(0, 0) == [0, 2]
    kv.seq_rm(0, 0, -1)
    kv.seq_rm(2, 0, -1)
    assert kv.state.n_used(0) == 0
    code, sp = kv.split([0], [[1]])
    assert sp.cells == [[0]]                  # freed cells are reused first-fit



def test_seq_cp_equals_storing_with_every_id():
    # BATCH-ZH, Part E: "Hello world" stored once for sequences {0, 1, 2}.  Storing
    # it for sequence 0 and copying it to 1 and 2 must give the same cells, and
    # each decode row then sees the page's three cells.
    g = golden("prefix_sharing.json")
    mk = lambda: OracleKV(n_ctx=16, n_batch=16, n_ubatch=16, n_seq_max=3, n_stream=1,
                          n_layer=1, n_head=2, n_head_kv=1, head_dim=4, keep_kv=False)
    shared, copied = mk(), mk()
    assert shared.split(g["prefill"]["pos"], g["prefill"]["seq"], n_seq_id=[3, 3])[0] == 0
    assert copied.split(g["prefill"]["pos"], [[0]] * len(g["prefill"]["pos"]))[0] == 0
    assert copied.seq_cp(0, 1, 0, -1) == 0 and copied.seq_cp(0, 2, 0, -1) == 0
    assert copied.state.same_as(shared.state)
    code, sp = copied.split(g["decode"]["pos"], g["decode"]["seq"])
    vis = (copied.mask(sp, 0) == M.F16_ZERO).sum(axis=1)
    assert list(vis) == [g["cells_visible_per_decode_row"]] * 3


def test_seq_cp_range_inverse_and_streams():
    kv = OracleKV(n_ctx=32, n_batch=32, n_ubatch=32, n_seq_max=4, n_stream=2,
                  n_layer=1, n_head=2, n_head_kv=1, head_dim=4, keep_kv=False,
                  seq_to_stream=[0, 0, 1, 1])
    kv.split(list(range(10)), [[0]] * 10)
    before = kv.state.copy()
    assert kv.seq_cp(0, 1, 3, 7) == 0
    # only positions 3 .. 6 gain sequence 1
    assert [j for j in range(10) if kv.state.seq_has(0, j, 1)] == [3, 4, 5, 6]
    assert kv.state.seq_pos_max(1) == 6
    assert kv.seq_cp(0, 1, 0, -1) == 0        # cells already holding 1 stay as they are
    assert all(kv.state.seqs_of(0, j) == [0, 1] for j in range(10))
    kv.seq_rm(1, 0, -1)                       # removing the copy restores the state
    assert kv.state.same_as(before)
    assert kv.seq_cp(0, 2, 0, -1) == "cross-stream" and kv.state.same_as(before)

# ----------------------------------------------------------------------------
# cache layout and the pages' measurements
# ----------------------------------------------------------------------------

def test_kv_layout_pins():
    g = golden("kv_sizes.json")
    r = g["row"]
    assert L.row_values(r["n_head_kv"], r["head_dim"]) == r["values"]
    assert L.row_bytes(r["n_head_kv"], r["head_dim"]) == r["bytes"]
    t = g["per_token"]
    assert L.bytes_per_token(t["n_layer"], 8, 128) == t["bytes"]
    assert t["tokens"] * L.bytes_per_token(t["n_layer"], 8, 128) == t["bytes_for_tokens"]
    c = g["cache"]
    assert L.cache_bytes(c["n_cells"], c["n_layer"], 8, 128) == c["total_bytes"]
    assert c["n_cells"] * L.row_bytes(8, 128) * c["n_layer"] == c["k_bytes"]
    s = g["strides"]
    assert list(L.shape(8, 128, s["kv_size"], 1)) == s["ne"]
    assert list(L.strides(8, 128, s["kv_size"])) == s["nb"]
    o = g["offset"]
    assert L.byte_offset(0, o["cell"], o["head"], o["elem"], 8, 128, 4096) == o["bytes"]
    u = g["streams"]
    assert list(L.shape(8, 128, u["n_ctx"], 1)) == u["unified"]
    assert list(L.shape(8, 128, u["n_ctx"], 4)) == u["non_unified"]
    assert L.cache_bytes(u["n_ctx"], 28, 8, 128) == u["bytes_each"]
    m = g["mha_vs_gqa"]
    assert L.bytes_per_token(m["n_layer"], 1, m["mha_width"]) == m["mha_bytes_per_token"]
    assert 4096 * L.bytes_per_token(m["n_layer"], 1, m["mha_width"]) == m["mha_bytes_4096"]
    assert L.bytes_per_token(m["n_layer"], m["gqa_n_head_kv"], m["gqa_head_dim"]) == m["gqa_bytes_per_token"]
    assert 4096 * L.bytes_per_token(m["n_layer"], 8, 128) == m["gqa_bytes_4096"]


def test_stream_offset_matches_numpy_layout():
    # the byte offset formula agrees with numpy's own C-order addressing of the
    # oracle's [n_stream, kv_size, n_head_kv, head_dim] fp16 array
    arr = np.zeros((3, 40, 8, 128), dtype=np.float16)
    for (s, j, h, e) in [(0, 37, 3, 10), (2, 5, 7, 127), (1, 39, 0, 0)]:
        want = (s * arr.strides[0] + j * arr.strides[1] + h * arr.strides[2] + e * arr.strides[3])
        assert L.byte_offset(s, j, h, e, 8, 128, 40) == want


def test_duty_cycle_pin():
    for c in golden("duty_cycle.json")["cases"]:
        assert L.duty_cycle(c["lengths"]) == (c["useful"], c["executed"])
        if "approx" in c:
            assert round(c["useful"] / c["executed"], 2) == c["approx"]



def _drive(sched, check=None):
    """Run the loop to the end, checking the budgets at every pass."""
    def on_batch(retired, pos, seq):
        assert len(pos) <= sched.token_budget
        assert len(sched.running) <= sched.max_seqs and sched.free_cells >= 0
        assert len(set(seq)) == len(sched.running)
        if check is not None:
            check(retired, pos, seq)
    return S.run(sched, on_batch)


def test_fixed_batch_duty_cycle_pin():
    # ITER: the page's fixed batches, run through the scheduler loop in fixed mode
    for c in golden("duty_cycle.json")["cases"]:
        n = len(c["lengths"])
        sch = S.Scheduler(kv_size=1 << 16, n_seq_max=n, max_seqs=n, token_budget=4096, fixed=True)
        for N in c["lengths"]:
            assert sch.submit(16, N) is not None
        _drive(sch)
        assert (sch.useful, sch.passes * sch.max_seqs) == (c["useful"], c["executed"])


def test_continuous_equals_fixed_for_equal_lengths():
    # equal output lengths leave nothing to refill: k full batches take k N passes
    for fixed in (True, False):
        sch = S.Scheduler(kv_size=4096, n_seq_max=8, max_seqs=4, token_budget=256, fixed=fixed)
        for _ in range(12):
            sch.submit(10, 7)
        _drive(sch)
        assert sch.passes == 3 * 7 and sch.duty_cycle() == 1.0


def test_continuous_refills_slots():
    # the page's eight lengths, eight requests each: the fixed batch stays at its
    # 5568 / 16384 per group, the loop refills freed slots at once; useful
    # positions are the same and equal the sum of the batch sizes
    lengths = [64, 128, 256, 512, 512, 1024, 1024, 2048]
    out = {}
    for fixed in (True, False):
        sch = S.Scheduler(kv_size=1 << 16, n_seq_max=8, max_seqs=8, token_budget=4096, fixed=fixed)
        for _ in range(8):
            for N in lengths:
                sch.submit(32, N)
        sizes = []
        _drive(sch, lambda r, pos, seq: sizes.append(len(set(seq))) if pos else None)
        assert sch.useful == 8 * sum(lengths) == sum(sizes)
        out[fixed] = sch
    assert out[True].passes == 8 * 2048 and out[True].duty_cycle() == 5568 / 16384
    # neither budget binds here: while requests wait every pass runs eight
    # sequences, and the drain after the last admission lasts at most one
    # longest request
    lo = -(-8 * sum(lengths) // 8)
    assert lo <= out[False].passes <= lo + max(lengths)


def test_scheduler_budgets_and_retirement():
    # worked by hand: kv_size 100 cells, 40 positions per pass, four slots;
    # A = (30 prompt, 10 new), B = (30, 10), C = (5, 3), D = (20, 2)
    sch = S.Scheduler(kv_size=100, n_seq_max=4, max_seqs=4, token_budget=40, fixed=False)
    assert sch.submit(41, 1) is None and sch.submit(60, 41) is None     # can never run
    for L, N in [(30, 10), (30, 10), (5, 3), (20, 2)]:
        assert sch.submit(L, N) is not None
    expect = {
        1: ([], [0] * 30, list(range(30))),                               # B: 30 + 30 > 40 positions
        2: ([], [0] + [1] * 30 + [2] * 5, [30] + list(range(30)) + list(range(5))),   # D: 36 + 20 > 40
        3: ([], [0, 1, 2], [31, 30, 5]),                                   # D: 22 cells > 12 free
        4: ([], [0, 1, 2], [32, 31, 6]),
        5: ([2], [0, 1], [33, 32]),                                        # C retired: 20 free < 22
        11: ([0], [1] + [0] * 20, [38] + list(range(20))),                 # A retired: D takes id 0
    }
    n = 0
    while True:
        retired, pos, seq = sch.next_batch()
        if not pos:
            break
        n += 1
        if n in expect:
            assert (retired, seq, pos) == expect[n], n
        sch.advance()
    assert n == 12 and sch.useful == 10 + 10 + 3 + 2 and not sch.waiting

def test_f16_dump_pin():
    g = golden("f16_dump.json")
    raw = bytes.fromhex(g["hex"].replace(" ", ""))
    vals = np.frombuffer(raw, dtype="<f2").astype(np.float64)
    assert [round(float(v), 4) for v in vals] == g["values_4dp"]
    assert int(np.frombuffer(raw[:2], dtype="<u2")[0]) == int(g["first_bits"], 16)


# ----------------------------------------------------------------------------
# the mask
# ----------------------------------------------------------------------------

def test_prefix_sharing_pin():
    g = golden("prefix_sharing.json")
    kv = OracleKV(n_ctx=16, n_batch=16, n_ubatch=16, n_seq_max=3, n_stream=1,
                  n_layer=1, n_head=2, n_head_kv=1, head_dim=4, keep_kv=False)
    code, sp = kv.split(g["prefill"]["pos"], g["prefill"]["seq"], n_seq_id=[3, 3])
    assert code == 0 and kv.state.n_used(0) == 2 * g["kv_copies_of_prefix"]
    code, sp = kv.split(g["decode"]["pos"], g["decode"]["seq"])
    m = kv.mask(sp, 0)
    vis = (m == M.F16_ZERO).sum(axis=1)
    assert list(vis) == [g["cells_visible_per_decode_row"]] * 3
    # each decode row sees the two shared cells and its own cell only
    own = sp.cells[0]
    for i in range(3):
        assert set(np.flatnonzero(m[i] == 0)) == {0, 1, own[i]}


def test_mask_rule_cases():
    st = C.CellState(1, 8, 3)
    st.fill(0, 0, 0, [0])
    st.fill(0, 1, 1, [0, 1])
    st.fill(0, 2, 5, [0])
    st.fill(0, 3, 2, [1])
    # cell 4.. empty
    m = M.kq_mask(st, [1, 2], [0, 1], [0, 0], 8, causal=True)
    assert list(m[0]) == [0, 0, 0xFC00, 0xFC00, 0xFC00, 0xFC00, 0xFC00, 0xFC00]
    assert list(m[1]) == [0xFC00, 0, 0xFC00, 0, 0xFC00, 0xFC00, 0xFC00, 0xFC00]
    m = M.kq_mask(st, [1], [0], [0], 8, causal=False)   # non-causal drops pos
    assert list(m[0][:4]) == [0, 0, 0, 0xFC00]
    # the query masks with its first id only (UBATCH, "The mask is doing the work")
    assert M.kq_mask(st, [9], [1], [0], 4, True)[0].tolist() == [0xFC00, 0, 0xFC00, 0]


def test_mask_vector_equals_pairwise_random():
    rng = np.random.default_rng(3)
    for trial in range(30):
        n_seq = int(rng.integers(1, 5))
        st = C.CellState(2, 24, n_seq)
        for s in range(2):
            for j in range(24):
                if rng.random() < 0.6:
                    k = int(rng.integers(1, n_seq + 1))
                    st.fill(s, j, int(rng.integers(0, 10)),
                            sorted(rng.choice(n_seq, size=k, replace=False).tolist()))
        n = int(rng.integers(1, 6))
        rp = rng.integers(0, 10, n).tolist()
        rq = rng.integers(0, n_seq, n).tolist()
        rs = rng.integers(0, 2, n).tolist()
        for causal in (True, False):
            for n_swa in (0, 1, 3, 7):
                a = M.kq_mask(st, rp, rq, rs, 24, causal, n_swa)
                b = M.kq_mask_bruteforce(st, rp, rq, rs, 24, causal, n_swa)
                assert np.array_equal(a, b)


def test_sliding_window_closed_form():
    # one sequence, 20 prompt cells, a window of w = 5 positions: causal row i
    # sees cells max(0, i - 4) .. i, min(i + 1, 5) of them; without causality
    # the window still drops cells more than 4 positions back, nothing ahead
    w, T = 5, 20
    for causal in (True, False):
        kv = OracleKV(n_ctx=32, n_batch=32, n_ubatch=32, n_layer=1, n_head=2, n_head_kv=1,
                      head_dim=4, keep_kv=False, causal=causal, n_swa=w)
        code, sp = kv.split(list(range(T)), [[0]] * T)
        m = kv.mask(sp, 0) == M.F16_ZERO
        for i in range(T):
            hi = i if causal else T - 1
            assert set(np.flatnonzero(m[i])) == set(range(max(0, i - w + 1), hi + 1)), (causal, i)
        if causal:
            assert m.sum(axis=1).tolist() == [min(i + 1, w) for i in range(T)]


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def _torch_sdpa(q, k, v, attn_mask=None, is_causal=False):
    torch = pytest.importorskip("torch")
    tq = torch.from_numpy(q.astype(np.float64)).transpose(0, 1)   # [H, T, d]
    tk = torch.from_numpy(k.astype(np.float64)).transpose(0, 1)   # [Hkv, S, d]
    tv = torch.from_numpy(v.astype(np.float64)).transpose(0, 1)
    m = None if attn_mask is None else torch.from_numpy(attn_mask)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq.unsqueeze(0), tk.unsqueeze(0), tv.unsqueeze(0), attn_mask=m,
        is_causal=is_causal, enable_gqa=True)
    return out[0].transpose(0, 1).numpy()


@pytest.mark.parametrize("n_head,n_head_kv", [(16, 8), (32, 8), (4, 4), (6, 2)])
def test_attention_single_seq_causal_equals_sdpa(n_head, n_head_kv):
    d, T = 16, 37
    kv = OracleKV(n_ctx=64, n_batch=64, n_ubatch=64, n_seq_max=1, n_layer=1,
                  n_head=n_head, n_head_kv=n_head_kv, head_dim=d)
    q = gen.uniform_f16(1, (T, n_head, d), -2, 2)
    k = gen.uniform_f16(2, (T, n_head_kv, d), -2, 2)
    v = gen.uniform_f16(3, (T, n_head_kv, d), -2, 2)
    code, sp = kv.split(list(range(T)), [[0]] * T)
    kv.store(sp, 0, 0, k.reshape(T, -1), v.reshape(T, -1))
    out = kv.attention(sp, 0, 0, q)
    ref = _torch_sdpa(q, k, v, is_causal=True)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_attention_chunked_with_explicit_mask_equals_sdpa():
    # a chunk of U rows against C cached cells: the [U, C+U] score matrix
    # (UBATCH, "Chunked prefill is the same mechanism")
    d, H, Hk, Ccache, U = 8, 4, 2, 11, 5
    kv = OracleKV(n_ctx=32, n_batch=32, n_ubatch=32, n_layer=1, n_head=H, n_head_kv=Hk, head_dim=d)
    k = gen.uniform_f16(4, (Ccache + U, Hk, d))
    v = gen.uniform_f16(5, (Ccache + U, Hk, d))
    q = gen.uniform_f16(6, (Ccache + U, H, d))
    code, sp = kv.split(list(range(Ccache)), [[0]] * Ccache)
    kv.store(sp, 0, 0, k[:Ccache].reshape(Ccache, -1), v[:Ccache].reshape(Ccache, -1))
    code, sp = kv.split(list(range(Ccache, Ccache + U)), [[0]] * U)
    kv.store(sp, 0, 0, k[Ccache:].reshape(U, -1), v[Ccache:].reshape(U, -1))
    out = kv.attention(sp, 0, 0, q[Ccache:])
    allowed = np.zeros((U, Ccache + U), dtype=bool)
    for i in range(U):
        allowed[i, :Ccache + i + 1] = True
    ref = _torch_sdpa(q[Ccache:], k, v, attn_mask=allowed)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)



def test_attention_sliding_window_equals_banded_sdpa():
    # a causal prompt under a window of 6 positions: the softmax over each row's
    # last six keys, which SDPA gives with an explicit banded mask
    d, H, Hk, T, w = 8, 4, 2, 23, 6
    kv = OracleKV(n_ctx=32, n_batch=32, n_ubatch=32, n_layer=1, n_head=H, n_head_kv=Hk,
                  head_dim=d, n_swa=w)
    k = gen.uniform_f16(14, (T, Hk, d))
    v = gen.uniform_f16(15, (T, Hk, d))
    q = gen.uniform_f16(16, (T, H, d))
    code, sp = kv.split(list(range(T)), [[0]] * T)
    kv.store(sp, 0, 0, k.reshape(T, -1), v.reshape(T, -1))
    out = kv.attention(sp, 0, 0, q)
    band = np.zeros((T, T), dtype=bool)
    for i in range(T):
        band[i, max(0, i - w + 1):i + 1] = True
    np.testing.assert_allclose(out, _torch_sdpa(q, k, v, attn_mask=band), rtol=1e-12, atol=1e-12)

def test_attention_loops_equal_vectorised():
    rng = np.random.default_rng(11)
    H, Hk, d, m = 4, 2, 5, 6
    q = rng.standard_normal((H, d))
    keys = rng.standard_normal((m, Hk, d))
    vals = rng.standard_normal((m, Hk, d))
    kc = keys[None].astype(np.float64)
    vc = vals[None].astype(np.float64)
    vis = np.array([True, False, True, True, False, True])
    a = A.attend_row(q, kc, vc, 0, vis, H, Hk)
    idx = np.flatnonzero(vis)
    b = A.attend_row_loops(q.tolist(), keys[idx].tolist(), vals[idx].tolist(), H, Hk)
    np.testing.assert_allclose(a, np.array(b), rtol=1e-12, atol=1e-13)
    z = A.attend_row(q, kc, vc, 0, np.zeros(m, dtype=bool), H, Hk)
    assert not z.any()


def test_attention_softmax_closed_form_two_keys():
    # two visible keys: weights are the logistic function of the score gap
    d = 4
    q = np.array([[1.0, 0, 0, 0]])
    keys = np.array([[[2.0, 0, 0, 0]], [[0.0, 0, 0, 0]]])[None][0][None]
    vals = np.array([[[1.0, 0, 0, 0]], [[0.0, 1.0, 0, 0]]])[None][0][None]
    o = A.attend_row(q, keys, vals, 0, np.array([True, True]), 1, 1)
    w0 = 1.0 / (1.0 + math.exp(-(2.0 - 0.0) / math.sqrt(d)))
    np.testing.assert_allclose(o[0], [w0, 1 - w0, 0, 0], rtol=1e-14)


def _run_calls(kv, cfg_id, calls, layer_rows_q, n_head, width_kv, width_q):
    outs = {}
    for call in calls:
        code, sp = kv.split(call["pos"], call["seq"], n_seq_id=[len(s) for s in call["seq"]])
        assert code == 0
        for k, ub in enumerate(sp.ubatches):
            rows = ub["rows"]
            pos = [call["pos"][r] for r in rows]
            con = [call["content"][r] for r in rows]
            kk = gen.batch_rows(cfg_id, 0, gen.KIND_K, pos, con, width_kv)
            vv = gen.batch_rows(cfg_id, 0, gen.KIND_V, pos, con, width_kv)
            kv.store(sp, k, 0, kk, vv)
            qq = gen.batch_rows(cfg_id, 0, gen.KIND_Q, pos, con, width_q).reshape(len(rows), n_head, -1)
            o = kv.attention(sp, k, 0, qq)
            for n, r in enumerate(rows):
                key = (tuple(call["seq"][r]), call["pos"][r])
                outs[key] = o[n]
    return outs


def _kvo(n_ctx=256, n_ubatch=64, n_seq_max=4, n_stream=1, s2s=None, H=4, Hk=2, d=8):
    return OracleKV(n_ctx=n_ctx, n_batch=n_ctx, n_ubatch=n_ubatch, n_seq_max=n_seq_max,
                    n_stream=n_stream, n_layer=1, n_head=H, n_head_kv=Hk, head_dim=d,
                    seq_to_stream=s2s)


def _prompt(seq, p0, n, content=None, seqs=None):
    return {"pos": list(range(p0, p0 + n)), "seq": [list(seqs or [seq])] * n,
            "content": [seq if content is None else content] * n}


def test_invariant_chunked_equals_whole_equals_token_by_token():
    H, Hk, d = 4, 2, 8
    whole = _run_calls(_kvo(n_ubatch=64), 9, [_prompt(0, 0, 40)], None, H, Hk * d, H * d)
    chunked = _run_calls(_kvo(n_ubatch=7), 9, [_prompt(0, 0, 40)], None, H, Hk * d, H * d)
    tbt = _run_calls(_kvo(n_ubatch=64), 9, [_prompt(0, p, 1) for p in range(40)], None, H, Hk * d, H * d)
    for key in whole:
        np.testing.assert_allclose(chunked[key], whole[key], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(tbt[key], whole[key], rtol=1e-12, atol=1e-14)


def test_invariant_sequence_isolation():
    H, Hk, d = 4, 2, 8
    alone = _run_calls(_kvo(), 9, [_prompt(0, 0, 20), _prompt(0, 20, 1)], None, H, Hk * d, H * d)
    mixed_call = {"pos": [], "seq": [], "content": []}
    a, b = _prompt(0, 0, 20), _prompt(1, 0, 15)
    for i in range(20):   # interleave two sequences row by row in one batch
        for src in (a, b):
            if i < len(src["pos"]):
                for kk in mixed_call:
                    mixed_call[kk].append(src[kk][i])
    dec = {"pos": [15, 20], "seq": [[1], [0]], "content": [1, 0]}
    mixed = _run_calls(_kvo(n_ubatch=8), 9, [mixed_call, dec], None, H, Hk * d, H * d)
    for key, val in alone.items():
        np.testing.assert_allclose(mixed[key], val, rtol=1e-12, atol=1e-14)


def test_invariant_prefix_shared_equals_duplicated():
    H, Hk, d = 4, 2, 8
    shared = _run_calls(_kvo(), 9, [_prompt(0, 0, 12, content=0, seqs=[0, 1]),
                                    {"pos": [12, 12, 13, 13], "seq": [[0], [1], [0], [1]],
                                     "content": [5, 6, 5, 6]}], None, H, Hk * d, H * d)
    dup = _run_calls(_kvo(), 9, [_prompt(0, 0, 12, content=0), _prompt(1, 0, 12, content=0),
                                 {"pos": [12, 12, 13, 13], "seq": [[0], [1], [0], [1]],
                                  "content": [5, 6, 5, 6]}], None, H, Hk * d, H * d)
    for s in (0, 1):
        for p in (12, 13):
            np.testing.assert_allclose(shared[((s,), p)], dup[((s,), p)], rtol=1e-12, atol=1e-14)


def test_invariant_row_permutation():
    H, Hk, d = 4, 2, 8
    base = [_prompt(0, 0, 10), _prompt(1, 0, 7)]
    call = {"pos": [10, 7, 11, 8], "seq": [[0], [1], [0], [1]], "content": [0, 1, 0, 1]}
    perm = {k: [v[i] for i in (3, 1, 2, 0)] for k, v in call.items()}
    # (row order within a sequence must stay causal-consistent: the permuted
    # batch keeps pos 10 before 11 for seq 0 in the cache via separate calls)
    a = _run_calls(_kvo(), 9, base + [call], None, H, Hk * d, H * d)
    b = _run_calls(_kvo(), 9, base + [perm], None, H, Hk * d, H * d)
    for key in a:
        np.testing.assert_allclose(b[key], a[key], rtol=1e-12, atol=1e-14)


def test_invariant_streams_partition():
    # a non-unified cache: two sequences in two streams give the same outputs as
    # each sequence alone in a one-stream cache (KV-MEM, "Unified versus non-unified")
    H, Hk, d = 4, 2, 8
    two = _run_calls(_kvo(n_stream=2, n_seq_max=2, s2s=[0, 1]), 9,
                     [{"pos": list(range(9)) + list(range(6)), "seq": [[0]] * 9 + [[1]] * 6,
                       "content": [0] * 9 + [1] * 6}], None, H, Hk * d, H * d)
    for s, n in ((0, 9), (1, 6)):
        alone = _run_calls(_kvo(n_seq_max=2), 9, [_prompt(s, 0, n)], None, H, Hk * d, H * d)
        for key, val in alone.items():
            np.testing.assert_allclose(two[key], val, rtol=1e-12, atol=1e-14)
