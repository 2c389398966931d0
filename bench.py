#!/usr/bin/env python
"""Benchmark: ubatch attention over a cell-indexed KV cache on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
host splitting and cell reservation, then for every ubatch and every layer the
K/V store and the attention (the mask / attention plan is built once per
ubatch).  Default workload (configuration 2): a 5000-token single-sequence
prefill with a Qwen3-0.6B attention shape (16 query heads, 8 KV heads,
head_dim 128, 28 layers), n_batch 2048, n_ubatch 512 -> 3 decode calls, 10
ubatches; the step starts from an empty cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2|3|4|5]
                    [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no cross-GPU exchange); value = all ranks' tokens / the slowest
rank's time.  `--impl reference` times the CPU oracle (plain NumPy float64)
on a bounded sample of the same workload; rank 0 only.
"""

import argparse
import datetime
import json
import os
import re
import select
import statistics
import subprocess
import sys
import time

if "reference" in sys.argv:
    # the oracle runs single-threaded; BLAS reads these when NumPy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import configs  # noqa: E402

METRIC = "ubatch tokens/s"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="default workload only: skip the decode legs (the 256- and 8-sequence decode "
                         "workloads measured after it)")
    ap.add_argument("--decode-steps", type=int, default=20,
                    help="timed steps of each decode leg")
    ap.add_argument("--layers", type=int, default=None,
                    help="run fewer layers than the workload has (small cases for profiling only)")
    ap.add_argument("--ubatch", type=int, default=None,
                    help="override the workload's n_ubatch (the n_ubatch sweep)")
    ap.add_argument("--streams", type=int, default=None,
                    help="override n_stream (sequence q in stream q %% n_stream); with --kv-per-stream")
    ap.add_argument("--kv-per-stream", type=int, default=None,
                    help="with --streams: cells per stream (n_ctx = streams x this)")
    ap.add_argument("--loop", action="store_true",
                    help="iteration-level batching loop (native scheduler), fixed batch vs continuous")
    ap.add_argument("--loop-copies", type=int, default=2,
                    help="--loop: requests per output length (the page's eight lengths)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# workload bookkeeping (no attention arithmetic: counts only)
# ---------------------------------------------------------------------------

# workloads whose measured calls hold one decode row per sequence
# DRAM bytes (read + write) of one k_decode launch of the 256-sequence workload,
# from an ncu capture of the current kernel (profiles/k_decode_llama8b-decode-256seq-
# lognormal.md; a launch at decode step 2, 3.521 GB algorithmic).  Cleared to nothing
# whenever the kernel changes until it is captured again.
DECODE_TRAFFIC = {5: 3556978688}
# One k_prefill launch of the 5000-token prefill captured by ncu (profiles/k_prefill_
# qwen-prefill-5000-b2048-ub512.md: ubatch 5, layer 5): its DRAM bytes (read + write)
# and its algorithmic bytes.  The launches of a step differ in size, so the reported
# traffic is this ratio times the timed launches' mean algorithmic bytes (DRAM traffic
# grows with the K/V rows read; the O rows stay in L2 within a launch).  Cleared to
# nothing whenever the kernel changes until it is captured again.
PREFILL_TRAFFIC = {2: (14806272, 18874368)}

DECODE_BOUND = {3: True, 5: True}


def measured_tokens(cfg):
    return sum(len(c["pos"]) for c in cfg["measured"])


def row_visible_cells(pos):
    """Every workload stores positions 0..p of a row's sequence before the
    row attends, so a causal row at position p sees p + 1 cells."""
    return np.asarray(pos, dtype=np.int64) + 1


class Clocks:
    """nvidia-smi sampling during the timed region.  The sampler starts before the
    warm-up and the first sample is awaited there, so that nvidia-smi's own start-up
    (which can hold up the device for a while) stays out of the timed region; only
    samples stamped inside the timed window are kept."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.proc = None
        self.gpu = gpu
        self.first = ""
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        ready, _, _ = select.select([self.proc.stdout], [], [], 10.0)
        if ready:
            self.first = self.proc.stdout.readline()

    def mark(self, t0, t1):
        """The timed window, as datetime.now() before and after it."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        if self.window is not None:   # let a sample land after a window shorter than the period
            wait = 0.3 - (datetime.datetime.now() - self.window[1]).total_seconds()
            if wait > 0:
                time.sleep(wait)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in (self.first + out).strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None   # unreadable stamp: the sample is kept unfiltered
            rows.append((ts, sm, mx, parts[4:8]))
        if self.window is not None and all(r[0] is not None for r in rows):
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
            # a window shorter than the sampling period: the two samples around it
            before = [r for r in rows if r[0] < self.window[0]]
            after = [r for r in rows if r[0] > self.window[1]]
            rows = inside or before[-1:] + after[:1]
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in rows]), "sm_max_mhz": max(r[2] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


class EventPool:
    """Start/end CUDA events created before the timed region (creating them
    inside it would put host work between the launches)."""

    def __init__(self, n):
        import torch
        self.ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
        self.meta = []

    def take(self, pairs, nbytes):
        i = len(self.meta)
        self.meta.append((pairs, nbytes))
        return self.ev[i]

    def results(self):
        """(ms, pairs, bytes) per recorded launch."""
        return [(self.ev[i][0].elapsed_time(self.ev[i][1]), p, b) for i, (p, b) in enumerate(self.meta)]


def max_over_ranks(ms, device):
    """The slowest replica's time (every rank gets it).  Replicas share no
    data: this reduction of one timing value is the only collective."""
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class OursArm:
    def __init__(self, cfg, device):
        import torch
        import continuous_batching_kv_gb300 as kv
        self.torch, self.kv, self.cfg = torch, kv, cfg
        sh, prm = cfg["shape"], cfg["params"]
        self.H, self.Hk, self.d, self.L = sh["n_head"], sh["n_head_kv"], sh["head_dim"], sh["n_layer"]
        self.dev = device
        width = self.Hk * self.d
        self.kc = [torch.zeros((prm["n_ctx"], width), dtype=torch.float16, device=device) for _ in range(self.L)]
        self.vc = [torch.zeros((prm["n_ctx"], width), dtype=torch.float16, device=device) for _ in range(self.L)]
        self.c = kv.kv_init(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                            n_seq_max=prm["n_seq_max"], n_stream=prm["n_stream"], n_layer=self.L,
                            n_head=self.H, n_head_kv=self.Hk, head_dim=self.d,
                            seq_to_stream=prm.get("seq_to_stream"), k_layers=self.kc, v_layers=self.vc)
        # a stream of its own (not the legacy default stream, which would serialise
        # with the end-to-end mode's copy stream)
        self.stream = torch.cuda.Stream(device)
        self.decode_loop = DECODE_BOUND.get(cfg["id"], False)
        self.step_no = -1
        self.gen = torch.Generator(device=device)
        self.gen.manual_seed(1234)
        with torch.cuda.stream(self.stream):   # inputs are made on the stream that uses them
            self._setup()
            self._prepare_inputs()

    def close(self):
        """Free the library cache and this arm's device tensors."""
        if self.c is not None:
            self.torch.cuda.synchronize()
            self.kv.kv_free(self.c)
            self.c = None
        self.kc = self.vc = self.calls = None

    def _randn(self, *shape):
        return self.torch.randn(*shape, generator=self.gen, device=self.dev, dtype=self.torch.float32).half()

    def _setup(self):
        """Fill the cache with the workload's setup calls (untimed)."""
        kv = self.kv
        width = self.Hk * self.d
        for call in self.cfg["setup"]:
            s = kv.kv_split_ubatches(self.c, call["pos"], call["seq"])
            assert kv.kv_prepare_cells(self.c, s) == 0
            for k in range(kv.kv_split_count(s)):
                n = kv.kv_split_ubatch(s, k)["n_tokens"]
                for layer in range(self.L):
                    kk = self._randn(n, width)
                    vv = self._randn(n, width)
                    kv.kv_store(self.c, s, k, layer, kk, vv, self.stream)
            kv.kv_split_free(s)
        self.torch.cuda.synchronize()
        self.base_pos_max = {}
        for call in self.cfg["measured"]:
            for seqs in call["seq"]:
                q = seqs[0]
                self.base_pos_max[q] = kv.kv_seq_pos_max(self.c, q)
        # decode iterations that fit in the free cells of the fullest stream
        prm = self.cfg["params"]
        kv_size = prm["n_ctx"] // prm["n_stream"]
        per_stream = {}
        for call in self.cfg["measured"]:
            for seqs in call["seq"]:
                st = (prm.get("seq_to_stream") or [i % prm["n_stream"] for i in range(prm["n_seq_max"])])[seqs[0]]
                per_stream[st] = per_stream.get(st, 0) + 1
        free = min(kv_size - kv.kv_stream_n_kv(self.c, st) for st in per_stream) if per_stream else 0
        self.max_steps = max(0, free // max(per_stream.values()) - 1) if per_stream else 0

    def _prepare_inputs(self):
        """Per measured call: the marshalled batch, its ubatch shapes, and
        resident per-(ubatch, layer) Q/K/V/O device tensors."""
        kv = self.kv
        self.calls = []
        self.flops_per_ub = []
        for call in self.cfg["measured"]:
            s = kv.kv_split_ubatches(self.c, call["pos"], call["seq"])
            ubs = []
            for k in range(kv.kv_split_count(s)):
                u = kv.kv_split_ubatch(s, k)
                rows = list(u["rows"])
                n = len(rows)
                # all layers' Q, K and V of the ubatch in one device buffer (the end-to-end
                # mode copies it from the host in one piece); per layer: Q, K, V
                lq, lk = n * self.H * self.d, n * self.Hk * self.d
                per = lq + 2 * lk
                buf = self._randn(self.L * per)
                t = {"n": n, "dev": buf, "per": per, "lq": lq, "lk": lk,
                     "o": self.torch.empty((n, self.H, self.d), dtype=self.torch.float32, device=self.dev),
                     "pairs": int(row_visible_cells([call["pos"][r] for r in rows]).sum()),
                     "bytes": self._kv_bytes(call, rows, n),
                     "row_kv_bytes": len({call["seq"][r][0] for r in rows}) * 2 * self.Hk * self.d * 2}
                t["q"], t["k"], t["v"] = self._views(t, buf)
                ubs.append(t)
            kv.kv_split_free(s)
            # the batch is marshalled once (numpy arrays, ids as a flat list plus
            # counts); each step re-splits it in the library
            marsh = (np.asarray(call["pos"], dtype=np.int32),
                     (np.fromiter((q for ids in call["seq"] for q in ids), dtype=np.int32),
                      np.asarray([len(ids) for ids in call["seq"]], dtype=np.int32)))
            self.calls.append((call, ubs, marsh))
        self.torch.cuda.synchronize()

    def _kv_bytes(self, call, rows, n):
        """Least HBM traffic of one attention launch: every sequence's visible
        K and V rows read once for all its query heads, plus Q in and O out."""
        cells = {}
        for r in rows:
            q = call["seq"][r][0]
            cells[q] = max(cells.get(q, 0), call["pos"][r] + 1)
        kv_rows = sum(cells.values())
        return int(kv_rows * 2 * self.Hk * self.d * 2 + n * self.H * self.d * (2 + 4))

    def _views(self, t, buf):
        """Per layer Q [n, H, d], K and V [n, Hk*d] inside one ubatch input buffer."""
        n, per, lq, lk = t["n"], t["per"], t["lq"], t["lk"]
        return ([buf[l * per:l * per + lq].view(n, self.H, self.d) for l in range(self.L)],
                [buf[l * per + lq:l * per + lq + lk].view(n, self.Hk * self.d) for l in range(self.L)],
                [buf[l * per + lq + lk:(l + 1) * per].view(n, self.Hk * self.d) for l in range(self.L)])

    def input_bytes(self):
        return sum(t["dev"].numel() * 2 for _, ubs, _ in self.calls for t in ubs)

    def enable_host_inputs(self):
        """End-to-end mode: a pinned host copy of every ubatch's input buffer and of
        its output, two device input buffers per ubatch (a step computes from one
        while the next step's inputs arrive in the other), a copy stream and events."""
        torch = self.torch
        for _, ubs, _ in self.calls:
            for t in ubs:
                t["host"] = t["dev"].cpu().pin_memory()
                dev2 = torch.empty_like(t["dev"])
                t["sets"] = [(t["dev"], t["q"], t["k"], t["v"]), (dev2,) + self._views(t, dev2)]
                t["in_ev"] = [torch.cuda.Event(), torch.cuda.Event()]
                t["ohost"] = torch.empty(t["o"].shape, dtype=t["o"].dtype).pin_memory()
                t["out_ev"] = torch.cuda.Event()
                t["d2h_ev"] = torch.cuda.Event()
        self.copy_stream = torch.cuda.Stream(self.dev)
        self.set_ev = [torch.cuda.Event(), torch.cuda.Event()]
        self.restart_host_steps()

    def restart_host_steps(self):
        """The next end-to-end step copies its own inputs (nothing prefetched)."""
        self.e2e_n = 0
        self.prefetched = False
        for ev in self.set_ev:
            ev.record(self.stream)
        for _, ubs, _ in self.calls:
            for t in ubs:
                t["d2h_ev"].record(self.stream)

    def _copy_inputs(self, set_i):
        """Copy every ubatch's inputs into input buffer set set_i once the step that
        last used that set has finished."""
        torch = self.torch
        self.copy_stream.wait_event(self.set_ev[set_i])
        with torch.cuda.stream(self.copy_stream):
            for _, ubs, _ in self.calls:
                for t in ubs:
                    t["sets"][set_i][0].copy_(t["host"], non_blocking=True)
                    t["in_ev"][set_i].record(self.copy_stream)

    def reset(self):
        """Before a step: return the cache to its post-setup state, or, for the
        decode workloads, advance one token (each step is the next decode
        iteration of the same sequences, as a serving loop runs; the cache is
        rolled back only when it would run out of cells)."""
        kv = self.kv
        if self.decode_loop:
            self.step_no += 1
            if self.step_no <= self.max_steps:
                return
            self.step_no = 0
            for q, pmax in self.base_pos_max.items():
                kv.kv_seq_rm(self.c, q, pmax + 1, -1)
            return
        if not self.cfg["setup"]:
            kv.kv_seq_rm(self.c, -1, 0, -1)
        else:
            for q, pmax in self.base_pos_max.items():
                kv.kv_seq_rm(self.c, q, pmax + 1, -1)

    def rewind(self):
        """Return the cache to its post-setup state and the decode loop to its
        first iteration, so that a second pass replays the same steps."""
        for q, pmax in self.base_pos_max.items():
            self.kv.kv_seq_rm(self.c, q, pmax + 1, -1)
        self.step_no = -1

    def timed_calls_per_step(self):
        return sum(len(ubs) for _, ubs, _ in self.calls) * (self.L - 1 if self.L > 1 else 1)

    def step(self, timers=None, host=False, prefetch=False):
        """One pass of the whole path.  timers: an EventPool that brackets the
        attention calls that launch no planning kernels (layers >= 1; with a single
        layer, layer 0, whose calls also plan).
        host: end-to-end mode -- every ubatch's inputs come from pinned host memory
        over a copy stream, and every ubatch's output goes back to pinned host
        memory over the same stream; the attention stream waits for each ubatch's
        inputs.  prefetch: also copy the next step's inputs into the other input
        buffers, so that they arrive while this step computes."""
        kv, torch = self.kv, self.torch
        self.reset()
        last = []
        off = max(0, self.step_no) if self.decode_loop else 0
        # algorithmic work of this step's attention launches, all layers (counts only)
        self.step_work = [0, 0]
        for _, ubs, _ in self.calls:
            for t in ubs:
                self.step_work[0] += self.L * (t["pairs"] + off * t["n"])
                self.step_work[1] += self.L * (t["bytes"] + off * t["row_kv_bytes"])
        cur = self.e2e_n & 1 if host else 0
        if host:
            if not self.prefetched:
                self._copy_inputs(cur)
            self.prefetched = False
            if prefetch:
                self._copy_inputs(cur ^ 1)
                self.prefetched = True
        for ci, (call, ubs, marsh) in enumerate(self.calls):
            s = kv.kv_split_ubatches(self.c, marsh[0] + off if off else marsh[0], marsh[1])
            assert kv.kv_prepare_cells(self.c, s) == 0
            for k, t in enumerate(ubs):
                qs, ks, vs = t["q"], t["k"], t["v"]
                if host:
                    _, qs, ks, vs = t["sets"][cur]
                    self.stream.wait_event(t["in_ev"][cur])
                    self.stream.wait_event(t["d2h_ev"])   # last step's read of o is done
                for layer in range(self.L):
                    kv.kv_store(self.c, s, k, layer, ks[layer], vs[layer], self.stream)
                    if timers is not None and (layer > 0 or self.L == 1):
                        e0, e1 = timers.take(t["pairs"] + off * t["n"], t["bytes"] + off * t["row_kv_bytes"])
                        e0.record(self.stream)
                        kv.ubatch_attention(self.c, s, k, layer, qs[layer], t["o"], None, self.stream)
                        e1.record(self.stream)
                    else:
                        kv.ubatch_attention(self.c, s, k, layer, qs[layer], t["o"], None, self.stream)
                if host:
                    t["out_ev"].record(self.stream)
                    self.copy_stream.wait_event(t["out_ev"])
                    with torch.cuda.stream(self.copy_stream):
                        t["ohost"].copy_(t["o"], non_blocking=True)
                        t["d2h_ev"].record(self.copy_stream)
                    last.append(t["ohost"])
            kv.kv_split_free(s)
        if host:
            self.set_ev[cur].record(self.stream)
            self.e2e_n += 1
        return last


def apply_overrides(cfg, args):
    """--ubatch / --streams: the same workload at another n_ubatch, or with one
    cache stream per sequence group instead of the unified cache (KV-MEM,
    "Unified versus non-unified"); the workload's name records the change."""
    prm = cfg["params"]
    if args.ubatch is not None:
        prm["n_ubatch"] = args.ubatch
        cfg["name"] = re.sub(r"-ub\d+", "", cfg["name"]) + "-ub%d" % args.ubatch
    if args.streams is not None:
        per = args.kv_per_stream or prm["n_ctx"] // args.streams
        prm["n_stream"] = args.streams
        prm["n_ctx"] = args.streams * per
        prm.pop("seq_to_stream", None)
        cfg["name"] += "-streams%dx%d" % (args.streams, per)
    return cfg


def run_ours(args, rank, world, device):
    import torch
    import continuous_batching_kv_gb300 as kv
    torch.cuda.set_device(device)
    cfg = apply_overrides(configs.config(args.config, n_layer=args.layers), args)
    arm = OursArm(cfg, device)
    hbm, tflops, peak_src = load_peaks()
    dist = world > 1

    def barrier():
        if dist:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    clocks = Clocks(device if isinstance(device, int) else torch.cuda.current_device())
    clocks.start()
    for _ in range(max(args.warmup, 3)):
        arm.step()
    barrier()
    launches0 = kv.kv_launch_count(arm.c)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w0 = datetime.datetime.now()
    t0.record(arm.stream)
    work = [0, 0]
    for _ in range(args.steps):
        arm.step()
        work[0] += arm.step_work[0]
        work[1] += arm.step_work[1]
    t1.record(arm.stream)
    barrier()
    clocks.mark(w0, datetime.datetime.now())
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    launches = kv.kv_launch_count(arm.c) - launches0
    assert kv.kv_device_error(arm.c) == 0
    ms_max = max_over_ranks(ms_total, device) if dist else ms_total
    tokens = measured_tokens(cfg) * args.steps * world
    value = tokens / (ms_max / 1e3)

    # The attention launches' own durations come from a second pass over the
    # same steps: an event recorded between kv_store and ubatch_attention sits
    # between two kernels that otherwise overlap (the attention kernel's
    # start-up runs under the store's tail), so bracketing every call would
    # slow the pass whose total is the headline value.
    arm.rewind()
    for _ in range(max(args.warmup, 3)):
        arm.step()
    timers = EventPool(arm.timed_calls_per_step() * args.steps)
    barrier()
    for _ in range(args.steps):
        arm.step(timers=timers)
    barrier()
    assert kv.kv_device_error(arm.c) == 0

    # roofline of the dominant kernel (attention), timed live above
    res = timers.results()
    durs = [ms for ms, _, _ in res]
    secs = sum(durs) / 1e3
    if DECODE_BOUND.get(cfg["id"], False):
        # decode: one query row per sequence, so the launch streams K/V from HBM
        moved = sum(b for _, _, b in res)
        achieved = moved / secs / 1e9 if durs else 0.0
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": DECODE_TRAFFIC.get(cfg["id"]),
                "kernel": "ubatch_attention (k_decode)",
                "algorithmic_bytes_per_launch": int(moved / max(1, len(durs)))}
    else:
        per_pair_flops = 4 * arm.d * arm.H
        achieved = (sum(p for _, p, _ in res) * per_pair_flops) / secs / 1e12 if durs else 0.0
        alg_bytes = sum(b for _, _, b in res) / max(1, len(durs))
        tr = PREFILL_TRAFFIC.get(cfg["id"]) if args.ubatch is None and args.streams is None else None
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tflops, "unit": "TFLOP/s",
                "frac": round(achieved / tflops, 4),
                "traffic": int(alg_bytes * tr[0] / tr[1]) if tr else None,
                "kernel": "ubatch_attention (k_prefill)",
                "algorithmic_bytes_per_launch": int(alg_bytes)}
    roof.update({"peak_source": peak_src, "launches_timed": len(durs),
                 "timing": ("CUDA events around each attention launch of layers >= 1, " if arm.L > 1 else
                            "CUDA events around each attention launch (one layer: its plan kernels included), ")
                           + "on a second pass over the same steps",
                 "avg_launch_us": round(1e3 * sum(durs) / max(1, len(durs)), 2)})
    # The same algorithmic work over the whole unbracketed timed region (split,
    # reservation, stores, plans and attention of every step): a lower bound on
    # the attention launches' own rate, free of the bracketing events' cost.
    step_s = ms_total / 1e3
    if roof["bound"] == "hbm":
        st_ach = work[1] / step_s / 1e9
    else:
        st_ach = work[0] * 4 * arm.d * arm.H / step_s / 1e12
    roof["step_level"] = {"achieved": round(st_ach, 2 if roof["bound"] == "tensor" else 1),
                          "frac": round(st_ach / roof["peak"], 4), "unit": roof["unit"],
                          "basis": "algorithmic %s of every attention launch of the timed steps / the "
                                   "timed region (whole steps: host work, stores, plans included)"
                                   % ("bytes" if roof["bound"] == "hbm" else "flops")}

    e2e = None
    if not args.no_e2e:
        arm.enable_host_inputs()
        arm.step(host=True)
        barrier()
        t0.record(arm.stream)
        arm.restart_host_steps()   # the first timed step's copies start inside the timed region
        out = None
        for i in range(args.steps):
            # each step's inputs are copied inside the timed region: the first step's by
            # itself, the others' by the step before (the last step prefetches nothing)
            out = arm.step(host=True, prefetch=i + 1 < args.steps)
        # the results are read back on the copy stream; the timed region ends after them
        arm.stream.wait_stream(arm.copy_stream)
        t1.record(arm.stream)
        barrier()
        ms_e2e = t0.elapsed_time(t1)
        if dist:
            ms_e2e = max_over_ranks(ms_e2e, device)
        e2e = {"value": round(tokens / (ms_e2e / 1e3), 1), "unit": UNIT,
               "h2d_bytes_per_step": arm.input_bytes(),
               "d2h_bytes_per_step": int(sum(x.numel() * 4 for x in out))}

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 in, f32 accumulate/out",
            "data": "synthetic N(0,1) fp16 Q/K/V (seeded); no weights",
            "config": {"workload": cfg["name"], "config_id": cfg["id"],
                       "n_layer": arm.L, "n_head": arm.H, "n_head_kv": arm.Hk, "head_dim": arm.d,
                       "tokens_per_step": measured_tokens(cfg), **{k: v for k, v in cfg["params"].items()
                                                                    if k != "seq_to_stream"},
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "inputs larger than L2 (%.2f GB resident per step)" % (arm.input_bytes() / 1e9)},
            "roofline": roof, "gpu_launches": int(launches), "clocks": clk, "e2e": e2e}
    return line, arm


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(cfg, rows_per_ub):
    """Run the oracle's whole path for one layer on a bounded sample; return
    (seconds, extrapolated tokens/s, description)."""
    from oracle.session import OracleKV
    from workloads import gen
    sh, prm = cfg["shape"], cfg["params"]
    H, Hk, d, L = sh["n_head"], sh["n_head_kv"], sh["head_dim"], sh["n_layer"]
    o = OracleKV(n_ctx=prm["n_ctx"], n_batch=prm["n_batch"], n_ubatch=prm["n_ubatch"],
                 n_seq_max=prm["n_seq_max"], n_stream=prm["n_stream"], n_layer=1, n_head=H,
                 n_head_kv=Hk, head_dim=d, seq_to_stream=prm.get("seq_to_stream"))
    for call in cfg["setup"]:
        code, sp = o.split(call["pos"], call["seq"], keep_snapshots=False)
        for k, ub in enumerate(sp.ubatches):
            pos = [call["pos"][r] for r in ub["rows"]]
            con = [call["content"][r] for r in ub["rows"]]
            o.store(sp, k, 0, gen.batch_rows(cfg["id"], 0, 1, pos, con, Hk * d),
                    gen.batch_rows(cfg["id"], 0, 2, pos, con, Hk * d))
    t_split = t_store = t_attn = 0.0
    n_att = 0
    for call in cfg["measured"]:
        t = time.perf_counter()
        code, sp = o.split(call["pos"], call["seq"])
        t_split += time.perf_counter() - t
        for k, ub in enumerate(sp.ubatches):
            rows = ub["rows"]
            pos = [call["pos"][r] for r in rows]
            con = [call["content"][r] for r in rows]
            kk = gen.batch_rows(cfg["id"], 0, 1, pos, con, Hk * d)
            vv = gen.batch_rows(cfg["id"], 0, 2, pos, con, Hk * d)
            t = time.perf_counter()
            o.store(sp, k, 0, kk, vv)
            t_store += time.perf_counter() - t
            n = len(rows)
            sel = list(range(n)) if n <= rows_per_ub else \
                sorted(set(np.linspace(0, n - 1, rows_per_ub).astype(int).tolist()))
            q = gen.batch_rows(cfg["id"], 0, 0, pos, con, H * d).reshape(n, H, d)
            t = time.perf_counter()
            o.attention(sp, k, 0, q, rows=sel)
            t_attn += time.perf_counter() - t
            n_att += len(sel)
    ntok = measured_tokens(cfg)
    per_step = t_split + L * (t_store + t_attn * ntok / max(1, n_att))
    desc = ("oracle (NumPy float64, 1 thread): split+prepare of all %d tokens, 1 of %d layers stored, "
            "attention for %d of %d rows (<= %d per ubatch); extrapolated to %d layers x %d rows"
            % (ntok, L, n_att, ntok, rows_per_ub, L, ntok))
    return t_split + t_store + t_attn, ntok / per_step, desc


def _oracle_run(cfg, threads):
    """The oracle's bounded sample of the workload in a fresh process with `threads`
    BLAS threads; returns (cpu seconds, tokens/s, description) or an error string."""
    t = str(threads)
    env = dict(os.environ, OMP_NUM_THREADS=t, OPENBLAS_NUM_THREADS=t, MKL_NUM_THREADS=t)
    code = ("import json,sys; sys.path.insert(0, %r); import bench; from workloads import configs; "
            "s, v, d = bench.oracle_sample(configs.config(%d), %d); print(json.dumps([s, v, d]))"
            % (ROOT, cfg["id"], 160 if cfg["id"] == 2 else 64))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return "failed: " + (r.stderr.strip().splitlines()[-1][:200] if r.stderr.strip() else "no output")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(cfg):
    """The oracle as it stands on the host: one BLAS thread (the reported figure)
    and, beside it, every host core."""
    one = _oracle_run(cfg, 1)
    if isinstance(one, str):
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": one}
    secs, val, desc = one
    out = {"value": round(val, 2), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc,
           "cpu_seconds": round(secs, 2), "host_cores_available": os.cpu_count()}
    ncpu = os.cpu_count() or 1
    if ncpu > 1:
        allc = _oracle_run(cfg, ncpu)
        if not isinstance(allc, str):
            out["all_cores"] = {"value": round(allc[1], 2), "cores": ncpu, "cpu_seconds": round(allc[0], 2)}
    return out


def run_reference(args, cfg):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    rows = 8
    for _ in range(args.warmup):
        oracle_sample(cfg, rows)
    vals, secs = [], 0.0
    desc = ""
    for _ in range(args.steps):
        s, v, desc = oracle_sample(cfg, rows)
        vals.append(v)
        secs += s
    value = statistics.mean(vals)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic N(0,1) fp16 Q/K/V (seeded); no weights",
            "config": {"workload": cfg["name"], "config_id": cfg["id"]},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


LOOP_LENGTHS = [64, 128, 256, 512, 512, 1024, 1024, 2048]   # ITER: the fixed batch's eight output lengths


def run_loop(args, device):
    """The iteration-level batching loop through the native scheduler and the
    attention path: requests with the page's eight output lengths (each
    --loop-copies times, first come first served, 128-token prompts), eight
    sequences at a time, 2048 positions per pass, Qwen3-0.6B attention shape over
    28 layers.  Each pass: kv_sched_next, split + prepare, kv_store and
    ubatch_attention per ubatch and layer, kv_sched_advance.  Run once as a fixed
    batch (admission only into an empty batch) and once continuously; reports
    tokens/s (new tokens over the loop's device time) and the duty cycle
    (new tokens over passes x 8 slots: ITER, "Two resources idled by a fixed
    batch")."""
    import torch
    import continuous_batching_kv_gb300 as kv
    torch.cuda.set_device(device)
    sh = configs.QWEN
    H, Hk, d, L = sh["n_head"], sh["n_head_kv"], sh["head_dim"], sh["n_layer"]
    max_seqs, budget, prompt = 8, 2048, 128
    n_ctx = 24576                       # >= 8 reservations of prompt + 2048
    gen = torch.Generator(device=device)
    gen.manual_seed(7)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).half()
    q = [rnd(budget, H, d) for _ in range(L)]
    kk = [rnd(budget, Hk * d) for _ in range(L)]
    vv = [rnd(budget, Hk * d) for _ in range(L)]
    o = torch.empty(budget, H, d, device=device)
    kc = [torch.zeros(n_ctx, Hk * d, dtype=torch.float16, device=device) for _ in range(L)]
    vc = [torch.zeros_like(t) for t in kc]

    def loop(fixed, requests):
        c = kv.kv_init(n_ctx=n_ctx, n_batch=budget, n_ubatch=512, n_seq_max=max_seqs, n_layer=L,
                       n_head=H, n_head_kv=Hk, head_dim=d, k_layers=kc, v_layers=vc)
        sch = kv.kv_sched_init(c, max_seqs, budget, fixed)
        for n_new in requests:
            kv.kv_sched_submit(sch, prompt, n_new)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_host = time.perf_counter()
        e0.record()
        while True:
            b = kv.kv_sched_next(sch)
            if b.n_tokens == 0:
                break
            sp = kv.kv_split_sched_batch(c, b)
            assert kv.kv_prepare_cells(c, sp) == 0
            for k in range(kv.kv_split_count(sp)):
                n = kv.kv_split_ubatch(sp, k)["n_tokens"]
                for layer in range(L):
                    kv.kv_store(c, sp, k, layer, kk[layer][:n], vv[layer][:n])
                    kv.ubatch_attention(c, sp, k, layer, q[layer][:n], o[:n])
            kv.kv_split_free(sp)
            kv.kv_sched_advance(sch)
        e1.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_host
        st = kv.kv_sched_stats(sch)
        assert kv.kv_device_error(c) == 0
        launches = kv.kv_launch_count(c)
        kv.kv_sched_free(sch)
        kv.kv_free(c)
        ms = e0.elapsed_time(e1)
        return {"passes": st["passes"], "new_tokens": st["useful"],
                "duty_cycle": round(st["useful"] / (st["passes"] * max_seqs), 4),
                "ms": round(ms, 1), "host_wall_ms": round(1e3 * wall, 1),
                "tokens_per_s": round(st["useful"] / (ms / 1e3), 1), "gpu_launches": launches}

    loop(False, [64, 8, 8])             # warm-up (kernels loaded, clocks up)
    requests = [n for _ in range(args.loop_copies) for n in LOOP_LENGTHS]
    clocks = Clocks(device)
    clocks.start()
    w0 = datetime.datetime.now()
    fixed = loop(True, requests)
    cont = loop(False, requests)
    clocks.mark(w0, datetime.datetime.now())
    return {"metric": "iteration-loop new tokens/s", "value": cont["tokens_per_s"], "unit": "tokens/s",
            "higher_is_better": True, "n_gpus": 1, "dtype": "f16 in, f32 accumulate",
            "data": "synthetic N(0,1) fp16 Q/K/V (seeded); no weights",
            "config": {"workload": "iteration-loop-qwen-%dx8req" % args.loop_copies,
                       "output_lengths": LOOP_LENGTHS, "copies": args.loop_copies, "prompt_len": prompt,
                       "max_seqs": max_seqs, "token_budget": budget, "n_layer": L, "n_head": H,
                       "n_head_kv": Hk, "head_dim": d, "cache_budget": "prompt + max_new reserved at admission"},
            "continuous": cont, "fixed": fixed,
            "speedup_vs_fixed": round(cont["tokens_per_s"] / fixed["tokens_per_s"], 3),
            "clocks": clocks.stop()}


def decode_legs(args, rank, world, device):
    """The decode side of the metric, measured in the same run after the
    default workload: the 256-sequence Llama-shape decode (lognormal
    contexts, 32 layers) and the 8-sequence Qwen-shape decode, each through
    run_ours with its own timed region, per-launch roofline, step-level
    roofline and clock record (no end-to-end pass, no oracle)."""
    import argparse as _ap
    import torch
    out = {}
    for cid in (5, 3):
        sub = _ap.Namespace(**vars(args))
        sub.config, sub.no_e2e, sub.steps = cid, True, args.decode_steps
        l, a = run_ours(sub, rank, world, device)
        a.close()
        del a
        torch.cuda.empty_cache()
        out[l["config"]["workload"]] = {
            "metric": "decode KV-attention GB/s", "tokens_per_s": l["value"], "ms_per_step": l["ms_per_step"],
            "steps": l["steps"], "warmup": l["warmup"], "config": l["config"], "roofline": l["roofline"],
            "gpu_launches": l["gpu_launches"], "clocks": l["clocks"]}
    return out


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = apply_overrides(configs.config(args.config, n_layer=args.layers), args)
    if args.ubatch is not None or args.streams is not None:
        args.no_cpu = True      # the oracle sample reads the stock workload
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, cfg)), flush=True)
        return
    if args.loop:
        if rank == 0:
            print(json.dumps(run_loop(args, local)), flush=True)
        return
    import torch
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line, arm = run_ours(args, rank, world, local)
    if args.config == 2 and not args.no_decode and args.layers is None and args.ubatch is None \
            and args.streams is None:
        arm.close()
        del arm
        line["decode"] = decode_legs(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(cfg)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
