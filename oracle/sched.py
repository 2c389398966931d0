"""Iteration-level (continuous) batching: the scheduler loop, plain Python.

Test infrastructure only (like everything under oracle/): the library's native
scheduler is checked against this one, iteration by iteration.

ITER ("Iteration-Level Batching: Reforming the Batch at Every Token"), "The loop
that replaces the batch": before every forward pass the scheduler (1) retires the
finished sequences and releases their cache, (2) admits waiting sequences while
the token budget and the cache budget both allow it, (3) assembles the batch: a
newly admitted sequence contributes its whole prompt, a running one one token.
The pass then gives every sequence in the batch one more token.  "The budget that
actually binds": the token budget counts positions per pass (L for a prompt of L
tokens, 1 per running sequence).  "Two resources idled by a fixed batch": a fixed
batch admits a group together and runs it until its longest member ends; its duty
cycle is the useful positions over passes x slots (5,568 of 16,384 for the
page's eight lengths; (20 + 2000) / (2 x 2000) for its pair).

Readings (the page gives a sketch, not a specification):
* the cache budget is the page's conservative one: admission reserves
  prompt + max_new cells (its worst case), released at retirement;
* the waiting queue is first come, first served with no overtaking (the sketch
  stops at the first request that does not fit);
* a request of L prompt tokens and N new tokens takes N passes: its prompt pass
  yields token 1 and each later pass one more (at position L + generated - 1);
  it is retired at the start of the pass after its N-th token;
* sequence ids: a newly admitted sequence takes the smallest id not running;
* fixed mode admits only into an empty batch (the classical batch).

Pins (tests/test_oracle_pins.py): the page's two duty cycles in fixed mode; with
equal output lengths, continuous and fixed batching take the same passes (k N for
k full batches, duty 1); budgets hold at every pass; useful positions equal the
sum of the batch sizes over passes.
"""

from collections import deque


class Request:
    def __init__(self, rid, prompt_len, max_new):
        self.rid, self.L, self.N = rid, prompt_len, max_new
        self.seq = -1
        self.generated = 0


class Scheduler:
    def __init__(self, kv_size, n_seq_max, max_seqs, token_budget, fixed=False):
        assert 1 <= max_seqs <= n_seq_max and max_seqs <= token_budget
        self.kv_size, self.n_seq_max = kv_size, n_seq_max
        self.max_seqs, self.token_budget, self.fixed = max_seqs, token_budget, fixed
        self.free_cells = kv_size
        self.waiting = deque()
        self.running = []              # in admission order
        self.next_rid = 0
        self.passes = self.useful = 0
        self.batch_seqs = []           # sequences in the last assembled batch

    def submit(self, prompt_len, max_new):
        """Queue a request; returns its id, or None when it can never run."""
        if prompt_len < 1 or max_new < 1 or prompt_len > self.token_budget or prompt_len + max_new > self.kv_size:
            return None
        r = Request(self.next_rid, prompt_len, max_new)
        self.next_rid += 1
        self.waiting.append(r)
        return r.rid

    def next_batch(self):
        """One iteration: returns (retired sequence ids, positions, sequence ids
        of the batch's tokens); an empty batch means nothing is left."""
        retired = [r.seq for r in self.running if r.generated == r.N]
        for r in [r for r in self.running if r.generated == r.N]:
            self.running.remove(r)
            self.free_cells += r.L + r.N
        tokens = len(self.running)     # one decode position per running sequence
        new = []
        if not self.fixed or not self.running:
            while self.waiting:
                r = self.waiting[0]
                if (len(self.running) + len(new) >= self.max_seqs or r.L + r.N > self.free_cells
                        or tokens + r.L > self.token_budget):
                    break
                self.waiting.popleft()
                used = {x.seq for x in self.running} | {x.seq for x in new}
                r.seq = min(q for q in range(self.n_seq_max) if q not in used)
                self.free_cells -= r.L + r.N
                tokens += r.L
                new.append(r)
        pos, seq = [], []
        for r in self.running:
            pos.append(r.L + r.generated - 1)
            seq.append(r.seq)
        for r in new:
            pos.extend(range(r.L))
            seq.extend([r.seq] * r.L)
        self.running.extend(new)
        self.batch_seqs = [r for r in self.running]
        return retired, pos, seq

    def advance(self):
        """The pass ran: every sequence of the batch has one more token."""
        if not self.batch_seqs:
            return
        for r in self.batch_seqs:
            r.generated += 1
        self.passes += 1
        self.useful += len(self.batch_seqs)
        self.batch_seqs = []

    def duty_cycle(self):
        return self.useful / (self.passes * self.max_seqs) if self.passes else 0.0


def run(sched, on_batch=None):
    """Drive the loop to the end; on_batch(retired, pos, seq) sees every batch."""
    while True:
        retired, pos, seq = sched.next_batch()
        if on_batch is not None:
            on_batch(retired, pos, seq)
        if not pos:
            return sched
        sched.advance()
