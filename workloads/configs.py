"""The five workloads: model shapes, cache parameters and decode calls.

A *call* is one batch handed to the library: a dict with ``pos`` (list of
int), ``seq`` (list of sequence-id lists, first id first) and ``content``
(which sequence's token stream the row's Q/K/V values come from; a sequence
that copies another's tokens names the original).  ``setup`` calls fill the
cache; ``measured`` calls are the ones attention is checked and timed on.

Attention shapes (no weights are involved; Q/K/V are synthetic):
* Qwen3-0.6B: 16 query heads, 8 KV heads, head_dim 128, 28 layers;
* Llama-3-8B: 32 query heads, 8 KV heads, head_dim 128, 32 layers.
"""

import numpy as np

QWEN = dict(name="qwen3-0.6b", n_head=16, n_head_kv=8, head_dim=128, n_layer=28)
LLAMA = dict(name="llama-3-8b", n_head=32, n_head_kv=8, head_dim=128, n_layer=32)


def _prompt(seq, p0, n, content=None, seqs=None):
    c = seq if content is None else content
    s = [seq] if seqs is None else list(seqs)
    return {"pos": list(range(p0, p0 + n)), "seq": [list(s) for _ in range(n)],
            "content": [c] * n}


def _concat(calls):
    out = {"pos": [], "seq": [], "content": []}
    for c in calls:
        for k in out:
            out[k].extend(c[k])
    return out


def _chunk(call, n_batch):
    """A caller splits an over-long list into decode calls of at most n_batch."""
    out = []
    n = len(call["pos"])
    for a in range(0, n, n_batch):
        out.append({k: v[a:a + n_batch] for k, v in call.items()})
    return out


def config(cid, n_layer=None):
    """Workload ``cid`` (1..5).  ``n_layer`` overrides the layer count (the
    per-layer work is identical, so parity tests may run fewer layers)."""
    if cid == 1:
        # Single layer, one sequence: a 7-token prompt then 4 decode steps.
        shape = dict(QWEN, n_layer=1)
        prm = dict(n_ctx=64, n_batch=2048, n_ubatch=512, n_seq_max=1, n_stream=1)
        measured = [_prompt(0, 0, 7)] + [_prompt(0, p, 1) for p in (7, 8, 9, 10)]
        setup = []
        name = "qwen-1layer-kv64-prompt7-decode4"
    elif cid == 2:
        # 5000-token single-sequence prefill in three decode calls.
        shape = dict(QWEN)
        prm = dict(n_ctx=8192, n_batch=2048, n_ubatch=512, n_seq_max=1, n_stream=1)
        setup = []
        measured = _chunk(_prompt(0, 0, 5000), 2048)
        name = "qwen-prefill-5000-b2048-ub512"
    elif cid == 3:
        # Eight sequences prefilled one after another, then one decode row each.
        shape = dict(QWEN)
        lens = [64, 128, 256, 512, 512, 1024, 1024, 2048]
        prm = dict(n_ctx=8192, n_batch=2048, n_ubatch=512, n_seq_max=8, n_stream=1)
        setup = [_prompt(s, 0, L) for s, L in enumerate(lens)]
        measured = [_concat([_prompt(s, L, 1) for s, L in enumerate(lens)])]
        name = "qwen-decode-8seq-unified"
    elif cid == 4:
        # Prefix sharing over four streams, then a mixed iteration.
        shape = dict(QWEN)
        s2s = []
        for s in range(64):
            if s < 16:
                s2s.append(0)
            elif s < 32:
                s2s.append(1 + (s - 16) % 3)
            elif s == 32:
                s2s.append(2)
            elif s == 33:
                s2s.append(3)
            else:
                s2s.append(s % 4)
        prm = dict(n_ctx=4 * 8192, n_batch=4096, n_ubatch=512, n_seq_max=64, n_stream=4,
                   seq_to_stream=s2s)
        prefix = _prompt(0, 0, 1024, content=0, seqs=range(16))
        divergent = _concat([_prompt(s, 1024, 256) for s in range(16)])
        twins = _concat([_concat([_prompt(s, 0, 1024, content=0),
                                  _prompt(s, 1024, 256, content=s - 16)])
                         for s in range(16, 32)])
        setup = [prefix, divergent] + _chunk(twins, 4096)
        decode = _concat([_prompt(s, 1280, 1, content=(s if s < 16 else s - 16))
                          for s in range(32)])
        measured = [_concat([decode, _prompt(32, 0, 1500), _prompt(33, 0, 1500)])]
        name = "qwen-mixed-prefix16-4streams"
    elif cid == 5:
        # 256 sequences with lognormal contexts, one decode row each.
        shape = dict(LLAMA)
        lens = context_lengths_cfg5()
        prm = dict(n_ctx=1 << 20, n_batch=2048, n_ubatch=512, n_seq_max=256, n_stream=1)
        setup = []
        for s, L in enumerate(lens):
            setup.extend(_chunk(_prompt(s, 0, int(L)), 2048))
        measured = [_concat([_prompt(s, int(L), 1) for s, L in enumerate(lens)])]
        name = "llama8b-decode-256seq-lognormal"
    else:
        raise ValueError(cid)
    if n_layer is not None:
        shape = dict(shape, n_layer=n_layer)
    return {"id": cid, "name": name, "shape": shape, "params": prm,
            "setup": setup, "measured": measured}


def context_lengths_cfg5(seed=0, n=256):
    """Lognormal contexts, median 2048, sigma 1.0, clipped to [128, 32768]."""
    rng = np.random.default_rng(seed)
    x = rng.lognormal(np.log(2048.0), 1.0, n)
    return np.clip(np.round(x), 128, 32768).astype(np.int64)
